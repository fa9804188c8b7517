"""The C-ABI library without a GPU: it loads, exports every function include/moe_fp8.h
declares (with the binding's argument counts), and rejects bad arguments on the host
before touching CUDA."""

import ctypes as C
import os
import re

import pytest

import fp8_block_scaled_bias_b300 as m
from fp8_block_scaled_bias_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_fp8.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    decls = {}
    for mt in re.finditer(r"^\s*(?:const\s+)?[\w\s\*]+?\b(\w+)\s*\(([^;{]*?)\)\s*;", src, re.M):
        name, args = mt.group(1), mt.group(2).strip()
        n = 0 if args in ("", "void") else args.count(",") + 1
        decls[name] = n
    return decls


def test_header_parses():
    d = _declared()
    assert len(d) >= 17
    for name in ("moe_route", "moe_permute", "fp8_quant_1x128", "fp8_blockscaled_grouped_gemm",
                 "moe_swiglu_fp8_fwd", "moe_combine", "moe_bias_update", "moe_router_logits"):
        assert name in d


def test_library_exports_every_declared_symbol():
    lib = m.load()
    for name, nargs in _declared().items():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"
        assert len(_lib.SIGNATURES[name][1]) == nargs, name
    assert set(_lib.SIGNATURES) == set(_declared())


def test_status_strings_and_version():
    lib = m.load()
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = lib.moe_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.moe_status_string(7).decode() == "unknown status"
    assert lib.moe_version() >= 100


def test_host_argument_checks_need_no_gpu():
    lib = m.load()
    P = C.c_void_p(16)          # never dereferenced: every call below fails validation
    # route: E not divisible by groups, K too large, too many experts
    assert lib.moe_route(P, 0, P, 4, 15, 4, 2, 2, 4, 1.0, P, P, None) == -1
    assert lib.moe_route(P, 0, P, 4, 16, 4, 2, 2, 9, 1.0, P, P, None) == -1
    assert lib.moe_route(P, 0, P, 4, 2048, 32, 2, 2, 4, 1.0, P, P, None) == -2
    assert lib.moe_route(None, 0, None, 4, 16, 4, 2, 2, 4, 1.0, None, None, None) == -1
    # quantisation: columns not a multiple of 128, null pointers
    assert lib.fp8_quant_1x128(P, 4, 100, 100, P, P, None) == -1
    assert lib.fp8_quant_1x128(None, 4, 128, 128, P, P, None) == -1
    assert lib.fp8_quant_128x128(P, 100, 128, P, P, None) == -1
    # GEMM: bad N/K, too many groups, missing workspace for a gather
    assert lib.fp8_blockscaled_grouped_gemm(P, P, 1, None, P, P, P, 1, 128, 100, 128, P, 128,
                                            None, None, 0, None) == -1
    assert lib.fp8_blockscaled_grouped_gemm(P, P, 1, None, P, P, P, 2000, 128, 128, 128, P, 128,
                                            None, None, 0, None) == -2
    assert lib.fp8_blockscaled_grouped_gemm(P, P, 4, P, P, P, P, 1, 128, 128, 128, P, 128,
                                            None, None, 0, None) == -5
    assert lib.fp8_blockscaled_grouped_gemm(P, P, 1, None, P, P, P, 1, 128, 128, 128, P, 100,
                                            None, None, 0, None) == -1
    # experts: missing workspace
    assert lib.moe_swiglu_fp8_fwd(P, P, 8, P, P, 16, P, P, P, P, 2, 128, 128, P, P, P, None,
                                  None, 0, None) == -5
    # permute: too many experts / slots, missing workspace
    assert lib.moe_permute(P, 8, 4, 2000, 1, P, P, P, P, None, P, 1 << 20, None) == -2
    assert lib.moe_permute(P, 8, 40, 16, 1, P, P, P, P, None, P, 1 << 20, None) == -2
    assert lib.moe_permute(P, 8, 4, 16, 1, P, P, P, P, None, None, 0, None) == -5
    # allocation-free permute: scratch need beyond its static array
    assert lib.moe_permute_noalloc(P, 128 * 257, 2, 1024, 1, P, P, P, P, None, None) == -2
    # combine: K too large, d not a multiple of 8
    assert lib.moe_combine(P, 8, P, P, 4, 33, 128, -1, P, None, None) == -2
    assert lib.moe_combine(P, 8, P, P, 4, 4, 100, -1, P, None, None) == -1
    # router logits: E above the tensor-core tile
    assert lib.moe_router_logits(P, 4, 128, P, 512, P, None, None, 0, None) == -2
    assert lib.moe_bias_update(None, P, 16, 4, 2, 0.001, None) == -1


def test_empty_inputs_are_no_ops():
    lib = m.load()
    assert lib.moe_route(None, 0, None, 0, 16, 4, 2, 2, 4, 1.0, None, None, None) == 0
    assert lib.fp8_quant_1x128(None, 0, 128, 128, None, None, None) == 0
    assert lib.moe_combine(None, 0, None, None, 0, 4, 128, -1, None, None, None) == 0
    assert lib.fp8_blockscaled_grouped_gemm(None, None, 0, None, None, None, None, 1, 0, 128,
                                            128, None, 128, None, None, 0, None) == 0


def test_workspace_sizes():
    lib = m.load()
    T, K, E, d, f = 4096, 8, 256, 7168, 2048
    rows = T * K + T
    sw = lib.moe_swiglu_ws_bytes(rows, d, f)
    assert sw >= rows * d + rows * (d // 128) * 4
    assert lib.moe_workspace_bytes(T, K, E, d, f) >= max(sw, lib.moe_permute_ws_bytes(T, K, E))
    assert lib.fp8_grouped_gemm_ws_bytes(1000, 512, 0) == 0
    assert lib.fp8_grouped_gemm_ws_bytes(1000, 512, 1) >= 1000 * 512 + 1000 * 4 * 4


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.dirname(m.__file__)
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, fn)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle", src, re.M), fn
                assert "oracle/" not in src, fn
