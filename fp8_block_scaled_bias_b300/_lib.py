"""ctypes binding of libmoe_fp8.so (include/moe_fp8.h).

Argument marshalling only: every step of the forward runs in the library's CUDA
kernels.  The library is built in-tree (``python -m fp8_block_scaled_bias_b300.build``);
loading fails loudly if it is missing.
"""

import ctypes as C
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_fp8.so")

_P = C.c_void_p
_I = C.c_int
_F = C.c_float
_SZ = C.c_size_t
_LL = C.c_longlong

# name -> (restype, argtypes); mirrors include/moe_fp8.h
SIGNATURES = {
    "moe_status_string": (C.c_char_p, [_I]),
    "moe_version": (_I, []),
    "moe_router_logits": (_I, [_P, _I, _I, _P, _I, _P, _P, _P, _SZ, _P]),
    "moe_router_logits_ws_bytes": (_SZ, [_I, _I, _I]),
    "moe_router_split_bf16": (_I, [_P, _LL, _P, _P]),
    "moe_route": (_I, [_P, _I, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P]),
    "moe_permute": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_permute_ws_bytes": (_SZ, [_I, _I, _I]),
    "moe_permute_noalloc": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "fp8_quant_1x128": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "fp8_quant_scatter_1x128": (_I, [_P, _I, _I, _I, _P, _I, _I, _I, _P, _P, _P, _P]),
    "fp8_quant_128x128": (_I, [_P, _I, _I, _P, _P, _P]),
    "fp8_quant_1x128_pow2": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "fp8_quant_128x128_pow2": (_I, [_P, _I, _I, _P, _P, _P]),
    "fp8_mx_grouped_gemm": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P, _P]),
    "fp8_quant_scatter_1x128_pow2": (_I, [_P, _I, _I, _I, _P, _I, _I, _I, _P, _P, _P, _P]),
    "moe_gate_up_mx": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _P, _P, _P, _P]),
    "fp8_blockscaled_grouped_gemm": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P, _I,
                                          _P, _P, _SZ, _P]),
    "fp8_grouped_gemm_ws_bytes": (_SZ, [_I, _I, _I]),
    "moe_gate_up_fp8_train": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "fp8_transpose_128x128": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_padded_rows_cap": (_I, [_I, _I]),
    "moe_segment_pad_offsets": (_I, [_P, _I, _P, _P, _P]),
    "moe_combine_bwd_rows": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "fp8_quant_128x1_pow2": (_I, [_P, _I, _P, _I, _P, _P, _I, _I, _P, _P, _P, _P]),
    "moe_swiglu_bwd_fp8": (_I, [_P, _P, _P, _I, _I, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P,
                                _P]),
    "fp8_wgrad_grouped_gemm": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_set_gemm_tiling": (_I, [_I]),
    "moe_get_gemm_tiling": (_I, []),
    "moe_test_gemm_wait_expiry": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _I, _P,
                                       C.c_ulonglong, _P]),
    "moe_swiglu_fp8_fwd": (_I, [_P, _P, _I, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P,
                                _P, _P, _SZ, _P]),
    "moe_swiglu_ws_bytes": (_SZ, [_I, _I, _I]),
    "moe_gather_rows_fp8": (_I, [_P, _P, _I, _P, _P, _I, _I, _P, _P, _P, _P]),
    "moe_gate_up_fp8": (_I, [_P, _P, _P, _I, _P, _P, _I, _I, _I, _P, _P, _P, _P]),
    "moe_combine": (_I, [_P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_bias_update": (_I, [_P, _P, _I, _I, _I, _F, _P]),
    "moe_seq_balance_stats": (_I, [_P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _SZ, _P]),
    "moe_seq_balance_stats_ws_bytes": (_SZ, [_I, _I, _I]),
    "moe_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
}

STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_CUDA",
          -4: "MOE_ERR_DEVICE_TIMEOUT", -5: "MOE_ERR_WORKSPACE", -6: "MOE_ERR_DEVICE_DATA"}


class MoEError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({msg})")
        self.status = status


_lib = None


def load():
    """Load the library once; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m fp8_block_scaled_bias_b300.build`")
        lib = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def call(name, *args):
    """Call an int-returning entry point and raise MoEError on a non-zero status."""
    lib = load()
    st = getattr(lib, name)(*args)
    if st != 0:
        raise MoEError(name, st, lib.moe_status_string(st).decode())
    return st
