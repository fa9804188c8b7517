"""PyTorch-facing wrappers of the C-ABI entry points.

Each wrapper checks dtypes, shapes, device and contiguity, allocates its outputs with
torch (the library itself never allocates), and passes raw device pointers plus the
current CUDA stream.  No arithmetic of the method happens here.
"""

import torch

from ._lib import call, load

_U8, _F32, _I32, _BF16 = torch.uint8, torch.float32, torch.int32, torch.bfloat16


def _ptr(t):
    return t.data_ptr() if t is not None else None


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _check(t, dtype, name, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


class Workspace:
    """A growing per-device scratch buffer handed to calls that need workspace."""

    def __init__(self):
        self._buf = {}

    def get(self, nbytes, device):
        if nbytes <= 0:
            return None, 0
        key = torch.device(device).index or 0
        b = self._buf.get(key)
        if b is None or b.numel() < nbytes:
            b = torch.empty(nbytes, dtype=_U8, device=device)
            self._buf[key] = b
        return b.data_ptr(), b.numel()


WS = Workspace()


def new_status(device):
    """int32 device status word (0 = OK) for calls that report device-side errors."""
    return torch.zeros(1, dtype=_I32, device=device)


def status_value(status):
    return int(status.item())


# ---- router -----------------------------------------------------------------------------

def router_split_bf16(w):
    """FP32 centroids [E, d] -> BF16 planes [2, E, d] = (bf16(w), bf16(w - hi))."""
    _check(w, _F32, "w", 2)
    out = torch.empty((2,) + tuple(w.shape), dtype=_BF16, device=w.device)
    call("moe_router_split_bf16", _ptr(w), w.numel(), _ptr(out), _stream())
    return out


def router_logits(x, w_hilo, status=None, out=None):
    """z [T, E] FP32 = x [T, d] (BF16) . (hi + lo)^T."""
    _check(x, _BF16, "x", 2)
    _check(w_hilo, _BF16, "w_hilo", 3)
    T, d = x.shape
    E = w_hilo.shape[1]
    if w_hilo.shape != (2, E, d):
        raise ValueError("w_hilo must be [2, E, d]")
    z = out if out is not None else torch.empty(T, E, dtype=_F32, device=x.device)
    lib = load()
    ws, wsb = WS.get(lib.moe_router_logits_ws_bytes(T, d, E), x.device)
    call("moe_router_logits", _ptr(x), T, d, _ptr(w_hilo), E, _ptr(z), _ptr(status), ws, wsb,
         _stream())
    return z


def route(scores, bias, n_groups, topk_groups, K, group_topn=None, route_scale=1.0,
          affinities=False, out=None):
    """(idx int32 [T, K], gate FP32 [T, K]) from logits (or affinities) [T, E]."""
    _check(scores, _F32, "scores", 2)
    _check(bias, _F32, "bias", 1)
    T, E = scores.shape
    if group_topn is None:
        group_topn = K // topk_groups
    if out is None:
        idx = torch.empty(T, K, dtype=_I32, device=scores.device)
        gate = torch.empty(T, K, dtype=_F32, device=scores.device)
    else:
        idx, gate = out
    call("moe_route", _ptr(scores), int(bool(affinities)), _ptr(bias), T, E, n_groups,
         topk_groups, group_topn, K, float(route_scale), _ptr(idx), _ptr(gate), _stream())
    return idx, gate


def bias_update(bias, counts, T, K, gamma):
    """In place: bias += gamma * sign(T*K/E - counts)."""
    _check(bias, _F32, "bias", 1)
    _check(counts, _I32, "counts", 1)
    call("moe_bias_update", _ptr(bias), _ptr(counts), bias.numel(), T, K, float(gamma), _stream())
    return bias


def seq_balance_stats(scores, K, seq_len, alpha=1e-4, affinities=False, out=None):
    """(f [S, E], P [S, E], loss [S]) FP32 statistics of the sequence-wise balance loss for
    scores [T, E] (logits, or affinities), S = T / seq_len sequences."""
    _check(scores, _F32, "scores", 2)
    T, E = scores.shape
    S = T // seq_len if seq_len > 0 else 0
    dev = scores.device
    if out is None:
        f = torch.empty(S, E, dtype=_F32, device=dev)
        P = torch.empty(S, E, dtype=_F32, device=dev)
        loss = torch.empty(S, dtype=_F32, device=dev)
    else:
        f, P, loss = out
    lib = load()
    ws, wsb = WS.get(lib.moe_seq_balance_stats_ws_bytes(T, E, seq_len), dev)
    call("moe_seq_balance_stats", _ptr(scores), int(bool(affinities)), T, E, K, seq_len,
         float(alpha), _ptr(f), _ptr(P), _ptr(loss), ws, wsb, _stream())
    return f, P, loss


# ---- dispatch ---------------------------------------------------------------------------

def permute(idx, E, include_shared=True, status=None, out=None):
    """(counts [E], offsets [E+2], row_token [rows], row_of [T, K]) for idx [T, K]."""
    _check(idx, _I32, "idx", 2)
    T, K = idx.shape
    dev = idx.device
    rows = T * K + (T if include_shared else 0)
    if out is None:
        counts = torch.empty(E, dtype=_I32, device=dev)
        offsets = torch.empty(E + 2, dtype=_I32, device=dev)
        row_token = torch.empty(rows, dtype=_I32, device=dev)
        row_of = torch.empty(T, K, dtype=_I32, device=dev)
    else:
        counts, offsets, row_token, row_of = out
    lib = load()
    ws, wsb = WS.get(lib.moe_permute_ws_bytes(T, K, E), dev)
    call("moe_permute", _ptr(idx), T, K, E, int(bool(include_shared)), _ptr(counts),
         _ptr(offsets), _ptr(row_token), _ptr(row_of), _ptr(status), ws, wsb, _stream())
    return counts, offsets, row_token, row_of


# ---- quantisation -----------------------------------------------------------------------

def quant_1x128(x, out=None, pow2=False):
    """BF16 [rows, cols] -> (E4M3 codes uint8 [rows, cols], scales FP32 [cols/128, rows]);
    pow2: power-of-two scales (the MX-native variant)."""
    _check(x, _BF16, "x", 2)
    rows, cols = x.shape
    if out is None:
        q = torch.empty(rows, cols, dtype=_U8, device=x.device)
        s = torch.empty(cols // 128, rows, dtype=_F32, device=x.device)
    else:
        q, s = out
    call("fp8_quant_1x128_pow2" if pow2 else "fp8_quant_1x128", _ptr(x), rows, cols, cols,
         _ptr(q), _ptr(s), _stream())
    return q, s


def quant_scatter_1x128(x, row_of, n_rows, shared_row_base=None, status=None, out=None,
                        pow2=False):
    """Quantise each token row of x once and write it to rows row_of[t, :] and (if
    shared_row_base is not None) shared_row_base + t: bit for bit quant_1x128 followed by
    gather_rows with the inverse map."""
    _check(x, _BF16, "x", 2)
    _check(row_of, _I32, "row_of", 2)
    T, cols = x.shape
    K = row_of.shape[1]
    if out is None:
        q = torch.empty(n_rows, cols, dtype=_U8, device=x.device)
        s = torch.empty(cols // 128, n_rows, dtype=_F32, device=x.device)
    else:
        q, s = out
    base = -1 if shared_row_base is None else int(shared_row_base)
    call("fp8_quant_scatter_1x128_pow2" if pow2 else "fp8_quant_scatter_1x128", _ptr(x), T,
         cols, cols, _ptr(row_of), K, base, n_rows, _ptr(q), _ptr(s), _ptr(status), _stream())
    return q, s


def quant_128x128(w, pow2=False):
    """FP32 [rows, cols] -> (E4M3 codes uint8, scales FP32 [rows/128, cols/128]); pow2:
    power-of-two scales (the MX-native variant)."""
    _check(w, _F32, "w", 2)
    rows, cols = w.shape
    q = torch.empty(rows, cols, dtype=_U8, device=w.device)
    s = torch.empty(rows // 128, cols // 128, dtype=_F32, device=w.device)
    call("fp8_quant_128x128_pow2" if pow2 else "fp8_quant_128x128", _ptr(w), rows, cols,
         _ptr(q), _ptr(s), _stream())
    return q, s


# ---- GEMM and experts -------------------------------------------------------------------

def grouped_gemm(A, sA, B, sB, seg_offsets, M, a_rows=None, status=None, out=None):
    """BF16 C [M, N] = block-scaled A . B_g^T per segment (see include/moe_fp8.h).

    A uint8 [M_a, K], sA FP32 [K/128, M_a], B uint8 [G, N, K], sB FP32 [G, N/128, K/128],
    seg_offsets int32 [G+1], a_rows int32 [M] or None.
    """
    _check(A, _U8, "A", 2)
    _check(sA, _F32, "sA", 2)
    _check(B, _U8, "B", 3)
    _check(sB, _F32, "sB", 3)
    _check(seg_offsets, _I32, "seg_offsets", 1)
    G, N, K = B.shape
    if a_rows is not None:
        _check(a_rows, _I32, "a_rows", 1)
    C = out if out is not None else torch.empty(M, N, dtype=_BF16, device=A.device)
    lib = load()
    ws, wsb = WS.get(lib.fp8_grouped_gemm_ws_bytes(M, K, int(a_rows is not None)), A.device)
    call("fp8_blockscaled_grouped_gemm", _ptr(A), _ptr(sA), A.shape[0], _ptr(a_rows), _ptr(B),
         _ptr(sB), _ptr(seg_offsets), G, M, N, K, _ptr(C), C.stride(0), _ptr(status), ws, wsb,
         _stream())
    return C


def mx_grouped_gemm(A, sA, B, sB, seg_offsets, M, status=None, out=None):
    """MX-native variant of grouped_gemm (power-of-two scales applied by the tensor core);
    A rows already in segment order."""
    _check(A, _U8, "A", 2)
    _check(sA, _F32, "sA", 2)
    _check(B, _U8, "B", 3)
    _check(sB, _F32, "sB", 3)
    _check(seg_offsets, _I32, "seg_offsets", 1)
    G, N, K = B.shape
    C = out if out is not None else torch.empty(M, N, dtype=_BF16, device=A.device)
    call("fp8_mx_grouped_gemm", _ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(seg_offsets), G, M,
         N, K, _ptr(C), C.stride(0), _ptr(status), _stream())
    return C


def swiglu_fwd(xq, sx, row_token, offsets, rows, w13, s13, w2, s2, status=None, out=None):
    """SwiGLU experts over expert segments: returns (hq, sh, y_rows)."""
    for t, dt, n in ((xq, _U8, "xq"), (sx, _F32, "sx"), (row_token, _I32, "row_token"),
                     (offsets, _I32, "offsets"), (w13, _U8, "w13"), (s13, _F32, "s13"),
                     (w2, _U8, "w2"), (s2, _F32, "s2")):
        _check(t, dt, n)
    T, d = xq.shape
    S, f2, d2 = w13.shape
    f = f2 // 2
    dev = xq.device
    if out is None:
        hq = torch.empty(rows, f, dtype=_U8, device=dev)
        sh = torch.empty(f // 128, rows, dtype=_F32, device=dev)
        y_rows = torch.empty(rows, d, dtype=_BF16, device=dev)
    else:
        hq, sh, y_rows = out
    lib = load()
    ws, wsb = WS.get(lib.moe_swiglu_ws_bytes(rows, d, f), dev)
    call("moe_swiglu_fp8_fwd", _ptr(xq), _ptr(sx), T, _ptr(row_token), _ptr(offsets), rows,
         _ptr(w13), _ptr(s13), _ptr(w2), _ptr(s2), S, d, f, _ptr(hq), _ptr(sh), _ptr(y_rows),
         _ptr(status), ws, wsb, _stream())
    return hq, sh, y_rows


def gather_rows(src, src_scale, rows, row_limit=None, status=None, out=None):
    """FP8 rows in a new order: dst[r] = src[rows[r]] with their 1x128 scales."""
    _check(src, _U8, "src", 2)
    _check(src_scale, _F32, "src_scale", 2)
    _check(rows, _I32, "rows", 1)
    n, cols = rows.numel(), src.shape[1]
    if out is None:
        dst = torch.empty(n, cols, dtype=_U8, device=src.device)
        dsc = torch.empty(cols // 128, n, dtype=_F32, device=src.device)
    else:
        dst, dsc = out
    call("moe_gather_rows_fp8", _ptr(src), _ptr(src_scale), src.shape[0], _ptr(rows),
         _ptr(row_limit), n, cols, _ptr(dst), _ptr(dsc), _ptr(status), _stream())
    return dst, dsc


def gate_up(xq_rows, sx_rows, offsets, w13, s13, status=None, out=None, mx=False):
    """hq, sh = requantised silu(gate) * up over expert segments (rows in segment order);
    mx: the MX-native variant (power-of-two scales in and out)."""
    for t, dt, n in ((xq_rows, _U8, "xq_rows"), (sx_rows, _F32, "sx_rows"),
                     (offsets, _I32, "offsets"), (w13, _U8, "w13"), (s13, _F32, "s13")):
        _check(t, dt, n)
    rows, d = xq_rows.shape
    S, f2, _ = w13.shape
    f = f2 // 2
    if out is None:
        hq = torch.empty(rows, f, dtype=_U8, device=xq_rows.device)
        sh = torch.empty(f // 128, rows, dtype=_F32, device=xq_rows.device)
    else:
        hq, sh = out
    call("moe_gate_up_mx" if mx else "moe_gate_up_fp8", _ptr(xq_rows), _ptr(sx_rows),
         _ptr(offsets), rows, _ptr(w13), _ptr(s13), S, d, f, _ptr(hq), _ptr(sh), _ptr(status),
         _stream())
    return hq, sh


def combine(y_rows, row_of, gate, shared_row_base, status=None, out=None):
    """BF16 y [T, d] = shared + sum_k gate * expert rows (FP32 accumulation)."""
    _check(y_rows, _BF16, "y_rows", 2)
    _check(row_of, _I32, "row_of", 2)
    _check(gate, _F32, "gate", 2)
    T, K = row_of.shape
    d = y_rows.shape[1]
    y = out if out is not None else torch.empty(T, d, dtype=_BF16, device=y_rows.device)
    call("moe_combine", _ptr(y_rows), y_rows.shape[0], _ptr(row_of), _ptr(gate), T, K, d,
         int(shared_row_base), _ptr(y), _ptr(status), _stream())
    return y


# ---- backward of the experts (training) -------------------------------------------------

def gate_up_train(xq_rows, sx_rows, offsets, w13, s13, status=None, out=None):
    """Training-forward gate/up: (hq, sh) as gate_up, plus the SwiGLU inputs cached in FP8:
    guq uint8 [rows, 2f] (gate columns first) with 1x128 scales sgu [2f/128, rows]."""
    for t, dt, n in ((xq_rows, _U8, "xq_rows"), (sx_rows, _F32, "sx_rows"),
                     (offsets, _I32, "offsets"), (w13, _U8, "w13"), (s13, _F32, "s13")):
        _check(t, dt, n)
    rows, d = xq_rows.shape
    S, f2, _ = w13.shape
    f = f2 // 2
    dev = xq_rows.device
    if out is None:
        hq = torch.empty(rows, f, dtype=_U8, device=dev)
        sh = torch.empty(f // 128, rows, dtype=_F32, device=dev)
        guq = torch.empty(rows, 2 * f, dtype=_U8, device=dev)
        sgu = torch.empty(2 * f // 128, rows, dtype=_F32, device=dev)
    else:
        hq, sh, guq, sgu = out
    call("moe_gate_up_fp8_train", _ptr(xq_rows), _ptr(sx_rows), _ptr(offsets), rows, _ptr(w13),
         _ptr(s13), S, d, f, _ptr(hq), _ptr(sh), _ptr(guq), _ptr(sgu), _ptr(status), _stream())
    return hq, sh, guq, sgu


def transpose_128x128(w, s, gate_up_interleaved=False):
    """Transposed FP8 weights with transposed 128x128 block scales: w uint8 [G, R, C], s FP32
    [G, R/128, C/128] -> (wT [G, C, R], sT [G, C/128, R/128]); gate_up_interleaved: w is the
    64-row interleaved gate/up matrix and wT's columns come out gate first."""
    _check(w, _U8, "w", 3)
    _check(s, _F32, "s", 3)
    G, R, C = w.shape
    wT = torch.empty(G, C, R, dtype=_U8, device=w.device)
    sT = torch.empty(G, C // 128, R // 128, dtype=_F32, device=w.device)
    call("fp8_transpose_128x128", _ptr(w), _ptr(s), G, R, C, int(bool(gate_up_interleaved)),
         _ptr(wT), _ptr(sT), _stream())
    return wT, sT


def padded_rows_cap(rows, G):
    """Columns to allocate for the 128x1 (padded) layout of `rows` rows in G segments."""
    cap = load().moe_padded_rows_cap(int(rows), int(G))
    if cap < 0:
        raise ValueError("bad rows / G")
    return cap


def segment_pad_offsets(offsets, G, status=None, out=None):
    """int32 [G+1]: every segment's first padded row (128-row blocks per segment)."""
    _check(offsets, _I32, "offsets", 1)
    pad = out if out is not None else torch.empty(G + 1, dtype=_I32, device=offsets.device)
    call("moe_segment_pad_offsets", _ptr(offsets), G, _ptr(pad), _ptr(status), _stream())
    return pad


def combine_bwd_rows(dy, gate, row_of, shared_row_base, n_rows, status=None, out=None):
    """BF16 [n_rows, d] gradient of the expert output rows: gate * dy per routed row, dy
    per shared row."""
    _check(dy, _BF16, "dy", 2)
    _check(gate, _F32, "gate", 2)
    _check(row_of, _I32, "row_of", 2)
    T, d = dy.shape
    K = row_of.shape[1]
    dy_rows = out if out is not None else torch.empty(n_rows, d, dtype=_BF16, device=dy.device)
    call("moe_combine_bwd_rows", _ptr(dy), _ptr(gate), _ptr(row_of), T, K, d,
         int(shared_row_base), n_rows, _ptr(dy_rows), _ptr(status), _stream())
    return dy_rows


def quant_128x1_pow2(src, offsets, pad, kcap, rows=None, status=None, out=None):
    """128x1 power-of-two tiles of the segment-order rows (src[rows[r]] when gathering),
    transposed: (qT uint8 [cols, kcap], sT FP32 [kcap/128, cols])."""
    _check(src, _BF16, "src", 2)
    _check(offsets, _I32, "offsets", 1)
    _check(pad, _I32, "pad", 1)
    if rows is not None:
        _check(rows, _I32, "rows", 1)
    cols = src.shape[1]
    G = offsets.numel() - 1
    if out is None:
        qT = torch.empty(cols, kcap, dtype=_U8, device=src.device)
        sT = torch.empty(kcap // 128, cols, dtype=_F32, device=src.device)
    else:
        qT, sT = out
    call("fp8_quant_128x1_pow2", _ptr(src), src.shape[0], _ptr(rows), cols, _ptr(offsets),
         _ptr(pad), G, kcap, _ptr(qT), _ptr(sT), _ptr(status), _stream())
    return qT, sT


def swiglu_bwd(guq, sgu, dh, offsets, pad, kcap, out=None):
    """SwiGLU backward with recomputation: (dguq, sdgu, hT, shT, dguT, sdguT), see
    include/moe_fp8.h."""
    _check(guq, _U8, "guq", 2)
    _check(sgu, _F32, "sgu", 2)
    _check(dh, _BF16, "dh", 2)
    rows, f = dh.shape
    G = offsets.numel() - 1
    dev = dh.device
    if out is None:
        out = (torch.empty(rows, 2 * f, dtype=_U8, device=dev),
               torch.empty(2 * f // 128, rows, dtype=_F32, device=dev),
               torch.empty(f, kcap, dtype=_U8, device=dev),
               torch.empty(kcap // 128, f, dtype=_F32, device=dev),
               torch.empty(2 * f, kcap, dtype=_U8, device=dev),
               torch.empty(kcap // 128, 2 * f, dtype=_F32, device=dev))
    dguq, sdgu, hT, shT, dguT, sdguT = out
    call("moe_swiglu_bwd_fp8", _ptr(guq), _ptr(sgu), _ptr(dh), rows, f, _ptr(offsets),
         _ptr(pad), G, kcap, _ptr(dguq), _ptr(sdgu), _ptr(hT), _ptr(shT), _ptr(dguT),
         _ptr(sdguT), _stream())
    return out


def wgrad(aT, saT, bT, sbT, pad, status=None, out=None):
    """FP32 dW [G, I, J] = per expert, sum over its 128-row blocks of the block-scaled
    aT . bT^T (128x1 power-of-two scales applied by the tensor core)."""
    _check(aT, _U8, "aT", 2)
    _check(bT, _U8, "bT", 2)
    _check(saT, _F32, "saT", 2)
    _check(sbT, _F32, "sbT", 2)
    _check(pad, _I32, "pad", 1)
    I, kcap = aT.shape
    J = bT.shape[0]
    G = pad.numel() - 1
    dW = out if out is not None else torch.empty(G, I, J, dtype=_F32, device=aT.device)
    call("fp8_wgrad_grouped_gemm", _ptr(aT), _ptr(saT), _ptr(bT), _ptr(sbT), _ptr(pad), G, I, J,
         kcap, _ptr(dW), _ptr(status), _stream())
    return dW
