"""One DeepSeek-V3 MoE FFN layer forward, assembled from the C-ABI calls.

The order is the one the pages give for a MoE layer ("DeepSeek-V3" book, ch. 7 and
ch. 15; "DeepSeek-V3" summary, core ideas 1, 2 and 6): router logits kept above FP8,
sigmoid affinities with the selection-only bias and the group limit, normalised gates,
FP8 quantisation of the activations before dispatch, grouping of rows by expert,
SwiGLU experts as block-scaled FP8 grouped GEMMs (routed experts and the shared expert
as one more segment), and the gate-weighted BF16 combine.  The layer output excludes
the residual; ``forward(..., residual=True)`` adds x afterwards.

Weights are prepared once (not timed): expert matrices are quantised 128x128 on the
GPU and the gate/up matrices are interleaved in 64-row blocks so one 128-column GEMM
tile holds matching gate and up columns.

``mx=True`` runs the MX-native variant: power-of-two scales for x, the weights and h,
applied by the tensor core (tcgen05 kind::mxf8f6f4) instead of by software promotion;
its weights come from ``make_weights(..., pow2=True)``.

``train=True`` makes ``forward`` keep the SwiGLU inputs in FP8 and enables ``backward``:
the experts' input and weight gradients from the three FP8 GEMMs of each linear layer
("DeepSeek-V3" book, ch. 17 "One linear layer creates three GEMMs", "SwiGLU
recomputation"; ch. 16 "Why transposition is not trivial").  The router and gate
gradients are not computed.
"""

from dataclasses import dataclass

import torch

from . import ops


@dataclass
class MoEWeights:
    centroids: torch.Tensor   # FP32 [E, d]
    w_hilo: torch.Tensor      # BF16 [2, E, d]
    bias: torch.Tensor        # FP32 [E]
    w13: torch.Tensor         # E4M3 [E+1, 2f, d], gate/up interleaved in 64-row blocks
    s13: torch.Tensor         # FP32 [E+1, 2f/128, d/128]
    w2: torch.Tensor          # E4M3 [E+1, d, f]
    s2: torch.Tensor          # FP32 [E+1, d/128, f/128]


def save_bias(bias, path):
    """Write the selection bias b [E] (FP32), the layer's only state that training
    updates step by step ("DeepSeek-V3" summary, core idea 2), to a ``.npy`` file."""
    import numpy as np
    if bias.dtype != torch.float32 or bias.dim() != 1:
        raise ValueError("bias must be a 1-D float32 tensor")
    np.save(path, bias.detach().cpu().numpy())


def load_bias(path, out):
    """Read a bias saved by ``save_bias`` into ``out`` (a float32 [E] tensor on any device,
    e.g. ``weights.bias``) in place; the stored length must equal E."""
    import numpy as np
    b = np.load(path)
    if b.dtype != np.float32 or b.shape != tuple(out.shape) or out.dtype != torch.float32:
        raise ValueError(f"stored bias {b.dtype}{list(b.shape)} does not fit "
                         f"{out.dtype}{list(out.shape)}")
    out.copy_(torch.from_numpy(b))
    return out


def interleave_gate_up(q1, s1, q3, s3):
    """Gate [f, d] and up [f, d] codes/scales -> the layout the gate/up GEMM takes.

    Codes alternate in 64-row blocks (rows [128j, 128j+64) = gate rows [64j, 64j+64),
    rows [128j+64, 128j+128) = the matching up rows), so every 128-column GEMM tile holds
    matching gate and up columns.  Scales stay per 128x128 block of the original
    matrices, alternating gate block i, up block i."""
    f, d = q1.shape
    w13 = torch.stack([q1.view(f // 64, 64, d), q3.view(f // 64, 64, d)], dim=1)
    s13 = torch.stack([s1, s3], dim=1)
    return w13.reshape(2 * f, d), s13.reshape(2 * f // 128, d // 128)


def quantise_expert(w1, w3, w2, pow2=False):
    """FP32 (w1 [f,d], w3 [f,d], w2 [d,f]) on the GPU -> (w13, s13, w2q, s2) via the library
    (pow2: power-of-two scales, for the MX-native variant)."""
    q1, s1 = ops.quant_128x128(w1.contiguous(), pow2=pow2)
    q3, s3 = ops.quant_128x128(w3.contiguous(), pow2=pow2)
    q2, s2 = ops.quant_128x128(w2.contiguous(), pow2=pow2)
    w13, s13 = interleave_gate_up(q1, s1, q3, s3)
    return w13, s13, q2, s2


def make_weights(cfg, device="cuda", base_seed=0, expert_fn=None, pow2=False):
    """Seeded synthetic weights for ``cfg`` (a workloads.MoEConfig), quantised on the GPU.

    ``expert_fn(e)`` may override the FP32 expert generator (returns w1, w3, w2)."""
    import workloads
    dev = torch.device(device)
    cen = workloads.gen_centroids(cfg, base_seed).to(dev)
    bias = workloads.gen_bias(cfg, base_seed).to(dev)
    E, d, f = cfg.E, cfg.d, cfg.f
    w13 = torch.empty(E + 1, 2 * f, d, dtype=torch.uint8, device=dev)
    s13 = torch.empty(E + 1, 2 * f // 128, d // 128, dtype=torch.float32, device=dev)
    w2 = torch.empty(E + 1, d, f, dtype=torch.uint8, device=dev)
    s2 = torch.empty(E + 1, d // 128, f // 128, dtype=torch.float32, device=dev)
    for e in range(E + 1):
        if expert_fn is None:
            w = workloads.gen_expert_f32(cfg, e, device=dev, base_seed=base_seed)
        else:
            w = tuple(t.to(dev) for t in expert_fn(e))
        w13[e], s13[e], w2[e], s2[e] = quantise_expert(*w, pow2=pow2)
        del w
    return MoEWeights(cen, ops.router_split_bf16(cen), bias, w13, s13, w2, s2)


class MoELayer:
    """Buffers and the sequence of library calls for one layer forward."""

    def __init__(self, cfg, weights, T=None, mx=False, train=False):
        self.cfg = cfg
        self.w = weights
        self.mx = mx
        self.train = train
        if train and mx:
            raise ValueError("the training path uses the FP32-scale recipe")
        self.T = cfg.T if T is None else T
        T, E, K, d, f = self.T, cfg.E, cfg.K, cfg.d, cfg.f
        dev = weights.w13.device
        self.rows = T * K + T
        emp = lambda *s, dt=torch.float32: torch.empty(*s, dtype=dt, device=dev)
        self.z = emp(T, E)
        self.idx = emp(T, K, dt=torch.int32)
        self.gate = emp(T, K)
        self.counts = emp(E, dt=torch.int32)
        self.offsets = emp(E + 2, dt=torch.int32)
        self.row_token = emp(self.rows, dt=torch.int32)
        self.row_of = emp(T, K, dt=torch.int32)
        self.xq_rows = emp(self.rows, d, dt=torch.uint8)
        self.sx_rows = emp(d // 128, self.rows)
        self.hq = emp(self.rows, f, dt=torch.uint8)
        self.sh = emp(f // 128, self.rows)
        self.y_rows = emp(self.rows, d, dt=torch.bfloat16)
        self.y = emp(T, d, dt=torch.bfloat16)
        self.status = ops.new_status(dev)
        self.seg_end = self.offsets[cfg.E + 1:cfg.E + 2]     # device int32: rows in use
        if train:
            self.guq = emp(self.rows, 2 * f, dt=torch.uint8)     # SwiGLU inputs, FP8
            self.sgu = emp(2 * f // 128, self.rows)
            self.x = None
            self._wT = None
            self._ones = torch.ones(T, K, dtype=torch.float32, device=dev)

    # kernel launches of one forward, by stage (bias_update adds one more)
    STAGE_LAUNCHES = {"router_logits": 1, "route": 1, "permute": 3, "quant_dispatch": 1,
                      "gate_up": 1, "down": 1, "combine": 1}

    def forward(self, x, logits=None, residual=False, mark=None, out=None):
        """x BF16 [T, d] on the device -> y BF16 [T, d] (the layer's own buffer, or ``out``).

        ``mark(name)``, if given, is called after each stage's launches (the bench records
        a CUDA event there)."""
        cfg, w = self.cfg, self.w
        mark = mark or (lambda name: None)
        if logits is None:
            ops.router_logits(x, w.w_hilo, self.status, out=self.z)
            z = self.z
        else:
            z = logits
        mark("router_logits")
        ops.route(z, w.bias, cfg.n_groups, cfg.topk_groups, cfg.K, out=(self.idx, self.gate))
        mark("route")
        ops.permute(self.idx, cfg.E, True, self.status,
                    out=(self.counts, self.offsets, self.row_token, self.row_of))
        mark("permute")
        # 1x128 quantisation straight into segment order (one pass over x)
        ops.quant_scatter_1x128(x, self.row_of, self.rows, self.T * cfg.K, self.status,
                                out=(self.xq_rows, self.sx_rows), pow2=self.mx)
        mark("quant_dispatch")
        if self.train:
            ops.gate_up_train(self.xq_rows, self.sx_rows, self.offsets, w.w13, w.s13,
                              self.status, out=(self.hq, self.sh, self.guq, self.sgu))
            self.x = x
        else:
            ops.gate_up(self.xq_rows, self.sx_rows, self.offsets, w.w13, w.s13, self.status,
                        out=(self.hq, self.sh), mx=self.mx)
        mark("gate_up")
        down = ops.mx_grouped_gemm if self.mx else ops.grouped_gemm
        down(self.hq, self.sh, w.w2, w.s2, self.offsets, self.rows, status=self.status,
             out=self.y_rows)
        mark("down")
        y = self.y if out is None else out
        ops.combine(self.y_rows, self.row_of, self.gate, self.T * cfg.K, self.status, out=y)
        mark("combine")
        if residual:
            return y + x
        return y

    # kernel launches of one backward
    BACKWARD_LAUNCHES = 11

    def transposed_weights(self):
        """The Dgrad operands, made once: W2^T [E+1, f, d] and [W1; W3]^T [E+1, d, 2f] with
        their 128x128 block scales transposed."""
        if self._wT is None:
            w = self.w
            w2T, s2T = ops.transpose_128x128(w.w2, w.s2)
            w13T, s13T = ops.transpose_128x128(w.w13, w.s13, gate_up_interleaved=True)
            self._wT = (w2T, s2T, w13T, s13T)
        return self._wT

    def backward(self, dy, mark=None):
        """dy BF16 [T, d] (gradient of the layer output) -> dict of dx BF16 [T, d] (through
        the experts, not the router), dw13 FP32 [E+1, 2f, d] ([dW1; dW3], gate rows first)
        and dw2 FP32 [E+1, d, f], plus the intermediate tensors (the layer's own buffers,
        overwritten by the next backward).  Needs a forward with train=True first."""
        if not self.train or self.x is None:
            raise RuntimeError("backward needs a forward of a layer built with train=True")
        cfg, T, K, E = self.cfg, self.T, self.cfg.K, self.cfg.E
        rows, G = self.rows, E + 1
        mark = mark or (lambda name: None)
        w2T, s2T, w13T, s13T = self.transposed_weights()
        st = self.status
        b = self._backward_buffers(dy.device)
        kcap = b["kcap"]
        ops.combine_bwd_rows(dy, self.gate, self.row_of, T * K, rows, status=st, out=b["dy_rows"])
        ops.quant_1x128(b["dy_rows"], out=(b["dyq"], b["sdy"]))
        ops.grouped_gemm(b["dyq"], b["sdy"], w2T, s2T, self.offsets, rows, status=st, out=b["dh"])
        mark("down_dgrad")
        ops.segment_pad_offsets(self.offsets, G, status=st, out=b["pad"])
        ops.swiglu_bwd(self.guq, self.sgu, b["dh"], self.offsets, b["pad"], kcap,
                       out=(b["dguq"], b["sdgu"], b["hT"], b["shT"], b["dguT"], b["sdguT"]))
        mark("swiglu_bwd")
        ops.grouped_gemm(b["dguq"], b["sdgu"], w13T, s13T, self.offsets, rows, status=st,
                         out=b["dx_rows"])
        ops.combine(b["dx_rows"], self.row_of, self._ones, T * K, st, out=b["dx"])  # gates 1
        mark("gate_up_dgrad")
        ops.quant_128x1_pow2(b["dy_rows"], self.offsets, b["pad"], kcap, status=st,
                             out=(b["dyT"], b["sdyT"]))
        ops.wgrad(b["dyT"], b["sdyT"], b["hT"], b["shT"], b["pad"], status=st, out=b["dw2"])
        mark("down_wgrad")
        ops.quant_128x1_pow2(self.x, self.offsets, b["pad"], kcap, rows=self.row_token,
                             status=st, out=(b["xT"], b["sxT"]))
        ops.wgrad(b["dguT"], b["sdguT"], b["xT"], b["sxT"], b["pad"], status=st, out=b["dw13"])
        mark("gate_up_wgrad")
        return b

    def _backward_buffers(self, dev):
        """The backward's outputs and intermediates, allocated on the first backward."""
        if getattr(self, "_bwd", None) is None:
            cfg, T, E, d, f = self.cfg, self.T, self.cfg.E, self.cfg.d, self.cfg.f
            rows, G = self.rows, E + 1
            kcap = ops.padded_rows_cap(rows, G)
            emp = lambda *sh, dt=torch.float32: torch.empty(*sh, dtype=dt, device=dev)
            u8, bf, i32 = torch.uint8, torch.bfloat16, torch.int32
            self._bwd = dict(
                kcap=kcap, dy_rows=emp(rows, d, dt=bf), dyq=emp(rows, d, dt=u8),
                sdy=emp(d // 128, rows), dh=emp(rows, f, dt=bf), pad=emp(G + 1, dt=i32),
                dguq=emp(rows, 2 * f, dt=u8), sdgu=emp(2 * f // 128, rows),
                hT=emp(f, kcap, dt=u8), shT=emp(kcap // 128, f),
                dguT=emp(2 * f, kcap, dt=u8), sdguT=emp(kcap // 128, 2 * f),
                dx_rows=emp(rows, d, dt=bf), dx=emp(T, d, dt=bf),
                dyT=emp(d, kcap, dt=u8), sdyT=emp(kcap // 128, d),
                xT=emp(d, kcap, dt=u8), sxT=emp(kcap // 128, d),
                dw2=emp(G, d, f), dw13=emp(G, 2 * f, d))
        return self._bwd

    def bias_update(self, gamma):
        """Aux-loss-free bias step from this forward's expert loads (in place)."""
        ops.bias_update(self.w.bias, self.counts, self.T, self.cfg.K, gamma)

    def check_status(self):
        st = ops.status_value(self.status)
        if st != 0:
            from ._lib import STATUS
            raise RuntimeError(f"device status {STATUS.get(st, st)}")
