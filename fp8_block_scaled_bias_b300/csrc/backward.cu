// Backward of the SwiGLU experts in FP8: the data movement and elementwise kernels around
// the Dgrad and Wgrad GEMMs ("DeepSeek-V3" book, ch. 17 "One linear layer creates three
// GEMMs", "SwiGLU recomputation"; ch. 16 "Why transposition is not trivial").
//
//   seg_pad_kernel       padded offsets: each segment's rows cut into 128-row blocks that
//                        start at the segment's first row (the Wgrad K blocks)
//   transpose_kernel     FP8 [G][R][C] -> [G][C][R] with the 128x128 block scales
//                        transposed: a weight's Dgrad operand (setup, not per step)
//   dispatch_grad_kernel gradient of the combine w.r.t. the expert output rows:
//                        dy_rows[row_of[t][k]] = bf16(g[t][k] * dy[t]), shared rows dy[t]
//   regroup_kernel       BF16 rows (optionally gathered) -> 128x1 tiles with power-of-two
//                        scales, stored transposed [C][R_pad] (the Wgrad operands)
//   swiglu_bwd_kernel    recomputes h = silu(g) u from the FP8-cached g, u; dG, dU from dh;
//                        writes [dG | dU] in 1x128 tiles (the gate/up Dgrad operand) and
//                        h^T, [dG | dU]^T in 128x1 power-of-two tiles (the Wgrad operands)
//
// The 128x1 tiles use power-of-two scales, which the pages give for the regrouped
// backward tensors; they are quantised from the higher-precision values (BF16 or FP32),
// one scale per (128-row block, column).  Padded rows of a block hold code 0.
#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr int kTile = 128;             // rows and columns of a regrouping tile
constexpr int kBwdThreads = 256;

// Padded row block rb -> (segment e, first row r0, valid rows nv); false past the end.
MOE_DEV bool block_of(const int32_t* __restrict__ seg, const int32_t* __restrict__ pad, int G,
                      int rb, int& e, int& r0, int& nv) {
  const int p0 = rb * kTile;
  if (p0 >= pad[G]) return false;
  int lo = 0, hi = G - 1;                 // largest e with pad[e] <= p0 (and a non-empty range)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pad[mid] <= p0) lo = mid;
    else hi = mid - 1;
  }
  e = lo;
  r0 = seg[e] + (p0 - pad[e]);
  nv = min(kTile, seg[e + 1] - r0);
  return true;
}

// FP32 -> E4M3 byte (round to nearest even, saturating).
MOE_DEV uint32_t e4m3_byte(float v) { return f32x2_to_e4m3x2(v, 0.0f) & 0xFFu; }

MOE_DEV float e4m3_value(uint32_t code) {
  // E4M3 fn: bias 7, 3 mantissa bits, subnormals below 2^-6 (codes 0x7F/0xFF are NaN)
  const uint32_t s = code & 0x80u, e = (code >> 3) & 0xFu, m = code & 7u;
  float v;
  if (e == 0) v = static_cast<float>(m) * 0.001953125f;                 // m * 2^-9
  else v = __uint_as_float(((e + 120u) << 23) | (m << 20));             // 2^(e-7) * 1.m
  if ((code & 0x7Fu) == 0x7Fu) v = __uint_as_float(0x7FC00000u);
  return s ? -v : v;
}

}  // namespace

// ---- padded segment offsets ------------------------------------------------------------

__global__ void __launch_bounds__(1024) seg_pad_kernel(const int32_t* __restrict__ seg, int G,
                                                       int32_t* __restrict__ pad,
                                                       int32_t* __restrict__ status) {
  __shared__ int wsum[32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int cnt = t < G ? seg[t + 1] - seg[t] : 0;
  if (t < G && cnt < 0) set_status(status, MOE_ERR_DEVICE_DATA);
  const int v = t < G ? (max(cnt, 0) + kTile - 1) / kTile * kTile : 0;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += wsum[w];
  if (t == 0) pad[0] = 0;
  if (t < G) pad[t + 1] = base + incl;
}

// ---- weight transpose (setup) ------------------------------------------------------------

// Row r of the gate-first matrix [gate; up] in the 64-row interleaved layout.
MOE_DEV int interleaved_row(int r, int R) {
  const int half = R / 2;
  return r < half ? (r / 64) * 128 + (r % 64) : ((r - half) / 64) * 128 + 64 + (r - half) % 64;
}

// One 64 x 64 byte tile per block: dst[g][c][r] = src[g][row(r)][c], row(r) = r, or the
// interleaved position of gate-first row r.
__global__ void __launch_bounds__(256) transpose_kernel(const uint8_t* __restrict__ src, int R,
                                                        int C, int interleaved,
                                                        uint8_t* __restrict__ dst) {
  __shared__ uint8_t tile[64][65];
  const long long g = blockIdx.z;
  const int r0 = blockIdx.y * 64, c0 = blockIdx.x * 64;
  const uint8_t* s = src + g * R * static_cast<long long>(C);
  uint8_t* d = dst + g * R * static_cast<long long>(C);
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int rr = i >> 6, cc = i & 63;
    const int sr = interleaved ? interleaved_row(r0 + rr, R) : r0 + rr;
    tile[rr][cc] = s[static_cast<long long>(sr) * C + c0 + cc];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int cc = i >> 6, rr = i & 63;
    d[static_cast<long long>(c0 + cc) * R + r0 + rr] = tile[rr][cc];
  }
}

// sT[g][cb][rb] = s[g][blk(rb)][cb]; with the interleaved source the block scales alternate
// gate block i (2i), up block i (2i + 1), so gate-first block rb is 2 rb, or 2 (rb - RB/2) + 1.
__global__ void transpose_scales_kernel(const float* __restrict__ s, int RB, int CB, int G,
                                        int interleaved, float* __restrict__ sT) {
  const long long n = static_cast<long long>(G) * RB * CB;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long g = i / (RB * CB);
    const int rem = static_cast<int>(i % (RB * CB));
    const int rb = rem / CB, cb = rem % CB;
    const int sb = interleaved ? (rb < RB / 2 ? 2 * rb : 2 * (rb - RB / 2) + 1) : rb;
    sT[(g * CB + cb) * RB + rb] = s[(g * RB + sb) * CB + cb];
  }
}

// ---- gradient of the combine w.r.t. the expert output rows -------------------------------

// One block per token: row_of[t][k] gets bf16(fl32(gate[t][k] * dy[t][c])); the shared row
// (shared_row_base + t, when >= 0) gets dy[t] unchanged.
__global__ void __launch_bounds__(256) dispatch_grad_kernel(
    const uint16_t* __restrict__ dy, const float* __restrict__ gate,
    const int32_t* __restrict__ row_of, int K, int d, int shared_row_base, int n_rows,
    uint16_t* __restrict__ dy_rows, int32_t* __restrict__ status) {
  const int t = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(dy + static_cast<long long>(t) * d);
  for (int k = -1; k < K; ++k) {
    int row;
    float g = 1.0f;
    if (k < 0) {
      if (shared_row_base < 0) continue;
      row = shared_row_base + t;
    } else {
      row = row_of[static_cast<long long>(t) * K + k];
      g = gate[static_cast<long long>(t) * K + k];
    }
    if (row < 0 || row >= n_rows) {
      if (threadIdx.x == 0) set_status(status, MOE_ERR_DEVICE_DATA);
      continue;
    }
    uint4* dst = reinterpret_cast<uint4*>(dy_rows + static_cast<long long>(row) * d);
    for (int i = threadIdx.x; i < d / 8; i += blockDim.x) {
      uint4 v = src[i];
      if (k >= 0) {
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          w[j] = pack_bf16x2(__fmul_rn(g, __uint_as_float(w[j] << 16)),
                             __fmul_rn(g, __uint_as_float(w[j] & 0xFFFF0000u)));
        v = make_uint4(w[0], w[1], w[2], w[3]);
      }
      dst[i] = v;
    }
  }
}

// ---- 128x1 regrouping of BF16 rows ---------------------------------------------------------

// Block (rb, cb): rows [r0, r0 + nv) of the segment holding padded block rb (source row
// rows[r] when gathering), columns [128 cb, 128 cb + 128).  Column c's scale over the
// block is the power-of-two rule on its max |x|; codes go to qT[col][rb * 128 + r].
template <bool GATHER>
__global__ void __launch_bounds__(kBwdThreads) regroup_kernel(
    const uint16_t* __restrict__ src, int src_rows, const int32_t* __restrict__ rows, int C,
    const int32_t* __restrict__ seg, const int32_t* __restrict__ pad, int G, int ldq,
    uint8_t* __restrict__ qT, float* __restrict__ sT, int32_t* __restrict__ status) {
  __shared__ __align__(16) uint16_t tile[kTile][kTile + 8];
  __shared__ float part[2][kTile];
  int e, r0, nv;
  if (!block_of(seg, pad, G, blockIdx.x, e, r0, nv)) return;
  const int cb = blockIdx.y;
  const int tid = threadIdx.x;
  // load 128 rows x 256 bytes: 16 uint4 per row
  for (int i = tid; i < kTile * 16; i += kBwdThreads) {
    const int r = i >> 4, v = i & 15;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (r < nv) {
      int sr = r0 + r;
      if (GATHER) sr = rows[sr];
      if (sr >= 0 && sr < src_rows)
        val = *reinterpret_cast<const uint4*>(src + static_cast<long long>(sr) * C + cb * kTile +
                                              v * 8);
      else if (v == 0)
        set_status(status, MOE_ERR_DEVICE_DATA);
    }
    *reinterpret_cast<uint4*>(&tile[r][v * 8]) = val;
  }
  __syncthreads();
  const int c = tid & (kTile - 1), half = tid >> 7;
  float amax = 0.0f;
  for (int r = half * 64; r < half * 64 + 64; ++r)
    amax = fmaxf(amax, fabsf(bf16_bits_to_f32(tile[r][c])));
  part[half][c] = amax;
  __syncthreads();
  const float s = pow2_scale_from_amax(fmaxf(part[0][c], part[1][c]));
  const float rs = __frcp_rn(s);                          // exact: s is a power of two
  const int col = cb * kTile + c;
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int r = half * 64 + 4 * i;
    w[i] = e4m3_byte(bf16_bits_to_f32(tile[r][c]) * rs) |
           (e4m3_byte(bf16_bits_to_f32(tile[r + 1][c]) * rs) << 8) |
           (e4m3_byte(bf16_bits_to_f32(tile[r + 2][c]) * rs) << 16) |
           (e4m3_byte(bf16_bits_to_f32(tile[r + 3][c]) * rs) << 24);
  }
  uint4* dst = reinterpret_cast<uint4*>(qT + static_cast<long long>(col) * ldq +
                                        blockIdx.x * kTile + half * 64);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  if (half == 0) sT[static_cast<long long>(blockIdx.x) * C + col] = s;
}

// ---- SwiGLU backward with recomputation -----------------------------------------------------

namespace {
struct SwigluVals {
  float h, dg, du;
};

// g, u from their E4M3 codes and 1x128 scales; sigmoid with expf and IEEE division.
MOE_DEV SwigluVals swiglu_bwd_at(uint32_t qg, uint32_t qu, float sg, float su, float dh) {
  const float g = __fmul_rn(e4m3_value(qg), sg);
  const float u = __fmul_rn(e4m3_value(qu), su);
  const float sig = __fdiv_rn(1.0f, 1.0f + expf(-g));
  const float silu = g * sig;
  SwigluVals v;
  v.h = silu * u;
  v.du = dh * silu;
  v.dg = dh * u * sig * fmaf(g, 1.0f - sig, 1.0f);
  return v;
}

MOE_DEV void smem_max(float* p, float v) {
  atomicMax(reinterpret_cast<int*>(p), __float_as_int(v));   // v >= 0: int order = float order
}
}  // namespace

// Block (rb, cb): the segment rows of padded block rb, hidden columns [128 cb, 128 cb + 128).
// Pass 1 finds the row max-abs of dG and dU (their 1x128 groups) and the column max-abs of
// h, dG and dU (their 128x1 groups); pass 2 recomputes the values and writes the codes.
__global__ void __launch_bounds__(kBwdThreads) swiglu_bwd_kernel(
    const uint8_t* __restrict__ guq, const float* __restrict__ sgu,
    const uint16_t* __restrict__ dh, int R, int f, const int32_t* __restrict__ seg,
    const int32_t* __restrict__ pad, int G, int ldq, uint8_t* __restrict__ dguq,
    float* __restrict__ sdgu, uint8_t* __restrict__ hT, float* __restrict__ shT,
    uint8_t* __restrict__ dguT, float* __restrict__ sdguT) {
  // dynamic shared memory: the tile's g codes, u codes (rows padded to 144 bytes) and dh
  // (rows padded to 136 BF16 values), 71,680 bytes
  extern __shared__ __align__(16) uint8_t bwd_smem[];
  auto tg = reinterpret_cast<uint8_t(*)[kTile + 16]>(bwd_smem);
  auto tu = reinterpret_cast<uint8_t(*)[kTile + 16]>(bwd_smem + kTile * (kTile + 16));
  auto tdh = reinterpret_cast<uint16_t(*)[kTile + 8]>(bwd_smem + 2 * kTile * (kTile + 16));
  __shared__ float sg_s[kTile], su_s[kTile];
  __shared__ float rmax_g[kTile], rmax_u[kTile];
  __shared__ float cpart[3][2][kTile];
  int e, r0, nv;
  if (!block_of(seg, pad, G, blockIdx.x, e, r0, nv)) return;
  const int cb = blockIdx.y, tid = threadIdx.x;
  const int NB = f / kTile;                     // 1x128 groups of g (and of u)
  for (int i = tid; i < kTile * 8; i += kBwdThreads) {   // codes: 8 uint4 per row each
    const int r = i >> 3, v = i & 7;
    uint4 a = make_uint4(0, 0, 0, 0), b = a;
    if (r < nv) {
      const uint8_t* row = guq + static_cast<long long>(r0 + r) * 2 * f;
      a = *reinterpret_cast<const uint4*>(row + cb * kTile + v * 16);
      b = *reinterpret_cast<const uint4*>(row + f + cb * kTile + v * 16);
    }
    *reinterpret_cast<uint4*>(&tg[r][v * 16]) = a;
    *reinterpret_cast<uint4*>(&tu[r][v * 16]) = b;
  }
  for (int i = tid; i < kTile * 16; i += kBwdThreads) {  // dh: 16 uint4 per row
    const int r = i >> 4, v = i & 15;
    uint4 a = make_uint4(0, 0, 0, 0);
    if (r < nv)
      a = *reinterpret_cast<const uint4*>(dh + static_cast<long long>(r0 + r) * f + cb * kTile +
                                          v * 8);
    *reinterpret_cast<uint4*>(&tdh[r][v * 8]) = a;
  }
  if (tid < kTile) {
    const bool ok = tid < nv;
    sg_s[tid] = ok ? sgu[static_cast<long long>(cb) * R + r0 + tid] : 0.0f;
    su_s[tid] = ok ? sgu[static_cast<long long>(NB + cb) * R + r0 + tid] : 0.0f;
    rmax_g[tid] = 0.0f;
    rmax_u[tid] = 0.0f;
  }
  __syncthreads();

  const int c = tid & (kTile - 1), half = tid >> 7, lane = tid & 31;
  float cm_h = 0.0f, cm_g = 0.0f, cm_u = 0.0f;
  for (int r = half * 64; r < half * 64 + 64; ++r) {
    const SwigluVals v = swiglu_bwd_at(tg[r][c], tu[r][c], sg_s[r], su_s[r],
                                       bf16_bits_to_f32(tdh[r][c]));
    cm_h = fmaxf(cm_h, fabsf(v.h));
    cm_g = fmaxf(cm_g, fabsf(v.dg));
    cm_u = fmaxf(cm_u, fabsf(v.du));
    float mg = fabsf(v.dg), mu = fabsf(v.du);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      mg = fmaxf(mg, __shfl_xor_sync(0xFFFFFFFFu, mg, off));
      mu = fmaxf(mu, __shfl_xor_sync(0xFFFFFFFFu, mu, off));
    }
    if (lane == 0) {
      smem_max(&rmax_g[r], mg);
      smem_max(&rmax_u[r], mu);
    }
  }
  cpart[0][half][c] = cm_h;
  cpart[1][half][c] = cm_g;
  cpart[2][half][c] = cm_u;
  __syncthreads();

  // 128x1 scales of this thread's column, 1x128 scales of every row
  const float s_h = pow2_scale_from_amax(fmaxf(cpart[0][0][c], cpart[0][1][c]));
  const float s_g = pow2_scale_from_amax(fmaxf(cpart[1][0][c], cpart[1][1][c]));
  const float s_u = pow2_scale_from_amax(fmaxf(cpart[2][0][c], cpart[2][1][c]));
  const float rs_h = __frcp_rn(s_h), rs_g = __frcp_rn(s_g), rs_u = __frcp_rn(s_u);
  const int col = cb * kTile + c;
  uint32_t wh[16], wg[16], wu[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) { wh[i] = 0; wg[i] = 0; wu[i] = 0; }
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    const int r = half * 64 + j;
    const SwigluVals v = swiglu_bwd_at(tg[r][c], tu[r][c], sg_s[r], su_s[r],
                                       bf16_bits_to_f32(tdh[r][c]));
    const int sh = 8 * (j & 3);
    wh[j >> 2] |= e4m3_byte(v.h * rs_h) << sh;
    wg[j >> 2] |= e4m3_byte(v.dg * rs_g) << sh;
    wu[j >> 2] |= e4m3_byte(v.du * rs_u) << sh;
    if (r < nv) {   // the rows' 1x128 codes (FP32-scale rule, correctly rounded division)
      const float sgr = e4m3_scale_from_amax(rmax_g[r]);
      const float sur = e4m3_scale_from_amax(rmax_u[r]);
      uint8_t* out = dguq + static_cast<long long>(r0 + r) * 2 * f;
      out[col] = static_cast<uint8_t>(e4m3_byte(__fdiv_rn(v.dg, sgr)));
      out[f + col] = static_cast<uint8_t>(e4m3_byte(__fdiv_rn(v.du, sur)));
    }
  }
  const long long p = static_cast<long long>(blockIdx.x) * kTile + half * 64;
  uint4* dh_t = reinterpret_cast<uint4*>(hT + static_cast<long long>(col) * ldq + p);
  uint4* dg_t = reinterpret_cast<uint4*>(dguT + static_cast<long long>(col) * ldq + p);
  uint4* du_t = reinterpret_cast<uint4*>(dguT + static_cast<long long>(f + col) * ldq + p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    dh_t[i] = make_uint4(wh[4 * i], wh[4 * i + 1], wh[4 * i + 2], wh[4 * i + 3]);
    dg_t[i] = make_uint4(wg[4 * i], wg[4 * i + 1], wg[4 * i + 2], wg[4 * i + 3]);
    du_t[i] = make_uint4(wu[4 * i], wu[4 * i + 1], wu[4 * i + 2], wu[4 * i + 3]);
  }
  if (half == 0) {
    shT[static_cast<long long>(blockIdx.x) * f + col] = s_h;
    sdguT[static_cast<long long>(blockIdx.x) * 2 * f + col] = s_g;
    sdguT[static_cast<long long>(blockIdx.x) * 2 * f + f + col] = s_u;
  }
  if (tid < kTile && tid < nv) {
    sdgu[static_cast<long long>(cb) * R + r0 + tid] = e4m3_scale_from_amax(rmax_g[tid]);
    sdgu[static_cast<long long>(NB + cb) * R + r0 + tid] = e4m3_scale_from_amax(rmax_u[tid]);
  }
}

// ---- host launchers ------------------------------------------------------------------------

int launch_seg_pad(const int32_t* seg, int G, int32_t* pad, int32_t* status, cudaStream_t stream) {
  seg_pad_kernel<<<1, 1024, 0, stream>>>(seg, G, pad, status);
  return check_launch();
}

int launch_transpose_fp8(const uint8_t* src, const float* s, int G, int R, int C, bool interleaved,
                         uint8_t* dst, float* sT, cudaStream_t stream) {
  transpose_kernel<<<dim3(C / 64, R / 64, G), 256, 0, stream>>>(src, R, C, interleaved ? 1 : 0,
                                                                dst);
  int st = check_launch();
  if (st != MOE_OK) return st;
  const long long n = static_cast<long long>(G) * (R / 128) * (C / 128);
  const int blocks = static_cast<int>(min(4096LL, (n + 255) / 256));
  transpose_scales_kernel<<<blocks, 256, 0, stream>>>(s, R / 128, C / 128, G,
                                                      interleaved ? 1 : 0, sT);
  return check_launch();
}

int launch_dispatch_grad(const uint16_t* dy, const float* gate, const int32_t* row_of, int T,
                         int K, int d, int shared_row_base, int n_rows, uint16_t* dy_rows,
                         int32_t* status, cudaStream_t stream) {
  dispatch_grad_kernel<<<T, 256, 0, stream>>>(dy, gate, row_of, K, d, shared_row_base, n_rows,
                                              dy_rows, status);
  return check_launch();
}

int launch_regroup_128x1(const uint16_t* src, int src_rows, const int32_t* rows, int C,
                         const int32_t* seg, const int32_t* pad, int G, int max_blocks, int ldq,
                         uint8_t* qT, float* sT, int32_t* status, cudaStream_t stream) {
  const dim3 grid(max_blocks, C / kTile);
  if (rows)
    regroup_kernel<true><<<grid, kBwdThreads, 0, stream>>>(src, src_rows, rows, C, seg, pad, G,
                                                           ldq, qT, sT, status);
  else
    regroup_kernel<false><<<grid, kBwdThreads, 0, stream>>>(src, src_rows, rows, C, seg, pad, G,
                                                            ldq, qT, sT, status);
  return check_launch();
}

int launch_swiglu_bwd(const uint8_t* guq, const float* sgu, const uint16_t* dh, int R, int f,
                      const int32_t* seg, const int32_t* pad, int G, int max_blocks, int ldq,
                      uint8_t* dguq, float* sdgu, uint8_t* hT, float* shT, uint8_t* dguT,
                      float* sdguT, cudaStream_t stream) {
  constexpr int smem = 2 * kTile * (kTile + 16) + kTile * (kTile + 8) * 2;
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(swiglu_bwd_kernel), smem) != MOE_OK)
    return MOE_ERR_CUDA;
  swiglu_bwd_kernel<<<dim3(max_blocks, f / kTile), kBwdThreads, smem, stream>>>(
      guq, sgu, dh, R, f, seg, pad, G, ldq, dguq, sdgu, hT, shT, dguT, sdguT);
  return check_launch();
}

}  // namespace moe
