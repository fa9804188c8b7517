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
#include <cuda_fp16.h>

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

// Four E4M3 codes (bytes of q, lowest first) -> their exact values (hardware conversion to
// FP16, which holds every E4M3 value exactly).
MOE_DEV void e4m3x4_decode(uint32_t q, float (&v)[4]) {
  uint32_t lo, hi;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"(static_cast<uint16_t>(q & 0xFFFFu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"(static_cast<uint16_t>(q >> 16)));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}

// From the decoded g, u codes and their 1x128 scales: g and u (fl32(dec * s)), the sigmoid
// with expf and IEEE division, h, dG, dU.  (The fast exponential and division move enough
// dG, dU codes across E4M3 boundaries to cost the gate/up Dgrad its 2e-2 bound.)
MOE_DEV SwigluVals swiglu_bwd_at(float dg_code, float du_code, float sg, float su, float dh) {
  const float g = __fmul_rn(dg_code, sg);
  const float u = __fmul_rn(du_code, su);
  const float sig = __fdiv_rn(1.0f, 1.0f + expf(-g));
  const float silu = g * sig;
  SwigluVals v;
  v.h = silu * u;
  v.du = dh * silu;
  v.dg = dh * u * sig * fmaf(g, 1.0f - sig, 1.0f);
  return v;
}

}  // namespace

// One tile is (rb, cb): the segment rows of padded block rb, hidden columns
// [128 cb, 128 cb + 128).  512 threads; warp w owns rows 8 w .. 8 w + 7, lane l columns
// 4 l .. 4 l + 3, so every value is computed once and kept in registers: the rows' 1x128
// max-abs of dG and dU come from a warp reduction per row, the columns' 128x1 max-abs of
// h, dG and dU from a shared-memory reduction over the 16 warps.  The row-major stores
// are coalesced; the transposed codes go out as 8 contiguous bytes per column and thread.
//
// The kernel is persistent (one block per SM, the register file holds one tile's values)
// and streams its tiles through two shared-memory input buffers: the next tile's g, u, dh
// rows and scales are copied in with cp.async while the current one is computed, so the
// loads of a whole tile are in flight together instead of one row of them at a time.
constexpr int kSwThreads = 512;

struct SwTile {                          // one tile's inputs; rows past the segment are 0
  uint8_t g[kTile * kTile];              // gate codes [row][column]
  uint8_t u[kTile * kTile];              // up codes
  uint16_t dh[kTile * kTile];            // dh (BF16)
  float sg[kTile], su[kTile];            // the rows' 1x128 scales of g and u
};
constexpr int kSwSmem = 2 * static_cast<int>(sizeof(SwTile));

namespace {
// 16- and 4-byte asynchronous copies; a copy with valid == false reads nothing and writes
// zeros (the source operand is then only a placeholder inside the tensor).
MOE_DEV void cp_async_16z(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
MOE_DEV void cp_async_4z(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}
}  // namespace

__global__ void __launch_bounds__(kSwThreads, 1) swiglu_bwd_kernel(
    const uint8_t* __restrict__ guq, const float* __restrict__ sgu,
    const uint16_t* __restrict__ dh, int R, int f, const int32_t* __restrict__ seg,
    const int32_t* __restrict__ pad, int G, int ldq, uint8_t* __restrict__ dguq,
    float* __restrict__ sdgu, uint8_t* __restrict__ hT, float* __restrict__ shT,
    uint8_t* __restrict__ dguT, float* __restrict__ sdguT) {
  extern __shared__ __align__(16) uint8_t sw_smem[];
  __shared__ float cpart[16][3][kTile];          // per-warp column max: h, dG, dU
  __shared__ float cscale[3][kTile];             // the columns' power-of-two scales
  SwTile* const buf = reinterpret_cast<SwTile*>(sw_smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NB = f / kTile;
  const int ntiles = pad[G] / kTile * NB;

  // tile t -> (padded row block rb, column block cb, segment rows r0 .. r0 + nv - 1)
  auto tile_of = [&](int t, int& rb, int& cb, int& r0, int& nv) {
    rb = t / NB;
    cb = t - rb * NB;
    int e;
    block_of(seg, pad, G, rb, e, r0, nv);
  };
  auto load_tile = [&](SwTile* in, int r0, int nv, int cb) {
    for (int i = threadIdx.x; i < kTile * 8; i += kSwThreads) {      // g and u: 8 x 16 B a row
      const int r = i >> 3, c = i & 7;
      const bool v = r < nv;
      const uint8_t* src = v ? guq + static_cast<long long>(r0 + r) * 2 * f + cb * kTile + c * 16
                             : guq;
      cp_async_16z(smem_u32(in->g + r * kTile + c * 16), src, v);
      cp_async_16z(smem_u32(in->u + r * kTile + c * 16), v ? src + f : guq, v);
    }
    for (int i = threadIdx.x; i < kTile * 16; i += kSwThreads) {     // dh: 16 x 16 B a row
      const int r = i >> 4, c = i & 15;
      const bool v = r < nv;
      const uint16_t* src = v ? dh + static_cast<long long>(r0 + r) * f + cb * kTile + c * 8 : dh;
      cp_async_16z(smem_u32(in->dh + r * kTile + c * 8), src, v);
    }
    if (threadIdx.x < 2 * kTile) {
      const int r = threadIdx.x & (kTile - 1), which = threadIdx.x >> 7;
      const bool v = r < nv;
      const float* src = v ? sgu + static_cast<long long>(which ? NB + cb : cb) * R + r0 + r : sgu;
      cp_async_4z(smem_u32((which ? in->su : in->sg) + r), src, v);
    }
  };

  int t = blockIdx.x;
  if (t < ntiles) {
    int rb, cb, r0, nv;
    tile_of(t, rb, cb, r0, nv);
    load_tile(buf, r0, nv, cb);
  }
  cp_async_commit();
  for (int i = 0; t < ntiles; t += gridDim.x, ++i) {
    const int tn = t + static_cast<int>(gridDim.x);
    if (tn < ntiles) {                          // the next tile's inputs, into the other buffer
      int rb, cb, r0, nv;
      tile_of(tn, rb, cb, r0, nv);
      load_tile(buf + ((i + 1) & 1), r0, nv, cb);
    }
    cp_async_commit();                          // one group per iteration (possibly empty)
    cp_async_wait<1>();                         // this tile's group has landed
    __syncthreads();
    const SwTile* in = buf + (i & 1);
    int rb, cb, r0, nv;
    tile_of(t, rb, cb, r0, nv);
    const int c0 = cb * kTile + 4 * lane;         // this lane's first hidden column
    float hv[8][4], gv[8][4], uv[8][4];           // h, dG, dU of the warp's 8 rows
    float cm[3][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float rs_g[8], rs_u[8];                       // the rows' 1x128 scales
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int r = 8 * warp + k;
      const uint32_t qg = *reinterpret_cast<const uint32_t*>(in->g + r * kTile + 4 * lane);
      const uint32_t qu = *reinterpret_cast<const uint32_t*>(in->u + r * kTile + 4 * lane);
      const uint2 d2 = *reinterpret_cast<const uint2*>(in->dh + r * kTile + 4 * lane);
      const float sg = in->sg[r], su = in->su[r];
      float cg[4], cu[4];
      e4m3x4_decode(qg, cg);
      e4m3x4_decode(qu, cu);
      const float dhv[4] = {bf16_bits_to_f32(static_cast<uint16_t>(d2.x & 0xFFFFu)),
                            bf16_bits_to_f32(static_cast<uint16_t>(d2.x >> 16)),
                            bf16_bits_to_f32(static_cast<uint16_t>(d2.y & 0xFFFFu)),
                            bf16_bits_to_f32(static_cast<uint16_t>(d2.y >> 16))};
      float mg = 0.0f, mu = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const SwigluVals v = swiglu_bwd_at(cg[j], cu[j], sg, su, dhv[j]);
        hv[k][j] = v.h;
        gv[k][j] = v.dg;
        uv[k][j] = v.du;
        mg = fmaxf(mg, fabsf(v.dg));
        mu = fmaxf(mu, fabsf(v.du));
        cm[0][j] = fmaxf(cm[0][j], fabsf(v.h));
        cm[1][j] = fmaxf(cm[1][j], fabsf(v.dg));
        cm[2][j] = fmaxf(cm[2][j], fabsf(v.du));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        mg = fmaxf(mg, __shfl_xor_sync(0xFFFFFFFFu, mg, off));
        mu = fmaxf(mu, __shfl_xor_sync(0xFFFFFFFFu, mu, off));
      }
      const float s_g = e4m3_scale_from_amax(mg), s_u = e4m3_scale_from_amax(mu);
      rs_g[k] = s_g;
      rs_u[k] = s_u;
      if (lane == 0 && r < nv) {
        sdgu[static_cast<long long>(cb) * R + r0 + r] = s_g;
        sdgu[static_cast<long long>(NB + cb) * R + r0 + r] = s_u;
      }
    }
#pragma unroll
    for (int k = 0; k < 3; ++k)
#pragma unroll
      for (int j = 0; j < 4; ++j) cpart[warp][k][4 * lane + j] = cm[k][j];
    __syncthreads();
    if (threadIdx.x < 3 * kTile) {
      const int k = threadIdx.x / kTile, c = threadIdx.x % kTile;
      float m = 0.0f;
#pragma unroll
      for (int w = 0; w < 16; ++w) m = fmaxf(m, cpart[w][k][c]);
      const float sc = pow2_scale_from_amax(m);
      cscale[k][c] = sc;
      float* dst = k == 0 ? shT + static_cast<long long>(rb) * f
                          : sdguT + static_cast<long long>(rb) * 2 * f + (k - 1) * f;
      dst[cb * kTile + c] = sc;
    }
    __syncthreads();
    // row-major 1x128 codes of dG and dU (correctly rounded division, the quantiser's rule)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int r = 8 * warp + k;
      if (r < nv) {
        uint32_t wg = 0, wu = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          wg |= e4m3_byte(__fdiv_rn(gv[k][j], rs_g[k])) << (8 * j);
          wu |= e4m3_byte(__fdiv_rn(uv[k][j], rs_u[k])) << (8 * j);
        }
        uint8_t* out = dguq + static_cast<long long>(r0 + r) * 2 * f;
        *reinterpret_cast<uint32_t*>(out + c0) = wg;
        *reinterpret_cast<uint32_t*>(out + f + c0) = wu;
      }
    }
    // transposed 128x1 codes: 8 rows (bytes) per column and thread; padded rows are 0
    const long long pcol = static_cast<long long>(rb) * kTile + 8 * warp;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = c0 + j;
      const float rh = __frcp_rn(cscale[0][4 * lane + j]);    // exact: powers of two
      const float rg = __frcp_rn(cscale[1][4 * lane + j]);
      const float ru = __frcp_rn(cscale[2][4 * lane + j]);
      uint32_t h0 = 0, h1 = 0, g0 = 0, g1 = 0, u0 = 0, u1 = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        h0 |= e4m3_byte(hv[k][j] * rh) << (8 * k);
        h1 |= e4m3_byte(hv[k + 4][j] * rh) << (8 * k);
        g0 |= e4m3_byte(gv[k][j] * rg) << (8 * k);
        g1 |= e4m3_byte(gv[k + 4][j] * rg) << (8 * k);
        u0 |= e4m3_byte(uv[k][j] * ru) << (8 * k);
        u1 |= e4m3_byte(uv[k + 4][j] * ru) << (8 * k);
      }
      *reinterpret_cast<uint2*>(hT + static_cast<long long>(col) * ldq + pcol) = make_uint2(h0, h1);
      *reinterpret_cast<uint2*>(dguT + static_cast<long long>(col) * ldq + pcol) = make_uint2(g0, g1);
      *reinterpret_cast<uint2*>(dguT + static_cast<long long>(f + col) * ldq + pcol) =
          make_uint2(u0, u1);
    }
    __syncthreads();                            // cscale and this input buffer are reused
  }
  cp_async_wait<0>();
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
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(swiglu_bwd_kernel), kSwSmem) != MOE_OK)
    return MOE_ERR_CUDA;
  // persistent: one block per SM (or per tile when there are fewer), tiles counted on the
  // device from the padded offsets
  long long grid = static_cast<long long>(max_blocks) * (f / kTile);
  if (grid > num_sms()) grid = num_sms();
  if (grid < 1) grid = 1;
  swiglu_bwd_kernel<<<static_cast<unsigned>(grid), kSwThreads, kSwSmem, stream>>>(
      guq, sgu, dh, R, f, seg, pad, G, ldq, dguq, sdgu, hT, shT, dguT, sdguT);
  return check_launch();
}

}  // namespace moe
