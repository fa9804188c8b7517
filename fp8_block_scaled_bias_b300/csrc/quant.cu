// Online FP8 quantisation: BF16 activations in 1x128 tiles (fp8_quant_1x128) and FP32
// weights in 128x128 blocks (fp8_quant_128x128, setup only).
//
// The scale of a group is its max-abs divided by the E4M3 maximum 448, so the largest
// element lands on +-448 ("DeepSeek-V3" summary, core idea 6(a) fine-grained tiles and
// 6(d) online scaling; "DeepSeek-V3" book, ch. 16 "V3's grouping", "Online scales",
// "Scaling a group").  Quantised values are E4M3 round-to-nearest-even with saturation.
#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {
template <bool POW2>
MOE_DEV float scale_rule(float amax) {
  return POW2 ? pow2_scale_from_amax(amax) : e4m3_scale_from_amax(amax);
}
}  // namespace

// Half a warp per 1x128 tile: 16 lanes x 8 BF16 values.  Tiles are numbered with the
// column block fastest so a warp reads 512 contiguous bytes of one row.
template <bool POW2>
__global__ void __launch_bounds__(256) quant_1x128_kernel(const uint16_t* __restrict__ x,
                                                           int rows, int ncb, int ldx,
                                                           uint8_t* __restrict__ q,
                                                           float* __restrict__ scale,
                                                           long long ntiles) {
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4;
  const int hl = lane & 15;
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const long long cols = static_cast<long long>(ncb) * 128;
  for (long long p = warp; 2 * p < ntiles; p += nwarps) {
    const long long t = 2 * p + half;
    const bool valid = t < ntiles;
    const long long r = valid ? t / ncb : 0;
    const int cb = valid ? static_cast<int>(t % ncb) : 0;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (valid)
      v = __ldcs(reinterpret_cast<const uint4*>(x + r * ldx + cb * 128 + hl * 8));
    float f[8];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
    for (int off = 8; off > 0; off >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    const float s = scale_rule<POW2>(amax);
    uint32_t out[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t a = f32x2_to_e4m3x2(__fdiv_rn(f[4 * i], s), __fdiv_rn(f[4 * i + 1], s));
      const uint32_t b = f32x2_to_e4m3x2(__fdiv_rn(f[4 * i + 2], s), __fdiv_rn(f[4 * i + 3], s));
      out[i] = a | (b << 16);
    }
    if (valid) {
      *reinterpret_cast<uint2*>(q + r * cols + cb * 128 + hl * 8) = make_uint2(out[0], out[1]);
      if (hl == 0) scale[static_cast<long long>(cb) * rows + r] = s;
    }
  }
}

// Quantise-and-dispatch: each token's row of x is quantised 1x128 once and written to
// every row that uses it -- its K routed rows row_of[t][k] and, when shared_row_base >=
// 0, its shared-expert row shared_row_base + t -- of the permuted activation matrix (the
// pages quantise activations before dispatch, "DeepSeek-V3" book, ch. 17 "FP8 dispatch,
// BF16 combine").  Bit for bit the same as quant_1x128_kernel followed by a row gather
// with the inverse map: the same per-tile arithmetic, written to more places.
// One block per token (grid-stride); eight lanes per 1x128 tile, 16 values each, so every
// destination row gets 16-byte stores; the token's K destination rows are loaded once
// (one per lane) and passed around with shuffles.
template <bool POW2>
__global__ void __launch_bounds__(512) quant_scatter_1x128_kernel(
    const uint16_t* __restrict__ x, int T, int ldx, int ncb, const int32_t* __restrict__ row_of,
    int K, int shared_row_base, int n_rows, uint8_t* __restrict__ q, float* __restrict__ scale,
    int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int slot = threadIdx.x >> 3;          // tile slot of this block iteration
  const int el = threadIdx.x & 7;             // 16 values of the tile
  const int slots = blockDim.x >> 3;
  const long long cols = static_cast<long long>(ncb) * 128;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const int my_row = lane < K ? row_of[static_cast<long long>(t) * K + lane] : 0;
    for (int cb0 = 0; cb0 < ncb; cb0 += slots) {  // same trip count in every warp
      const int cb = cb0 + slot;
      const bool valid = cb < ncb;
      uint4 v[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
      if (valid) {
        const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<long long>(t) * ldx +
                                                          cb * 128 + el * 16);
        v[0] = __ldcs(src);
        v[1] = __ldcs(src + 1);
      }
      float f[16];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t w[4] = {v[h].x, v[h].y, v[h].z, v[h].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          f[8 * h + 2 * i] = __uint_as_float(w[i] << 16);
          f[8 * h + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
      }
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
      for (int off = 4; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
      const float s = scale_rule<POW2>(amax);
      uint32_t out[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t a = f32x2_to_e4m3x2(__fdiv_rn(f[4 * i], s), __fdiv_rn(f[4 * i + 1], s));
        const uint32_t b = f32x2_to_e4m3x2(__fdiv_rn(f[4 * i + 2], s), __fdiv_rn(f[4 * i + 3], s));
        out[i] = a | (b << 16);
      }
      const uint4 o = make_uint4(out[0], out[1], out[2], out[3]);
      for (int k = 0; k <= K; ++k) {
        int r;
        if (k < K) r = __shfl_sync(0xFFFFFFFFu, my_row, k);
        else if (shared_row_base >= 0) r = shared_row_base + t;
        else break;
        if (!valid) continue;
        if (r < 0 || r >= n_rows) {
          if (el == 0 && cb == 0) set_status(status, MOE_ERR_DEVICE_DATA);
          continue;
        }
        *reinterpret_cast<uint4*>(q + r * cols + cb * 128 + el * 16) = o;
        if (el == 0) scale[static_cast<long long>(cb) * n_rows + r] = s;
      }
    }
  }
}

int launch_quant_scatter_1x128(const uint16_t* x, int T, int cols, int ldx, const int32_t* row_of,
                               int K, int shared_row_base, int n_rows, uint8_t* q, float* scale,
                               bool pow2, int32_t* status, cudaStream_t stream) {
  if (T == 0 || cols == 0) return MOE_OK;
  // One block per token (the hardware block scheduler balances the tail; a grid-stride
  // loop over a resident grid left a quarter of the SMs idle in the last round: 0.71 vs
  // 0.64 of the copy rate at V3 shapes).  Tile slots per pass: an even split of the row's
  // tiles into <= 64 per pass (d = 7168: 56 slots, 448 threads, one pass).
  const int ncb = cols / 128;
  const int passes = (ncb + 63) / 64;
  const int slots = (ncb + passes - 1) / passes;
  const int threads = (slots * 8 + 31) / 32 * 32;
  const int blocks = T;
  if (pow2)
    quant_scatter_1x128_kernel<true><<<blocks, threads, 0, stream>>>(
        x, T, ldx, ncb, row_of, K, shared_row_base, n_rows, q, scale, status);
  else
    quant_scatter_1x128_kernel<false><<<blocks, threads, 0, stream>>>(
        x, T, ldx, ncb, row_of, K, shared_row_base, n_rows, q, scale, status);
  return check_launch();
}

// One block per 128x128 weight block; thread t covers row t/2, 64 columns.
template <bool POW2>
__global__ void __launch_bounds__(256) quant_128x128_kernel(const float* __restrict__ w,
                                                             int rows, int cols,
                                                             uint8_t* __restrict__ q,
                                                             float* __restrict__ scale) {
  const int rb = blockIdx.y, cb = blockIdx.x;
  const int r = rb * 128 + (threadIdx.x >> 1);
  const int c0 = cb * 128 + (threadIdx.x & 1) * 64;
  const float* src = w + static_cast<long long>(r) * cols + c0;
  float amax = 0.0f;
  for (int i = 0; i < 64; i += 4) {
    const float4 v = *reinterpret_cast<const float4*>(src + i);
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  __shared__ float wmax[8];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = wmax[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, wmax[i]);
  const float s = scale_rule<POW2>(amax);
  uint8_t* dst = q + static_cast<long long>(r) * cols + c0;
  for (int i = 0; i < 64; i += 4) {
    const float4 v = *reinterpret_cast<const float4*>(src + i);
    const uint32_t a = f32x2_to_e4m3x2(__fdiv_rn(v.x, s), __fdiv_rn(v.y, s));
    const uint32_t b = f32x2_to_e4m3x2(__fdiv_rn(v.z, s), __fdiv_rn(v.w, s));
    *reinterpret_cast<uint32_t*>(dst + i) = a | (b << 16);
  }
  if (threadIdx.x == 0) scale[static_cast<long long>(rb) * (cols / 128) + cb] = s;
}

int launch_quant_1x128(const uint16_t* x, int rows, int cols, int ldx, uint8_t* q,
                       float* scale, bool pow2, cudaStream_t stream) {
  const long long ntiles = static_cast<long long>(rows) * (cols / 128);
  if (ntiles == 0) return MOE_OK;
  const long long pairs = (ntiles + 1) / 2;
  long long blocks = (pairs + 7) / 8;                 // 8 warps per block
  const long long cap = static_cast<long long>(num_sms()) * 16;
  if (blocks > cap) blocks = cap;
  if (pow2)
    quant_1x128_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        x, rows, cols / 128, ldx, q, scale, ntiles);
  else
    quant_1x128_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        x, rows, cols / 128, ldx, q, scale, ntiles);
  return check_launch();
}

int launch_quant_128x128(const float* w, int rows, int cols, uint8_t* q, float* scale,
                         bool pow2, cudaStream_t stream) {
  if (rows == 0 || cols == 0) return MOE_OK;
  dim3 grid(cols / 128, rows / 128);
  if (pow2)
    quant_128x128_kernel<true><<<grid, 256, 0, stream>>>(w, rows, cols, q, scale);
  else
    quant_128x128_kernel<false><<<grid, 256, 0, stream>>>(w, rows, cols, q, scale);
  return check_launch();
}

}  // namespace moe
