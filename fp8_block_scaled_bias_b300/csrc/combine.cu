// Row movement around the expert GEMMs:
//   moe_combine  -- gate-weighted sum of each token's expert outputs plus the shared
//                   expert, BF16 in and out, FP32 accumulation in a fixed order
//                   ("DeepSeek-V3" book, ch. 7 "Selecting and combining experts";
//                   ch. 15 "What combine must do"; ch. 17 "FP8 dispatch, BF16 combine").
//   gather       -- copy FP8 rows (and their 1x128 scales) into expert-segment order
//                   before the grouped GEMM ("DeepSeek-V3" book, ch. 15: the receiver
//                   groups rows by expert).
#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {
constexpr int kCombineThreads = 128;
constexpr int kMaxK = 32;
}  // namespace

// One block per token (SLICED: per token and column slice, blockIdx.y); each thread owns
// 8 consecutive columns at a time.
template <bool SLICED>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    const uint16_t* __restrict__ y_rows, int n_rows, const int32_t* __restrict__ row_of,
    const float* __restrict__ gate, int K, int d, int shared_row_base,
    uint16_t* __restrict__ y, int32_t* status) {
  __shared__ long long rows[kMaxK + 1];
  __shared__ float g[kMaxK];
  __shared__ int bad;
  const int t = blockIdx.x;
  if (threadIdx.x == 0) bad = 0;
  __syncthreads();
  if (threadIdx.x < K) {
    const int r = row_of[static_cast<long long>(t) * K + threadIdx.x];
    if (r < 0 || r >= n_rows) { bad = 1; set_status(status, MOE_ERR_DEVICE_DATA); }
    rows[threadIdx.x] = static_cast<long long>(r) * d;
    g[threadIdx.x] = gate[static_cast<long long>(t) * K + threadIdx.x];
  }
  if (threadIdx.x == 0 && shared_row_base >= 0) {
    const long long r = static_cast<long long>(shared_row_base) + t;
    if (r >= n_rows) { bad = 1; set_status(status, MOE_ERR_DEVICE_DATA); }
    rows[kMaxK] = r * d;
  }
  __syncthreads();
  if (bad) return;
  const int nv = d / 8;
  const int v0 = SLICED ? static_cast<int>(blockIdx.y * blockDim.x + threadIdx.x)
                        : static_cast<int>(threadIdx.x);
  const int vstep = SLICED ? static_cast<int>(gridDim.y * blockDim.x) : static_cast<int>(blockDim.x);
  for (int v = v0; v < nv; v += vstep) {
    float acc[8];
    if (shared_row_base >= 0) {
      const uint4 u = __ldcs(reinterpret_cast<const uint4*>(y_rows + rows[kMaxK]) + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __uint_as_float(w[i] << 16);
        acc[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    }
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
      const uint4 u = __ldcs(reinterpret_cast<const uint4*>(y_rows + rows[k]) + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      const float gk = g[k];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] = __fmaf_rn(gk, __uint_as_float(w[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = __fmaf_rn(gk, __uint_as_float(w[i] & 0xFFFF0000u), acc[2 * i + 1]);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    reinterpret_cast<uint4*>(y + static_cast<long long>(t) * d)[v] = o;
  }
}

int launch_combine(const uint16_t* y_rows, int n_rows, const int32_t* row_of,
                   const float* gate, int T, int K, int d, int shared_row_base, uint16_t* y,
                   int32_t* status, cudaStream_t stream) {
  if (T == 0) return MOE_OK;
  // Decode-sized batches: a token's row is split over several blocks (up to one 8-column
  // vector per thread) until the grid fills the SMs, so a thread's K + 1 row loads are
  // most of the latency (T = 128: 25 -> 12 us).  Large batches keep one block per token.
  const int max_slices = (d / 8 + kCombineThreads - 1) / kCombineThreads;
  const long long want = (static_cast<long long>(num_sms()) * 16 + T - 1) / T;
  const int slices = static_cast<int>(want < 1 ? 1 : (want > max_slices ? max_slices : want));
  if (slices > 1)
    combine_kernel<true><<<dim3(T, slices), kCombineThreads, 0, stream>>>(
        y_rows, n_rows, row_of, gate, K, d, shared_row_base, y, status);
  else
    combine_kernel<false><<<T, kCombineThreads, 0, stream>>>(y_rows, n_rows, row_of, gate, K, d,
                                                            shared_row_base, y, status);
  return check_launch();
}

// One warp per destination row: 16-byte copies of the FP8 row, then its scales.
__global__ void __launch_bounds__(256) gather_rows_fp8_kernel(
    const uint8_t* __restrict__ src, const float* __restrict__ src_scale, int src_rows,
    const int32_t* __restrict__ rows, const int32_t* __restrict__ row_limit, int n_rows,
    int cols, uint8_t* __restrict__ dst, float* __restrict__ dst_scale, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int limit = row_limit ? min(*row_limit, n_rows) : n_rows;
  const int nv = cols / 16;
  const int ncb = cols / 128;
  for (long long r = warp; r < limit; r += nwarps) {
    const int s = rows[r];
    if (s < 0 || s >= src_rows) {
      if (lane == 0) set_status(status, MOE_ERR_DEVICE_DATA);
      continue;
    }
    const uint4* in = reinterpret_cast<const uint4*>(src + static_cast<long long>(s) * cols);
    uint4* out = reinterpret_cast<uint4*>(dst + r * cols);
    for (int v = lane; v < nv; v += 32) out[v] = __ldg(in + v);
    for (int cb = lane; cb < ncb; cb += 32)
      dst_scale[static_cast<long long>(cb) * n_rows + r] =
          __ldg(src_scale + static_cast<long long>(cb) * src_rows + s);
  }
}

int launch_gather_rows_fp8(const uint8_t* src, const float* src_scale, int src_rows,
                           const int32_t* rows, const int32_t* row_limit, int n_rows, int cols,
                           uint8_t* dst, float* dst_scale, int32_t* status,
                           cudaStream_t stream) {
  if (n_rows == 0) return MOE_OK;
  long long blocks = (static_cast<long long>(n_rows) + 7) / 8;
  const long long cap = static_cast<long long>(num_sms()) * 16;
  if (blocks > cap) blocks = cap;
  gather_rows_fp8_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      src, src_scale, src_rows, rows, row_limit, n_rows, cols, dst, dst_scale, status);
  return check_launch();
}

}  // namespace moe
