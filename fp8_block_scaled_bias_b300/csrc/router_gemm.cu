// Router logits z = x . E^T with FP32 accumulation.
//
// The router is kept above FP8 ("DeepSeek-V3" book, ch. 17 "High-precision
// exceptions", "Router precision has discrete consequences"; "DeepSeek-V3" summary,
// core idea 6).  The FP32 centroids arrive as two BF16 planes hi + lo (16 significant
// bits); x is BF16, so every product hi*x and lo*x is exact in FP32.
//
// This kernel is a CUDA-core tiled GEMM: a 64-token x 64-expert block tile, 4x4 outputs
// per thread, K staged through shared memory 32 at a time.
#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {
constexpr int RT_M = 64, RT_N = 64, RT_K = 32;
}

__global__ void __launch_bounds__(256) router_logits_simt_kernel(
    const uint16_t* __restrict__ x, int T, int d, const uint16_t* __restrict__ w_hilo, int E,
    float* __restrict__ z) {
  __shared__ float xs[RT_K][RT_M + 4];
  __shared__ float ws[RT_K][RT_N + 4];
  const int t0 = blockIdx.y * RT_M, e0 = blockIdx.x * RT_N;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const uint16_t* w_lo = w_hilo + static_cast<long long>(E) * d;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += RT_K) {
    // 64 rows x 32 k for x and for w: 2048 values each, 8 per thread
    for (int i = threadIdx.x; i < RT_M * RT_K; i += 256) {
      const int r = i / RT_K, k = i % RT_K;
      const int t = t0 + r, e = e0 + r;
      xs[k][r] = (t < T) ? bf16_bits_to_f32(x[static_cast<long long>(t) * d + k0 + k]) : 0.0f;
      float wv = 0.0f;
      if (e < E) {
        const long long o = static_cast<long long>(e) * d + k0 + k;
        wv = bf16_bits_to_f32(w_hilo[o]) + bf16_bits_to_f32(w_lo[o]);   // exact
      }
      ws[k][r] = wv;
    }
    __syncthreads();
#pragma unroll 8
    for (int k = 0; k < RT_K; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = xs[k][ty * 4 + i]; b[i] = ws[k][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = __fmaf_rn(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) z[static_cast<long long>(t) * E + e] = acc[i][j];
    }
  }
}

size_t router_logits_ws_bytes(int T, int d, int E) {
  (void)T; (void)d; (void)E;
  return 0;
}

int launch_router_logits(const uint16_t* x, int T, int d, const uint16_t* w_hilo, int E,
                         float* z, void* ws, cudaStream_t stream) {
  (void)ws;
  if (T == 0) return MOE_OK;
  dim3 grid((E + RT_N - 1) / RT_N, (T + RT_M - 1) / RT_M);
  router_logits_simt_kernel<<<grid, 256, 0, stream>>>(x, T, d, w_hilo, E, z);
  return check_launch();
}

__global__ void router_split_kernel(const float* __restrict__ w, long long n,
                                    uint16_t* __restrict__ hilo) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float v = w[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    hilo[i] = *reinterpret_cast<const uint16_t*>(&hi);
    hilo[n + i] = *reinterpret_cast<const uint16_t*>(&lo);
  }
}

int launch_router_split(const float* w, long long n, uint16_t* w_hilo, cudaStream_t stream) {
  if (n == 0) return MOE_OK;
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  router_split_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(w, n, w_hilo);
  return check_launch();
}

}  // namespace moe
