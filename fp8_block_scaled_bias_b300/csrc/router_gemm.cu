// Router logits z = x . E^T with FP32 accumulation, on tcgen05 BF16 tensor cores.
//
// The router is kept above FP8 ("DeepSeek-V3" book, ch. 17 "High-precision
// exceptions", "Router precision has discrete consequences"; "DeepSeek-V3" summary,
// core idea 6).  The FP32 centroids arrive as two BF16 planes hi + lo (16 significant
// bits); x is BF16, so every product hi*x and lo*x is exact and both planes accumulate
// into one FP32 TMEM accumulator: z = sum_k x_k hi_k + x_k lo_k.
//
// One CTA per 128-token x BN-expert tile (BN = min(64, E)) and K range, with a 6-stage TMA
// pipeline (x tile 128x64 BF16, hi and lo tiles BNx64).  When there are fewer tiles than
// SMs (decode batches: T = 128 gives 4 tiles) the K loop is split across CTAs
// (blockIdx.z) into FP32 partial tiles in the workspace, summed afterwards in split order
// by a second kernel, so the result does not depend on timing.
//   warp 0      TMA producer
//   warp 1      TMEM allocation; one thread issues 8 MMAs (M128 N=BN K16) per 64-deep
//               K block: 4 K steps on the hi plane and 4 on the lo plane
//   warps 2..5  epilogue: TMEM -> registers -> z (FP32)
#include <cuda.h>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace rk {
constexpr int BM = 128, BK = 64;                  // BK in BF16 elements = 128 bytes
constexpr int MAX_BN = 64;
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;              // 16 KB
constexpr int B_BYTES = MAX_BN * BK * 2;          // 8 KB per plane
constexpr int STAGE_BYTES = A_BYTES + 2 * B_BYTES;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 64;
constexpr int OFF_BAR = STAGES * STAGE_BYTES;
constexpr int OFF_MISC = OFF_BAR + (2 * STAGES + 2) * 8;
constexpr int SMEM_ALLOC = OFF_MISC + 16 + 1024;
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
}  // namespace rk

struct RouterParams {
  float* z;
  int T, d, E, BN;
  int32_t* status;
  float* part;           // split K: [splits][T][E] partial sums (else NULL: write z)
  int kb_per;            // K blocks per split
};

__global__ void __launch_bounds__(rk::THREADS, 1)
    router_logits_kernel(const __grid_constant__ CUtensorMap tmX,
                         const __grid_constant__ CUtensorMap tmW, const RouterParams p) {
  using namespace rk;
  extern __shared__ uint8_t router_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(router_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t acc_bar = bar0 + 8u * (2 * STAGES);
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BN = p.BN;
  const int m0 = blockIdx.y * BM;
  const int n0 = blockIdx.x * BN;
  const int kb0 = static_cast<int>(blockIdx.z) * p.kb_per;   // this CTA's K range
  const int KB = min(p.d / BK - kb0, p.kb_per);
  const uint32_t stage_tx = A_BYTES + 2u * BN * BK * 2;
  float* const out = p.part ? p.part + static_cast<long long>(blockIdx.z) * p.T * p.E : p.z;

  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) { mbar_init(full_bar(s), 1); mbar_init(empty_bar(s), 1); }
    mbar_init(acc_bar, 1);
    mbar_init(drain_bar, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      int kb = 0;
      for (; kb < KB; ++kb) {
        const int s = kb % STAGES;
        const uint32_t ph = (kb / STAGES) & 1;
        if (!mbar_wait(empty_bar(s), ph ^ 1, abort_flag, p.status)) { ok = false; break; }
        const uint32_t st = sbase + s * STAGE_BYTES;
        mbar_arrive_expect_tx(full_bar(s), stage_tx);
        const int kx = (kb0 + kb) * BK;
        tma_load_2d(st, &tmX, kx, m0, full_bar(s));
        tma_load_2d(st + A_BYTES, &tmW, kx, n0, full_bar(s));              // hi plane
        tma_load_2d(st + A_BYTES + B_BYTES, &tmW, kx, p.E + n0, full_bar(s));  // lo plane
      }
      if (!ok) {
        const int first = kb > STAGES ? kb - STAGES : 0;
        for (int i = first; i < kb; ++i) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(full_bar(i % STAGES), (i / STAGES) & 1))
            if (globaltimer_ns() - t0 > kWaitLimitNs) break;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = make_idesc(BM, BN, 1u, 1u);     // BF16 x BF16 -> F32
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % STAGES;
        const uint32_t ph = (kb / STAGES) & 1;
        if (!mbar_wait(full_bar(s), ph, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t st = sbase + s * STAGE_BYTES;
        const uint64_t adesc = smem_desc_sw128(st);
        const uint64_t hdesc = smem_desc_sw128(st + A_BYTES);
        const uint64_t ldesc = smem_desc_sw128(st + A_BYTES + B_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {       // 16 BF16 = 32 bytes per MMA: +2 encoded
          mma_bf16(tmem_base, adesc + 2 * k, hdesc + 2 * k, idesc, (kb | k) ? 1u : 0u);
          mma_bf16(tmem_base, adesc + 2 * k, ldesc + 2 * k, idesc, 1u);
        }
        mma_commit(empty_bar(s));
      }
      mma_commit(acc_bar);
      mma_commit(drain_bar);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain_bar, 0))
        if (globaltimer_ns() - t0 > kWaitLimitNs) break;
    }
  } else {
    const int q = warp & 3;
    const int row = q * 32 + lane;
    if (mbar_wait(acc_bar, 0, abort_flag, p.status)) {
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const int t = m0 + row;
      for (int c = 0; c < BN; c += 32) {
        uint32_t v[32];
        if (BN - c >= 32) {
          tmem_ld_32x32b_x32(tb + c, v);
          tmem_ld_wait();
          if (t < p.T) {
            float4* dst = reinterpret_cast<float4*>(out + static_cast<long long>(t) * p.E + n0 + c);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                   __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          }
        } else {
          // 16-column tail (BN = 16 or 48): load 32 columns, keep 16
          tmem_ld_32x32b_x32(tb + c, v);     // columns c..c+31 lie inside the 64 allocated
          tmem_ld_wait();
          if (t < p.T) {
            float4* dst = reinterpret_cast<float4*>(out + static_cast<long long>(t) * p.E + n0 + c);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                   __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* ptr,
                    uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                    uint32_t box_outer);   // runtime.cu

namespace {
// widest multiple of 16 <= 64 dividing E
int router_bn(int E) {
  for (int b = rk::MAX_BN; b >= 16; b -= 16)
    if (E % b == 0) return b;
  return 16;
}

// K splits for T tokens: enough CTAs to cover the SMs, at least 4 K blocks per split.
// Returns the number of splits (1: no split) and the K blocks per split.
int router_splits(int T, int d, int E, int* kb_per) {
  const int KB = d / rk::BK;
  const long long tiles = static_cast<long long>(E / router_bn(E)) * ((T + rk::BM - 1) / rk::BM);
  long long S = tiles > 0 ? num_sms() / tiles : 1;
  if (S > KB / 4) S = KB / 4;
  if (S < 2) { *kb_per = KB; return 1; }
  const int per = static_cast<int>((KB + S - 1) / S);
  *kb_per = per;
  return (KB + per - 1) / per;
}

// z = sum of the split partials, added in split order
__global__ void router_reduce_kernel(const float4* __restrict__ part, int S, long long n4,
                                     float4* __restrict__ z) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    float4 a = part[i];
    for (int s = 1; s < S; ++s) {
      const float4 b = part[static_cast<long long>(s) * n4 + i];
      a.x = __fadd_rn(a.x, b.x);
      a.y = __fadd_rn(a.y, b.y);
      a.z = __fadd_rn(a.z, b.z);
      a.w = __fadd_rn(a.w, b.w);
    }
    z[i] = a;
  }
}
}  // namespace

size_t router_logits_ws_bytes(int T, int d, int E) {
  if (T <= 0 || d <= 0 || E <= 0) return 0;
  int per = 0;
  const int S = router_splits(T, d, E, &per);
  return S > 1 ? static_cast<size_t>(S) * T * E * sizeof(float) : 0;
}

int launch_router_logits(const uint16_t* x, int T, int d, const uint16_t* w_hilo, int E,
                         float* z, int32_t* status, void* ws, cudaStream_t stream) {
  using namespace rk;
  if (T == 0) return MOE_OK;
  const int BN = router_bn(E);
  if (E % BN != 0) return MOE_ERR_UNSUPPORTED;
  int kb_per = 0;
  const int S = router_splits(T, d, E, &kb_per);
  if (S > 1 && !ws) return MOE_ERR_WORKSPACE;
  CUtensorMap tmX, tmW;
  if (!encode_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, d, T, 2ull * d, BK, BM))
    return MOE_ERR_CUDA;
  if (!encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, w_hilo, d, 2ull * E, 2ull * d, BK,
                      BN))
    return MOE_ERR_CUDA;
  RouterParams p{z, T, d, E, BN, status, S > 1 ? static_cast<float*>(ws) : nullptr, kb_per};
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(router_logits_kernel), SMEM_ALLOC) !=
      MOE_OK)
    return MOE_ERR_CUDA;
  dim3 grid(E / BN, (T + BM - 1) / BM, S);
  router_logits_kernel<<<grid, THREADS, SMEM_ALLOC, stream>>>(tmX, tmW, p);
  if (S > 1) {
    const int st = check_launch();
    if (st != MOE_OK) return st;
    const long long n4 = static_cast<long long>(T) * E / 4;
    long long blocks = (n4 + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    router_reduce_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const float4*>(ws), S, n4, reinterpret_cast<float4*>(z));
  }
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
