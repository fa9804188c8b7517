// FP8 E4M3 block-scaled grouped GEMM on tcgen05 tensor cores (sm_103a).
//
//   C[r][n] = sum_kb sA[kb][r] * sB[g][n/128][kb] * P_kb[r][n],
//   P_kb    = sum_{k in K-block kb} A[r][k] * B[g][n][k]       (128-deep K blocks)
//
// for the rows r of segment g.  The scales vary along K, so every 128-deep partial
// product needs its own scale product before it joins the sum ("DeepSeek-V3" book,
// ch. 16 "Scales along the GEMM inner dimension"); partials are promoted to FP32 at
// that interval ("DeepSeek-V3" summary, core idea 6(b); book ch. 16 "Periodic
// high-precision promotion").  The pages did this on Hopper with two warpgroups taking
// turns on register accumulators; here the tensor core writes each K block's partial
// into one of two TMEM buffers while the epilogue warps fold the other into FP32
// registers.
//
// Kernel shape (one CTA per SM, persistent):
//   warp 0      TMA producer: A tile 128x128 and B tile 256x128 per K block, 4 stages
//   warp 1      TMEM allocation; one thread issues 4 MMAs (M128 N256 K32) per K block
//               into TMEM buffer (kb & 1) and commits to the stage / buffer barriers
//   warps 2..9  promotion + epilogue: warp w reads TMEM lanes 32*(w%4).. (its rows);
//               warps 2-5 own one half of the 256 columns, warps 6-9 the other
// Tiles are 128 rows x 256 columns.  The tile list walks segments in order, then
// N tiles, with the M tiles of a segment fastest so CTAs working at the same time share
// the expert's weight tile through L2.  Segments need not be multiples of 128 rows:
// rows past a segment's end are computed and not stored.
//
// Epilogues:
//   kEpiBF16    C = BF16(acc)
//   kEpiSwiGLU  the B rows of N tile j are 128 gate rows then the matching 128 up rows;
//               h = silu(gate) * up (FP32) is requantised in 1x128 groups along the
//               hidden dimension (one group per N tile) -> hq (E4M3) and sh (FP32).
#include <cuda.h>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace gk {
constexpr int BM = 128, BN = 256, BK = 128;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + EPI_WARPS * 32;
constexpr int MAX_G = 1024;
constexpr uint32_t TMEM_COLS = 512;      // two 256-column FP32 partial buffers

// Shared-memory layout, offsets from a 1024-byte aligned base.
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
// barriers: full[STAGES], empty[STAGES], tfull[2], tempty[2], amax[2], drain
constexpr int NUM_BARS = 2 * STAGES + 7;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;          // tmem slot, abort flag, total
constexpr int OFF_SEG = OFF_MISC + 16;
constexpr int OFF_TSTART = OFF_SEG + (MAX_G + 1) * 4;
constexpr int OFF_AMAX = OFF_TSTART + (MAX_G + 1) * 4;    // [2 buffers][2 groups][128]
constexpr int SMEM_USED = OFF_AMAX + 2 * 2 * BM * 4;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;               // slack for 1024-B alignment
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
}  // namespace gk

struct GemmParams {
  const float* sA;
  const float* sB;
  const int32_t* seg;
  int G, M, N, K;
  uint16_t* C;
  int ldc;
  uint8_t* hq;
  float* sh;
  int32_t* status;
};

namespace {

MOE_DEV float silu_f32(float g) { return __fdiv_rn(g, 1.0f + expf(-g)); }

// Tile -> (segment, first row, valid rows, N tile).  tstart[g] = first tile of segment
// g (non-decreasing); the largest g with tstart[g] <= tile is non-empty.
MOE_DEV void decode_tile(int tile, const int* tstart, const int* seg, int G, int& g, int& m0,
                         int& rows_valid, int& nt) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tstart[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  g = lo;
  const int cnt = seg[g + 1] - seg[g];
  const int mt = (cnt + gk::BM - 1) / gk::BM;
  const int local = tile - tstart[g];
  const int m = local % mt;
  nt = local / mt;
  m0 = seg[g] + m * gk::BM;
  rows_valid = min(gk::BM, seg[g + 1] - m0);
}

// Bounded wait used only while shutting down after an abort: ignores the abort flag.
MOE_DEV void mbar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

}  // namespace

template <int EPI>
__global__ void __launch_bounds__(gk::THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  using namespace gk;
  extern __shared__ uint8_t gemm_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(gemm_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
  auto amax_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 4 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 6);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  int* total_tiles = reinterpret_cast<int*>(smem + OFF_MISC + 8);
  int* bad = reinterpret_cast<int*>(smem + OFF_MISC + 12);
  int* seg = reinterpret_cast<int*>(smem + OFF_SEG);
  int* tstart = reinterpret_cast<int*>(smem + OFF_TSTART);
  float* amax_x = reinterpret_cast<float*>(smem + OFF_AMAX);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G;
  const int NT = (p.N + BN - 1) / BN;
  const int KB = p.K / BK;

  // ---- segment table and tile prefix (every CTA computes its own copy) ----
  if (tid == 0) { *abort_flag = 0; *bad = 0; }
  for (int i = tid; i <= G; i += THREADS) seg[i] = p.seg[i];
  __syncthreads();
  {
    // each thread sums the tile counts of a run of segments; block-wide exclusive scan
    const int per = (G + THREADS - 1) / THREADS;
    const int g0 = min(G, tid * per), g1 = min(G, g0 + per);
    int local = 0;
    for (int g = g0; g < g1; ++g) {
      const int cnt = seg[g + 1] - seg[g];
      if (cnt < 0) *bad = 1;
      local += (cnt + BM - 1) / BM * NT;
    }
    if (tid == 0 && (seg[0] != 0 || seg[G] > p.M)) *bad = 1;
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += o;
    }
    int* wsum = reinterpret_cast<int*>(amax_x);   // scratch before the epilogue uses it
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += wsum[w];
    int run = wbase + incl - local;
    for (int g = g0; g < g1; ++g) {
      tstart[g] = run;
      run += (max(seg[g + 1] - seg[g], 0) + BM - 1) / BM * NT;
    }
    if (tid == THREADS - 1) {
      int tot = 0;
      for (int w = 0; w < THREADS / 32; ++w) tot += wsum[w];
      *total_tiles = tot;
      tstart[G] = tot;
    }
  }
  __syncthreads();
  if (*bad) {
    if (tid == 0) set_status(p.status, MOE_ERR_DEVICE_DATA);
    return;
  }
  const int total = *total_tiles;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(full_bar(s), 1); mbar_init(empty_bar(s), 1); }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), EPI_WARPS);
      mbar_init(amax_bar(b), EPI_WARPS * 32);
    }
    mbar_init(drain_bar, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int g, m0, rv, nt;
        decode_tile(tile, tstart, seg, G, g, m0, rv, nt);
        const int brow = g * p.N + nt * BN;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(empty_bar(s), ph ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(full_bar(s), STAGE_BYTES);
          tma_load_2d(sbase + OFF_A + s * A_BYTES, &tmA, kb * BK, m0, full_bar(s));
          tma_load_2d(sbase + OFF_B + s * B_BYTES, &tmB, kb * BK, brow, full_bar(s));
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA's shared memory is released
        const uint32_t first = it > STAGES ? it - STAGES : 0;
        for (uint32_t i = first; i < it; ++i) mbar_drain(full_bar(i % STAGES), (i / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(BM, BN, 0u, 0u);   // E4M3 x E4M3 -> F32
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          const int b = it & 1;
          const uint32_t bph = (it >> 1) & 1;
          if (!mbar_wait(tempty_bar(b), bph ^ 1, abort_flag, p.status)) { ok = false; break; }
          if (!mbar_wait(full_bar(s), ph, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(sbase + OFF_A + s * A_BYTES);
          const uint64_t bdesc = smem_desc_sw128(sbase + OFF_B + s * B_BYTES);
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)   // K = 32 bytes per MMA: +2 in the >>4 address
            mma_f8f6f4(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
          mma_commit(empty_bar(s));
          mma_commit(tfull_bar(b));
        }
      }
      // every MMA issued so far must finish before TMEM is released
      mma_commit(drain_bar);
      mbar_drain(drain_bar, 0);
    }
  } else {
    // ---------------- promotion + epilogue ----------------
    const int ew = warp - 2;
    const int grp = ew >> 2;            // column half
    const int q = warp & 3;             // TMEM lane window
    const int row = q * 32 + lane;      // row within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const int NB = p.N / 128;           // N blocks of 128 (weight scale rows)
    uint32_t it = 0;
    int tcount = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++tcount) {
      int g, m0, rv, nt;
      decode_tile(tile, tstart, seg, G, g, m0, rv, nt);
      const int arow = min(m0 + row, p.M - 1);
      const float* sa_col = p.sA + arow;
      const float* sb_g = p.sB + static_cast<long long>(g) * NB * KB;
      // weight-scale rows used by this thread's columns
      int nb0, nb1;
      if (EPI == kEpiSwiGLU) { nb0 = 2 * nt; nb1 = 2 * nt + 1; }
      else { nb0 = nb1 = 2 * nt + grp; }
      const bool nb_ok = nb1 < NB;
      // FP32 accumulators as pairs: the promotion runs as packed FP32 FMAs (two lanes'
      // worth per instruction, each rounded like a single FMA)
      float2 acc2[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc2[i] = make_float2(0.0f, 0.0f);
      float sa_next = __ldg(sa_col);
      float sb0_next = nb_ok ? __ldg(sb_g + static_cast<long long>(nb0) * KB) : 0.0f;
      float sb1_next = nb_ok ? __ldg(sb_g + static_cast<long long>(nb1) * KB) : 0.0f;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const float sa = sa_next, sb0 = sb0_next, sb1 = sb1_next;
        if (kb + 1 < KB) {
          sa_next = __ldg(sa_col + static_cast<long long>(kb + 1) * p.M);
          if (nb_ok) {
            sb0_next = __ldg(sb_g + static_cast<long long>(nb0) * KB + kb + 1);
            sb1_next = __ldg(sb_g + static_cast<long long>(nb1) * KB + kb + 1);
          }
        }
        const float sc0 = __fmul_rn(sa, sb0), sc1 = __fmul_rn(sa, sb1);
        const int b = it & 1;
        const uint32_t bph = (it >> 1) & 1;
        if (!mbar_wait(tfull_bar(b), bph, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tb = tmem_base + lane_addr + static_cast<uint32_t>(b * BN);
        // 16-column chunks keep the staging registers small enough that the 128
        // accumulators stay in registers (the 10-warp CTA allows 168 per thread)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          int col;
          if (EPI == kEpiSwiGLU) col = (c < 4 ? 0 : 128) + grp * 64 + (c & 3) * 16;
          else col = grp * 128 + c * 16;
          const float sc = (EPI == kEpiSwiGLU && c >= 4) ? sc1 : sc0;
          const float2 sc2 = make_float2(sc, sc);
          uint32_t v[16];
          tmem_ld_32x32b_x16(tb + static_cast<uint32_t>(col), v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            acc2[c * 8 + i] = __ffma2_rn(
                sc2, make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                acc2[c * 8 + i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(b));
      }
      if (!ok) break;
      float* acc = reinterpret_cast<float*>(acc2);

      if (EPI == kEpiBF16) {
        const int col0 = nt * BN + grp * 128;
        if (row < rv && col0 < p.N) {
          uint4* dst = reinterpret_cast<uint4*>(p.C + static_cast<long long>(m0 + row) * p.ldc + col0);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            uint4 o;
            o.x = pack_bf16x2(acc[8 * j + 0], acc[8 * j + 1]);
            o.y = pack_bf16x2(acc[8 * j + 2], acc[8 * j + 3]);
            o.z = pack_bf16x2(acc[8 * j + 4], acc[8 * j + 5]);
            o.w = pack_bf16x2(acc[8 * j + 6], acc[8 * j + 7]);
            dst[j] = o;
          }
        }
      } else {
        // h = silu(gate) * up for this thread's 64 hidden columns
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          acc[i] = __fmul_rn(silu_f32(acc[i]), acc[64 + i]);
          amax = fmaxf(amax, fabsf(acc[i]));
        }
        const int buf = tcount & 1;
        amax_x[(buf * 2 + grp) * BM + row] = amax;
        mbar_arrive(amax_bar(buf));
        if (!mbar_wait(amax_bar(buf), (tcount >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
        amax = fmaxf(amax, amax_x[(buf * 2 + (grp ^ 1)) * BM + row]);
        const float s = e4m3_scale_from_amax(amax);
        if (row < rv) {
          const int f = p.N / 2;
          uint4* dst = reinterpret_cast<uint4*>(p.hq + static_cast<long long>(m0 + row) * f +
                                                nt * 128 + grp * 64);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int e = 16 * j + 4 * i;
              const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(acc[e], s), __fdiv_rn(acc[e + 1], s));
              const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(acc[e + 2], s), __fdiv_rn(acc[e + 3], s));
              w[i] = lo | (hi << 16);
            }
            dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          if (grp == 0) p.sh[static_cast<long long>(nt) * p.M + m0 + row] = s;
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

// ---- host side ------------------------------------------------------------------------

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* ptr,
                    uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                    uint32_t box_outer);   // runtime.cu

int launch_fp8_gemm(const GemmArgs& a, GemmEpilogue epi, cudaStream_t stream) {
  using namespace gk;
  if (a.M == 0) return MOE_OK;
  CUtensorMap tmA, tmB;
  if (!encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A, a.K, a.M, a.K, BK, BM))
    return MOE_ERR_CUDA;
  if (!encode_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B,
                      a.K, static_cast<uint64_t>(a.G) * a.N, a.K, BK, BN))
    return MOE_ERR_CUDA;
  GemmParams p;
  p.sA = a.sA; p.sB = a.sB; p.seg = a.seg;
  p.G = a.G; p.M = a.M; p.N = a.N; p.K = a.K;
  p.C = a.C; p.ldc = a.ldc; p.hq = a.hq; p.sh = a.sh; p.status = a.status;

  const int NT = (a.N + BN - 1) / BN;
  const long long max_tiles = (static_cast<long long>(a.M) / BM + a.G) * NT;
  int grid = num_sms();
  if (max_tiles < grid) grid = static_cast<int>(max_tiles);
  if (grid < 1) grid = 1;

  auto kern = (epi == kEpiSwiGLU) ? fp8_gemm_kernel<kEpiSwiGLU> : fp8_gemm_kernel<kEpiBF16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_ALLOC) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  kern<<<grid, THREADS, SMEM_ALLOC, stream>>>(tmA, tmB, p);
  return check_launch();
}

}  // namespace moe
