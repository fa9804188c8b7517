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
// Kernel shape (one CTA per SM, persistent, in clusters of cs = 1, 2 or 4 CTAs):
//   warp 0      TMA producer: A tile 128x128 and B tile 256x128 (FP8) per K block,
//               4 stages.  The cs CTAs of a cluster work
//               on neighbouring N tiles of the same row block, so they need the same A
//               tile: each loads 128/cs of its rows and multicasts them to all, which
//               divides the A traffic from L2 by cs.
//   warp 1      TMEM allocation; one thread issues 4 MMAs (M128 N256 K32) per K block
//               into TMEM buffer (kb mod 2) and commits to the buffer barrier and to the
//               stage barrier of every CTA of the cluster (a stage is refilled only when
//               all cs CTAs have consumed it).  This warp never touches shared memory in
//               its loop: on this tensor core a shared-memory access by the issuing warp
//               (an mbarrier wait included) waits behind the operand reads of its MMAs in
//               flight and leaves the pipe idle.
//   warp 10     MMA scheduler: waits on the stage and TMEM-buffer mbarriers for each K
//               block and releases warp 1 through a named barrier (lockstep; its OR-
//               reduction carries an abort, so both warps leave the loop together)
//   warps 2..9  promotion + epilogue: warp w reads TMEM lanes 32*(w%4).. (its rows);
//               warps 2-5 own 128 of the 256 columns, warps 6-9 the other 128.  Each
//               thread adds its partials into 128 FP32 accumulators with packed FMAs,
//               16 columns per TMEM load; the scales arrive through cp.async rings.
// Tiles are 128 rows x 256 columns; the per-K-block synchronisation costs about the
// same for any tile width, so the wider tile amortises it over twice the MMA work.  The tile list walks segments in order, then N
// tiles, with the M tiles of a segment fastest so CTAs working at the same time share
// the expert's weight tile through L2.  Segments need not be multiples of 128 rows:
// rows past a segment's end are computed and not stored.
//
// Epilogues:
//   kEpiBF16    C = BF16(acc)
//   kEpiSwiGLU  B rows [128j, 128j+64) are gate rows [64j, 64j+64) and rows
//               [128j+64, 128j+128) the matching up rows, so N tile p (256 columns)
//               covers hidden columns [128p, 128p+128), one 1x128 group, and each
//               thread holds 64 gate and the 64 matching up accumulators of its row:
//               h = silu(gate) * up.  The two threads of a row exchange their max-abs
//               through shared memory and requantise h -> hq (E4M3) and sh (FP32).
#include <cuda.h>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace gk {
constexpr int BM = 128, BN = 256, BK = 128;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int SCHED_WARP = 2 + EPI_WARPS;          // waits on barriers for the MMA warp
constexpr int THREADS = 64 + EPI_THREADS + 32;
constexpr int MMA_BAR = 1;                         // named barrier: MMA warp + scheduler
constexpr int SPF = 8;                             // K blocks of scales prefetched ahead
constexpr int MAX_G = 1024;
constexpr int TBUF = 2;                  // TMEM partial buffers of BN columns
constexpr uint32_t TMEM_COLS = 512;

template <int EPI>
struct Layout {
  static constexpr int STAGES = 4;
  static constexpr int STASH = 0;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_STASH = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BAR = OFF_STASH + STASH;
  // barriers: full[STAGES], empty[STAGES], tfull[TBUF], tempty[TBUF], amax[2], drain
  static constexpr int NUM_BARS = 2 * STAGES + 2 * TBUF + 3;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;   // tmem slot, abort, total, bad
  static constexpr int OFF_SEG = OFF_MISC + 16;
  static constexpr int OFF_TSTART = OFF_SEG + (MAX_G + 1) * 4;
  static constexpr int OFF_AMAX = OFF_TSTART + (MAX_G + 1) * 4;   // [2 bufs][2 groups][128]
  // per-thread rings of prefetched scales: sA [SPF][EPI_THREADS], sB [SPF][EPI_WARPS][2]
  static constexpr int OFF_SCALE_A = OFF_AMAX + 2 * 2 * BM * 4;
  static constexpr int OFF_SCALE_B = OFF_SCALE_A + SPF * EPI_THREADS * 4;
  static constexpr int SMEM_USED = OFF_SCALE_B + SPF * EPI_WARPS * 2 * 4;
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024;              // 1024-B alignment slack
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};
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

// silu on the tile-end critical path: the fast exponential and division (a few ulps;
// h is compared with the oracle's float64 silu within a tolerance, never bit for bit)
MOE_DEV float silu_f32(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Cluster work unit -> (segment, first row, valid rows, unit index within the row
// block).  ustart[g] = first unit of segment g (non-decreasing); the largest g with
// ustart[g] <= unit is non-empty.  Units of a segment run M blocks fastest.
MOE_DEV void decode_unit(int unit, const int* ustart, const int* seg, int G, int& g, int& m0,
                         int& rows_valid, int& nu) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ustart[mid] <= unit) lo = mid;
    else hi = mid - 1;
  }
  g = lo;
  const int cnt = seg[g + 1] - seg[g];
  const int mt = (cnt + gk::BM - 1) / gk::BM;
  const int local = unit - ustart[g];
  const int m = local % mt;
  nu = local / mt;
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

// h requantisation: multiply by the correctly rounded reciprocal of the group scale (one
// rounding more than x / s; it can move a code only when x / s sits within an FP32 ulp of
// an E4M3 rounding boundary, and h itself carries the GEMM's FP32 rounding anyway)
MOE_DEV uint32_t e4m3x4(float a, float b, float c, float d, float rs) {
  const uint32_t lo = f32x2_to_e4m3x2(__fmul_rn(a, rs), __fmul_rn(b, rs));
  const uint32_t hi = f32x2_to_e4m3x2(__fmul_rn(c, rs), __fmul_rn(d, rs));
  return lo | (hi << 16);
}

}  // namespace

template <int EPI>
__global__ void __launch_bounds__(gk::THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  using namespace gk;
  using L = Layout<EPI>;
  constexpr int STAGES = L::STAGES;
  constexpr int TPU = 1;                             // N tiles per work unit
  extern __shared__ uint8_t gemm_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(gemm_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + TBUF + b); };
  auto amax_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 * TBUF + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * TBUF + 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  int* total_units = reinterpret_cast<int*>(smem + L::OFF_MISC + 8);
  int* bad = reinterpret_cast<int*>(smem + L::OFF_MISC + 12);
  int* seg = reinterpret_cast<int*>(smem + L::OFF_SEG);
  int* ustart = reinterpret_cast<int*>(smem + L::OFF_TSTART);
  float* amax_x = reinterpret_cast<float*>(smem + L::OFF_AMAX);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G;
  const int NT = (p.N + BN - 1) / BN;      // N tiles (the last may be half-filled)
  const int cs = static_cast<int>(cluster_nctarank());
  const int crank = static_cast<int>(cluster_ctarank());
  const int NU = NT / TPU / cs;            // cluster work units per M block
  const int KB = p.K / BK;
  const uint16_t cmask = static_cast<uint16_t>((1u << cs) - 1u);
  const int a_rows = BM / cs;              // A rows this CTA loads and multicasts

  // ---- segment table and unit prefix (every CTA computes its own copy) ----
  if (tid == 0) { *abort_flag = 0; *bad = 0; }
  for (int i = tid; i <= G; i += THREADS) seg[i] = p.seg[i];
  __syncthreads();
  {
    // each thread sums the unit counts of a run of segments; block-wide exclusive scan
    const int per = (G + THREADS - 1) / THREADS;
    const int g0 = min(G, tid * per), g1 = min(G, g0 + per);
    int local = 0;
    for (int g = g0; g < g1; ++g) {
      const int cnt = seg[g + 1] - seg[g];
      if (cnt < 0) *bad = 1;
      local += (max(cnt, 0) + BM - 1) / BM * NU;
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
      ustart[g] = run;
      run += (max(seg[g + 1] - seg[g], 0) + BM - 1) / BM * NU;
    }
    if (tid == THREADS - 1) {
      int tot = 0;
      for (int w = 0; w < THREADS / 32; ++w) tot += wsum[w];
      *total_units = tot;
      ustart[G] = tot;
    }
  }
  __syncthreads();
  if (*bad) {
    if (tid == 0) set_status(p.status, MOE_ERR_DEVICE_DATA);
    return;
  }
  const int total = *total_units;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(full_bar(s), 1); mbar_init(empty_bar(s), cs); }
    for (int b = 0; b < TBUF; ++b) { mbar_init(tfull_bar(b), 1); mbar_init(tempty_bar(b), EPI_WARPS); }
    for (int b = 0; b < 2; ++b) mbar_init(amax_bar(b), EPI_THREADS);
    mbar_init(drain_bar, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  cluster_sync();          // every CTA's barriers exist before any multicast reaches it
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int first_unit = static_cast<int>(cluster_id_x());
  const int unit_stride = static_cast<int>(ncluster_x());

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
        int g, m0, rv, cu;
        decode_unit(unit, ustart, seg, G, g, m0, rv, cu);
        const int nu = cu * cs + crank;
        for (int t = 0; ok && t < TPU; ++t) {
          const int brow = g * p.N + (nu * TPU + t) * BN;
          for (int kb = 0; kb < KB; ++kb, ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            if (!mbar_wait(empty_bar(s), ph ^ 1, abort_flag, p.status)) { ok = false; break; }
            mbar_arrive_expect_tx(full_bar(s), STAGE_BYTES);   // whole A tile + own B tile
            const uint32_t a_dst = sbase + L::OFF_A + s * A_BYTES;
            if (cs == 1)
              tma_load_2d(a_dst, &tmA, kb * BK, m0, full_bar(s));
            else
              tma_load_2d_multicast(a_dst + crank * a_rows * BK, &tmA, kb * BK,
                                    m0 + crank * a_rows, full_bar(s), cmask);
            tma_load_2d(sbase + L::OFF_B + s * B_BYTES, &tmB, kb * BK, brow, full_bar(s));
          }
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA's shared memory is released
        const uint32_t first = it > STAGES ? it - STAGES : 0;
        for (uint32_t i = first; i < it; ++i) mbar_drain(full_bar(i % STAGES), (i / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (no shared-memory access in the loop) ----------------
    constexpr uint32_t idesc = make_idesc(BM, BN, 0u, 0u);   // E4M3 x E4M3 -> F32
    uint32_t it = 0;
    bool ok = true;
    for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
      for (int t = 0; ok && t < TPU; ++t) {
        for (int kb = 0; kb < KB; ++kb, ++it) {
          // released by the scheduler once stage s is full and TMEM buffer b is free
          if (named_bar_sync_or(MMA_BAR, 64, false)) { ok = false; break; }
          if (lane == 0) {
            const int s = it % STAGES;
            const int b = it % TBUF;
            tc_fence_after();
            const uint64_t adesc = smem_desc_sw128(sbase + L::OFF_A + s * A_BYTES);
            const uint64_t bdesc = smem_desc_sw128(sbase + L::OFF_B + s * B_BYTES);
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
#pragma unroll
            for (int k = 0; k < BK / 32; ++k)   // K = 32 bytes per MMA: +2 in the >>4 address
              mma_f8f6f4(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
            if (cs == 1) mma_commit(empty_bar(s));
            else mma_commit_multicast(empty_bar(s), cmask);
            mma_commit(tfull_bar(b));
          }
          __syncwarp();
        }
      }
    }
    // every MMA issued so far must finish before TMEM is released
    if (lane == 0) {
      mma_commit(drain_bar);
      mbar_drain(drain_bar, 0);
    }
    __syncwarp();
  } else if (warp == SCHED_WARP) {
    // ---------------- MMA scheduler ----------------
    // Same iteration sequence as the MMA warp; one named barrier per K block.
    uint32_t it = 0;
    bool ok = true;
    for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
      for (int t = 0; ok && t < TPU; ++t) {
        for (int kb = 0; kb < KB; ++kb, ++it) {
          int good = 1;
          if (lane == 0) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            const int b = it % TBUF;
            const uint32_t bph = (it / TBUF) & 1;
            good = mbar_wait(tempty_bar(b), bph ^ 1, abort_flag, p.status) &&
                   mbar_wait(full_bar(s), ph, abort_flag, p.status);
          }
          good = __shfl_sync(0xFFFFFFFFu, good, 0);
          tc_fence_before();
          if (named_bar_sync_or(MMA_BAR, 64, good == 0)) { ok = false; break; }
        }
      }
    }
  } else if (warp >= 2 && warp < 2 + EPI_WARPS) {
    // ---------------- promotion + epilogue ----------------
    const int etid = tid - 64;
    const int grp = (warp - 2) >> 2;    // column half of the tile
    const int q = warp & 3;             // TMEM lane window
    const int row = q * 32 + lane;      // row within the tile
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const int NB = p.N / 128;           // weight-scale rows per segment
    // TMEM columns of this thread's eight 16-column chunks (SwiGLU: 4 gate then 4 up)
    int cols[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
      cols[c] = (EPI == kEpiSwiGLU) ? grp * 128 + (c < 4 ? 0 : 64) + (c & 3) * 16
                                    : grp * 128 + c * 16;
    // Scale prefetch: every K block needs sA[kb][row] (this thread's row) and the one or
    // two weight scales of the tile's N blocks.  They are copied into shared-memory rings
    // SPF K blocks ahead with cp.async, following the same (unit, tile, K block) sequence
    // as the promotion loop, so the L2 latency never sits on the critical path.
    const uint32_t ring_a = sbase + L::OFF_SCALE_A + static_cast<uint32_t>(etid) * 4;
    const uint32_t ring_b = sbase + L::OFF_SCALE_B + static_cast<uint32_t>(warp - 2) * 8;
    const float* ring_a_f = reinterpret_cast<const float*>(smem + L::OFF_SCALE_A) + etid;
    const float* ring_b_f = reinterpret_cast<const float*>(smem + L::OFF_SCALE_B) + (warp - 2) * 2;
    int pf_unit = first_unit, pf_t = 0, pf_kb = 0;       // prefetch cursor
    int pf_g = 0, pf_m0 = 0, pf_nu = 0;
    bool pf_live = pf_unit < total;
    if (pf_live) {
      int rv_unused, cu;
      decode_unit(pf_unit, ustart, seg, G, pf_g, pf_m0, rv_unused, cu);
      pf_nu = cu * cs + crank;
    }
    uint32_t pf_it = 0;
    auto prefetch_one = [&]() {
      // issue the copies of the cursor's K block into ring slot pf_it % SPF, then advance
      if (pf_live) {
        const int nt = pf_nu * TPU + pf_t;
        // (a half-filled last tile has no second N block: read a valid scale, unused)
        const int nb0 = (EPI == kEpiSwiGLU) ? 2 * nt : min(2 * nt + grp, NB - 1);
        const int nb1 = (EPI == kEpiSwiGLU) ? 2 * nt + 1 : nb0;
        const int slot = static_cast<int>(pf_it % SPF);
        const int arow = min(pf_m0 + row, p.M - 1);
        cp_async_4(ring_a + slot * EPI_THREADS * 4,
                   p.sA + static_cast<long long>(pf_kb) * p.M + arow);
        if (lane == 0) {
          const float* sb = p.sB + static_cast<long long>(pf_g) * NB * KB + pf_kb;
          cp_async_4(ring_b + slot * EPI_WARPS * 8, sb + static_cast<long long>(nb0) * KB);
          cp_async_4(ring_b + slot * EPI_WARPS * 8 + 4, sb + static_cast<long long>(nb1) * KB);
        }
        if (++pf_kb == KB) {
          pf_kb = 0;
          if (++pf_t == TPU) {
            pf_t = 0;
            pf_unit += unit_stride;
            pf_live = pf_unit < total;
            if (pf_live) {
              int rv_unused, cu;
              decode_unit(pf_unit, ustart, seg, G, pf_g, pf_m0, rv_unused, cu);
              pf_nu = cu * cs + crank;
            }
          }
        }
      }
      cp_async_commit();                                 // one group per K block, maybe empty
      ++pf_it;
    };
    for (int i = 0; i < SPF - 1; ++i) prefetch_one();
    // the scales of the first K block, read one block ahead from then on
    cp_async_wait<SPF - 2>();
    __syncwarp();
    float nsa = ring_a_f[0], nsb0 = ring_b_f[0], nsb1 = ring_b_f[1];

    uint32_t it = 0;
    int ucount = 0;
    bool ok = true;
    for (int unit = first_unit; ok && unit < total; unit += unit_stride, ++ucount) {
      int g, m0, rv, cu;
      decode_unit(unit, ustart, seg, G, g, m0, rv, cu);
      const int nu = cu * cs + crank;
      (void)g;
      for (int t = 0; ok && t < TPU; ++t) {
        const int nt = nu * TPU + t;
        float2 acc2[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc2[i] = make_float2(0.0f, 0.0f);
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const float sa = nsa, sb0 = nsb0, sb1 = nsb1;
          const int b = it % TBUF;
          const uint32_t bph = (it / TBUF) & 1;
          if (!mbar_wait_warp(tfull_bar(b), bph, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const float sc0 = __fmul_rn(sa, sb0);
          const float sc1 = __fmul_rn(sa, sb1);
          const uint32_t tb = tmem_base + lane_addr + static_cast<uint32_t>(b * BN);
          // two 16-column loads in flight per wait: four TMEM round trips per K block
#pragma unroll
          for (int c = 0; c < 8; c += 2) {
            const float sc = (c < 4) ? sc0 : sc1;
            const float2 sc2 = make_float2(sc, sc);
            uint32_t v[2][16];
            tmem_ld_32x32b_x16(tb + static_cast<uint32_t>(cols[c]), v[0]);
            tmem_ld_32x32b_x16(tb + static_cast<uint32_t>(cols[c + 1]), v[1]);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int i = 0; i < 8; ++i)
                acc2[(c + h) * 8 + i] = __ffma2_rn(
                    sc2,
                    make_float2(__uint_as_float(v[h][2 * i]), __uint_as_float(v[h][2 * i + 1])),
                    acc2[(c + h) * 8 + i]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(b));     // the buffer is folded in
          // scales of K block it + 1: their shared-memory latency overlaps the next wait
          prefetch_one();                                // K block it + SPF - 1
          cp_async_wait<SPF - 2>();                      // this thread's copies for it + 1
          __syncwarp();                                  // lane 0's weight scales too
          const int nslot = static_cast<int>((it + 1) % SPF);
          nsa = ring_a_f[nslot * EPI_THREADS];
          nsb0 = ring_b_f[nslot * EPI_WARPS * 2];
          nsb1 = ring_b_f[nslot * EPI_WARPS * 2 + 1];
        }
        if (!ok) break;
        float* acc = reinterpret_cast<float*>(acc2);

        if (EPI == kEpiBF16) {
          if (row < rv && nt * BN + grp * 128 < p.N) {
            uint4* dst = reinterpret_cast<uint4*>(p.C + static_cast<long long>(m0 + row) * p.ldc +
                                                  nt * BN + grp * 128);
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
          const int buf = ucount & 1;
          amax_x[(buf * 2 + grp) * BM + row] = amax;
          mbar_arrive(amax_bar(buf));
          if (!mbar_wait_warp(amax_bar(buf), (ucount >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
          amax = fmaxf(amax, amax_x[(buf * 2 + (grp ^ 1)) * BM + row]);
          const float s = e4m3_scale_from_amax(amax);
          const float rs = __frcp_rn(s);
          if (row < rv) {
            const int f = p.N / 2;
            uint4* dst = reinterpret_cast<uint4*>(p.hq + static_cast<long long>(m0 + row) * f +
                                                  nt * 128 + grp * 64);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float* h = acc + 16 * j;
              dst[j] = make_uint4(e4m3x4(h[0], h[1], h[2], h[3], rs),
                                  e4m3x4(h[4], h[5], h[6], h[7], rs),
                                  e4m3x4(h[8], h[9], h[10], h[11], rs),
                                  e4m3x4(h[12], h[13], h[14], h[15], rs));
            }
            if (grp == 0) p.sh[static_cast<long long>(nt) * p.M + m0 + row] = s;
          }
        }
      }
    }
    cp_async_wait<0>();                                  // no copy may land after exit
  }

  tc_fence_before();
  cluster_sync();          // no CTA leaves while a cluster peer may still write into it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---- host side ------------------------------------------------------------------------

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* ptr,
                    uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                    uint32_t box_outer);   // runtime.cu

namespace {

// Largest cluster size in {4, 2, 1} that divides the work units of one row block.
int pick_cluster(int units_per_block) {
  // Clusters share the A tile through multicast, which cuts L2 traffic but not the
  // shared-memory traffic that bounds this kernel, and 4-CTA clusters leave SMs idle
  // (fewer can be resident at once); one-CTA clusters measured faster.
  (void)units_per_block;
  return 1;
}

template <int EPI>
int launch_gemm_kernel(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p,
                       int cs, long long max_units, cudaStream_t stream) {
  constexpr int smem = gk::Layout<EPI>::SMEM_ALLOC;
  auto kern = fp8_gemm_kernel<EPI>;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(gk::THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // as many clusters as can be resident at once (the kernel is persistent)
  static int max_clusters[5] = {0, 0, 0, 0, 0};
  if (max_clusters[cs] == 0) {
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms() / cs * cs), 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) n = num_sms() / cs;
    max_clusters[cs] = n;
  }
  long long clusters = max_clusters[cs];
  if (max_units < clusters) clusters = max_units;
  if (clusters < 1) clusters = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * cs), 1, 1);
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p) != cudaSuccess) return MOE_ERR_CUDA;
  return check_launch();
}

}  // namespace

int launch_fp8_gemm(const GemmArgs& a, GemmEpilogue epi, cudaStream_t stream) {
  using namespace gk;
  if (a.M == 0) return MOE_OK;
  if (a.N % 128 != 0 || (epi == kEpiSwiGLU && a.N % BN != 0)) return MOE_ERR_UNSUPPORTED;
  const int units = (a.N + BN - 1) / BN;                        // CTA units per row block
  const int cs = pick_cluster(units);
  CUtensorMap tmA, tmB;
  if (!encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A, a.K, a.M, a.K, BK, BM / cs))
    return MOE_ERR_CUDA;
  if (!encode_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B,
                      a.K, static_cast<uint64_t>(a.G) * a.N, a.K, BK, BN))
    return MOE_ERR_CUDA;
  GemmParams p;
  p.sA = a.sA; p.sB = a.sB; p.seg = a.seg;
  p.G = a.G; p.M = a.M; p.N = a.N; p.K = a.K;
  p.C = a.C; p.ldc = a.ldc; p.hq = a.hq; p.sh = a.sh; p.status = a.status;
  const long long max_units = (static_cast<long long>(a.M) / BM + a.G) * (units / cs);
  if (epi == kEpiSwiGLU) return launch_gemm_kernel<kEpiSwiGLU>(tmA, tmB, p, cs, max_units, stream);
  return launch_gemm_kernel<kEpiBF16>(tmA, tmB, p, cs, max_units, stream);
}

}  // namespace moe
