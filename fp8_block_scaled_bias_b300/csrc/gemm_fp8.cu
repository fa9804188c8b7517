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
// Two tilings of the same kernel (one CTA per SM, persistent):
//   single  one CTA per 128-row x 256-column tile: per K block it loads A 128x128 and
//           B 256x128 (48 KB) and issues M128 N256 MMAs (tcgen05 cta_group::1).
//   pair    two CTAs (a cluster of 2) per 256-row x 256-column tile: one tcgen05
//           cta_group::2 MMA (M256 N256) reads A rows [0, 128) and B rows [0, 128) from
//           the first CTA's shared memory and A rows [128, 256), B rows [128, 256) from
//           the second's, and writes rows [0, 128) of the accumulator into the first
//           CTA's TMEM and rows [128, 256) into the second's.  Each CTA loads 32 KB per K
//           block for the same MMA work per SM (a third fewer bytes through L2), and still
//           promotes its own 128 rows.  The pace of both tilings is the TMEM buffer round
//           trip (promotion reads, MMA, barrier latencies), which the pair lengthens with
//           its cross-CTA release: measured slower than the single tiling on B300.
// Warp roles:
//   warp 0      TMA producer of this CTA's A and B rows, STAGES-deep ring.  In the pair
//               tiling both CTAs' loads complete on the first CTA's stage barrier.
//   warp 1      TMEM allocation; one thread waits for the stage and for TMEM buffer
//               (kb mod 2), issues 4 MMAs (K32 each) per K block into that buffer and
//               commits to the stage and buffer barriers (of both CTAs in the pair
//               tiling; only the first CTA issues).
//   warps 2..9  promotion + epilogue: warp w reads TMEM lanes 32*(w%4).. (its rows);
//               warps 2-5 own 128 of the 256 columns, warps 6-9 the other 128.  Each
//               thread adds its partials into 128 FP32 accumulators with packed FMAs,
//               16 columns per TMEM load; each K block's scales are loaded from global
//               memory into registers during the K block before (measured faster on
//               this B300 than cp.async rings in shared memory or a feeder warp).
// The tile list walks segments in order, then N tiles, with the M tiles of a segment
// fastest so CTAs working at the same time share the expert's weight tile through L2.
// Segments need not be multiples of the tile height: rows past a segment's end are
// computed and not stored.
//
// Epilogues:
//   kEpiBF16    C = BF16(acc)
//   kEpiSwiGLU  B rows [128j, 128j+64) are gate rows [64j, 64j+64) and rows
//               [128j+64, 128j+128) the matching up rows, so N tile p (256 columns)
//               covers hidden columns [128p, 128p+128), one 1x128 group, and each
//               thread holds 64 gate and the 64 matching up accumulators of its row:
//               h = silu(gate) * up.  The two threads of a row exchange their max-abs
//               through shared memory and requantise h -> hq (E4M3) and sh (FP32).
//
// Every mbarrier wait is bounded (GemmParams::wait_ns); on expiry the kernel records
// MOE_ERR_DEVICE_TIMEOUT, stops issuing work, lets its copies and MMAs in flight land,
// frees TMEM and returns.
#include <atomic>
#include <cuda.h>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace gk {
constexpr int BN = 256, BK = 128;
constexpr int ROWS = 128;                          // accumulator rows per CTA (TMEM lanes)
constexpr int A_BYTES = ROWS * BK;
constexpr int EPI_WARPS = 8;
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int THREADS = 64 + EPI_THREADS;
constexpr int MAX_G = 1024;
constexpr int TBUF = 2;                            // TMEM partial buffers of BN columns
constexpr uint32_t TMEM_COLS = 512;

template <bool PAIR>
struct Layout {
  static constexpr int BM = PAIR ? 2 * ROWS : ROWS;     // rows per work unit
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;     // B rows this CTA loads
  static constexpr int B_BYTES = B_ROWS * BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES; // bytes this CTA loads per K block
  static constexpr int STAGES = PAIR ? 6 : 4;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
  // barriers: full[STAGES], empty[STAGES], tfull[TBUF], tempty[TBUF], amax[2], drain, stall
  static constexpr int NUM_BARS = 2 * STAGES + 2 * TBUF + 4;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;   // tmem slot, abort, total, bad
  static constexpr int OFF_SEG = OFF_MISC + 16;
  static constexpr int OFF_TSTART = OFF_SEG + (MAX_G + 1) * 4;
  // row max-abs exchange: [2 bufs][h, gate, up][2 column halves][128 rows]
  static constexpr int OFF_AMAX = OFF_TSTART + (MAX_G + 1) * 4;
  static constexpr int SMEM_USED = OFF_AMAX + 2 * 3 * 2 * ROWS * 4;
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
  uint8_t* guq;          // training forward: g, u cached as E4M3 [M][N] (gate cols first)
  float* sgu;            // and their 1x128 scales [N/128][M]
  int32_t* status;
  uint64_t wait_ns;      // limit of every mbarrier wait
  int stall;             // != 0: the MMA issuer waits on a barrier nothing arrives on
};

namespace {

// silu on the tile-end critical path: the fast exponential and division (a few ulps;
// h is compared with the oracle's float64 silu within a tolerance, never bit for bit)
MOE_DEV float silu_f32(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Work unit -> (segment, first row of the unit, N tile).  ustart[g] = first unit of
// segment g (non-decreasing); the largest g with ustart[g] <= unit is non-empty.  Units
// of a segment run M blocks (of BM rows) fastest.
template <int BM>
MOE_DEV void decode_unit(int unit, const int* ustart, const int* seg, int G, int& g, int& m0,
                         int& nt) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ustart[mid] <= unit) lo = mid;
    else hi = mid - 1;
  }
  g = lo;
  const int cnt = seg[g + 1] - seg[g];
  const int mt = (cnt + BM - 1) / BM;
  const int local = unit - ustart[g];
  nt = local / mt;
  m0 = seg[g] + (local % mt) * BM;
}

// Bounded wait used only while shutting down after an abort: ignores the abort flag.
MOE_DEV void mbar_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
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

// The activation quantiser's rule exactly: q = E4M3(fl32(x / s)), correctly rounded division.
MOE_DEV uint32_t e4m3x4_div(const float* x, float s) {
  const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(x[0], s), __fdiv_rn(x[1], s));
  const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(x[2], s), __fdiv_rn(x[3], s));
  return lo | (hi << 16);
}

// ---- tcgen05 forms of the two tilings (one kernel uses one cta_group throughout) ----

template <bool PAIR>
MOE_DEV void tmem_alloc_g(uint32_t dst, uint32_t ncols) {
  if (PAIR) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else {
    tmem_alloc(dst, ncols);
  }
}

template <bool PAIR>
MOE_DEV void tmem_dealloc_g(uint32_t taddr, uint32_t ncols) {
  if (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  else
    tmem_dealloc(taddr, ncols);
}

template <bool PAIR>
MOE_DEV void mma_fp8_g(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                       uint32_t accumulate) {
  if (PAIR)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  else
    mma_f8f6f4(d_tmem, adesc, bdesc, idesc, accumulate);
}

// Arrive once on the mbarrier at shared::cluster address `bar` (either CTA of the pair)
// when every MMA issued so far by this thread has completed.
template <bool PAIR>
MOE_DEV void mma_commit_g(uint32_t bar) {
  if (PAIR)
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
  else
    mma_commit(bar);
}

}  // namespace

template <int EPI, bool PAIR>
__global__ void __launch_bounds__(gk::THREADS, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  using namespace gk;
  using L = Layout<PAIR>;
  constexpr int STAGES = L::STAGES, BM = L::BM;
  // SwiGLU epilogue; CACHE: also keep its inputs g, u in FP8 (training forward)
  constexpr bool SWIGLU = EPI == kEpiSwiGLU || EPI == kEpiSwiGLUCache;
  constexpr bool CACHE = EPI == kEpiSwiGLUCache;
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
  const uint32_t stall_bar = bar0 + 8u * (2 * STAGES + 2 * TBUF + 3);
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
  const int KB = p.K / BK;
  const uint64_t wait_ns = p.wait_ns;
  // pair tiling: rank 0 issues the MMAs and owns the stage barriers; rank 1 is its peer
  const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
  const bool issuer = crank == 0;

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
      local += (max(cnt, 0) + BM - 1) / BM * NT;
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
      run += (max(seg[g + 1] - seg[g], 0) + BM - 1) / BM * NT;
    }
    if (tid == THREADS - 1) {
      int tot = 0;
      for (int w = 0; w < THREADS / 32; ++w) tot += wsum[w];
      *total_units = tot;
      ustart[G] = tot;
    }
  }
  __syncthreads();
  // Both CTAs of a pair read the same segment table, so they leave here together,
  // before either touches the other's shared memory.
  if (*bad) {
    if (tid == 0) set_status(p.status, MOE_ERR_DEVICE_DATA);
    return;
  }
  const int total = *total_units;

  if (tid == 0) {
    // full: one arrival per loading CTA (plus the bytes); empty: one MMA commit;
    // tempty: every promotion warp of the CTA(s) sharing the accumulator
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), PAIR ? 2 : 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < TBUF; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), (PAIR ? 2 : 1) * EPI_WARPS);
    }
    for (int b = 0; b < 2; ++b) mbar_init(amax_bar(b), EPI_THREADS);
    mbar_init(drain_bar, 1);
    mbar_init(stall_bar, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc_g<PAIR>(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  if (PAIR) cluster_sync();   // both CTAs' barriers exist before either signals the other
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int first_unit = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int unit_stride = PAIR ? static_cast<int>(ncluster_x()) : static_cast<int>(gridDim.x);
  const int row_off = static_cast<int>(crank) * ROWS;   // this CTA's rows within the unit

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
        int g, m0, nt;
        decode_unit<BM>(unit, ustart, seg, G, g, m0, nt);
        const int arow = m0 + row_off;
        const int brow = g * p.N + nt * BN + static_cast<int>(crank) * L::B_ROWS;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait<PAIR>(empty_bar(s), ph ^ 1, abort_flag, p.status, wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = sbase + L::OFF_A + s * A_BYTES;
          const uint32_t b_dst = sbase + L::OFF_B + s * L::B_BYTES;
          if (PAIR) {
            const uint32_t fb = mapa_shared(full_bar(s), 0);
            mbar_arrive_expect_tx_cluster(fb, L::STAGE_BYTES);
            tma_load_2d_pair(a_dst, &tmA, kb * BK, arow, fb);
            tma_load_2d_pair(b_dst, &tmB, kb * BK, brow, fb);
          } else {
            mbar_arrive_expect_tx(full_bar(s), L::STAGE_BYTES);
            tma_load_2d(a_dst, &tmA, kb * BK, arow, full_bar(s));
            tma_load_2d(b_dst, &tmB, kb * BK, brow, full_bar(s));
          }
        }
      }
      if (!ok && issuer) {
        // let the copies already issued land before the CTA's shared memory is released
        // (the second CTA of a pair gives up only after a full wait limit without
        // progress, long after its last copies landed)
        const uint32_t first = it > STAGES ? it - STAGES : 0;
        for (uint32_t i = first; i < it; ++i)
          mbar_drain(full_bar(i % STAGES), (i / STAGES) & 1, wait_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // One thread waits for stage s (full) and TMEM buffer b (released by the promotion
    // warps), then issues the K block's four MMAs and the commits.  Waiting here directly
    // takes a hop out of the buffer round trip that sets the pace: a separate waiting
    // warp releasing this one through a named barrier measured ~450 cycles slower per
    // round trip on this B300.
    if (issuer && lane == 0) {
      constexpr uint32_t idesc = make_idesc(BM, BN, 0u, 0u);   // E4M3 x E4M3 -> F32
      uint32_t it = 0;
      bool ok = true;
      for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          const int b = it % TBUF;
          const uint32_t bph = (it / TBUF) & 1;
          // (failure-path test: a barrier nothing arrives on)
          if (!((!p.stall || mbar_wait(stall_bar, 0, abort_flag, p.status, wait_ns)) &&
                mbar_wait<PAIR>(full_bar(s), ph, abort_flag, p.status, wait_ns) &&
                mbar_wait<PAIR>(tempty_bar(b), bph ^ 1, abort_flag, p.status, wait_ns))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(sbase + L::OFF_A + s * A_BYTES);
          const uint64_t bdesc = smem_desc_sw128(sbase + L::OFF_B + s * L::B_BYTES);
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)   // K = 32 bytes per MMA: +2 in the >>4 address
            mma_fp8_g<PAIR>(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
          if (PAIR) {
            mma_commit_g<true>(mapa_shared(empty_bar(s), 0));
            mma_commit_g<true>(mapa_shared(empty_bar(s), 1));
            mma_commit_g<true>(mapa_shared(tfull_bar(b), 0));
            mma_commit_g<true>(mapa_shared(tfull_bar(b), 1));
          } else {
            mma_commit(empty_bar(s));
            mma_commit(tfull_bar(b));
          }
        }
      }
      // every MMA issued so far must finish before TMEM is released
      mma_commit_g<PAIR>(drain_bar);
      mbar_drain(drain_bar, 0, wait_ns);
    }
    __syncwarp();
  } else if (warp >= 2 && warp < 2 + EPI_WARPS) {
    // ---------------- promotion + epilogue ----------------
    const int grp = (warp - 2) >> 2;    // column half of the tile
    const int q = warp & 3;             // TMEM lane window
    const int row = q * 32 + lane;      // row within this CTA's 128 rows
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    const int NB = p.N / 128;           // weight-scale rows per segment
    // the arrival that releases a TMEM buffer goes to the MMA-issuing CTA
    const uint32_t tempty_dst[TBUF] = {PAIR ? mapa_shared(tempty_bar(0), 0) : tempty_bar(0),
                                       PAIR ? mapa_shared(tempty_bar(1), 0) : tempty_bar(1)};
    // TMEM columns of this thread's eight 16-column chunks, from its half's first column
    // (SwiGLU: 4 gate then 4 up)
    auto col_of = [](int c) {
      return static_cast<uint32_t>((SWIGLU) ? (c < 4 ? 0 : 64) + (c & 3) * 16 : c * 16);
    };
    // Scales: every K block needs sA[kb][row] (this thread's row) and the one or two
    // weight scales of the tile's N blocks.  They are loaded from global memory into
    // registers one K block ahead: the loads for K block it + 1 are issued before the wait
    // for K block it, so a K block of waiting and folding covers most of their latency.
    // (The weight scales are the same address in every lane: one broadcast load.)
    auto load_scales = [&](int g_, int m0_, int nt_, int kb_, float& a, float& b0, float& b1) {
      const int nb0 = (SWIGLU) ? 2 * nt_ : min(2 * nt_ + grp, NB - 1);
      const int nb1 = (SWIGLU) ? 2 * nt_ + 1 : nb0;
      const int arow = min(m0_ + row_off + row, p.M - 1);
      a = __ldg(p.sA + static_cast<long long>(kb_) * p.M + arow);
      const float* sb = p.sB + static_cast<long long>(g_) * NB * KB + kb_;
      b0 = __ldg(sb + static_cast<long long>(nb0) * KB);
      b1 = __ldg(sb + static_cast<long long>(nb1) * KB);
    };
    float csa = 1.0f, csb0 = 1.0f, csb1 = 1.0f;          // scales of the current K block
    if (first_unit < total) {
      int g, m0, nt;
      decode_unit<BM>(first_unit, ustart, seg, G, g, m0, nt);
      load_scales(g, m0, nt, 0, csa, csb0, csb1);
    }

    uint32_t it = 0;
    uint32_t xch = 0;                                    // row max-abs exchanges so far
    bool ok = true;
    for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
      int g, m0, nt;
      decode_unit<BM>(unit, ustart, seg, G, g, m0, nt);
      const int r0 = m0 + row_off;                       // first row of this CTA's part
      const int rv = min(ROWS, seg[g + 1] - r0);         // its valid rows (may be <= 0)
      float2 acc2[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc2[i] = make_float2(0.0f, 0.0f);
      for (int kb = 0; kb < KB; ++kb, ++it) {
        float nsa = 1.0f, nsb0 = 1.0f, nsb1 = 1.0f;
        if (kb + 1 < KB) {
          load_scales(g, m0, nt, kb + 1, nsa, nsb0, nsb1);
        } else if (unit + unit_stride < total) {         // the next unit's first K block
          int ng, nm0, nnt;
          decode_unit<BM>(unit + unit_stride, ustart, seg, G, ng, nm0, nnt);
          load_scales(ng, nm0, nnt, 0, nsa, nsb0, nsb1);
        }
        const int b = it % TBUF;
        const uint32_t bph = (it / TBUF) & 1;
        if (!mbar_wait_warp<PAIR>(tfull_bar(b), bph, abort_flag, p.status, wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float sc0 = __fmul_rn(csa, csb0);
        const float sc1 = __fmul_rn(csa, csb1);
        const uint32_t tb = tmem_base + lane_addr + static_cast<uint32_t>(b * BN + grp * 128);
        // four 16-column loads in flight per wait: two TMEM round trips per K block
        // (chunks 0-3 take the first N block's scale, 4-7 the second's)
#pragma unroll
        for (int c = 0; c < 8; c += 4) {
          uint32_t v[4][16];
#pragma unroll
          for (int h = 0; h < 4; ++h) tmem_ld_32x32b_x16(tb + col_of(c + h), v[h]);
          const float sc = (c < 4) ? sc0 : sc1;
          const float2 sc2 = make_float2(sc, sc);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 4; ++h)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              acc2[(c + h) * 8 + i] = __ffma2_rn(
                  sc2,
                  make_float2(__uint_as_float(v[h][2 * i]), __uint_as_float(v[h][2 * i + 1])),
                  acc2[(c + h) * 8 + i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {                                 // the buffer is folded in
          if (PAIR) mbar_arrive_cluster(tempty_dst[b]);
          else mbar_arrive(tempty_dst[b]);
        }
        csa = nsa;
        csb0 = nsb0;
        csb1 = nsb1;
      }
      if (!ok) break;
      float* acc = reinterpret_cast<float*>(acc2);

      if (EPI == kEpiBF16) {
        if (row < rv && nt * BN + grp * 128 < p.N) {
          uint16_t* crow = p.C + static_cast<long long>(r0 + row) * p.ldc + nt * BN + grp * 128;
          // a row's 128 values leave as 32-byte stores when C and its row pitch allow
          // (a warp's store instruction covers 32 rows, one sector each), else 16-byte
          if (((reinterpret_cast<uintptr_t>(p.C) | static_cast<uintptr_t>(p.ldc) * 2) & 31) == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float* v = acc + 16 * j;
              st_global_v8(crow + 16 * j, pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                           pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]),
                           pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]),
                           pack_bf16x2(v[12], v[13]), pack_bf16x2(v[14], v[15]));
            }
          } else {
            uint4* dst = reinterpret_cast<uint4*>(crow);
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
        }
      } else {
        const int f = p.N / 2;
        // The two threads of a row (column halves grp 0 and 1) exchange row max-abs values
        // through shared memory; exchange xch uses buffer xch & 1.
        auto exchange = [&](float v0, float v1, float& m0, float& m1) {
          float* ax = amax_x + (xch & 1) * 3 * 2 * ROWS;  // [value][half][row]
          ax[grp * ROWS + row] = v0;
          ax[(2 + grp) * ROWS + row] = v1;
          mbar_arrive(amax_bar(xch & 1));
          const bool okx =
              mbar_wait_warp(amax_bar(xch & 1), (xch >> 1) & 1, abort_flag, p.status, wait_ns);
          m0 = fmaxf(v0, ax[(grp ^ 1) * ROWS + row]);
          m1 = fmaxf(v1, ax[(2 + (grp ^ 1)) * ROWS + row]);
          ++xch;
          return okx;
        };
        if (CACHE) {
          // training forward: the SwiGLU inputs g, u (gate and up columns of this row) are
          // kept in FP8 for the backward, one 1x128 scale per 128 hidden columns
          float ag = 0.0f, au = 0.0f;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            ag = fmaxf(ag, fabsf(acc[i]));
            au = fmaxf(au, fabsf(acc[64 + i]));
          }
          if (!exchange(ag, au, ag, au)) { ok = false; break; }
          const float sg = e4m3_scale_from_amax(ag), su = e4m3_scale_from_amax(au);
          if (row < rv) {
            uint8_t* gr = p.guq + static_cast<long long>(r0 + row) * p.N + nt * 128 + grp * 64;
            uint4* gd = reinterpret_cast<uint4*>(gr);
            uint4* ud = reinterpret_cast<uint4*>(gr + f);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float* gv = acc + 16 * j;
              const float* uv = acc + 64 + 16 * j;
              gd[j] = make_uint4(e4m3x4_div(gv, sg), e4m3x4_div(gv + 4, sg),
                                 e4m3x4_div(gv + 8, sg), e4m3x4_div(gv + 12, sg));
              ud[j] = make_uint4(e4m3x4_div(uv, su), e4m3x4_div(uv + 4, su),
                                 e4m3x4_div(uv + 8, su), e4m3x4_div(uv + 12, su));
            }
            if (grp == 0) {
              p.sgu[static_cast<long long>(nt) * p.M + r0 + row] = sg;
              p.sgu[static_cast<long long>(f / 128 + nt) * p.M + r0 + row] = su;
            }
          }
        }
        // h = silu(gate) * up for this thread's 64 hidden columns
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          acc[i] = __fmul_rn(silu_f32(acc[i]), acc[64 + i]);
          amax = fmaxf(amax, fabsf(acc[i]));
        }
        float unused;
        if (!exchange(amax, 0.0f, amax, unused)) { ok = false; break; }
        const float s = e4m3_scale_from_amax(amax);
        const float rs = __frcp_rn(s);
        if (row < rv) {
          uint4* dst = reinterpret_cast<uint4*>(p.hq + static_cast<long long>(r0 + row) * f +
                                                nt * 128 + grp * 64);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float* h = acc + 16 * j;
            dst[j] = make_uint4(e4m3x4(h[0], h[1], h[2], h[3], rs),
                                e4m3x4(h[4], h[5], h[6], h[7], rs),
                                e4m3x4(h[8], h[9], h[10], h[11], rs),
                                e4m3x4(h[12], h[13], h[14], h[15], rs));
          }
          if (grp == 0) p.sh[static_cast<long long>(nt) * p.M + r0 + row] = s;
        }
      }
    }
  }

  tc_fence_before();
  if (PAIR) cluster_sync();   // neither CTA leaves while the other may still signal it
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_g<PAIR>(tmem_base, TMEM_COLS);
  }
}

// ---- host side ------------------------------------------------------------------------

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* ptr,
                    uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                    uint32_t box_outer);   // runtime.cu

namespace {

std::atomic<int> g_tiling{0};   // moe_set_gemm_tiling

// Resident CTA pairs of the pair-tiled kernel on the current device (cached per device).
template <int EPI>
int max_pairs() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms() / 2;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms() / 2 * 2), 1, 1);
    cfg.blockDim = dim3(gk::THREADS, 1, 1);
    cfg.dynamicSmemBytes = gk::Layout<true>::SMEM_ALLOC;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_kernel<EPI, true>, &cfg) != cudaSuccess ||
        n <= 0) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

template <int EPI, bool PAIR>
int launch_gemm_kernel(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p,
                       long long units, cudaStream_t stream) {
  constexpr int smem = gk::Layout<PAIR>::SMEM_ALLOC;
  auto kern = fp8_gemm_kernel<EPI, PAIR>;
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(kern), smem) != MOE_OK)
    return MOE_ERR_CUDA;
  if (!PAIR) {
    long long grid = num_sms();                    // persistent: one CTA per SM
    if (units < grid) grid = units;
    if (grid < 1) grid = 1;
    kern<<<static_cast<unsigned>(grid), gk::THREADS, smem, stream>>>(tmA, tmB, p);
    return check_launch();
  }
  long long pairs = max_pairs<EPI>();
  if (units < pairs) pairs = units;
  if (pairs < 1) pairs = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.blockDim = dim3(gk::THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p) != cudaSuccess) return MOE_ERR_CUDA;
  return check_launch();
}

template <bool PAIR>
int launch_tiling(const GemmArgs& a, GemmEpilogue epi, const GemmParams& p,
                  cudaStream_t stream) {
  using namespace gk;
  using L = Layout<PAIR>;
  CUtensorMap tmA, tmB;
  if (!encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A, a.K, a.M, a.K, BK, ROWS))
    return MOE_ERR_CUDA;
  if (!encode_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B,
                      a.K, static_cast<uint64_t>(a.G) * a.N, a.K, BK, L::B_ROWS))
    return MOE_ERR_CUDA;
  // an upper bound of the work units (each segment adds at most one partial M block)
  const long long units = (static_cast<long long>(a.M) / L::BM + a.G) * ((a.N + BN - 1) / BN);
  if (epi == kEpiSwiGLU) return launch_gemm_kernel<kEpiSwiGLU, PAIR>(tmA, tmB, p, units, stream);
  if (epi == kEpiSwiGLUCache)
    return launch_gemm_kernel<kEpiSwiGLUCache, PAIR>(tmA, tmB, p, units, stream);
  return launch_gemm_kernel<kEpiBF16, PAIR>(tmA, tmB, p, units, stream);
}

}  // namespace

void set_gemm_tiling(int mode) { g_tiling.store(mode); }
int gemm_tiling() { return g_tiling.load(); }

int launch_fp8_gemm(const GemmArgs& a, GemmEpilogue epi, cudaStream_t stream) {
  using namespace gk;
  if (a.M == 0) return MOE_OK;
  if (a.N % 128 != 0 || (epi != kEpiBF16 && a.N % BN != 0)) return MOE_ERR_UNSUPPORTED;
  if (epi == kEpiSwiGLUCache && (!a.guq || !a.sgu)) return MOE_ERR_INVALID_ARG;
  GemmParams p;
  p.sA = a.sA; p.sB = a.sB; p.seg = a.seg;
  p.G = a.G; p.M = a.M; p.N = a.N; p.K = a.K;
  p.C = a.C; p.ldc = a.ldc; p.hq = a.hq; p.sh = a.sh; p.status = a.status;
  p.guq = a.guq; p.sgu = a.sgu;
  p.wait_ns = a.wait_ns ? a.wait_ns : kWaitLimitNs;
  p.stall = a.stall;
  // Automatic choice: the single tiling.  With the buffer round trip bound by the
  // promotion's TMEM reads, the pair tiling's smaller B loads buy nothing and its
  // cross-CTA release costs time: measured on this B300, single beats pair on the five
  // dense sweep shapes (by 2-15%) and on the skewed MoE layer.  The pair stays selectable.
  const int mode = g_tiling.load();
  // segments of a few rows (decode batches): weight rows on the MMA's M side
  const bool swap_ok = a.N % 256 == 0 && epi != kEpiSwiGLUCache;
  if (swap_ok && (mode == 3 || (mode == 0 && static_cast<long long>(a.M) <= 16LL * a.G)))
    return launch_fp8_gemm_swap(a, epi, false, stream);
  const bool pair = mode == 2;
  return pair ? launch_tiling<true>(a, epi, p, stream) : launch_tiling<false>(a, epi, p, stream);
}

}  // namespace moe
