// MX-native variant of the grouped FP8 GEMM: the block scales are applied by the tensor
// core itself (tcgen05.mma kind::mxf8f6f4 with UE8M0 scale factors), so the FP32
// accumulator stays in TMEM for the whole K loop and there is no per-K-block
// promotion round trip.
//
//   C[r][n] = sum_kb sA[kb][r] * sB[g][n/128][kb] * P_kb[r][n]      (same formula as the
//                                                                    FP32-scale GEMM)
// with every scale a power of two.  The pages note that V3's 1x128 / 128x128 groups match
// the microscaling formats Blackwell tensor cores take natively ("DeepSeek-V3" summary,
// core idea 6(a)) and ask for native group-scaled MMA (core idea 8, hardware wishlist).
// The hardware scale block is 32 deep along K, so the four 32-deep steps of a 128-deep
// block read the same scale.
//
// Kernel shape (one CTA per SM, persistent):
//   warp 0       TMA producer: A tile 128x128 and B tile 256x128 (FP8) per K block
//   warp 1       TMEM allocation; one thread issues 4 block-scaled MMAs (M128 N256 K32)
//                per K block into the one accumulator; never touches shared memory in
//                its loop (a named barrier with the scheduler releases it)
//   warps 2-5    scale writers: per K block, the exponent bytes of the tile's 128 row
//                scales and 256 column scales go into a ring of TMEM scale slots
//                (tcgen05.st; one warp per TMEM lane quarter, all four write the same
//                words, so each quarter holds a full copy)
//   warps 6-13   epilogue: TMEM accumulator -> BF16 C, then release the accumulator
//   warp 14      scheduler: waits for the stage, the scale slot and (at a tile's first
//                K block) the accumulator, then releases warp 1
// TMEM: columns [0, 256) accumulator; scale slot j at 256 + 16 j: 4 columns of row scales
// (word (lane l, column c) = rows l % 32 + 32 c, the byte repeated for the four 32-deep
// steps), then 8 columns of column scales laid out the same way for 256 B rows.
//
// kEpiF32 is the Wgrad of the expert backward ("DeepSeek-V3" book, ch. 17 "One linear layer
// creates three GEMMs"; ch. 16 "Why transposition is not trivial"): the contraction runs
// over token rows, so both operands arrive transposed, K-major over each expert's rows
// padded to 128-row blocks, with one power-of-two scale per (row block, output row) and
// per (row block, output column) -- the 128x1 regrouping.  A unit is (expert, 128-row
// tile, 256-column tile) and its K loop covers that expert's row blocks only; an expert
// without rows gets zeros.  The block scales of B vary per column, which the tensor
// core's per-column scale factors take directly.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace mx {
constexpr int BK = 128;
constexpr int SF_SLOTS = 4;
constexpr int SF_WARP0 = 2, SF_WARPS = 4;
constexpr int EPI_WARP0 = 6, EPI_WARPS = 8;
constexpr int SCHED_WARP = 14;
constexpr int THREADS = 15 * 32;
constexpr int MMA_BAR = 1;
constexpr int EPI_BAR = 2;                          // named barrier of the 8 epilogue warps
constexpr int MAX_G = 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_SLOT_COLS = 16;

// Tile shapes.  Single: one 128 x 256 accumulator per CTA (the SwiGLU epilogue needs the
// 256-column gate/up pairing).  Pair: two 128-row sub-tiles of one 256-row block share
// each B tile (two MMAs per K step, two 128 x 224 accumulators): 60 KB per K block for
// twice the MMA work of the single tile's 48 KB, so fewer bytes ride the shared-memory
// ring per multiply-add -- the ring is what bounds these kernels.
template <bool PAIR, bool F32OUT = false>
struct Tile {
  static constexpr int BM = PAIR ? 256 : 128;       // rows per CTA tile
  static constexpr int BN = PAIR ? 224 : 256;       // columns per accumulator
  // FP32 output (Wgrad): short K loops, so 3 stages, and room for the store staging
  static constexpr int STAGES = (PAIR || F32OUT) ? 3 : 4;
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // TMEM: accumulators at [0, (PAIR ? 2 : 1) * BN); scale slots after them, 16 columns
  // each: row scales of sub-tile 0 (4 columns), [of sub-tile 1 (4)], column scales (8)
  static constexpr uint32_t SF_COL0 = (PAIR ? 2 : 1) * BN;
  static constexpr uint32_t SFA1_OFF = 4;
  static constexpr uint32_t SFB_OFF = PAIR ? 8 : 4;
  static_assert(SF_COL0 + SF_SLOTS * SF_SLOT_COLS <= TMEM_COLS, "TMEM budget");
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
  // full[STAGES], empty[STAGES], sf_full[SF_SLOTS], sf_empty[SF_SLOTS], tfull, tempty, drain
  static constexpr int NUM_BARS = 2 * STAGES + 2 * SF_SLOTS + 3;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;   // tmem slot, abort, total, bad
  static constexpr int OFF_SEG = OFF_MISC + 16;
  static constexpr int OFF_USTART = OFF_SEG + (MAX_G + 1) * 4;
  static constexpr int OFF_WSUM = OFF_USTART + (MAX_G + 1) * 4;
  static constexpr int OFF_AMAX = OFF_WSUM + 32 * 4;         // [2 tiles][2 halves][128 rows]
  // FP32 output: per epilogue warp two 4 KB boxes (32 rows x 32 floats, 128-byte swizzle)
  // that TMA stores write out; 1024-byte aligned like the swizzle atom
  static constexpr int STG_BOX = 32 * 32 * 4;
  static constexpr int OFF_STG = (OFF_AMAX + 2 * 2 * 128 * 4 + 1023) & ~1023;
  static constexpr int SMEM_USED = OFF_STG + (F32OUT ? EPI_WARPS * 2 * STG_BOX : 0);
  static constexpr int SMEM_ALLOC = SMEM_USED + 1024;
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
};

// Instruction descriptor of a block-scaled MMA (kind::mxf8f6f4; D is FP32): bits [4,6)
// scale byte of B, [7,10) A type, [10,13) B type (0 = E4M3), [17,23) N >> 3, bit 23 scale
// type (1 = UE8M0), [24,29) M >> 4, [29,31) scale byte of A.  The scale byte picks one of
// the four bytes of each 32-bit scale word in TMEM.
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, uint32_t a_byte, uint32_t b_byte) {
  return (b_byte << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) | (a_byte << 29);
}
}  // namespace mx

struct MxParams {
  const float* sA;
  const float* sB;
  const int32_t* seg;
  int G, M, N, K;
  uint16_t* C;
  int ldc;
  uint8_t* hq;           // SwiGLU epilogue: [M][N/2] E4M3
  float* sh;             // SwiGLU epilogue: [N/256][M] power-of-two scales
  float* Cf;             // F32 epilogue (Wgrad): [G][M][ldc]
  int32_t* status;
};

namespace {

MOE_DEV void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                    uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

MOE_DEV void tmem_st_x4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}

MOE_DEV void tmem_st_x8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
               "r"(r[7])
               : "memory");
}

MOE_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2-D tiled store of one shared-memory box (bulk async-group completion); x, y >= 0.
MOE_DEV void tma_store_2d(const void* tmap, uint32_t src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}

MOE_DEV void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read their shared-memory source.
template <int N>
MOE_DEV void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N of this thread's bulk groups are still in flight.
template <int N>
MOE_DEV void bulk_wait_group() { asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory"); }


// A power-of-two FP32 scale as a UE8M0 byte repeated four times (one per 32-deep step).
// Anything else (zero, subnormal, inf/NaN, a mantissa bit set) is a data error.
MOE_DEV uint32_t ue8m0_word(float s, bool& bad) {
  const uint32_t b = __float_as_uint(s);
  const uint32_t e = (b >> 23) & 0xFFu;
  if ((b & 0x807FFFFFu) != 0 || e == 0 || e == 0xFFu) bad = true;
  return e * 0x01010101u;
}

MOE_DEV float silu_mx(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

template <int BM>
MOE_DEV void decode_unit(int unit, const int* ustart, const int* seg, int G, int& g, int& m0,
                         int& rows_valid, int& nt) {
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
  m0 = seg[g] + (local % mt) * BM;
  nt = local / mt;
  rows_valid = min(BM, seg[g + 1] - m0);
}

MOE_DEV void mbar_drain_mx(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

}  // namespace

template <int EPI, bool PAIR>
__global__ void __launch_bounds__(mx::THREADS, 1)
    fp8_mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmC, const MxParams p) {
  using namespace mx;
  using TL = Tile<PAIR, EPI == kEpiF32>;
  constexpr int BM = TL::BM, BN = TL::BN, STAGES = TL::STAGES;
  constexpr int A_BYTES = TL::A_BYTES, B_BYTES = TL::B_BYTES, STAGE_BYTES = TL::STAGE_BYTES;
  constexpr int OFF_A = TL::OFF_A, OFF_B = TL::OFF_B, OFF_BAR = TL::OFF_BAR;
  constexpr int OFF_MISC = TL::OFF_MISC, OFF_SEG = TL::OFF_SEG, OFF_USTART = TL::OFF_USTART;
  constexpr int OFF_WSUM = TL::OFF_WSUM, OFF_AMAX = TL::OFF_AMAX;
  constexpr uint32_t SF_COL0 = TL::SF_COL0, SFB_OFF = TL::SFB_OFF, SFA1_OFF = TL::SFA1_OFF;
  static_assert(!PAIR || EPI == kEpiBF16, "the paired tile has the BF16 epilogue only");
  constexpr bool WG = EPI == kEpiF32;        // Wgrad: per-expert K ranges, column scales
  extern __shared__ uint8_t mx_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(mx_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto sf_full_bar = [&](int j) { return bar0 + 8u * (2 * STAGES + j); };
  auto sf_empty_bar = [&](int j) { return bar0 + 8u * (2 * STAGES + SF_SLOTS + j); };
  const uint32_t tfull_bar = bar0 + 8u * (2 * STAGES + 2 * SF_SLOTS);
  const uint32_t tempty_bar = tfull_bar + 8u;
  const uint32_t drain_bar = tfull_bar + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  int* total_units = reinterpret_cast<int*>(smem + OFF_MISC + 8);
  int* bad = reinterpret_cast<int*>(smem + OFF_MISC + 12);
  int* seg = reinterpret_cast<int*>(smem + OFF_SEG);
  int* ustart = reinterpret_cast<int*>(smem + OFF_USTART);
  int* wsum = reinterpret_cast<int*>(smem + OFF_WSUM);
  float* amax_x = reinterpret_cast<float*>(smem + OFF_AMAX);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G;
  const int NT = (p.N + BN - 1) / BN;        // N tiles (the last may be half-filled)
  const int NB = p.N / 128;                  // weight-scale rows per segment
  const int KB = p.K / BK;
  const int MT = p.M / 128;                  // Wgrad: row tiles per expert

  // ---- segment table and unit prefix ----
  if (tid == 0) { *abort_flag = 0; *bad = 0; }
  for (int i = tid; i <= G; i += THREADS) seg[i] = p.seg[i];
  __syncthreads();
  if (WG) {
    // padded row offsets: start at 0, non-decreasing, whole 128-row blocks, within K
    for (int g = tid; g < G; g += THREADS)
      if (seg[g + 1] < seg[g] || (seg[g + 1] & (BK - 1)) != 0) *bad = 1;
    if (tid == 0) {
      if (seg[0] != 0 || seg[G] > p.K) *bad = 1;
      *total_units = G * MT * NT;
    }
  } else {
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
  if (*bad) {
    if (tid == 0) set_status(p.status, MOE_ERR_DEVICE_DATA);
    return;
  }
  const int total = *total_units;
  // unit -> (segment g, first row m0, valid rows rv, N tile nt, first K block kb0, K blocks)
  auto unit_info = [&](int unit, int& g, int& m0, int& rv, int& nt, int& kb0, int& nkb) {
    if (WG) {
      // N tiles fastest: the CTAs running together write whole rows of dW between them
      g = unit / (MT * NT);
      const int r = unit - g * MT * NT;
      const int mt = r / NT;
      nt = r - mt * NT;
      m0 = mt * 128;
      rv = 128;
      kb0 = seg[g] / BK;
      nkb = (seg[g + 1] - seg[g]) / BK;
    } else {
      decode_unit<BM>(unit, ustart, seg, G, g, m0, rv, nt);
      kb0 = 0;
      nkb = KB;
    }
  };

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(full_bar(s), 1); mbar_init(empty_bar(s), 1); }
    for (int j = 0; j < SF_SLOTS; ++j) {
      mbar_init(sf_full_bar(j), SF_WARPS);
      mbar_init(sf_empty_bar(j), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, EPI_WARPS);
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
  const int first_unit = blockIdx.x, unit_stride = gridDim.x;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
        int g, m0, rv, nt, kb0, nkb;
        unit_info(unit, g, m0, rv, nt, kb0, nkb);
        const int brow = (WG ? 0 : g * p.N) + nt * BN;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(empty_bar(s), ph ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(full_bar(s), STAGE_BYTES);
          tma_load_2d(sbase + OFF_A + s * A_BYTES, &tmA, (kb0 + kb) * BK, m0, full_bar(s));
          tma_load_2d(sbase + OFF_B + s * B_BYTES, &tmB, (kb0 + kb) * BK, brow, full_bar(s));
        }
      }
      if (!ok) {
        const uint32_t first = it > STAGES ? it - STAGES : 0;
        for (uint32_t i = first; i < it; ++i) mbar_drain_mx(full_bar(i % STAGES), (i / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    uint32_t it = 0;
    bool ok = true;
    for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
      int nkb = KB;
      if (WG) {                      // once per tile: the expert's K range
        int g, m0, rv, nt, kb0;
        unit_info(unit, g, m0, rv, nt, kb0, nkb);
      }
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        if (named_bar_sync_or(MMA_BAR, 64, false)) { ok = false; break; }
        if (lane == 0) {
          const int s = it % STAGES;
          const int j = it % SF_SLOTS;
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(sbase + OFF_A + s * A_BYTES);
          const uint64_t bdesc = smem_desc_sw128(sbase + OFF_B + s * B_BYTES);
          const uint32_t sfa = tmem_base + SF_COL0 + j * SF_SLOT_COLS;
#pragma unroll
          for (int k = 0; k < BK / 32; ++k) {
            mma_mx(tmem_base, adesc + 2 * k, bdesc + 2 * k, idesc_mx(128, BN, k, k), sfa,
                   sfa + SFB_OFF, (kb > 0 || k > 0) ? 1u : 0u);
            if (PAIR)     // rows [128, 256): the next 16 KB of the A stage, second accumulator
              mma_mx(tmem_base + BN, adesc + ((128 * 128) >> 4) + 2 * k, bdesc + 2 * k,
                     idesc_mx(128, BN, k, k), sfa + SFA1_OFF, sfa + SFB_OFF,
                     (kb > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(empty_bar(s));
          mma_commit(sf_empty_bar(j));
          if (kb == nkb - 1) mma_commit(tfull_bar);
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      mma_commit(drain_bar);
      mbar_drain_mx(drain_bar, 0);
    }
    __syncwarp();
  } else if (warp == SCHED_WARP) {
    // ---------------- MMA scheduler ----------------
    uint32_t it = 0, tt = 0;
    bool ok = true;
    for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
      int nkb = KB;
      if (WG) {
        int g, m0, rv, nt, kb0;
        unit_info(unit, g, m0, rv, nt, kb0, nkb);
        if (nkb == 0) continue;      // no accumulator use: the epilogue writes zeros
      }
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        int good = 1;
        if (lane == 0) {
          const int s = it % STAGES;
          const int j = it % SF_SLOTS;
          good = (kb != 0 || mbar_wait(tempty_bar, (tt & 1) ^ 1, abort_flag, p.status)) &&
                 mbar_wait(sf_full_bar(j), (it / SF_SLOTS) & 1, abort_flag, p.status) &&
                 mbar_wait(full_bar(s), (it / STAGES) & 1, abort_flag, p.status);
        }
        good = __shfl_sync(0xFFFFFFFFu, good, 0);
        tc_fence_before();
        if (named_bar_sync_or(MMA_BAR, 64, good == 0)) { ok = false; break; }
      }
      ++tt;
    }
  } else if (warp >= SF_WARP0 && warp < SF_WARP0 + SF_WARPS) {
    // ---------------- scale writers ----------------
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t it = 0;
    bool ok = true, badscale = false;
    for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
      int g, m0, rv, nt, kb0, nkb;
      unit_info(unit, g, m0, rv, nt, kb0, nkb);
      const int nb0 = 2 * nt, nb1 = min(2 * nt + 1, NB - 1);
      const int n0 = nt * BN;
      const float* sbg = p.sB + (WG ? 0LL : static_cast<long long>(g) * NB * KB);
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int kbg = kb0 + kb;                   // K block in the scale arrays
        const int j = it % SF_SLOTS;
        if (!mbar_wait_warp(sf_empty_bar(j), ((it / SF_SLOTS) & 1) ^ 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t wa[4], wa1[4], wb[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int r = min(m0 + lane + 32 * c, p.M - 1);
          wa[c] = ue8m0_word(__ldg(p.sA + static_cast<long long>(kbg) * p.M + r), badscale);
          if (PAIR) {
            const int r1 = min(m0 + 128 + lane + 32 * c, p.M - 1);
            wa1[c] = ue8m0_word(__ldg(p.sA + static_cast<long long>(kbg) * p.M + r1), badscale);
          }
        }
        // B row n of the tile is row 32 c + lane of column c.
        if (WG) {
          // one scale per column (output column n0 + n) of this row block
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int n = min(n0 + 32 * c + lane, p.N - 1);
            wb[c] = ue8m0_word(__ldg(p.sB + static_cast<long long>(kbg) * p.N + n), badscale);
          }
        } else if (PAIR) {
          // 224-row tiles: a row's weight block is (n0 + n) / 128 (rows past N: any block)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int nb = min((n0 + 32 * c + lane) / 128, NB - 1);
            wb[c] = ue8m0_word(__ldg(sbg + static_cast<long long>(nb) * KB + kb), badscale);
          }
        } else {
          // Plain layout: rows [0, 128) belong to weight block 2 nt, [128, 256) to 2 nt + 1.
          // SwiGLU (gate/up interleaved in 64-row blocks): rows [0, 64) and [128, 192) are
          // gate rows (block 2 nt of the scales, which alternate gate block, up block),
          // [64, 128) and [192, 256) up rows.
          const uint32_t b0 = ue8m0_word(__ldg(sbg + static_cast<long long>(nb0) * KB + kb), badscale);
          const uint32_t b1 = ue8m0_word(__ldg(sbg + static_cast<long long>(nb1) * KB + kb), badscale);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            wb[c] = (EPI == kEpiSwiGLU ? ((c >> 1) & 1) : (c >> 2)) ? b1 : b0;
        }
        const uint32_t col = tmem_base + lane_addr + SF_COL0 + j * SF_SLOT_COLS;
        tmem_st_x4(col, wa);
        if (PAIR) tmem_st_x4(col + SFA1_OFF, wa1);
        tmem_st_x8(col + SFB_OFF, wb);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sf_full_bar(j));
      }
    }
    if (__any_sync(0xFFFFFFFFu, badscale) && lane == 0) set_status(p.status, MOE_ERR_DEVICE_DATA);
  } else if (warp >= EPI_WARP0 && warp < EPI_WARP0 + EPI_WARPS) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;
    const int grp = (warp - EPI_WARP0) >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    uint32_t tt = 0;
    for (int unit = first_unit; unit < total; unit += unit_stride) {
      int g, m0, rv, nt, kb0, nkb;
      unit_info(unit, g, m0, rv, nt, kb0, nkb);
      if (WG && nkb == 0) {
        // an expert without rows: its weight gradient is zero (no accumulator use); each
        // store instruction writes 512 contiguous bytes of one of the warp's 32 rows
        if (nt * BN + grp * 128 < p.N) {
          float* c0 = p.Cf + (static_cast<long long>(g) * p.M + m0 + q * 32) * p.ldc + nt * BN +
                      grp * 128 + lane * 4;
#pragma unroll 8
          for (int r = 0; r < 32; ++r)
            *reinterpret_cast<float4*>(c0 + static_cast<long long>(r) * p.ldc) =
                make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        continue;
      }
      const bool good = mbar_wait_warp(tfull_bar, tt & 1, abort_flag, p.status);
      // all eight warps agree before any of them uses the barrier below
      if (named_bar_sync_or(EPI_BAR, EPI_WARPS * 32, !good)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + lane_addr + static_cast<uint32_t>(grp * 128);
      if (WG) {
        // FP32 weight gradient: the warp's 32 rows x 128 columns of its half, 32 columns at
        // a time.  Each 32 x 32 box goes into shared memory (row `lane`, 16-byte chunk k at
        // position k ^ (lane & 7): the 128-byte swizzle) and leaves by a TMA store, two boxes
        // in flight per warp.  The accumulator is released as soon as it has been read, so
        // the next tile's MMAs run while the stores drain.
        const bool store = nt * BN + grp * 128 < p.N;
        const uint32_t stg = sbase + TL::OFF_STG + (warp - EPI_WARP0) * 2 * TL::STG_BOX;
        uint8_t* stg_p = smem + TL::OFF_STG + (warp - EPI_WARP0) * 2 * TL::STG_BOX;
        const int y = g * p.M + m0 + q * 32;
#pragma unroll
        for (int c = 0; c < 8; c += 2) {
          uint32_t v[2][16];
          tmem_ld_32x32b_x16(tbase + c * 16, v[0]);
          tmem_ld_32x32b_x16(tbase + c * 16 + 16, v[1]);
          const int bx = (c >> 1) & 1;
          if (lane == 0) bulk_wait_group_read<1>();   // this box's store of two rounds ago
          __syncwarp();
          tmem_ld_wait();
          if (store) {
            uint8_t* row_p = stg_p + bx * TL::STG_BOX + lane * 128;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t* w = &v[k >> 2][(k & 3) * 4];
              *reinterpret_cast<uint4*>(row_p + ((k ^ (lane & 7)) * 16)) =
                  make_uint4(w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async();                      // visible to the TMA engine
          }
          __syncwarp();
          if (store && lane == 0) {
            tma_store_2d(&tmC, stg + bx * TL::STG_BOX, nt * BN + grp * 128 + c * 16, y);
            bulk_commit_group();
          }
        }
      } else if (PAIR) {
        // sub-tile grp (rows 128 grp + row of the block), all BN columns of its accumulator
        const int trow = grp * 128 + row;
        const uint32_t abase = tmem_base + lane_addr + static_cast<uint32_t>(grp * BN);
        uint16_t* crow = p.C + static_cast<long long>(m0 + trow) * p.ldc + nt * BN;
#pragma unroll
        for (int c = 0; c < BN / 16; c += 2) {
          uint32_t v[2][16];
          tmem_ld_32x32b_x16(abase + c * 16, v[0]);
          tmem_ld_32x32b_x16(abase + c * 16 + 16, v[1]);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (trow < rv && nt * BN + (c + h) * 16 < p.N) {
              uint4* dst = reinterpret_cast<uint4*>(crow + (c + h) * 16);
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                uint4 o;
                o.x = pack_bf16x2(__uint_as_float(v[h][8 * i + 0]), __uint_as_float(v[h][8 * i + 1]));
                o.y = pack_bf16x2(__uint_as_float(v[h][8 * i + 2]), __uint_as_float(v[h][8 * i + 3]));
                o.z = pack_bf16x2(__uint_as_float(v[h][8 * i + 4]), __uint_as_float(v[h][8 * i + 5]));
                o.w = pack_bf16x2(__uint_as_float(v[h][8 * i + 6]), __uint_as_float(v[h][8 * i + 7]));
                dst[i] = o;
              }
            }
          }
        }
      } else if (EPI == kEpiBF16) {
        const int col0 = nt * BN + grp * 128;
        const bool store = row < rv && col0 < p.N;
        uint4* dst =
            reinterpret_cast<uint4*>(p.C + static_cast<long long>(m0 + row) * p.ldc + col0);
#pragma unroll
        for (int c = 0; c < 8; c += 2) {
          uint32_t v[2][16];
          tmem_ld_32x32b_x16(tbase + c * 16, v[0]);
          tmem_ld_32x32b_x16(tbase + c * 16 + 16, v[1]);
          tmem_ld_wait();
          if (store) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int i = 0; i < 2; ++i) {
                uint4 o;
                o.x = pack_bf16x2(__uint_as_float(v[h][8 * i + 0]), __uint_as_float(v[h][8 * i + 1]));
                o.y = pack_bf16x2(__uint_as_float(v[h][8 * i + 2]), __uint_as_float(v[h][8 * i + 3]));
                o.z = pack_bf16x2(__uint_as_float(v[h][8 * i + 4]), __uint_as_float(v[h][8 * i + 5]));
                o.w = pack_bf16x2(__uint_as_float(v[h][8 * i + 6]), __uint_as_float(v[h][8 * i + 7]));
                dst[(c + h) * 2 + i] = o;
              }
          }
        }
      } else {
        // SwiGLU: columns [0, 64) of this half are gate rows, [64, 128) the matching up
        // rows (64-row interleave of w13).  Pass 1 finds the row's max |h| over its 128
        // hidden columns (64 here, 64 in the partner warp of the other half); pass 2
        // reloads the accumulator, recomputes the same h and writes E4M3 codes.
        float amax = 0.0f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[2][16];
          tmem_ld_32x32b_x16(tbase + c * 16, v[0]);
          tmem_ld_32x32b_x16(tbase + 64 + c * 16, v[1]);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            amax = fmaxf(amax, fabsf(__fmul_rn(silu_mx(__uint_as_float(v[0][i])),
                                               __uint_as_float(v[1][i]))));
        }
        float* ax = amax_x + (tt & 1) * 2 * BM;
        ax[grp * BM + row] = amax;
        named_bar_sync_or(EPI_BAR, EPI_WARPS * 32, false);
        amax = fmaxf(amax, ax[(grp ^ 1) * BM + row]);
        const float sc = pow2_scale_from_amax(amax);
        const float rs = __frcp_rn(sc);                     // exact: sc is a power of two
        const bool store = row < rv;
        const int f = p.N / 2;
        uint4* dst = reinterpret_cast<uint4*>(p.hq + static_cast<long long>(m0 + row) * f +
                                              nt * 128 + grp * 64);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[2][16];
          tmem_ld_32x32b_x16(tbase + c * 16, v[0]);
          tmem_ld_32x32b_x16(tbase + 64 + c * 16, v[1]);
          tmem_ld_wait();
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float h[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              h[i] = __fmul_rn(__fmul_rn(silu_mx(__uint_as_float(v[0][4 * j + i])),
                                         __uint_as_float(v[1][4 * j + i])),
                               rs);
            w[j] = f32x2_to_e4m3x2(h[0], h[1]) | (f32x2_to_e4m3x2(h[2], h[3]) << 16);
          }
          if (store) dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (store && grp == 0) p.sh[static_cast<long long>(nt) * p.M + m0 + row] = sc;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar);
      ++tt;
    }
    if (WG && lane == 0) bulk_wait_group<0>();     // every store complete before exit
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

namespace {
template <int EPI, bool PAIR>
int launch_mx_kernel(const uint8_t* A, const uint8_t* B, const MxParams& p, cudaStream_t stream) {
  using TL = mx::Tile<PAIR, EPI == kEpiF32>;
  constexpr bool WG = EPI == kEpiF32;
  CUtensorMap tmA, tmB;
  // Wgrad: A = a^T [M][K] and B = b^T [N][K] shared by every expert; else B is [G][N][K]
  if (!encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, p.K, p.M, p.K, mx::BK, TL::BM))
    return MOE_ERR_CUDA;
  if (!encode_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, p.K,
                      static_cast<uint64_t>(WG ? 1 : p.G) * p.N, p.K, mx::BK, TL::BN))
    return MOE_ERR_CUDA;
  // Wgrad: C is FP32 [G][M][ldc], written in 32 x 32 boxes; otherwise unused (a copy of A's)
  CUtensorMap tmC = tmA;
  if (WG && !encode_tmap_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.Cf, p.ldc,
                            static_cast<uint64_t>(p.G) * p.M, static_cast<uint64_t>(p.ldc) * 4,
                            32, 32))
    return MOE_ERR_CUDA;
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(fp8_mx_gemm_kernel<EPI, PAIR>),
                           TL::SMEM_ALLOC) != MOE_OK)
    return MOE_ERR_CUDA;
  const long long units =
      WG ? static_cast<long long>(p.G) * (p.M / 128) * ((p.N + TL::BN - 1) / TL::BN)
         : (static_cast<long long>(p.M) / TL::BM + p.G) * ((p.N + TL::BN - 1) / TL::BN);
  long long grid = num_sms();
  if (units < grid) grid = units;
  if (grid < 1) grid = 1;
  fp8_mx_gemm_kernel<EPI, PAIR>
      <<<static_cast<unsigned>(grid), mx::THREADS, TL::SMEM_ALLOC, stream>>>(tmA, tmB, tmC, p);
  return check_launch();
}
}  // namespace

int launch_mx_gemm(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                   const int32_t* seg, int G, int M, int N, int K, uint16_t* C, int ldc,
                   uint8_t* hq, float* sh, GemmEpilogue epi, int32_t* status,
                   cudaStream_t stream) {
  if (M == 0) return MOE_OK;
  if (N % 128 != 0 || (epi == kEpiSwiGLU && N % 256 != 0)) return MOE_ERR_UNSUPPORTED;
  // Segments of a few rows (decode batches): the swapped-operand kernel, whose software
  // promotion with power-of-two scales is exact, like the tensor core's block scaling.
  const int mode = gemm_tiling();
  if (N % 256 == 0 && (mode == 3 || (mode == 0 && static_cast<long long>(M) <= 16LL * G))) {
    GemmArgs a{};
    a.A = A; a.sA = sA; a.B = B; a.sB = sB; a.seg = seg;
    a.G = G; a.M = M; a.N = N; a.K = K; a.C = C; a.ldc = ldc; a.hq = hq; a.sh = sh;
    a.status = status;
    return launch_fp8_gemm_swap(a, epi, true, stream);
  }
  MxParams p;
  p.sA = sA; p.sB = sB; p.seg = seg;
  p.G = G; p.M = M; p.N = N; p.K = K;
  p.C = C; p.ldc = ldc; p.hq = hq; p.sh = sh; p.Cf = nullptr; p.status = status;
  // SwiGLU: the 256-column gate/up tile.  BF16 output: two 128-row sub-tiles per CTA share
  // each B tile when segments average at least 256 rows; shorter segments would leave the
  // second sub-tile mostly empty, so they keep the single tile (measured: V3's routed
  // segments, ~140 rows on average, run 10% slower on the paired tile, dense shapes up to
  // 1.5x faster).
  if (epi == kEpiSwiGLU) return launch_mx_kernel<kEpiSwiGLU, false>(A, B, p, stream);
  if (static_cast<long long>(M) >= 256LL * G)
    return launch_mx_kernel<kEpiBF16, true>(A, B, p, stream);
  return launch_mx_kernel<kEpiBF16, false>(A, B, p, stream);
}

int launch_wgrad_gemm(const uint8_t* aT, const float* sA, const uint8_t* bT, const float* sB,
                      const int32_t* pad, int G, int I, int J, int Kcap, float* C,
                      int32_t* status, cudaStream_t stream) {
  if (I % 128 != 0 || J % 128 != 0 || Kcap % 128 != 0) return MOE_ERR_UNSUPPORTED;
  MxParams p;
  p.sA = sA; p.sB = sB; p.seg = pad;
  p.G = G; p.M = I; p.N = J; p.K = Kcap;
  p.C = nullptr; p.ldc = J; p.hq = nullptr; p.sh = nullptr; p.Cf = C; p.status = status;
  return launch_mx_kernel<kEpiF32, false>(aT, bT, p, stream);
}

}  // namespace moe
