// Grouped block-scaled FP8 GEMM for short segments (decode batches), operands swapped:
//
//   D[n][r] = sum_kb sB[g][n/128][kb] * sA[kb][r] * sum_{k in kb} B[g][n][k] * A[r][k]
//
// the same result as the row-tiled kernel (C[r][n] = D[n][r]), for segments of a few rows.
// Per-expert decode batches are small, so the MoE part is memory-bound on the weights
// ("DeepSeek-V3" summary, core idea 8 on decode; the pages' hardware wishlist asks for
// transposed GEMM reads): a 128-row MMA tile of tokens would be mostly empty.  Here the
// weight rows fill the MMA's M side (two M128 halves of a 256-row weight tile) and the
// segment's tokens its N side (N = 32), so every MMA row is real and each K block moves
// 32 KB of weights against 4 KB of tokens.  Partials are promoted to FP32 every 128-deep
// K block ("DeepSeek-V3" book, ch. 16 "Periodic high-precision promotion"): the weight
// block's scale is one number per 64 or 128 weight rows (per 128-row half; per gate and up
// half-block on the gate/up interleave), the token scales one per column.
//
// Kernel shape (one CTA per SM, persistent):
//   warp 0      TMA producer: per K block the 256x128 weight tile and the 32x128 token
//               tile (rows of the segment from seg_start + 32 t), STAGES deep
//   warp 1      TMEM allocation; one thread issues 2 x 4 MMAs (M128 N32 K32) per K block
//               into TMEM buffer (kb mod 8): half h at columns (2 b + h) * 32
//   warp 10     MMA scheduler (stage full, TMEM buffer free -> named barrier with warp 1)
//   warp 11     scale feeder: per K block the 32 token scales and the 2 weight scales
//               into a shared-memory ring slot (cp.async, completion on the slot's mbarrier)
//   warps 2..9  promotion + epilogue: thread = one weight row (half (w-2)/4, TMEM lane
//               quarter w%4), 32 FP32 accumulators, one 32-column TMEM load per K block
// Epilogues: BF16 C[r][n] (a warp writes 64 contiguous bytes of one token row per store);
// SwiGLU on the 64-row gate/up interleave: the tile's 256 weight rows are gate and up rows
// of 128 hidden columns, so the up threads pass their values to the gate threads through
// shared memory, h = silu(gate) * up, and each token's 1x128 scale is the max over the
// tile's 128 hidden columns.
//
// POW2: the MX-native recipe's short segments.  Its scales are powers of two, so each
// promotion product sB * sA * partial is exact -- the scaling the tensor core's block
// scales would apply -- and h is requantised with the power-of-two rule.  A scale that is
// not a positive normal power of two is reported as MOE_ERR_DEVICE_DATA, as the MX
// kernel does.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace sw {
constexpr int BK = 128;
constexpr int WROWS = 256;                     // weight rows per tile (two M128 halves)
constexpr int TOK = 32;                        // tokens per tile (MMA N)
constexpr int W_BYTES = WROWS * BK;            // 32 KB
constexpr int T_BYTES = TOK * BK;              // 4 KB
constexpr int STAGE_BYTES = W_BYTES + T_BYTES;
constexpr int STAGES = 5;
constexpr int TBUF = 8;                        // TMEM buffers of 2 x 32 columns
constexpr int SR = 8;                          // scale ring slots
constexpr int SLOT_FLOATS = 36;                // 32 token scales, 2 weight scales, pad
constexpr int EPI_WARPS = 8;
constexpr int SCHED_WARP = 10, FEED_WARP = 11;
constexpr int THREADS = 12 * 32;
constexpr int MMA_BAR = 1, EPI_BAR = 2;
constexpr int MAX_G = 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr int OFF_W = 0;
constexpr int OFF_T = OFF_W + STAGES * W_BYTES;
constexpr int OFF_BAR = OFF_T + STAGES * T_BYTES;
// full[STAGES], empty[STAGES], tfull[TBUF], tempty[TBUF], sfull[SR], sempty[SR], drain
constexpr int NUM_BARS = 2 * STAGES + 2 * TBUF + 2 * SR + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;          // tmem slot, abort, total, bad
constexpr int OFF_SEG = OFF_MISC + 16;
constexpr int OFF_USTART = OFF_SEG + (MAX_G + 1) * 4;
constexpr int OFF_WSUM = OFF_USTART + (MAX_G + 1) * 4;
constexpr int OFF_RING = OFF_WSUM + 32 * 4;
constexpr int OFF_XCH = OFF_RING + SR * SLOT_FLOATS * 4;  // SwiGLU: up values [128][33]
constexpr int OFF_AMAX = OFF_XCH + 128 * 33 * 4;          // SwiGLU: [4 warps][32 tokens]
constexpr int SMEM_USED = OFF_AMAX + 4 * 32 * 4;
constexpr int SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory budget");
static_assert(2 * TBUF * TOK <= static_cast<int>(TMEM_COLS), "TMEM budget");
}  // namespace sw

struct SwapParams {
  const float* sA;       // [K/128][M] token scales
  const float* sB;       // [G][N/128][K/128] weight scales
  const int32_t* seg;
  int G, M, N, K;
  uint16_t* C;           // BF16: [M][ldc]
  int ldc;
  uint8_t* hq;           // SwiGLU: [M][N/2] E4M3
  float* sh;             // SwiGLU: [N/256][M]
  int32_t* status;
  uint64_t wait_ns;
};

namespace {

// unit -> (segment g, first token row r0, 256-row weight block wb).  Units of a segment
// run its token chunks fastest, so the chunks that share a weight tile are neighbours.
MOE_DEV void swap_unit(int unit, const int* ustart, const int* seg, int G, int NWB, int& g,
                       int& r0, int& wb) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ustart[mid] <= unit) lo = mid;
    else hi = mid - 1;
  }
  g = lo;
  const int chunks = (seg[g + 1] - seg[g] + sw::TOK - 1) / sw::TOK;
  const int local = unit - ustart[g];
  wb = local / chunks;
  r0 = seg[g] + (local % chunks) * sw::TOK;
  (void)NWB;
}

MOE_DEV void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

MOE_DEV float silu_swap(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

MOE_DEV bool is_pow2_scale(float s) {
  const uint32_t b = __float_as_uint(s), e = (b >> 23) & 0xFFu;
  return (b & 0x807FFFFFu) == 0 && e != 0 && e != 0xFFu;
}

}  // namespace

template <int EPI, bool POW2>
__global__ void __launch_bounds__(sw::THREADS, 1)
    fp8_gemm_swap_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, const SwapParams p) {
  using namespace sw;
  extern __shared__ uint8_t swap_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(swap_smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + OFF_BAR;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + TBUF + b); };
  auto sfull_bar = [&](int j) { return bar0 + 8u * (2 * STAGES + 2 * TBUF + j); };
  auto sempty_bar = [&](int j) { return bar0 + 8u * (2 * STAGES + 2 * TBUF + SR + j); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * TBUF + 2 * SR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  int* total_units = reinterpret_cast<int*>(smem + OFF_MISC + 8);
  int* bad = reinterpret_cast<int*>(smem + OFF_MISC + 12);
  int* seg = reinterpret_cast<int*>(smem + OFF_SEG);
  int* ustart = reinterpret_cast<int*>(smem + OFF_USTART);
  int* wsum = reinterpret_cast<int*>(smem + OFF_WSUM);
  float* ring = reinterpret_cast<float*>(smem + OFF_RING);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G;
  const int NWB = p.N / WROWS;              // 256-row weight blocks
  const int NB = p.N / 128;
  const int KB = p.K / BK;
  const uint64_t wait_ns = p.wait_ns;

  // ---- segment table and unit prefix: units of segment g = chunks * NWB ----
  if (tid == 0) { *abort_flag = 0; *bad = 0; }
  for (int i = tid; i <= G; i += THREADS) seg[i] = p.seg[i];
  __syncthreads();
  {
    const int per = (G + THREADS - 1) / THREADS;
    const int g0 = min(G, tid * per), g1 = min(G, g0 + per);
    int local = 0;
    for (int g = g0; g < g1; ++g) {
      const int cnt = seg[g + 1] - seg[g];
      if (cnt < 0) *bad = 1;
      local += (max(cnt, 0) + TOK - 1) / TOK * NWB;
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
      run += (max(seg[g + 1] - seg[g], 0) + TOK - 1) / TOK * NWB;
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
    for (int s = 0; s < STAGES; ++s) { mbar_init(full_bar(s), 1); mbar_init(empty_bar(s), 1); }
    for (int b = 0; b < TBUF; ++b) { mbar_init(tfull_bar(b), 1); mbar_init(tempty_bar(b), EPI_WARPS); }
    for (int j = 0; j < SR; ++j) { mbar_init(sfull_bar(j), 32); mbar_init(sempty_bar(j), EPI_WARPS); }
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
        int g, r0, wb;
        swap_unit(unit, ustart, seg, G, NWB, g, r0, wb);
        const int wrow = g * p.N + wb * WROWS;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % STAGES;
          if (!mbar_wait(empty_bar(s), ((it / STAGES) & 1) ^ 1, abort_flag, p.status, wait_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), STAGE_BYTES);
          tma_load_2d(sbase + OFF_W + s * W_BYTES, &tmB, kb * BK, wrow, full_bar(s));
          tma_load_2d(sbase + OFF_T + s * T_BYTES, &tmA, kb * BK, r0, full_bar(s));
        }
      }
      if (!ok) {
        const uint32_t first = it > STAGES ? it - STAGES : 0;
        for (uint32_t i = first; i < it; ++i)
          drain_wait(full_bar(i % STAGES), (i / STAGES) & 1, wait_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = make_idesc(128, TOK, 0u, 0u);   // E4M3 x E4M3 -> F32
    uint32_t it = 0;
    bool ok = true;
    for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
      for (int kb = 0; kb < KB; ++kb, ++it) {
        if (named_bar_sync_or(MMA_BAR, 64, false)) { ok = false; break; }
        if (lane == 0) {
          const int s = it % STAGES;
          const int b = it % TBUF;
          tc_fence_after();
          const uint64_t tdesc = smem_desc_sw128(sbase + OFF_T + s * T_BYTES);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint64_t wdesc = smem_desc_sw128(sbase + OFF_W + s * W_BYTES + h * 128 * BK);
            const uint32_t d = tmem_base + static_cast<uint32_t>((2 * b + h) * TOK);
#pragma unroll
            for (int k = 0; k < BK / 32; ++k)
              mma_f8f6f4(d, wdesc + 2 * k, tdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
          }
          mma_commit(empty_bar(s));
          mma_commit(tfull_bar(b));
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      mma_commit(drain_bar);
      drain_wait(drain_bar, 0, wait_ns);
    }
    __syncwarp();
  } else if (warp == SCHED_WARP) {
    // ---------------- MMA scheduler ----------------
    uint32_t it = 0;
    bool ok = true;
    for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
      for (int kb = 0; kb < KB; ++kb, ++it) {
        int good = 1;
        if (lane == 0) {
          const int s = it % STAGES, b = it % TBUF;
          good = mbar_wait(tempty_bar(b), ((it / TBUF) & 1) ^ 1, abort_flag, p.status, wait_ns) &&
                 mbar_wait(full_bar(s), (it / STAGES) & 1, abort_flag, p.status, wait_ns);
        }
        good = __shfl_sync(0xFFFFFFFFu, good, 0);
        tc_fence_before();
        if (named_bar_sync_or(MMA_BAR, 64, good == 0)) { ok = false; break; }
      }
    }
  } else if (warp == FEED_WARP) {
    // ---------------- scale feeder ----------------
    uint32_t it = 0;
    bool ok = true;
    for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
      int g, r0, wb;
      swap_unit(unit, ustart, seg, G, NWB, g, r0, wb);
      const int trow = min(r0 + lane, p.M - 1);
      const float* sbw = p.sB + (static_cast<long long>(g) * NB + 2 * wb) * KB;
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int j = it % SR;
        if (!mbar_wait_warp(sempty_bar(j), ((it / SR) & 1) ^ 1, abort_flag, p.status, wait_ns)) {
          ok = false;
          break;
        }
        const uint32_t dst = smem_u32(ring + j * SLOT_FLOATS);
        cp_async_4(dst + 4u * lane, p.sA + static_cast<long long>(kb) * p.M + trow);
        if (lane < 2) cp_async_4(dst + 4u * (TOK + lane), sbw + static_cast<long long>(lane) * KB + kb);
        cp_async_mbar_arrive(sfull_bar(j));
      }
    }
    cp_async_wait<0>();
  } else {
    // ---------------- promotion + epilogue (warps 2..9) ----------------
    const int h = (warp - 2) >> 2;                 // weight-row half of the tile
    const int q = warp & 3;                        // TMEM lane quarter
    const int wr = h * 128 + q * 32 + lane;        // this thread's weight row in the tile
    const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
    float* xch = reinterpret_cast<float*>(smem + OFF_XCH);
    float* amx = reinterpret_cast<float*>(smem + OFF_AMAX);
    uint32_t it = 0;
    bool ok = true, badscale = false;
    for (int unit = first_unit; ok && unit < total; unit += unit_stride) {
      int g, r0, wb;
      swap_unit(unit, ustart, seg, G, NWB, g, r0, wb);
      const int nv = min(TOK, seg[g + 1] - r0);    // valid tokens of this chunk
      float2 acc2[TOK / 2];
#pragma unroll
      for (int i = 0; i < TOK / 2; ++i) acc2[i] = make_float2(0.0f, 0.0f);
      for (int kb = 0; kb < KB; ++kb, ++it) {
        const int b = it % TBUF, j = it % SR;
        int good = 1;
        if (lane == 0)
          good = mbar_wait(sfull_bar(j), (it / SR) & 1, abort_flag, p.status, wait_ns) &&
                 mbar_wait(tfull_bar(b), (it / TBUF) & 1, abort_flag, p.status, wait_ns);
        if (!__shfl_sync(0xFFFFFFFFu, good, 0)) { ok = false; break; }
        tc_fence_after();
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + lane_addr + static_cast<uint32_t>((2 * b + h) * TOK), v);
        const float* sl = ring + j * SLOT_FLOATS;
        // weight block scale: per 128-row half for the plain layout; on the gate/up
        // interleave a half holds 64 gate rows (gate block, slot 0) and the matching 64 up
        // rows (up block, slot 1)
        const float swt = sl[TOK + (EPI == kEpiSwiGLU ? (q >> 1) : h)];
        if (POW2 && warp == 2)                      // one warp checks the slot's scales
          badscale |= !is_pow2_scale(sl[lane]) || (lane < 2 && !is_pow2_scale(sl[TOK + lane]));
        float2 sc2[TOK / 2];
#pragma unroll
        for (int i = 0; i < TOK / 4; ++i) {       // token scales x the weight scale
          const float4 s4 = reinterpret_cast<const float4*>(sl)[i];
          sc2[2 * i] = make_float2(__fmul_rn(swt, s4.x), __fmul_rn(swt, s4.y));
          sc2[2 * i + 1] = make_float2(__fmul_rn(swt, s4.z), __fmul_rn(swt, s4.w));
        }
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < TOK / 2; ++i)
          acc2[i] = __ffma2_rn(sc2[i], make_float2(__uint_as_float(v[2 * i]),
                                                   __uint_as_float(v[2 * i + 1])), acc2[i]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(tempty_bar(b));
          mbar_arrive(sempty_bar(j));
        }
      }
      // the SwiGLU epilogue's named barriers need every epilogue warp: agree first
      if (EPI == kEpiSwiGLU && named_bar_sync_or(EPI_BAR, EPI_WARPS * 32, !ok)) break;
      if (!ok) break;
      const float* acc = reinterpret_cast<const float*>(acc2);
      if (EPI == kEpiBF16) {
        // C[r0 + c][wb * 256 + wr]: for a fixed token, the warp's 32 lanes write 64
        // contiguous bytes
        uint16_t* col = p.C + static_cast<long long>(r0) * p.ldc + wb * WROWS + wr;
#pragma unroll
        for (int c = 0; c < TOK; ++c)
          if (c < nv) {
            const __nv_bfloat16 v16 = __float2bfloat16_rn(acc[c]);
            col[static_cast<long long>(c) * p.ldc] = *reinterpret_cast<const uint16_t*>(&v16);
          }
      } else {
        // SwiGLU.  Tile rows: [64 i, 64 i + 64) of half h are gate (i even) or up (i odd)
        // rows of hidden columns hc = wb * 128 + 64 h + (wr % 64); quarters 0-1 of each
        // half hold gate rows, quarters 2-3 the matching up rows.
        const bool is_gate = q < 2;
        const int hl = h * 64 + (q & 1) * 32 + lane;    // hidden column within the tile
        if (!is_gate) {
#pragma unroll
          for (int c = 0; c < TOK; ++c) xch[hl * 33 + c] = acc[c];
        }
        named_bar_sync_or(EPI_BAR, EPI_WARPS * 32, false);
        float hv[TOK];
        if (is_gate) {
          // h for this hidden column and the 32 tokens; per-token max over the gate warps
#pragma unroll
          for (int c = 0; c < TOK; ++c) {
            hv[c] = __fmul_rn(silu_swap(acc[c]), xch[hl * 33 + c]);
            float m = fabsf(hv[c]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
            if (lane == c) amx[(h * 2 + (q & 1)) * TOK + c] = m;
          }
        }
        named_bar_sync_or(EPI_BAR, EPI_WARPS * 32, false);
        if (is_gate) {
          const int f = p.N / 2;
          uint8_t* hrow = p.hq + static_cast<long long>(r0) * f + wb * 128 + hl;
#pragma unroll
          for (int c = 0; c < TOK; ++c) {
            const float amax = fmaxf(fmaxf(amx[c], amx[TOK + c]), fmaxf(amx[2 * TOK + c], amx[3 * TOK + c]));
            const float s = POW2 ? pow2_scale_from_amax(amax) : e4m3_scale_from_amax(amax);
            const float rs = __frcp_rn(s);                 // exact when s is a power of two
            if (c < nv) {
              hrow[static_cast<long long>(c) * f] =
                  static_cast<uint8_t>(f32x2_to_e4m3x2(__fmul_rn(hv[c], rs), 0.0f) & 0xFFu);
              if (hl == 0) p.sh[static_cast<long long>(wb) * p.M + r0 + c] = s;
            }
          }
        }
        named_bar_sync_or(EPI_BAR, EPI_WARPS * 32, false);   // xch / amx free again
      }
    }
    if (POW2 && __any_sync(0xFFFFFFFFu, badscale) && lane == 0)
      set_status(p.status, MOE_ERR_DEVICE_DATA);
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

int launch_fp8_gemm_swap(const GemmArgs& a, GemmEpilogue epi, bool pow2, cudaStream_t stream) {
  using namespace sw;
  if (a.M == 0) return MOE_OK;
  if (a.N % WROWS != 0 || (epi != kEpiBF16 && epi != kEpiSwiGLU)) return MOE_ERR_UNSUPPORTED;
  CUtensorMap tmA, tmB;
  if (!encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A, a.K, a.M, a.K, BK, TOK))
    return MOE_ERR_CUDA;
  if (!encode_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, a.K,
                      static_cast<uint64_t>(a.G) * a.N, a.K, BK, WROWS))
    return MOE_ERR_CUDA;
  SwapParams p;
  p.sA = a.sA; p.sB = a.sB; p.seg = a.seg;
  p.G = a.G; p.M = a.M; p.N = a.N; p.K = a.K;
  p.C = a.C; p.ldc = a.ldc; p.hq = a.hq; p.sh = a.sh; p.status = a.status;
  p.wait_ns = a.wait_ns ? a.wait_ns : kWaitLimitNs;
  const long long units = (static_cast<long long>(a.M) / TOK + a.G) * (a.N / WROWS);
  long long grid = num_sms();
  if (units < grid) grid = units;
  if (grid < 1) grid = 1;
  auto run = [&](auto kern) {
    if (set_max_dynamic_smem(reinterpret_cast<const void*>(kern), SMEM_ALLOC) != MOE_OK)
      return MOE_ERR_CUDA;
    kern<<<static_cast<unsigned>(grid), THREADS, SMEM_ALLOC, stream>>>(tmA, tmB, p);
    return check_launch();
  };
  if (epi == kEpiSwiGLU)
    return pow2 ? run(fp8_gemm_swap_kernel<kEpiSwiGLU, true>)
                : run(fp8_gemm_swap_kernel<kEpiSwiGLU, false>);
  return pow2 ? run(fp8_gemm_swap_kernel<kEpiBF16, true>)
              : run(fp8_gemm_swap_kernel<kEpiBF16, false>);
}

}  // namespace moe
