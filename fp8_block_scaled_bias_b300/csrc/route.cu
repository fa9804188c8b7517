// Router: sigmoid affinities, selection bias, group limit, top-k and normalised gates
// (moe_route), and the auxiliary-loss-free bias step (moe_bias_update).
//
// "DeepSeek-V3" summary, core idea 1 (sigmoid affinities, gates normalised over the
// chosen experts, at most M groups per token scored by the sum of their top K/M
// affinities) and core idea 2 (bias added for selection only; +-gamma by load);
// "DeepSeek-V3" book, ch. 7 "The router's affinity scores", "Selecting and combining
// experts"; ch. 8 "V3's routing-only bias", "Restricting target nodes", "The feedback
// update".
//
// One warp routes one token.  Every ranking orders by (score descending, index
// ascending), so ties go to the lower index; the chosen experts are emitted in that
// order, which also fixes the order of the gate denominator sum.
#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr int kRouteWarps = 4;

// (v, i) ranks strictly before (bv, bi): larger score, or equal score and lower index.
MOE_DEV bool ranks_before(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Warp-wide arg-best over one candidate per lane; lanes with ok == false take no part.
// Every lane returns the winner (index -1 if no lane had a candidate).
MOE_DEV void warp_best(float& v, int& i, bool ok) {
  if (!ok) { v = -INFINITY; i = -1; }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xFFFFFFFFu, v, off);
    const int oi = __shfl_xor_sync(0xFFFFFFFFu, i, off);
    if (oi >= 0 && (i < 0 || ranks_before(ov, oi, v, i))) { v = ov; i = oi; }
  }
}

}  // namespace

__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(
    const float* __restrict__ scores, int aff, const float* __restrict__ bias, int T, int E,
    int n_groups, int topk_groups, int group_topn, int K, float route_scale,
    int32_t* __restrict__ idx, float* __restrict__ gate) {
  extern __shared__ float route_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouteWarps + warp;
  if (t >= T) return;                       // warp-uniform; no block barrier follows
  float* s_s = route_smem + warp * 2 * E;   // affinities
  float* c_s = s_s + E;                     // selection scores
  const int gs = E / n_groups;

  // affinities and selection scores; the row's logits and the biases are loaded 256 at a
  // time (eight per lane, all in flight together) before any arithmetic
  const float* zrow = scores + static_cast<long long>(t) * E;
  for (int e0 = 0; e0 < E; e0 += 256) {
    float zz[8], bb[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + 32 * j + lane;
      zz[j] = e < E ? __ldg(zrow + e) : 0.0f;
      bb[j] = e < E ? __ldg(bias + e) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + 32 * j + lane;
      if (e < E) {
        const float s = aff ? zz[j] : __fdiv_rn(1.0f, 1.0f + expf(-zz[j]));
        s_s[e] = s;
        c_s[e] = __fadd_rn(s, bb[j]);
      }
    }
  }
  __syncwarp();

  // group score: sum of the group_topn best selection scores, added best first
  float gscore = -INFINITY;
  if (gs == 32 && group_topn <= 2) {
    // one expert of every group per lane (expert 32 j + lane of group j): the two best of
    // each group by a butterfly over the warp, every step keeping the best two of four
    // by the same (score descending, index ascending) order
    for (int j = 0; j < n_groups; ++j) {
      float v1 = c_s[j * 32 + lane], v2 = -INFINITY;
      int i1 = lane, i2 = -1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float o1 = __shfl_xor_sync(0xFFFFFFFFu, v1, off);
        const int p1 = __shfl_xor_sync(0xFFFFFFFFu, i1, off);
        const float o2 = __shfl_xor_sync(0xFFFFFFFFu, v2, off);
        const int p2 = __shfl_xor_sync(0xFFFFFFFFu, i2, off);
        // merge two ranked pairs (v1,i1) >= (v2,i2) and (o1,p1) >= (o2,p2)
        if (ranks_before(o1, p1, v1, i1)) {
          const bool second = p2 >= 0 && ranks_before(o2, p2, v1, i1);
          v2 = second ? o2 : v1;
          i2 = second ? p2 : i1;
          v1 = o1;
          i1 = p1;
        } else if (p1 >= 0 && (i2 < 0 || ranks_before(o1, p1, v2, i2))) {
          v2 = o1;
          i2 = p1;
        }
      }
      const float g = group_topn == 1 ? v1 : __fadd_rn(v1, v2);
      if (lane == j) gscore = g;
    }
  } else if (lane < n_groups) {
    const float* g = c_s + lane * gs;
    float pv = INFINITY;
    int pi = -1;
    float acc = 0.0f;
    for (int j = 0; j < group_topn; ++j) {
      float bv = -INFINITY;
      int bi = -1;
      for (int i = 0; i < gs; ++i) {
        const float v = g[i];
        const bool after = v < pv || (v == pv && i > pi);   // not yet taken
        if (after && (bi < 0 || ranks_before(v, i, bv, bi))) { bv = v; bi = i; }
      }
      acc = (j == 0) ? bv : __fadd_rn(acc, bv);
      pv = bv;
      pi = bi;
    }
    gscore = acc;
  }

  // keep the topk_groups best groups
  uint32_t kept = 0;
  for (int j = 0; j < topk_groups; ++j) {
    float v = gscore;
    int i = lane;
    warp_best(v, i, lane < n_groups && !((kept >> lane) & 1u));
    kept |= 1u << i;
  }

  // top-K experts among the kept groups
  uint32_t picked = 0;                      // bit j: expert lane + 32 j already chosen
  int my_idx = 0;
  float my_s = 0.0f;
  for (int k = 0; k < K; ++k) {
    float bv = -INFINITY;
    int bi = -1;
    for (int j = 0, e = lane; e < E; ++j, e += 32) {
      if (((kept >> (e / gs)) & 1u) && !((picked >> j) & 1u)) {
        const float v = c_s[e];
        if (bi < 0 || ranks_before(v, e, bv, bi)) { bv = v; bi = e; }
      }
    }
    warp_best(bv, bi, bi >= 0);
    if (lane == (bi & 31)) picked |= 1u << (bi >> 5);
    if (lane == k) { my_idx = bi; my_s = s_s[bi]; }
  }

  // gates: the chosen affinities over their sum, summed in list order
  float denom = __shfl_sync(0xFFFFFFFFu, my_s, 0);
  for (int k = 1; k < K; ++k) denom = __fadd_rn(denom, __shfl_sync(0xFFFFFFFFu, my_s, k));
  if (lane < K) {
    float g = __fdiv_rn(my_s, denom);
    if (route_scale != 1.0f) g = __fmul_rn(g, route_scale);
    idx[static_cast<long long>(t) * K + lane] = my_idx;
    gate[static_cast<long long>(t) * K + lane] = g;
  }
}

// Register-resident routing for E <= 32 * NJ: lane l holds experts l + 32 j (j < NJ) and
// their affinities and selection scores in registers.  Same rankings and tie-breaks as
// route_kernel; the top-K rounds keep a per-lane best, so after each warp-wide arg-best
// only the winning lane rescans its NJ candidates.
template <int NJ>
__global__ void __launch_bounds__(kRouteWarps * 32) route_reg_kernel(
    const float* __restrict__ scores, int aff, const float* __restrict__ bias, int T, int E,
    int n_groups, int topk_groups, int group_topn, int K, float route_scale,
    int32_t* __restrict__ idx, float* __restrict__ gate) {
  extern __shared__ float route_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouteWarps + warp;
  if (t >= T) return;                       // warp-uniform; no block barrier follows
  const int gs = E / n_groups;
  const float* zrow = scores + static_cast<long long>(t) * E;

  float s[NJ], c[NJ];
  uint32_t valid = 0;
  {
    float zz[NJ], bb[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {          // all loads in flight before any arithmetic
      const int e = 32 * j + lane;
      zz[j] = e < E ? __ldg(zrow + e) : 0.0f;
      bb[j] = e < E ? __ldg(bias + e) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      s[j] = aff ? zz[j] : __fdiv_rn(1.0f, 1.0f + expf(-zz[j]));
      c[j] = __fadd_rn(s[j], bb[j]);
      if (32 * j + lane < E) valid |= 1u << j;
    }
  }

  // group score: sum of the group_topn best selection scores, added best first
  float gscore = -INFINITY;
  if (gs == 32 && group_topn <= 2) {
    // group j is register slot j: the two best of every group by butterflies over the
    // warp, all groups interleaved
    float v1[NJ], v2[NJ];
    int i1[NJ], i2[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) { v1[j] = c[j]; i1[j] = lane; v2[j] = -INFINITY; i2[j] = -1; }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        if (j >= n_groups) continue;
        const float o1 = __shfl_xor_sync(0xFFFFFFFFu, v1[j], off);
        const int p1 = __shfl_xor_sync(0xFFFFFFFFu, i1[j], off);
        const float o2 = __shfl_xor_sync(0xFFFFFFFFu, v2[j], off);
        const int p2 = __shfl_xor_sync(0xFFFFFFFFu, i2[j], off);
        // merge two ranked pairs (v1,i1) >= (v2,i2) and (o1,p1) >= (o2,p2)
        if (ranks_before(o1, p1, v1[j], i1[j])) {
          const bool second = p2 >= 0 && ranks_before(o2, p2, v1[j], i1[j]);
          v2[j] = second ? o2 : v1[j];
          i2[j] = second ? p2 : i1[j];
          v1[j] = o1;
          i1[j] = p1;
        } else if (p1 >= 0 && (i2[j] < 0 || ranks_before(o1, p1, v2[j], i2[j]))) {
          v2[j] = o1;
          i2[j] = p1;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      if (j < n_groups && lane == j) gscore = group_topn == 1 ? v1[j] : __fadd_rn(v1[j], v2[j]);
  } else {
    // any other grouping: lane g scans group g from shared memory
    float* c_s = route_smem + warp * E;
#pragma unroll
    for (int j = 0; j < NJ; ++j)
      if (32 * j + lane < E) c_s[32 * j + lane] = c[j];
    __syncwarp();
    if (lane < n_groups) {
      const float* g = c_s + lane * gs;
      float pv = INFINITY;
      int pi = -1;
      float acc = 0.0f;
      for (int j = 0; j < group_topn; ++j) {
        float bv = -INFINITY;
        int bi = -1;
        for (int i = 0; i < gs; ++i) {
          const float v = g[i];
          const bool after = v < pv || (v == pv && i > pi);   // not yet taken
          if (after && (bi < 0 || ranks_before(v, i, bv, bi))) { bv = v; bi = i; }
        }
        acc = (j == 0) ? bv : __fadd_rn(acc, bv);
        pv = bv;
        pi = bi;
      }
      gscore = acc;
    }
  }

  // keep the topk_groups best groups
  uint32_t kept = 0;
  for (int j = 0; j < topk_groups; ++j) {
    float v = gscore;
    int i = lane;
    warp_best(v, i, lane < n_groups && !((kept >> lane) & 1u));
    kept |= 1u << i;
  }

  // candidates: this lane's experts in kept groups
  uint32_t avail = 0;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int grp = gs == 32 ? j : (32 * j + lane) / gs;
    if (((valid >> j) & 1u) && ((kept >> grp) & 1u)) avail |= 1u << j;
  }
  float bv = -INFINITY;
  int bi = -1;
  auto lane_best = [&]() {
    bv = -INFINITY;
    bi = -1;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = 32 * j + lane;
      if (((avail >> j) & 1u) && (bi < 0 || ranks_before(c[j], e, bv, bi))) { bv = c[j]; bi = e; }
    }
  };
  lane_best();

  // top-K experts among the kept groups
  int my_idx = 0;
  float my_s = 0.0f;
  for (int k = 0; k < K; ++k) {
    float wv = bv;
    int wi = bi;
    warp_best(wv, wi, wi >= 0);
    float ws = 0.0f;
    if (wi >= 0 && lane == (wi & 31)) {
      const int jw = wi >> 5;
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        if (j == jw) ws = s[j];
      avail &= ~(1u << jw);
      lane_best();
    }
    ws = __shfl_sync(0xFFFFFFFFu, ws, wi & 31);
    if (lane == k) { my_idx = wi; my_s = ws; }
  }

  // gates: the chosen affinities over their sum, summed in list order
  float denom = __shfl_sync(0xFFFFFFFFu, my_s, 0);
  for (int k = 1; k < K; ++k) denom = __fadd_rn(denom, __shfl_sync(0xFFFFFFFFu, my_s, k));
  if (lane < K) {
    float g = __fdiv_rn(my_s, denom);
    if (route_scale != 1.0f) g = __fmul_rn(g, route_scale);
    idx[static_cast<long long>(t) * K + lane] = my_idx;
    gate[static_cast<long long>(t) * K + lane] = g;
  }
}

int launch_route(const float* scores, int aff, const float* bias, int T, int E, int n_groups,
                 int topk_groups, int group_topn, int K, float route_scale, int32_t* idx,
                 float* gate, cudaStream_t stream) {
  if (T == 0) return MOE_OK;
  const unsigned blocks = static_cast<unsigned>((T + kRouteWarps - 1) / kRouteWarps);
  if (E <= 256) {
    const size_t smem = static_cast<size_t>(kRouteWarps) * E * sizeof(float);
    route_reg_kernel<8><<<blocks, kRouteWarps * 32, smem, stream>>>(
        scores, aff, bias, T, E, n_groups, topk_groups, group_topn, K, route_scale, idx, gate);
    return check_launch();
  }
  const size_t smem = static_cast<size_t>(kRouteWarps) * 2 * E * sizeof(float);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  route_kernel<<<blocks, kRouteWarps * 32, smem, stream>>>(
      scores, aff, bias, T, E, n_groups, topk_groups, group_topn, K, route_scale, idx, gate);
  return check_launch();
}

// b_i <- b_i + gamma * sign(T*K/E - load_i); the sign is taken exactly in integers.
__global__ void bias_update_kernel(float* __restrict__ bias, const int32_t* __restrict__ counts,
                                   int E, long long TK, float gamma) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= E) return;
  const long long diff = TK - static_cast<long long>(E) * counts[i];
  if (diff > 0) bias[i] = __fadd_rn(bias[i], gamma);
  else if (diff < 0) bias[i] = __fsub_rn(bias[i], gamma);
}

int launch_bias_update(float* bias, const int32_t* counts, int E, int T, int K, float gamma,
                       cudaStream_t stream) {
  if (E == 0) return MOE_OK;
  bias_update_kernel<<<(E + 255) / 256, 256, 0, stream>>>(
      bias, counts, E, static_cast<long long>(T) * K, gamma);
  return check_launch();
}

}  // namespace moe
