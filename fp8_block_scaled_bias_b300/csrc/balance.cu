// Sequence-wise balance statistics of the complementary balance loss, forward only
// ("DeepSeek-V3" book, ch. 8 "Routing and Load Balancing", section "The complementary
// sequence loss"; "DeepSeek-V3" summary, core idea 2, the safety-net paragraph).
//
// For each sequence of L consecutive tokens:
//   f_i  = N_r * (number of tokens whose plain top-K affinities include expert i) / (K L)
//   P_i  = mean over the sequence of s_i / sum_j s_j
//   loss = alpha * sum_i f_i P_i
// The frequency follows the ORIGINAL affinities (top-K over all routed experts, no bias,
// no group limit), as the pages define it.
//
// Two launches, both in a fixed order so the result is deterministic:
//   partial  one block per (chunk of kBalTokens tokens, sequence): a warp per token
//            forms sum_j s_j and the token's top-K (ties to the lower index), then a
//            thread per expert adds s_i / sum_j s_j over the chunk's tokens in order;
//            per-chunk sums and counts go to the workspace
//   final    one block per sequence: a thread per expert adds its chunks in order and
//            writes f_i, P_i; the loss is a fixed-shape tree over the experts
#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {
constexpr int kBalTokens = 64;
constexpr int kBalThreads = 256;
constexpr int kBalWarps = kBalThreads / 32;

int bal_chunks(int L) { return (L + kBalTokens - 1) / kBalTokens; }

MOE_DEV float affinity(const float* scores, int aff, long long i) {
  const float z = scores[i];
  return aff ? z : __fdiv_rn(1.0f, 1.0f + expf(-z));
}

// (v, i) ranks strictly before (bv, bi): larger value, or equal value and lower index.
MOE_DEV bool ranks_before(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}
}  // namespace

size_t seq_balance_ws_bytes(int T, int E, int L) {
  if (T <= 0 || L <= 0 || E <= 0) return 0;
  const long long S = T / L;
  return static_cast<size_t>(S) * bal_chunks(L) * E * (sizeof(float) + sizeof(int32_t));
}

__global__ void __launch_bounds__(kBalThreads) balance_partial_kernel(
    const float* __restrict__ scores, int aff, int E, int K, int L, float* __restrict__ part_p,
    int32_t* __restrict__ part_n) {
  __shared__ float denom[kBalTokens];
  extern __shared__ int32_t picks[];          // [E]
  const int chunk = blockIdx.x, seq = blockIdx.y, nch = gridDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long t0 = static_cast<long long>(seq) * L + static_cast<long long>(chunk) * kBalTokens;
  const int nt = min(kBalTokens, L - chunk * kBalTokens);
  for (int e = threadIdx.x; e < E; e += blockDim.x) picks[e] = 0;
  __syncthreads();

  for (int j = warp; j < nt; j += kBalWarps) {
    const float* row = scores + (t0 + j) * E;
    // sum_j s_j: each lane adds its experts in index order, then a fixed xor tree
    float part = 0.0f;
    for (int e = lane; e < E; e += 32) part = __fadd_rn(part, affinity(row, aff, e));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part = __fadd_rn(part, __shfl_xor_sync(0xFFFFFFFFu, part, off));
    if (lane == 0) denom[j] = part;
    // plain top-K: K rounds of a warp arg-best over the experts not yet taken
    int last_i = -1;
    float last_v = INFINITY;
    for (int k = 0; k < K; ++k) {
      float bv = -INFINITY;
      int bi = -1;
      for (int e = lane; e < E; e += 32) {
        const float v = affinity(row, aff, e);
        const bool left = ranks_before(last_v, last_i, v, e);   // ranks after the last pick
        if (left && (bi < 0 || ranks_before(v, e, bv, bi))) { bv = v; bi = e; }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
        if (oi >= 0 && (bi < 0 || ranks_before(ov, oi, bv, bi))) { bv = ov; bi = oi; }
      }
      if (bi < 0) break;
      if (lane == 0) atomicAdd(&picks[bi], 1);                  // integer: order-free
      last_v = bv;
      last_i = bi;
    }
  }
  __syncthreads();
  const long long slot = (static_cast<long long>(seq) * nch + chunk) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.0f;
    for (int j = 0; j < nt; ++j)                                // token order
      acc = __fadd_rn(acc, __fdiv_rn(affinity(scores + (t0 + j) * E, aff, e), denom[j]));
    part_p[slot + e] = acc;
    part_n[slot + e] = picks[e];
  }
}

__global__ void __launch_bounds__(kBalThreads) balance_final_kernel(
    const float* __restrict__ part_p, const int32_t* __restrict__ part_n, int E, int K, int L,
    int nch, float alpha, float* __restrict__ f, float* __restrict__ P,
    float* __restrict__ loss) {
  __shared__ float red[kBalThreads];
  const int seq = blockIdx.x;
  float mine = 0.0f;                          // this thread's experts, in index order
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.0f;
    long long n = 0;
    for (int c = 0; c < nch; ++c) {
      const long long slot = (static_cast<long long>(seq) * nch + c) * E + e;
      acc = __fadd_rn(acc, part_p[slot]);
      n += part_n[slot];
    }
    const float fe = __fdiv_rn(static_cast<float>(n * E), static_cast<float>(K) * L);
    const float pe = __fdiv_rn(acc, static_cast<float>(L));
    f[static_cast<long long>(seq) * E + e] = fe;
    P[static_cast<long long>(seq) * E + e] = pe;
    mine = __fadd_rn(mine, __fmul_rn(fe, pe));
  }
  red[threadIdx.x] = mine;
  __syncthreads();
  for (int w = kBalThreads / 2; w > 0; w >>= 1) {               // fixed tree
    if (threadIdx.x < w) red[threadIdx.x] = __fadd_rn(red[threadIdx.x], red[threadIdx.x + w]);
    __syncthreads();
  }
  if (threadIdx.x == 0) loss[seq] = __fmul_rn(alpha, red[0]);
}

int launch_seq_balance(const float* scores, int aff, int T, int E, int K, int L, float alpha,
                       float* f, float* P, float* loss, void* ws, cudaStream_t stream) {
  const int S = T / L, nch = bal_chunks(L);
  float* part_p = static_cast<float*>(ws);
  int32_t* part_n = reinterpret_cast<int32_t*>(part_p + static_cast<size_t>(S) * nch * E);
  balance_partial_kernel<<<dim3(nch, S), kBalThreads, E * sizeof(int32_t), stream>>>(
      scores, aff, E, K, L, part_p, part_n);
  if (check_launch() != MOE_OK) return MOE_ERR_CUDA;
  balance_final_kernel<<<S, kBalThreads, 0, stream>>>(part_p, part_n, E, K, L, nch, alpha, f, P,
                                                      loss);
  return check_launch();
}

}  // namespace moe
