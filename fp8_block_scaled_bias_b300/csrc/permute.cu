// Dispatch metadata: group the (token, slot) pairs into expert-contiguous segments
// ("DeepSeek-V3" book, ch. 15 "What dispatch must do" -- rows grouped by expert, with
// metadata naming the source token so combine can restore it; ch. 7 "Batches change
// what is active"; no token dropping, "DeepSeek-V3" summary, core idea 1).
//
// A stable counting sort keyed by expert, in three passes over token chunks:
//   count    per-chunk histograms
//   scan     per-expert totals, exclusive scan -> segment offsets, per-chunk bases
//   scatter  warps walk the chunk's pairs in (token, slot) order and hand out rows
// Every step is integer work in a fixed order, so the result is deterministic and equal
// to a stable sort whatever the launch timing.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {
constexpr int kChunkTokens = 128;
constexpr int kPermThreads = 256;
constexpr int kPermWarps = kPermThreads / 32;
constexpr int kScanThreads = 1024;

int n_chunks(int T) { return (T + kChunkTokens - 1) / kChunkTokens; }
}  // namespace

size_t permute_ws_bytes(int T, int K, int E) {
  (void)K;
  return static_cast<size_t>(n_chunks(T)) * E * sizeof(int32_t);
}

__global__ void __launch_bounds__(kPermThreads) permute_count_kernel(
    const int32_t* __restrict__ idx, int T, int K, int E, int32_t* __restrict__ chunk_counts,
    int32_t* status) {
  extern __shared__ int32_t hist[];
  const int c = blockIdx.x;
  const int t0 = c * kChunkTokens;
  const int np = min(kChunkTokens, T - t0) * K;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int32_t* src = idx + static_cast<long long>(t0) * K;
  for (int p = threadIdx.x; p < np; p += blockDim.x) {
    const int e = src[p];
    if (e < 0 || e >= E) set_status(status, MOE_ERR_DEVICE_DATA);
    else atomicAdd(&hist[e], 1);              // integer counts: order does not matter
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_counts[static_cast<long long>(c) * E + e] = hist[e];
}

// Block-wide exclusive scan of one value per thread (kScanThreads threads).
__device__ int block_exclusive_scan(int v, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < kScanThreads / 32) ? warp_sums[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, wi, off);
      if (lane >= off) wi += o;
    }
    warp_sums[lane] = wi - w;                  // exclusive prefix of warp totals
  }
  __syncthreads();
  return warp_sums[warp] + incl - v;
}

__global__ void __launch_bounds__(kScanThreads) permute_scan_kernel(
    int32_t* __restrict__ chunk_counts /* in: counts, out: bases */, int nchunks, int T, int K,
    int E, int include_shared, int32_t* __restrict__ counts, int32_t* __restrict__ offsets) {
  __shared__ int warp_sums[32];
  const int e = threadIdx.x;                   // E <= kScanThreads
  int total = 0;
  if (e < E) {
    for (int c = 0; c < nchunks; ++c) {
      int32_t* p = chunk_counts + static_cast<long long>(c) * E + e;
      const int n = *p;
      *p = total;                              // running base within the expert
      total += n;
    }
  }
  const int off = block_exclusive_scan(e < E ? total : 0, warp_sums);
  if (e < E) {
    counts[e] = total;
    offsets[e] = off;
    for (int c = 0; c < nchunks; ++c) chunk_counts[static_cast<long long>(c) * E + e] += off;
  }
  if (e == 0) {
    offsets[E] = T * K;
    offsets[E + 1] = T * K + (include_shared ? T : 0);
  }
}

// One block per chunk.  The chunk's pairs are split into kPermWarps contiguous runs, one
// per warp; a per-warp histogram and a prefix over the warps give each warp its first row
// in every expert segment.  Each warp then walks its run in windows of 32 pairs, in
// order: lanes holding the same expert find each other with __match_any_sync, take rows
// in lane order, and the highest such lane advances that expert's running row.  The rows
// handed out are those of a stable counting sort, independent of timing.
__global__ void __launch_bounds__(kPermThreads) permute_scatter_kernel(
    const int32_t* __restrict__ idx, int T, int K, int E, int include_shared,
    const int32_t* __restrict__ chunk_base, int32_t* __restrict__ row_token,
    int32_t* __restrict__ row_of) {
  extern __shared__ int32_t next_row[];        // [kPermWarps][E]
  const int c = blockIdx.x;
  const int t0 = c * kChunkTokens;
  const int nt = min(kChunkTokens, T - t0);
  const int np = nt * K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int run = ((np + kPermWarps - 1) / kPermWarps + 31) & ~31;
  const int p_begin = min(np, warp * run), p_end = min(np, p_begin + run);
  const int32_t* src = idx + static_cast<long long>(t0) * K;
  for (int i = threadIdx.x; i < kPermWarps * E; i += blockDim.x) next_row[i] = 0;
  __syncthreads();
  for (int p = p_begin + lane; p < p_end; p += 32) {
    const int e = src[p];
    if (e >= 0 && e < E) atomicAdd(&next_row[warp * E + e], 1);   // counts: order-free
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int row = chunk_base[static_cast<long long>(c) * E + e];
    for (int w = 0; w < kPermWarps; ++w) {
      const int n = next_row[w * E + e];
      next_row[w * E + e] = row;
      row += n;
    }
  }
  __syncthreads();
  int32_t* mine = next_row + warp * E;
  const unsigned lt = (1u << lane) - 1u;
  for (int base = p_begin; base < p_end; base += 32) {
    const int p = base + lane;
    int e = p < p_end ? src[p] : -1;
    const bool valid = e >= 0 && e < E;
    if (!valid) e = -1 - lane;                 // a key no other lane holds
    const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
    if (valid) {
      const int row = mine[e] + __popc(same & lt);
      row_of[static_cast<long long>(t0) * K + p] = row;
      row_token[row] = t0 + p / K;
    }
    __syncwarp();
    if (valid && lane == 31 - __clz(same)) mine[e] += __popc(same);
    __syncwarp();
  }
  if (include_shared) {
    const long long base = static_cast<long long>(T) * K;
    for (int i = threadIdx.x; i < nt; i += blockDim.x) row_token[base + t0 + i] = t0 + i;
  }
}

// A single chunk (T <= kChunkTokens, decode batches): the three passes in one block --
// per-warp histograms, the exclusive scan over experts (segment offsets), per-warp bases,
// then the same ordered hand-out as permute_scatter_kernel.  One launch instead of three.
__global__ void __launch_bounds__(kPermThreads) permute_single_kernel(
    const int32_t* __restrict__ idx, int T, int K, int E, int include_shared,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ row_token,
    int32_t* __restrict__ row_of, int32_t* status) {
  extern __shared__ int32_t next_row[];        // [kPermWarps][E]
  __shared__ int warp_tot[kPermWarps];
  const int np = T * K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int run = ((np + kPermWarps - 1) / kPermWarps + 31) & ~31;
  const int p_begin = min(np, warp * run), p_end = min(np, p_begin + run);
  for (int i = threadIdx.x; i < kPermWarps * E; i += blockDim.x) next_row[i] = 0;
  __syncthreads();
  for (int p = p_begin + lane; p < p_end; p += 32) {
    const int e = idx[p];
    if (e < 0 || e >= E) set_status(status, MOE_ERR_DEVICE_DATA);
    else atomicAdd(&next_row[warp * E + e], 1);   // counts: order-free
  }
  __syncthreads();
  // exclusive scan of the expert totals: thread i owns experts [i*per, i*per + per)
  const int per = (E + kPermThreads - 1) / kPermThreads;
  const int e0 = min(E, static_cast<int>(threadIdx.x) * per), e1 = min(E, e0 + per);
  int local = 0;
  for (int e = e0; e < e1; ++e)
    for (int w = 0; w < kPermWarps; ++w) local += next_row[w * E + e];
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = incl - local;
  for (int w = 0; w < warp; ++w) base += warp_tot[w];
  __syncthreads();                             // every thread has read the totals
  for (int e = e0; e < e1; ++e) {
    int row = base, n = 0;
    for (int w = 0; w < kPermWarps; ++w) {
      const int c = next_row[w * E + e];
      next_row[w * E + e] = row;               // this warp's first row in segment e
      row += c;
      n += c;
    }
    counts[e] = n;
    offsets[e] = base;
    base += n;
  }
  if (threadIdx.x == 0) {
    offsets[E] = T * K;
    offsets[E + 1] = T * K + (include_shared ? T : 0);
  }
  __syncthreads();
  int32_t* mine = next_row + warp * E;
  const unsigned lt = (1u << lane) - 1u;
  for (int b0 = p_begin; b0 < p_end; b0 += 32) {
    const int p = b0 + lane;
    int e = p < p_end ? idx[p] : -1;
    const bool valid = e >= 0 && e < E;
    if (!valid) e = -1 - lane;                 // a key no other lane holds
    const unsigned same = __match_any_sync(0xFFFFFFFFu, e);
    if (valid) {
      const int row = mine[e] + __popc(same & lt);
      row_of[p] = row;
      row_token[row] = p / K;
    }
    __syncwarp();
    if (valid && lane == 31 - __clz(same)) mine[e] += __popc(same);
    __syncwarp();
  }
  if (include_shared)
    for (int i = threadIdx.x; i < T; i += blockDim.x) row_token[static_cast<long long>(T) * K + i] = i;
}

int launch_permute(const int32_t* idx, int T, int K, int E, int include_shared,
                   int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* row_of,
                   int32_t* status, void* ws, cudaStream_t stream) {
  const int nc = n_chunks(T);
  if (nc == 1) {
    const size_t smem = static_cast<size_t>(kPermWarps) * E * sizeof(int32_t);
    permute_single_kernel<<<1, kPermThreads, smem, stream>>>(idx, T, K, E, include_shared,
                                                            counts, offsets, row_token, row_of,
                                                            status);
    return check_launch() == MOE_OK ? MOE_OK : MOE_ERR_CUDA;
  }
  int32_t* chunk = static_cast<int32_t*>(ws);
  if (nc > 0) {
    permute_count_kernel<<<nc, kPermThreads, E * sizeof(int32_t), stream>>>(idx, T, K, E, chunk,
                                                                            status);
    if (check_launch() != MOE_OK) return MOE_ERR_CUDA;
  }
  permute_scan_kernel<<<1, kScanThreads, 0, stream>>>(chunk, nc, T, K, E, include_shared, counts,
                                                       offsets);
  if (check_launch() != MOE_OK) return MOE_ERR_CUDA;
  if (nc > 0) {
    const size_t smem = static_cast<size_t>(kPermWarps) * E * sizeof(int32_t);
    permute_scatter_kernel<<<nc, kPermThreads, smem, stream>>>(idx, T, K, E, include_shared,
                                                                chunk, row_token, row_of);
    if (check_launch() != MOE_OK) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// ---- allocation-free variant -----------------------------------------------------------
//
// Scratch for moe_permute_noalloc: the per-chunk expert histograms live in this
// file-scope device array instead of caller memory.  Every GPU that loads the library
// holds it (1 MiB) until the process exits.  In host code the name is only a host-side
// stand-in, so its device address is looked up with cudaGetSymbolAddress while the
// device is current: on the first call on each device, and again whenever that device's
// CUDA context has changed since (cudaDeviceReset destroys the context that the address
// belonged to; context IDs are never reused within a process).

constexpr long long kNoAllocScratchInts = 262144;          // 1 MiB of int32
static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};
}  // namespace

long long permute_noalloc_max_ints() { return kNoAllocScratchInts; }

int permute_noalloc_scratch(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx);
  if (!g_scratch_ptr[dev] || !have_ctx || ctx != g_scratch_ctx[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_permute_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_scratch_ptr[dev] = static_cast<int32_t*>(ptr);
    // the lookup made the device's context current if none was
    g_scratch_ctx[dev] = current_context_id(&ctx) ? ctx : 0;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace moe
