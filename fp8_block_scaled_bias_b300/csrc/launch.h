// Host-side declarations shared by the kernel files and the C-ABI layer (api.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/moe_fp8.h"

namespace moe {

// Multiprocessor count of the current device (cached per device).
int num_sms();

// Raise a kernel's dynamic shared-memory limit on the current device (once per device).
int set_max_dynamic_smem(const void* func, int bytes);

// Unique ID of the current CUDA context (runtime.cu); false when none is current.
bool current_context_id(unsigned long long* id);

// MOE_OK if the last launch succeeded, else MOE_ERR_CUDA (and clears the error).
int check_launch();

// pow2: the power-of-two scale rule of the MX-native variant instead of amax / 448.
int launch_quant_1x128(const uint16_t* x, int rows, int cols, int ldx, uint8_t* q,
                       float* scale, bool pow2, cudaStream_t stream);
// Quantise each row t of x (BF16 [T][cols], row stride ldx) once and write it to rows
// row_of[t][0..K-1] and, if shared_row_base >= 0, shared_row_base + t of q / scale.
int launch_quant_scatter_1x128(const uint16_t* x, int T, int cols, int ldx, const int32_t* row_of,
                               int K, int shared_row_base, int n_rows, uint8_t* q, float* scale,
                               bool pow2, int32_t* status, cudaStream_t stream);
int launch_quant_128x128(const float* w, int rows, int cols, uint8_t* q, float* scale,
                         bool pow2, cudaStream_t stream);



int launch_route(const float* scores, int aff, const float* bias, int T, int E, int n_groups,
                 int topk_groups, int group_topn, int K, float route_scale, int32_t* idx,
                 float* gate, cudaStream_t stream);

size_t permute_ws_bytes(int T, int K, int E);
int launch_permute(const int32_t* idx, int T, int K, int E, int include_shared,
                   int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* row_of,
                   int32_t* status, void* ws, cudaStream_t stream);

// Allocation-free permutation scratch (permute.cu): capacity in int32 and the device
// address of the static array on the current device (looked up once per device).
long long permute_noalloc_max_ints();
int permute_noalloc_scratch(int32_t** out);

int launch_combine(const uint16_t* y_rows, int n_rows, const int32_t* row_of,
                   const float* gate, int T, int K, int d, int shared_row_base, uint16_t* y,
                   int32_t* status, cudaStream_t stream);

// Sequence-wise balance statistics (balance.cu): workspace bytes and the two launches.
size_t seq_balance_ws_bytes(int T, int E, int L);
int launch_seq_balance(const float* scores, int aff, int T, int E, int K, int L, float alpha,
                       float* f, float* P, float* loss, void* ws, cudaStream_t stream);

int launch_bias_update(float* bias, const int32_t* counts, int E, int T, int K, float gamma,
                       cudaStream_t stream);

// Copy rows: dst[r] = src[rows[r]] for r < min(n_rows, *row_limit) (row_limit on the
// device; NULL = n_rows), for an FP8 matrix of `cols` columns and its 1x128 scales
// ([cols/128][src_rows] -> [cols/128][n_rows]).
int launch_gather_rows_fp8(const uint8_t* src, const float* src_scale, int src_rows,
                           const int32_t* rows, const int32_t* row_limit, int n_rows, int cols,
                           uint8_t* dst, float* dst_scale, int32_t* status,
                           cudaStream_t stream);

// Grouped block-scaled GEMM (tcgen05).  Epilogue kinds:
enum GemmEpilogue { kEpiBF16 = 0, kEpiSwiGLU = 1, kEpiF32 = 2, kEpiSwiGLUCache = 3 };
struct GemmArgs {
  const uint8_t* A;      // [M][K] rows already in segment order
  const float* sA;       // [K/128][M]
  const uint8_t* B;      // [G][N][K]
  const float* sB;       // [G][N/128][K/128]
  const int32_t* seg;    // [G+1] device
  int G, M, N, K;
  uint16_t* C;           // kEpiBF16: [M][ldc] BF16
  int ldc;
  uint8_t* hq;           // kEpiSwiGLU: [M][N/2] E4M3
  float* sh;             // kEpiSwiGLU: [N/256][M]
  uint8_t* guq;          // kEpiSwiGLU, training: g | u as E4M3 [M][N] (NULL: not cached)
  float* sgu;            // and their 1x128 scales [N/128][M]
  int32_t* status;
  uint64_t wait_ns;      // 0: the default limit of every mbarrier wait
  int stall;             // failure-path test: the MMA issuer waits on a barrier nothing arrives on
};
int launch_fp8_gemm(const GemmArgs& a, GemmEpilogue epi, cudaStream_t stream);
// Grouped GEMM for short segments with the operands swapped (gemm_swap.cu): weight rows on
// the MMA's M side, 32 tokens on N.  BF16 and SwiGLU epilogues; N % 256 == 0.  pow2: h is
// requantised with the power-of-two rule (the MX-native recipe's short segments).
int launch_fp8_gemm_swap(const GemmArgs& a, GemmEpilogue epi, bool pow2, cudaStream_t stream);
// CTA tiling of the grouped GEMM: 0 automatic, 1 one CTA per 128-row tile, 2 CTA pairs
// per 256-row tile (tcgen05 cta_group::2), 3 swapped operands for short segments.
// Process-wide.
void set_gemm_tiling(int mode);
int gemm_tiling();

// MX-native grouped GEMM (gemm_mx.cu): power-of-two block scales applied by the tensor
// core.  A rows already in segment order.  kEpiBF16 writes C; kEpiSwiGLU writes hq / sh
// (power-of-two requantisation of h).
int launch_mx_gemm(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                   const int32_t* seg, int G, int M, int N, int K, uint16_t* C, int ldc,
                   uint8_t* hq, float* sh, GemmEpilogue epi, int32_t* status,
                   cudaStream_t stream);

// Expert backward helpers (backward.cu).
int launch_seg_pad(const int32_t* seg, int G, int32_t* pad, int32_t* status, cudaStream_t stream);
// interleaved: src is the gate/up matrix with gate and up rows alternating in 64-row blocks
// (and scales alternating gate block, up block); dst columns come out gate first, then up.
int launch_transpose_fp8(const uint8_t* src, const float* s, int G, int R, int C, bool interleaved,
                         uint8_t* dst, float* sT, cudaStream_t stream);
int launch_dispatch_grad(const uint16_t* dy, const float* gate, const int32_t* row_of, int T,
                         int K, int d, int shared_row_base, int n_rows, uint16_t* dy_rows,
                         int32_t* status, cudaStream_t stream);
int launch_regroup_128x1(const uint16_t* src, int src_rows, const int32_t* rows, int C,
                         const int32_t* seg, const int32_t* pad, int G, int max_blocks, int ldq,
                         uint8_t* qT, float* sT, int32_t* status, cudaStream_t stream);
int launch_swiglu_bwd(const uint8_t* guq, const float* sgu, const uint16_t* dh, int R, int f,
                      const int32_t* seg, const int32_t* pad, int G, int max_blocks, int ldq,
                      uint8_t* dguq, float* sdgu, uint8_t* hT, float* shT, uint8_t* dguT,
                      float* sdguT, cudaStream_t stream);

// Wgrad of the expert backward (gemm_mx.cu): per expert e, C[e] [I][J] (FP32, row pitch J)
// = sum over e's 128-row blocks rb of sA[rb][i] * sB[rb][j] * sum_p aT[i][p] * bT[j][p], with
// aT [I][Kcap], bT [J][Kcap] FP8 (K-major over padded rows), power-of-two scales
// [Kcap/128][I] and [Kcap/128][J], and pad [G+1] the experts' padded row offsets (device).
int launch_wgrad_gemm(const uint8_t* aT, const float* sA, const uint8_t* bT, const float* sB,
                      const int32_t* pad, int G, int I, int J, int Kcap, float* C,
                      int32_t* status, cudaStream_t stream);

int launch_router_logits(const uint16_t* x, int T, int d, const uint16_t* w_hilo, int E,
                         float* z, int32_t* status, void* ws, cudaStream_t stream);
size_t router_logits_ws_bytes(int T, int d, int E);
int launch_router_split(const float* w, long long n, uint16_t* w_hilo, cudaStream_t stream);

}  // namespace moe
