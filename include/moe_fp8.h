/*
 * moe_fp8.h -- C-ABI of libmoe_fp8.so: the forward pass of one DeepSeek-V3 MoE FFN
 * layer with FP8 E4M3 block-scaled experts, for NVIDIA B300 (sm_103a).
 *
 * The layer, in the order the entry points run it:
 *   moe_router_logits     z = x . E^T                       (router, kept above FP8)
 *   moe_route             sigmoid, bias for selection, group limit, top-k, gates
 *   moe_permute           (token, slot) pairs -> expert-contiguous rows
 *   fp8_quant_1x128       x -> E4M3 with one FP32 scale per 1x128 tile
 *   moe_swiglu_fp8_fwd    grouped gate/up GEMM + SwiGLU + requantise, grouped down GEMM
 *   moe_combine           y_t = shared_t + sum_k g_tk * expert_out
 *   moe_bias_update       aux-loss-free bias step after the forward
 * plus moe_seq_balance_stats (statistics of the complementary sequence-wise balance
 * loss), fp8_blockscaled_grouped_gemm (the GEMM on its own, dense when G = 1) and two
 * setup helpers that prepare weights (fp8_quant_128x128, moe_router_split_bf16).
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a DEVICE pointer owned by the caller.  The library never
 *     allocates device memory; scratch space comes from the caller through (ws,
 *     ws_bytes), sized by moe_workspace_bytes() or the per-call *_ws_bytes() helpers.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream) and never synchronises the host.
 *   - Return value: MOE_OK or a negative MOE_ERR_* code for errors found on the host
 *     (arguments, launch failures).  Errors found on the device (bad indices in device
 *     data, a bounded wait that expired) are written to the caller's `dev_status`
 *     (int32 on the device, 0 = OK) where a call takes one; read it after a sync.
 *     The first device error wins; later ones do not overwrite it.
 *   - Results are deterministic: the same inputs give the same bits on every run.
 *   - FP8 is E4M3 in the finite-number convention ("fn": max 448, no infinity, NaN =
 *     0x7F/0xFF), stored as uint8.  BF16 is stored as uint16 bit patterns.
 *   - Scales are FP32 dequantisation multipliers: x_hat = s * decode(q).
 *       activation scales (1x128 tiles):  s[cols/128][rows]   (K-block-major)
 *       weight scales (128x128 blocks):   s[G][N/128][K/128]
 *
 * Sources, cited by page title and section:
 *   [book]  "DeepSeek-V3" book (slop-6tp.pages.dev/papers-html/dsv3): ch. 7 "Fine-grained
 *           and Shared Experts", ch. 8 "Routing and Load Balancing", ch. 15 "Moving
 *           Tokens to Experts", ch. 16 "Understanding FP8 Numbers", ch. 17 "The Actual
 *           Mixed-precision Pipeline".
 *   [sum]   "DeepSeek-V3" summary (deepseek-2024.kryvik.com): core ideas 1 (DeepSeekMoE,
 *           node-limited routing), 2 (auxiliary-loss-free load balancing), 6 (FP8 mixed
 *           precision (a)-(d)).
 *   [pfd]   "DeepSeek-V3: the recipe, and the interconnect that shaped it"
 *           (paperfordummies.in): "The one formula", "Auxiliary-loss-free balancing",
 *           "FP8: the other half of the byte reduction".
 */
#ifndef MOE_FP8_H
#define MOE_FP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------------------ */
#define MOE_OK                   0
#define MOE_ERR_INVALID_ARG     -1  /* null pointer, misaligned pointer, bad dimension   */
#define MOE_ERR_UNSUPPORTED     -2  /* valid but outside what the kernels implement      */
#define MOE_ERR_CUDA            -3  /* a CUDA runtime/driver call or a launch failed     */
#define MOE_ERR_DEVICE_TIMEOUT  -4  /* device: a bounded wait inside a kernel expired    */
#define MOE_ERR_WORKSPACE       -5  /* ws is NULL or ws_bytes is too small               */
#define MOE_ERR_DEVICE_DATA     -6  /* device: index data out of range / inconsistent    */

/* Static description of a status code (never NULL). */
const char* moe_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int moe_version(void);

/* ---- router ------------------------------------------------------------------------ */

/* Router logits z[t][i] = sum_k x[t][k] * e_i[k], FP32 result.
 * The router is one of the places the method keeps above FP8 ([book] ch. 17 "High-
 * precision exceptions", "Router precision has discrete consequences"; [sum] core
 * idea 6).  x is BF16 [T][d] (row pitch d).  The FP32 centroids E [E][d] arrive split
 * into two BF16 planes, w_hilo = [hi; lo] with hi = bf16(E), lo = bf16(E - hi)
 * (moe_router_split_bf16), so the products run on BF16 tensor cores with FP32
 * accumulation and E keeps 16 significant bits.
 * Limits: d % 128 == 0, E % 16 == 0, E <= 256, T >= 0; x and w_hilo 16-byte aligned.
 * ws: moe_router_logits_ws_bytes(T, d, E) bytes, 16-byte aligned: nonzero when there are
 * fewer 128-token tiles than SMs (e.g. T = 128), where the K loop is split across CTAs into
 * FP32 partials that a second launch sums in a fixed order (the same bits every call).
 * z: FP32 [T][E], 16-byte aligned.  A bounded wait that expires inside the kernel sets
 * MOE_ERR_DEVICE_TIMEOUT in dev_status (may be NULL). */
int moe_router_logits(const uint16_t* x, int T, int d, const uint16_t* w_hilo, int E,
                      float* z, int32_t* dev_status, void* ws, size_t ws_bytes, void* stream);
size_t moe_router_logits_ws_bytes(int T, int d, int E);

/* Setup helper (not on the timed path): split FP32 centroids [E][d] into the two BF16
 * planes moe_router_logits takes: w_hilo[0][i][k] = bf16_rn(w), w_hilo[1][i][k] =
 * bf16_rn(w - hi).  n = E * d elements. */
int moe_router_split_bf16(const float* w, long long n, uint16_t* w_hilo, void* stream);

/* Route every token ([sum] core ideas 1-2; [book] ch. 7 "The router's affinity scores",
 * "Selecting and combining experts"; ch. 8 "V3's routing-only bias", "Restricting
 * target nodes"):
 *   s_i  = sigmoid(z_i)            (skipped when scores_are_affinities != 0)
 *   c_i  = s_i + bias_i            selection score; the bias never reaches the gate
 *   group score = sum of the group_topn largest c in the group (added in descending
 *                 order); the topk_groups best groups are kept
 *   idx  = the K largest c among experts of kept groups, listed in descending c
 *   gate_k = s_idx_k / (s_idx_0 + ... + s_idx_{K-1}) * route_scale
 * Ties in every ranking go to the lower index.  All arithmetic is FP32; divisions are
 * IEEE round-to-nearest.  With scores_are_affinities the results are bit-identical to
 * the plain definition above; from logits, sigmoid uses expf.
 * scores: FP32 [T][E]; bias: FP32 [E]; topk_idx: int32 [T][K]; topk_gate: FP32 [T][K].
 * Limits: E % n_groups == 0, n_groups <= 32, E <= 1024, 1 <= topk_groups <= n_groups,
 * 1 <= group_topn <= E/n_groups, 1 <= K <= min(32, topk_groups*E/n_groups). */
int moe_route(const float* scores, int scores_are_affinities, const float* bias,
              int T, int E, int n_groups, int topk_groups, int group_topn, int K,
              float route_scale, int32_t* topk_idx, float* topk_gate, void* stream);

/* ---- dispatch metadata ------------------------------------------------------------- */

/* Group the T*K (token, slot) pairs by expert ([book] ch. 15 "What dispatch must do";
 * ch. 7 "Batches change what is active"; no token is dropped, [sum] core idea 1).
 * A stable counting sort keyed by expert: rows of segment e are ordered by token.
 * When include_shared != 0 the shared expert is segment E: rows T*K + t hold token t.
 * Outputs (int32):
 *   counts[E]            pairs per routed expert
 *   offsets[E+2]         offsets[e] = first row of segment e; offsets[E] = T*K;
 *                        offsets[E+1] = T*K + (include_shared ? T : 0)
 *   row_token[T*K (+T)]  token held by each row
 *   row_of[T][K]         row holding pair (t, k)
 * An index outside [0, E) sets MOE_ERR_DEVICE_DATA in dev_status (outputs undefined).
 * Limits: E <= 1024, K <= 32.  ws: moe_permute_ws_bytes. */
int moe_permute(const int32_t* topk_idx, int T, int K, int E, int include_shared,
                int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* row_of,
                int32_t* dev_status, void* ws, size_t ws_bytes, void* stream);
size_t moe_permute_ws_bytes(int T, int K, int E);

/* moe_permute without caller workspace (the pages have no counterpart: this is a
 * convenience of this library).  Same arguments, results and errors as moe_permute,
 * minus (ws, ws_bytes).  For callers that cannot allocate device memory at the point of
 * the call -- code recorded into a CUDA graph, where cudaMalloc may not be called,
 * runtimes that own all device memory through their own allocator, or latency-critical
 * loops where an allocation would synchronise the device.
 *   - The scratch is a static device array of 1 MiB (262144 int32) inside the library;
 *     every GPU that loads the library holds it until the process exits.  Calls whose
 *     scratch need, ceil(T/128) * E int32, exceeds it return MOE_ERR_UNSUPPORTED.
 *   - The first call on each device looks up the array's device address (with that
 *     device current); make that first call before any stream capture.  The lookup is
 *     repeated when the device's CUDA context has changed (after cudaDeviceReset), so
 *     make the first call after a reset before any capture too.
 *   - Every call shares the one array and nothing in it needs to start at zero (each
 *     call writes every entry it reads).  Calls that overlap on the GPU, e.g. on two
 *     streams without ordering between them, race on it: serialise them.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine. */
int moe_permute_noalloc(const int32_t* topk_idx, int T, int K, int E, int include_shared,
                        int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* row_of,
                        int32_t* dev_status, void* stream);

/* ---- FP8 quantisation -------------------------------------------------------------- */

/* Quantise BF16 x [rows][cols] (row pitch ldx elements) to E4M3 with one FP32 scale per
 * 1x128 tile ([sum] core idea 6(a),(d); [book] ch. 16 "V3's grouping", "Online scales",
 * "Scaling a group"):  amax = max|x| over the tile; s = amax / 448 (IEEE division);
 * q = E4M3_rn_satfinite(x / s); amax == 0 gives s = 1, q = 0.
 * q: uint8 [rows][cols]; scale: FP32 [cols/128][rows].  cols % 128 == 0, ldx >= cols,
 * x 16-byte aligned with ldx % 8 == 0. */
int fp8_quant_1x128(const uint16_t* x, int rows, int cols, int ldx, uint8_t* q,
                    float* scale, void* stream);

/* Quantise-and-dispatch: each token row t of x is quantised as above once and written
 * to every row of the permuted matrix that uses it: rows row_of[t][0..K-1] and, when
 * shared_row_base >= 0, row shared_row_base + t.  With row_of and the shared rows from
 * moe_permute this is bit for bit fp8_quant_1x128 followed by moe_gather_rows_fp8 with
 * row_token, in one pass over x: the pages quantise activations before dispatch ([book]
 * ch. 17 "FP8 dispatch, BF16 combine").  x: BF16 [T][cols] (pitch ldx); row_of: int32
 * [T][K]; q: uint8 [n_rows][cols]; scale: FP32 [cols/128][n_rows].  A destination
 * outside [0, n_rows) sets MOE_ERR_DEVICE_DATA and is skipped.  K <= 32; x and q 16-byte
 * aligned, ldx % 8 == 0. */
int fp8_quant_scatter_1x128(const uint16_t* x, int T, int cols, int ldx, const int32_t* row_of,
                            int K, int shared_row_base, int n_rows, uint8_t* q, float* scale,
                            int32_t* dev_status, void* stream);

/* Setup helper: quantise FP32 w [rows][cols] in 128x128 blocks, same scale rule.
 * q: uint8 [rows][cols]; scale: FP32 [rows/128][cols/128].  rows, cols % 128 == 0. */
int fp8_quant_128x128(const float* w, int rows, int cols, uint8_t* q, float* scale,
                      void* stream);

/* Power-of-two-scale quantisers (the MX-native variant, for fp8_mx_grouped_gemm): the
 * same tiles, layouts and E4M3 rounding, with s = the smallest power of two such that
 * 448 * s >= amax (at least 2^-126; s = 1 when amax == 0), so x / s is exact and never
 * saturates.  The pages note that the 1x128 / 128x128 groups match the microscaling
 * formats Blackwell tensor cores take natively ([sum] core idea 6(a)) and mention
 * power-of-two scales ([book] ch. 17 "Attention-related saved activations").  The
 * scatter form is fp8_quant_scatter_1x128 with this rule. */
int fp8_quant_1x128_pow2(const uint16_t* x, int rows, int cols, int ldx, uint8_t* q,
                         float* scale, void* stream);
int fp8_quant_128x128_pow2(const float* w, int rows, int cols, uint8_t* q, float* scale,
                           void* stream);
int fp8_quant_scatter_1x128_pow2(const uint16_t* x, int T, int cols, int ldx,
                                 const int32_t* row_of, int K, int shared_row_base, int n_rows,
                                 uint8_t* q, float* scale, int32_t* dev_status, void* stream);

/* ---- FP8 block-scaled grouped GEMM ------------------------------------------------- */

/* C[r][n] = sum_kb sA[kb][r'] * sB[g][n/128][kb] * sum_{k in kb} A[r'][k] * B[g][n][k]
 * for every row r of segment g (seg_offsets[g] <= r < seg_offsets[g+1]), with
 * r' = a_rows ? a_rows[r] : r.  Each 128-deep K block is summed on the tensor cores,
 * then scaled and added into FP32 ("promotion" every 128 elements of K: [sum] core idea
 * 6(b); [book] ch. 16 "Scales along the GEMM inner dimension", "Periodic high-precision
 * promotion").  C is BF16 (round to nearest even), row pitch ldc.
 *   A:  uint8 [M_a][K] (M_a = M when a_rows is NULL, else the rows a_rows refers to),
 *   sA: FP32 [K/128][M_a];  B: uint8 [G][N][K];  sB: FP32 [G][N/128][K/128];
 *   seg_offsets: int32 [G+1] on the device, non-decreasing, seg_offsets[0] = 0,
 *                seg_offsets[G] <= M;  a_rows: int32 [M] or NULL;  C: [M][ldc].
 * G = 1 with seg_offsets = {0, M} is the dense GEMM.
 * Limits: N % 128 == 0, K % 128 == 0, 1 <= G <= 1024, ldc % 8 == 0, A/B/C 16-byte
 * aligned.  ws: fp8_grouped_gemm_ws_bytes (non-zero only when a_rows != NULL). */
int fp8_blockscaled_grouped_gemm(const uint8_t* A, const float* sA, int M_a,
                                 const int32_t* a_rows, const uint8_t* B, const float* sB,
                                 const int32_t* seg_offsets, int G, int M, int N, int K,
                                 uint16_t* C, int ldc, int32_t* dev_status,
                                 void* ws, size_t ws_bytes, void* stream);
size_t fp8_grouped_gemm_ws_bytes(int M, int K, int has_a_rows);

/* CTA tiling of fp8_blockscaled_grouped_gemm, moe_gate_up_fp8 and moe_swiglu_fp8_fwd
 * (a performance choice; results are the same bits either way):
 *   0  automatic (the default): tiling 3 when the segments average at most 16 rows
 *      (M <= 16 * G, decode batches) and N % 256 == 0, else tiling 1 (on B300 tiling 2
 *      measured 2-15% slower on dense shapes and slower on MoE segments);
 *   1  one CTA per 128-row x 256-column tile (tcgen05 cta_group::1);
 *   2  two CTAs of a cluster per 256-row x 256-column tile: one tcgen05 cta_group::2
 *      MMA over both CTAs' shared memory, each CTA loading half of the weight tile;
 *   3  operands swapped for short segments: 256 weight rows on the MMA's M side times 32
 *      tokens of a segment on N, so no MMA row is padding; per-expert decode batches are
 *      small and weight-bound ([sum] core idea 8: transposed GEMM reads).  Needs
 *      N % 256 == 0; otherwise tiling 1 runs.
 * The setting is process-wide and applies to calls made after it.  Returns
 * MOE_ERR_INVALID_ARG for any other mode. */
int moe_set_gemm_tiling(int mode);
int moe_get_gemm_tiling(void);

/* Failure-path test of the kernels' bounded waits; not for production use.  Runs
 * fp8_blockscaled_grouped_gemm (a_rows = NULL, same arguments) with every mbarrier wait
 * limited to wait_ns nanoseconds (1e5 <= wait_ns <= 2e9) and the MMA-issuing thread first
 * waiting on a barrier that nothing arrives on.  That wait expires: the kernel writes
 * MOE_ERR_DEVICE_TIMEOUT to dev_status (required), stops issuing work, lets its copies
 * and tensor-core operations in flight finish, frees its TMEM and returns, leaving C
 * partly unwritten.  The GPU stays usable for the next call. */
int moe_test_gemm_wait_expiry(const uint8_t* A, const float* sA, const uint8_t* B,
                              const float* sB, const int32_t* seg_offsets, int G, int M, int N,
                              int K, uint16_t* C, int ldc, int32_t* dev_status,
                              unsigned long long wait_ns, void* stream);

/* MX-native variant ([sum] core idea 6(a), core idea 8 "native group-scaled MMA"): the
 * same C as fp8_blockscaled_grouped_gemm (A rows in segment order, no a_rows) when every
 * scale is a power of two, with the scales applied inside the tensor core
 * (tcgen05.mma kind::mxf8f6f4, UE8M0 scale factors) and one FP32 accumulator per tile
 * for the whole K loop: no per-block promotion.  Scales must be positive normal powers
 * of two (fp8_quant_*_pow2); anything else sets MOE_ERR_DEVICE_DATA.  Same layouts and
 * limits as fp8_blockscaled_grouped_gemm; no workspace.  Segments of a few rows (decode
 * batches: M <= 16 * G, N % 256 == 0, see moe_set_gemm_tiling) run on the swapped-operand
 * kernel instead, whose per-block promotion with power-of-two scales is exact -- the same
 * scaling the tensor core would apply. */
int fp8_mx_grouped_gemm(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                        const int32_t* seg_offsets, int G, int M, int N, int K, uint16_t* C,
                        int ldc, int32_t* dev_status, void* stream);

/* MX-native gate/up: moe_gate_up_fp8 on power-of-two scales (x rows, w13), with h
 * requantised 1x128 by the power-of-two rule of fp8_quant_1x128_pow2, so hq / sh feed
 * fp8_mx_grouped_gemm for the down projection.  Same layouts and limits as
 * moe_gate_up_fp8; a scale that is not a power of two sets MOE_ERR_DEVICE_DATA. */
int moe_gate_up_mx(const uint8_t* xq_rows, const float* sx_rows, const int32_t* offsets,
                   int rows, const uint8_t* w13, const float* s13, int n_segments, int d, int f,
                   uint8_t* hq, float* sh, int32_t* dev_status, void* stream);

/* ---- experts ----------------------------------------------------------------------- */

/* SwiGLU experts on FP8 rows, one segment per expert ([book] ch. 2 "RMSNorm and
 * SwiGLU", ch. 7 "What one expert computes"; [sum] core idea 6):
 *   rows r of segment e take token row_token[r] of xq (quantised 1x128);
 *   [G | U] = xq_rows . w13_e^T   (grouped block-scaled GEMM, FP32 results)
 *   h = silu(G) * U               (FP32), requantised 1x128 along f -> hq, sh
 *   y_rows = hq . w2_e^T          (grouped block-scaled GEMM, BF16 results)
 * w13 interleaves the gate and up weights in 64-row blocks: rows [128j, 128j+64) of
 * expert e are gate rows [64j, 64j+64) and rows [128j+64, 128j+128) the matching up
 * rows, so every 128-column output tile holds matching gate and up columns.  The
 * scales stay per 128x128 block of the original matrices: s13[e][2i][kb] belongs to
 * gate rows [128i, 128i+128), s13[e][2i+1][kb] to the same up rows.
 *   xq: uint8 [T][d]; sx: FP32 [d/128][T]; row_token: int32 [rows]; offsets: int32
 *   [n_segments+1] (device), offsets[n_segments] <= rows;
 *   w13: uint8 [n_segments][2f][d]; s13: FP32 [n_segments][2f/128][d/128];
 *   w2: uint8 [n_segments][d][f];   s2: FP32 [n_segments][d/128][f/128];
 *   hq: uint8 [rows][f]; sh: FP32 [f/128][rows]; y_rows: BF16 [rows][d].
 * Rows past offsets[n_segments] are not written.
 * Limits: d % 128 == 0, f % 128 == 0, 1 <= n_segments <= 1024.
 * ws: moe_swiglu_ws_bytes. */
int moe_swiglu_fp8_fwd(const uint8_t* xq, const float* sx, int T, const int32_t* row_token,
                       const int32_t* offsets, int rows, const uint8_t* w13,
                       const float* s13, const uint8_t* w2, const float* s2,
                       int n_segments, int d, int f, uint8_t* hq, float* sh,
                       uint16_t* y_rows, int32_t* dev_status, void* ws, size_t ws_bytes,
                       void* stream);
size_t moe_swiglu_ws_bytes(int rows, int d, int f);

/* The three steps of moe_swiglu_fp8_fwd as separate calls (same kernels), for callers
 * that schedule or time them one by one:
 *   moe_gather_rows_fp8  dst[r] = src[rows[r]] (an FP8 matrix of `cols` columns with its
 *                        1x128 scales [cols/128][src_rows] -> [cols/128][n_rows]) for
 *                        r < min(n_rows, *row_limit); row_limit is a device int32 (NULL:
 *                        n_rows).  An index outside [0, src_rows) sets
 *                        MOE_ERR_DEVICE_DATA.  cols % 128 == 0; src, dst 16-byte aligned.
 *   moe_gate_up_fp8      hq, sh = requant_1x128( silu(G) * U ), [G | U] = xq_rows . w13_e^T
 *                        per segment, xq_rows already in segment order ([rows][d], scales
 *                        [d/128][rows]).  Layouts as in moe_swiglu_fp8_fwd.
 *   the down projection is fp8_blockscaled_grouped_gemm(hq, sh, rows, NULL, w2, s2,
 *   offsets, n_segments, rows, d, f, y_rows, d, ...). */
int moe_gather_rows_fp8(const uint8_t* src, const float* src_scale, int src_rows,
                        const int32_t* rows, const int32_t* row_limit, int n_rows, int cols,
                        uint8_t* dst, float* dst_scale, int32_t* dev_status, void* stream);
int moe_gate_up_fp8(const uint8_t* xq_rows, const float* sx_rows, const int32_t* offsets,
                    int rows, const uint8_t* w13, const float* s13, int n_segments, int d,
                    int f, uint8_t* hq, float* sh, int32_t* dev_status, void* stream);

/* ---- backward of the experts (training) -------------------------------------------- */

/* The three GEMMs of a linear layer in training -- Fprop, Dgrad (input gradient,
 * dX = dY W^T) and Wgrad (weight gradient, dW = X^T dY) -- all take FP8 inputs ([book]
 * ch. 17 "One linear layer creates three GEMMs"; [sum] core idea 6).  Activation
 * gradients keep 1x128 tiles ([book] ch. 17 "Backward grouping and gradient
 * sensitivity").  Wgrad contracts over token rows, so its operands are regrouped into
 * 128x1 tiles with power-of-two scales ([book] ch. 16 "Why transposition is not
 * trivial"; ch. 17 "Attention-related saved activations"), and the MoE caches the
 * SwiGLU inputs in FP8 and recomputes the SwiGLU output in backward ([book] ch. 17
 * "SwiGLU recomputation").  One expert backward, rows in segment order:
 *   moe_combine_bwd_rows    dY rows from dy and the gates
 *   fp8_quant_1x128         dY -> 1x128 tiles
 *   fp8_blockscaled_grouped_gemm(dYq, W2^T)           dh (BF16), down Dgrad
 *   moe_swiglu_bwd_fp8      h recomputed from the cache; dG, dU; [dG|dU] 1x128 for the
 *                           gate/up Dgrad; h^T and [dG|dU]^T 128x1 for the Wgrads
 *   fp8_blockscaled_grouped_gemm([dG|dU]q, [W1;W3]^T) dX rows (BF16), gate/up Dgrad
 *   moe_combine(dX rows, gates = 1)                   dx per token
 *   fp8_quant_128x1_pow2    dY^T and the input rows X^T in 128x1 tiles
 *   fp8_wgrad_grouped_gemm(dY^T, h^T) -> dW2;  (... [dG|dU]^T, X^T) -> [dW1; dW3]
 * Padded row layout of the 128x1 tensors: every segment's rows are cut into 128-row
 * blocks starting at its first row; block b of segment e sits at columns
 * [pad[e] + 128 b, pad[e] + 128 b + 128) of a [C][kcap] matrix (pad from
 * moe_segment_pad_offsets, kcap >= pad[G] from moe_padded_rows_cap); rows past a
 * segment's end hold code 0.  Scales are [kcap/128][C], one per (row block, column). */

/* The gate/up GEMM of a training forward: moe_gate_up_fp8, and also the SwiGLU inputs
 * g, u cached in E4M3 with 1x128 scales (the fp8_quant_1x128 rule):
 *   guq: uint8 [rows][2f], columns [0, f) = g, [f, 2f) = u;  sgu: FP32 [2f/128][rows]. */
int moe_gate_up_fp8_train(const uint8_t* xq_rows, const float* sx_rows, const int32_t* offsets,
                          int rows, const uint8_t* w13, const float* s13, int n_segments, int d,
                          int f, uint8_t* hq, float* sh, uint8_t* guq, float* sgu,
                          int32_t* dev_status, void* stream);

/* Setup helper: the transposed FP8 weights of the Dgrad GEMMs.  wT[g][c][r] = w[g][r][c]
 * and sT[g][cb][rb] = s[g][rb][cb]: a 128x128 block keeps its scale under transposition,
 * so no requantisation is needed.  With gate_up_interleaved, w is moe_swiglu_fp8_fwd's
 * w13 (gate and up rows alternating in 64-row blocks) and the output columns come out
 * gate first: wT = [W1; W3]^T [G][d][2f].  w: uint8 [G][rows][cols]; s: FP32
 * [G][rows/128][cols/128]; rows, cols % 128 == 0 (rows % 256 when interleaved). */
int fp8_transpose_128x128(const uint8_t* w, const float* s, int G, int rows, int cols,
                          int gate_up_interleaved, uint8_t* wT, float* sT, void* stream);

/* Host helper: a bound of the padded row count, ceil((rows + 127 G) / 128) * 128 (-1 on
 * a bad argument). */
int moe_padded_rows_cap(int rows, int G);

/* pad[0] = 0, pad[e+1] = pad[e] + ceil(count_e / 128) * 128 with count_e =
 * offsets[e+1] - offsets[e] (device int32 [G+1] -> [G+1]).  A negative count sets
 * MOE_ERR_DEVICE_DATA.  G <= 1024. */
int moe_segment_pad_offsets(const int32_t* offsets, int G, int32_t* pad, int32_t* dev_status,
                            void* stream);

/* Gradient of moe_combine w.r.t. the expert output rows: dy_rows[row_of[t][k]] =
 * bf16(fl32(topk_gate[t][k] * dy[t])) and, when shared_row_base >= 0, dy_rows[shared_row_base
 * + t] = dy[t].  dy: BF16 [T][d]; dy_rows: BF16 [n_rows][d].  A row outside [0, n_rows) sets
 * MOE_ERR_DEVICE_DATA and is skipped.  d % 8 == 0, K <= 32, 16-byte aligned. */
int moe_combine_bwd_rows(const uint16_t* dy, const float* topk_gate, const int32_t* row_of,
                         int T, int K, int d, int shared_row_base, int n_rows, uint16_t* dy_rows,
                         int32_t* dev_status, void* stream);

/* 128x1 regrouping: the rows of segment order (row r is src[rows[r]], or src[r] when rows
 * is NULL) quantised in 128x1 tiles with power-of-two scales (the smallest 2^k >= 2^-126
 * with 448 * 2^k >= the column's max |x| over the block; 1 for an all-zero column), stored
 * transposed: qT uint8 [cols][kcap], sT FP32 [kcap/128][cols], padded layout as above.
 * src: BF16 [src_rows][cols]; offsets [G+1] and pad [G+1] on the device.  A gathered row
 * outside [0, src_rows) sets MOE_ERR_DEVICE_DATA.  cols % 128 == 0, kcap % 128 == 0,
 * G <= 1024, src and qT 16-byte aligned. */
int fp8_quant_128x1_pow2(const uint16_t* src, int src_rows, const int32_t* rows, int cols,
                         const int32_t* offsets, const int32_t* pad, int G, int kcap,
                         uint8_t* qT, float* sT, int32_t* dev_status, void* stream);

/* SwiGLU backward with recomputation, per row r of segment order:
 *   g = fl32(dec(guq[r][c]) * s), u likewise (the cache of moe_gate_up_fp8_train);
 *   sig = 1 / (1 + expf(-g));  h = g sig u;  dU = dh g sig;  dG = dh u sig (1 + g (1 - sig))
 * (FP32), written as
 *   dguq uint8 [rows][2f] (dG columns first) with 1x128 scales sdgu [2f/128][rows] (the
 *        fp8_quant_1x128 rule) -- the gate/up Dgrad operand;
 *   hT uint8 [f][kcap], shT [kcap/128][f] and dguT uint8 [2f][kcap], sdguT [kcap/128][2f]
 *        in 128x1 power-of-two tiles, padded layout as above -- the Wgrad operands.
 * dh: BF16 [rows][f].  f % 128 == 0, kcap % 128 == 0, G <= 1024. */
int moe_swiglu_bwd_fp8(const uint8_t* guq, const float* sgu, const uint16_t* dh, int rows, int f,
                       const int32_t* offsets, const int32_t* pad, int G, int kcap,
                       uint8_t* dguq, float* sdgu, uint8_t* hT, float* shT, uint8_t* dguT,
                       float* sdguT, void* stream);

/* Wgrad: for every expert e, dW[e][i][j] = sum over e's row blocks rb of saT[rb][i] *
 * sbT[rb][j] * sum_{p in rb} dec(aT[i][p]) * dec(bT[j][p]), FP32, on tcgen05 tensor cores
 * with the power-of-two block scales applied by the hardware (kind::mxf8f6f4): one scale
 * per (row block, output row) and per (row block, output column), each row block's
 * product promoted with its own scales.  An expert without rows gets zeros.
 * aT uint8 [I][kcap], saT FP32 [kcap/128][I]; bT uint8 [J][kcap], sbT FP32 [kcap/128][J];
 * pad [G+1] (device); dW FP32 [G][I][J].  Scales must be positive normal powers of two
 * (else MOE_ERR_DEVICE_DATA); pad must start at 0, rise in whole 128-row blocks and stay
 * within kcap (else MOE_ERR_DEVICE_DATA).  I, J, kcap % 128 == 0; G <= 1024. */
int fp8_wgrad_grouped_gemm(const uint8_t* aT, const float* saT, const uint8_t* bT,
                           const float* sbT, const int32_t* pad, int G, int I, int J, int kcap,
                           float* dW, int32_t* dev_status, void* stream);

/* ---- combine and bias update ------------------------------------------------------- */

/* y[t] = bf16( y_rows[shared_row_base + t] + sum_{k=0..K-1} gate[t][k] * y_rows[row_of[t][k]] )
 * accumulated in FP32 in exactly that order ([book] ch. 7 "Selecting and combining
 * experts", ch. 15 "What combine must do", ch. 17 "FP8 dispatch, BF16 combine").
 * shared_row_base < 0: no shared expert.  The residual is not added.
 * y_rows: BF16 [n_rows][d]; row_of: int32 [T][K]; gate: FP32 [T][K]; y: BF16 [T][d].
 * A row index outside [0, n_rows) sets MOE_ERR_DEVICE_DATA in dev_status and leaves that
 * token's output unwritten.  d % 8 == 0, 1 <= K <= 32, y_rows and y 16-byte aligned. */
int moe_combine(const uint16_t* y_rows, int n_rows, const int32_t* row_of,
                const float* gate, int T, int K, int d, int shared_row_base, uint16_t* y,
                int32_t* dev_status, void* stream);

/* Aux-loss-free bias step ([sum] core idea 2; [book] ch. 8 "The feedback update";
 * [pfd] "Auxiliary-loss-free balancing"):
 *   bias[i] += gamma * sign(T*K/E - counts[i]),   sign(0) = 0,
 * with the comparison done exactly in integers (T*K - E*counts[i]). */
int moe_bias_update(float* bias, const int32_t* counts, int E, int T, int K, float gamma,
                    void* stream);

/* ---- sequence-wise balance statistics (forward only) ------------------------------- */

/* Statistics of the complementary sequence-wise balance loss ([book] ch. 8 "The
 * complementary sequence loss"; [sum] core idea 2, the safety-net paragraph), for
 * T / seq_len consecutive sequences of seq_len tokens each:
 *   s[t][i]  = scores[t][i] if scores_are_affinities, else fl32(1 / (1 + expf(-z)))
 *   f[q][i]  = fl32(E * n_i) / fl32(K * seq_len), n_i = tokens of sequence q whose K
 *              largest s (over all E experts, ties to the lower index; no bias, no
 *              group limit) include expert i
 *   P[q][i]  = (1/seq_len) * sum over the sequence of s[t][i] / sum_j s[t][j]
 *   loss[q]  = alpha * sum_i f[q][i] * P[q][i]                 (alpha = 1e-4 in V3)
 * All FP32, summed in a fixed order (deterministic).  scores: FP32 [T][E]; f, P: FP32
 * [T/seq_len][E]; loss: FP32 [T/seq_len].  Workspace: moe_seq_balance_stats_ws_bytes.
 * Errors: MOE_ERR_INVALID_ARG unless 1 <= K <= E and seq_len divides T;
 * MOE_ERR_UNSUPPORTED for E > 1024, K > 32 or more than 65,535 sequences. */
size_t moe_seq_balance_stats_ws_bytes(int T, int E, int seq_len);
int moe_seq_balance_stats(const float* scores, int scores_are_affinities, int T, int E, int K,
                          int seq_len, float alpha, float* f, float* P, float* loss, void* ws,
                          size_t ws_bytes, void* stream);

/* Workspace large enough for every call of one layer forward with these sizes. */
size_t moe_workspace_bytes(int T, int K, int E, int d, int f);

#ifdef __cplusplus
}
#endif
#endif /* MOE_FP8_H */
