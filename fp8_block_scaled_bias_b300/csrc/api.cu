// extern "C" entry points of libmoe_fp8.so (declared in include/moe_fp8.h): argument
// checks on the host, workspace carving, then the launches on the caller's stream.
#include <cstdint>

#include "common.cuh"
#include "launch.h"

namespace {

using moe::GemmArgs;

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// bytes of the gathered FP8 rows + their scales, as carved from a workspace
inline size_t gathered_bytes(long long rows, long long cols) {
  return align256(static_cast<size_t>(rows) * cols) +
         align256(static_cast<size_t>(rows) * (cols / 128) * sizeof(float));
}

}  // namespace

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size or configuration";
    case MOE_ERR_CUDA: return "CUDA call or kernel launch failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel expired";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_DEVICE_DATA: return "device index data out of range or inconsistent";
    default: return "unknown status";
  }
}

int moe_version(void) { return 100; }

// ---- router ------------------------------------------------------------------------

size_t moe_router_logits_ws_bytes(int T, int d, int E) {
  return moe::router_logits_ws_bytes(T, d, E);
}

int moe_router_logits(const uint16_t* x, int T, int d, const uint16_t* w_hilo, int E,
                      float* z, int32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  if (T < 0 || d <= 0 || E <= 0 || d % 128 != 0 || E % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (E > 256) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !w_hilo || !z || !aligned16(x) || !aligned16(w_hilo) || !aligned16(z))
    return MOE_ERR_INVALID_ARG;
  const size_t need = moe::router_logits_ws_bytes(T, d, E);
  if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws))) return MOE_ERR_WORKSPACE;
  return moe::launch_router_logits(x, T, d, w_hilo, E, z, dev_status, ws, as_stream(stream));
}

int moe_router_split_bf16(const float* w, long long n, uint16_t* w_hilo, void* stream) {
  if (n < 0) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (!w || !w_hilo) return MOE_ERR_INVALID_ARG;
  return moe::launch_router_split(w, n, w_hilo, as_stream(stream));
}

int moe_route(const float* scores, int scores_are_affinities, const float* bias, int T, int E,
              int n_groups, int topk_groups, int group_topn, int K, float route_scale,
              int32_t* topk_idx, float* topk_gate, void* stream) {
  if (T < 0 || E <= 0 || n_groups <= 0 || E % n_groups != 0) return MOE_ERR_INVALID_ARG;
  const int gs = E / n_groups;
  if (topk_groups < 1 || topk_groups > n_groups || group_topn < 1 || group_topn > gs || K < 1 ||
      K > topk_groups * gs)
    return MOE_ERR_INVALID_ARG;
  if (E > 1024 || n_groups > 32 || K > 32) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!scores || !bias || !topk_idx || !topk_gate) return MOE_ERR_INVALID_ARG;
  return moe::launch_route(scores, scores_are_affinities, bias, T, E, n_groups, topk_groups,
                           group_topn, K, route_scale, topk_idx, topk_gate, as_stream(stream));
}

// ---- dispatch metadata ---------------------------------------------------------------

size_t moe_permute_ws_bytes(int T, int K, int E) {
  if (T < 0 || K < 0 || E < 0) return 0;
  return moe::permute_ws_bytes(T, K, E);
}

int moe_permute(const int32_t* topk_idx, int T, int K, int E, int include_shared,
                int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* row_of,
                int32_t* dev_status, void* ws, size_t ws_bytes, void* stream) {
  if (T < 0 || K < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || K > 32) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(T) * (K + 1) > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !row_token || !row_of)) return MOE_ERR_INVALID_ARG;
  const size_t need = moe::permute_ws_bytes(T, K, E);
  if (need > 0 && (!ws || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  return moe::launch_permute(topk_idx, T, K, E, include_shared, counts, offsets, row_token,
                             row_of, dev_status, ws, as_stream(stream));
}

int moe_permute_noalloc(const int32_t* topk_idx, int T, int K, int E, int include_shared,
                        int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* row_of,
                        int32_t* dev_status, void* stream) {
  if (T < 0 || K < 1 || E < 1) return MOE_ERR_INVALID_ARG;
  if (E > 1024 || K > 32) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(T) * (K + 1) > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !row_token || !row_of)) return MOE_ERR_INVALID_ARG;
  const long long need = static_cast<long long>(moe::permute_ws_bytes(T, K, E) / sizeof(int32_t));
  if (need > moe::permute_noalloc_max_ints()) return MOE_ERR_UNSUPPORTED;
  int32_t* scratch = nullptr;
  const int st = moe::permute_noalloc_scratch(&scratch);
  if (st != MOE_OK) return st;
  return moe::launch_permute(topk_idx, T, K, E, include_shared, counts, offsets, row_token,
                             row_of, dev_status, scratch, as_stream(stream));
}

// ---- quantisation --------------------------------------------------------------------

static int quant_1x128_common(const uint16_t* x, int rows, int cols, int ldx, uint8_t* q,
                              float* scale, bool pow2, void* stream) {
  if (rows < 0 || cols < 0 || cols % 128 != 0 || ldx < cols || ldx % 8 != 0)
    return MOE_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return MOE_OK;
  if (!x || !q || !scale || !aligned16(x) || (reinterpret_cast<uintptr_t>(q) & 7u))
    return MOE_ERR_INVALID_ARG;
  return moe::launch_quant_1x128(x, rows, cols, ldx, q, scale, pow2, as_stream(stream));
}

int fp8_quant_1x128(const uint16_t* x, int rows, int cols, int ldx, uint8_t* q, float* scale,
                    void* stream) {
  return quant_1x128_common(x, rows, cols, ldx, q, scale, false, stream);
}

int fp8_quant_1x128_pow2(const uint16_t* x, int rows, int cols, int ldx, uint8_t* q,
                         float* scale, void* stream) {
  return quant_1x128_common(x, rows, cols, ldx, q, scale, true, stream);
}

static int quant_scatter_common(const uint16_t* x, int T, int cols, int ldx,
                                const int32_t* row_of, int K, int shared_row_base, int n_rows,
                                uint8_t* q, float* scale, bool pow2, int32_t* dev_status,
                                void* stream) {
  if (T < 0 || K < 0 || n_rows < 0 || cols < 0 || cols % 128 != 0 || ldx < cols || ldx % 8 != 0)
    return MOE_ERR_INVALID_ARG;
  if (K > 32) return MOE_ERR_UNSUPPORTED;
  if (T == 0 || cols == 0) return MOE_OK;
  if (!x || (K > 0 && !row_of) || !q || !scale || !aligned16(x) || !aligned16(q))
    return MOE_ERR_INVALID_ARG;
  return moe::launch_quant_scatter_1x128(x, T, cols, ldx, row_of, K, shared_row_base, n_rows, q,
                                         scale, pow2, dev_status, as_stream(stream));
}

int fp8_quant_scatter_1x128(const uint16_t* x, int T, int cols, int ldx, const int32_t* row_of,
                            int K, int shared_row_base, int n_rows, uint8_t* q, float* scale,
                            int32_t* dev_status, void* stream) {
  return quant_scatter_common(x, T, cols, ldx, row_of, K, shared_row_base, n_rows, q, scale,
                              false, dev_status, stream);
}

int fp8_quant_scatter_1x128_pow2(const uint16_t* x, int T, int cols, int ldx,
                                 const int32_t* row_of, int K, int shared_row_base, int n_rows,
                                 uint8_t* q, float* scale, int32_t* dev_status, void* stream) {
  return quant_scatter_common(x, T, cols, ldx, row_of, K, shared_row_base, n_rows, q, scale,
                              true, dev_status, stream);
}

static int quant_128x128_common(const float* w, int rows, int cols, uint8_t* q, float* scale,
                                bool pow2, void* stream) {
  if (rows < 0 || cols < 0 || rows % 128 != 0 || cols % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return MOE_OK;
  if (!w || !q || !scale || !aligned16(w) || (reinterpret_cast<uintptr_t>(q) & 3u))
    return MOE_ERR_INVALID_ARG;
  return moe::launch_quant_128x128(w, rows, cols, q, scale, pow2, as_stream(stream));
}

int fp8_quant_128x128(const float* w, int rows, int cols, uint8_t* q, float* scale,
                      void* stream) {
  return quant_128x128_common(w, rows, cols, q, scale, false, stream);
}

int fp8_quant_128x128_pow2(const float* w, int rows, int cols, uint8_t* q, float* scale,
                           void* stream) {
  return quant_128x128_common(w, rows, cols, q, scale, true, stream);
}

// ---- grouped GEMM --------------------------------------------------------------------

size_t fp8_grouped_gemm_ws_bytes(int M, int K, int has_a_rows) {
  if (!has_a_rows || M <= 0 || K <= 0) return 0;
  return gathered_bytes(M, K);
}

static int check_gemm_dims(int G, int M, int N, int K) {
  if (G < 1 || M < 0 || N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0)
    return MOE_ERR_INVALID_ARG;
  if (G > 1024) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(G) * N > INT32_MAX || K > (1 << 24)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int fp8_mx_grouped_gemm(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB,
                        const int32_t* seg_offsets, int G, int M, int N, int K, uint16_t* C,
                        int ldc, int32_t* dev_status, void* stream) {
  const int st = check_gemm_dims(G, M, N, K);
  if (st != MOE_OK) return st;
  if (M == 0) return MOE_OK;
  if (!A || !sA || !B || !sB || !seg_offsets || !C) return MOE_ERR_INVALID_ARG;
  if (ldc < N || ldc % 8 != 0 || !aligned16(A) || !aligned16(B) || !aligned16(C))
    return MOE_ERR_INVALID_ARG;
  return moe::launch_mx_gemm(A, sA, B, sB, seg_offsets, G, M, N, K, C, ldc, nullptr, nullptr,
                             moe::kEpiBF16, dev_status, as_stream(stream));
}

int fp8_blockscaled_grouped_gemm(const uint8_t* A, const float* sA, int M_a,
                                 const int32_t* a_rows, const uint8_t* B, const float* sB,
                                 const int32_t* seg_offsets, int G, int M, int N, int K,
                                 uint16_t* C, int ldc, int32_t* dev_status, void* ws,
                                 size_t ws_bytes, void* stream) {
  int st = check_gemm_dims(G, M, N, K);
  if (st != MOE_OK) return st;
  if (M == 0) return MOE_OK;
  if (!A || !sA || !B || !sB || !seg_offsets || !C) return MOE_ERR_INVALID_ARG;
  if (ldc < N || ldc % 8 != 0 || !aligned16(A) || !aligned16(B) || !aligned16(C))
    return MOE_ERR_INVALID_ARG;
  if (a_rows && M_a < 1) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  const uint8_t* Ause = A;
  const float* sAuse = sA;
  if (a_rows) {
    const size_t need = gathered_bytes(M, K);
    if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
    uint8_t* gA = static_cast<uint8_t*>(ws);
    float* gS = reinterpret_cast<float*>(gA + align256(static_cast<size_t>(M) * K));
    st = moe::launch_gather_rows_fp8(A, sA, M_a, a_rows, seg_offsets + G, M, K, gA, gS,
                                     dev_status, s);
    if (st != MOE_OK) return st;
    Ause = gA;
    sAuse = gS;
  }
  GemmArgs a{};
  a.A = Ause; a.sA = sAuse; a.B = B; a.sB = sB; a.seg = seg_offsets;
  a.G = G; a.M = M; a.N = N; a.K = K; a.C = C; a.ldc = ldc; a.status = dev_status;
  return moe::launch_fp8_gemm(a, moe::kEpiBF16, s);
}

int moe_set_gemm_tiling(int mode) {
  if (mode < 0 || mode > 3) return MOE_ERR_INVALID_ARG;
  moe::set_gemm_tiling(mode);
  return MOE_OK;
}

int moe_get_gemm_tiling(void) { return moe::gemm_tiling(); }

int moe_test_gemm_wait_expiry(const uint8_t* A, const float* sA, const uint8_t* B,
                              const float* sB, const int32_t* seg_offsets, int G, int M, int N,
                              int K, uint16_t* C, int ldc, int32_t* dev_status,
                              unsigned long long wait_ns, void* stream) {
  int st = check_gemm_dims(G, M, N, K);
  if (st != MOE_OK) return st;
  if (M == 0) return MOE_OK;
  if (!A || !sA || !B || !sB || !seg_offsets || !C || !dev_status) return MOE_ERR_INVALID_ARG;
  if (ldc < N || ldc % 8 != 0 || !aligned16(A) || !aligned16(B) || !aligned16(C))
    return MOE_ERR_INVALID_ARG;
  if (wait_ns < 100000ull || wait_ns > 2000000000ull) return MOE_ERR_INVALID_ARG;
  GemmArgs a{};
  a.A = A; a.sA = sA; a.B = B; a.sB = sB; a.seg = seg_offsets;
  a.G = G; a.M = M; a.N = N; a.K = K; a.C = C; a.ldc = ldc; a.status = dev_status;
  a.wait_ns = wait_ns;
  a.stall = 1;
  return moe::launch_fp8_gemm(a, moe::kEpiBF16, as_stream(stream));
}

// ---- experts -------------------------------------------------------------------------

size_t moe_swiglu_ws_bytes(int rows, int d, int f) {
  (void)f;
  if (rows <= 0 || d <= 0) return 0;
  return gathered_bytes(rows, d);
}

int moe_swiglu_fp8_fwd(const uint8_t* xq, const float* sx, int T, const int32_t* row_token,
                       const int32_t* offsets, int rows, const uint8_t* w13, const float* s13,
                       const uint8_t* w2, const float* s2, int n_segments, int d, int f,
                       uint8_t* hq, float* sh, uint16_t* y_rows, int32_t* dev_status, void* ws,
                       size_t ws_bytes, void* stream) {
  if (T < 0 || rows < 0 || d <= 0 || f <= 0 || d % 128 != 0 || f % 128 != 0 || n_segments < 1)
    return MOE_ERR_INVALID_ARG;
  int st = check_gemm_dims(n_segments, rows, 2 * f, d);
  if (st != MOE_OK) return st;
  st = check_gemm_dims(n_segments, rows, d, f);
  if (st != MOE_OK) return st;
  if (rows == 0) return MOE_OK;
  if (T == 0) return MOE_ERR_INVALID_ARG;
  if (!xq || !sx || !row_token || !offsets || !w13 || !s13 || !w2 || !s2 || !hq || !sh ||
      !y_rows)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(xq) || !aligned16(w13) || !aligned16(w2) || !aligned16(hq) || !aligned16(y_rows))
    return MOE_ERR_INVALID_ARG;
  const size_t need = gathered_bytes(rows, d);
  if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  uint8_t* xr = static_cast<uint8_t*>(ws);
  float* sxr = reinterpret_cast<float*>(xr + align256(static_cast<size_t>(rows) * d));
  st = moe::launch_gather_rows_fp8(xq, sx, T, row_token, offsets + n_segments, rows, d, xr, sxr,
                                   dev_status, s);
  if (st != MOE_OK) return st;

  GemmArgs up{};
  up.A = xr; up.sA = sxr; up.B = w13; up.sB = s13; up.seg = offsets;
  up.G = n_segments; up.M = rows; up.N = 2 * f; up.K = d;
  up.hq = hq; up.sh = sh; up.status = dev_status;
  st = moe::launch_fp8_gemm(up, moe::kEpiSwiGLU, s);
  if (st != MOE_OK) return st;

  GemmArgs down{};
  down.A = hq; down.sA = sh; down.B = w2; down.sB = s2; down.seg = offsets;
  down.G = n_segments; down.M = rows; down.N = d; down.K = f;
  down.C = y_rows; down.ldc = d; down.status = dev_status;
  return moe::launch_fp8_gemm(down, moe::kEpiBF16, s);
}

int moe_gather_rows_fp8(const uint8_t* src, const float* src_scale, int src_rows,
                        const int32_t* rows, const int32_t* row_limit, int n_rows, int cols,
                        uint8_t* dst, float* dst_scale, int32_t* dev_status, void* stream) {
  if (src_rows < 0 || n_rows < 0 || cols <= 0 || cols % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (n_rows == 0) return MOE_OK;
  if (!src || !src_scale || !rows || !dst || !dst_scale || !aligned16(src) || !aligned16(dst))
    return MOE_ERR_INVALID_ARG;
  return moe::launch_gather_rows_fp8(src, src_scale, src_rows, rows, row_limit, n_rows, cols, dst,
                                     dst_scale, dev_status, as_stream(stream));
}

int moe_gate_up_fp8(const uint8_t* xq_rows, const float* sx_rows, const int32_t* offsets,
                    int rows, const uint8_t* w13, const float* s13, int n_segments, int d, int f,
                    uint8_t* hq, float* sh, int32_t* dev_status, void* stream) {
  if (rows < 0 || d <= 0 || f <= 0 || d % 128 != 0 || f % 128 != 0 || n_segments < 1)
    return MOE_ERR_INVALID_ARG;
  const int st = check_gemm_dims(n_segments, rows, 2 * f, d);
  if (st != MOE_OK) return st;
  if (rows == 0) return MOE_OK;
  if (!xq_rows || !sx_rows || !offsets || !w13 || !s13 || !hq || !sh) return MOE_ERR_INVALID_ARG;
  if (!aligned16(xq_rows) || !aligned16(w13) || !aligned16(hq)) return MOE_ERR_INVALID_ARG;
  GemmArgs up{};
  up.A = xq_rows; up.sA = sx_rows; up.B = w13; up.sB = s13; up.seg = offsets;
  up.G = n_segments; up.M = rows; up.N = 2 * f; up.K = d;
  up.hq = hq; up.sh = sh; up.status = dev_status;
  return moe::launch_fp8_gemm(up, moe::kEpiSwiGLU, as_stream(stream));
}

int moe_gate_up_mx(const uint8_t* xq_rows, const float* sx_rows, const int32_t* offsets,
                   int rows, const uint8_t* w13, const float* s13, int n_segments, int d, int f,
                   uint8_t* hq, float* sh, int32_t* dev_status, void* stream) {
  if (rows < 0 || d <= 0 || f <= 0 || d % 128 != 0 || f % 128 != 0 || n_segments < 1)
    return MOE_ERR_INVALID_ARG;
  const int st = check_gemm_dims(n_segments, rows, 2 * f, d);
  if (st != MOE_OK) return st;
  if (rows == 0) return MOE_OK;
  if (!xq_rows || !sx_rows || !offsets || !w13 || !s13 || !hq || !sh) return MOE_ERR_INVALID_ARG;
  if (!aligned16(xq_rows) || !aligned16(w13) || !aligned16(hq)) return MOE_ERR_INVALID_ARG;
  return moe::launch_mx_gemm(xq_rows, sx_rows, w13, s13, offsets, n_segments, rows, 2 * f, d,
                             nullptr, 0, hq, sh, moe::kEpiSwiGLU, dev_status, as_stream(stream));
}

// ---- backward of the experts (training) ----------------------------------------------

int moe_gate_up_fp8_train(const uint8_t* xq_rows, const float* sx_rows, const int32_t* offsets,
                          int rows, const uint8_t* w13, const float* s13, int n_segments, int d,
                          int f, uint8_t* hq, float* sh, uint8_t* guq, float* sgu,
                          int32_t* dev_status, void* stream) {
  if (rows < 0 || d <= 0 || f <= 0 || d % 128 != 0 || f % 128 != 0 || n_segments < 1)
    return MOE_ERR_INVALID_ARG;
  const int st = check_gemm_dims(n_segments, rows, 2 * f, d);
  if (st != MOE_OK) return st;
  if (rows == 0) return MOE_OK;
  if (!xq_rows || !sx_rows || !offsets || !w13 || !s13 || !hq || !sh || !guq || !sgu)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(xq_rows) || !aligned16(w13) || !aligned16(hq) || !aligned16(guq))
    return MOE_ERR_INVALID_ARG;
  GemmArgs up{};
  up.A = xq_rows; up.sA = sx_rows; up.B = w13; up.sB = s13; up.seg = offsets;
  up.G = n_segments; up.M = rows; up.N = 2 * f; up.K = d;
  up.hq = hq; up.sh = sh; up.guq = guq; up.sgu = sgu; up.status = dev_status;
  return moe::launch_fp8_gemm(up, moe::kEpiSwiGLUCache, as_stream(stream));
}

int fp8_transpose_128x128(const uint8_t* w, const float* s, int G, int rows, int cols,
                          int gate_up_interleaved, uint8_t* wT, float* sT, void* stream) {
  if (G < 1 || rows < 0 || cols < 0 || rows % 128 != 0 || cols % 128 != 0)
    return MOE_ERR_INVALID_ARG;
  if (gate_up_interleaved && rows % 256 != 0) return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(G) > 65535) return MOE_ERR_UNSUPPORTED;
  if (rows == 0 || cols == 0) return MOE_OK;
  if (!w || !s || !wT || !sT) return MOE_ERR_INVALID_ARG;
  return moe::launch_transpose_fp8(w, s, G, rows, cols, gate_up_interleaved != 0, wT, sT,
                                   as_stream(stream));
}

int moe_padded_rows_cap(int rows, int G) {
  if (rows < 0 || G < 1) return -1;
  const long long cap = (static_cast<long long>(rows) + 127LL * G + 127) / 128 * 128;
  return cap > INT32_MAX ? -1 : static_cast<int>(cap);
}

int moe_segment_pad_offsets(const int32_t* offsets, int G, int32_t* pad, int32_t* dev_status,
                            void* stream) {
  if (G < 1) return MOE_ERR_INVALID_ARG;
  if (G > 1024) return MOE_ERR_UNSUPPORTED;
  if (!offsets || !pad) return MOE_ERR_INVALID_ARG;
  return moe::launch_seg_pad(offsets, G, pad, dev_status, as_stream(stream));
}

int moe_combine_bwd_rows(const uint16_t* dy, const float* topk_gate, const int32_t* row_of,
                         int T, int K, int d, int shared_row_base, int n_rows, uint16_t* dy_rows,
                         int32_t* dev_status, void* stream) {
  if (T < 0 || K < 1 || d <= 0 || d % 8 != 0 || n_rows < 0) return MOE_ERR_INVALID_ARG;
  if (K > 32) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!dy || !topk_gate || !row_of || !dy_rows || !aligned16(dy) || !aligned16(dy_rows))
    return MOE_ERR_INVALID_ARG;
  return moe::launch_dispatch_grad(dy, topk_gate, row_of, T, K, d, shared_row_base, n_rows,
                                   dy_rows, dev_status, as_stream(stream));
}

int fp8_quant_128x1_pow2(const uint16_t* src, int src_rows, const int32_t* rows, int cols,
                         const int32_t* offsets, const int32_t* pad, int G, int kcap,
                         uint8_t* qT, float* sT, int32_t* dev_status, void* stream) {
  if (src_rows < 0 || cols <= 0 || cols % 128 != 0 || G < 1 || kcap < 0 || kcap % 128 != 0)
    return MOE_ERR_INVALID_ARG;
  if (G > 1024 || cols / 128 > 65535) return MOE_ERR_UNSUPPORTED;
  if (kcap == 0) return MOE_OK;
  if (!src || !offsets || !pad || !qT || !sT || !aligned16(src) || !aligned16(qT))
    return MOE_ERR_INVALID_ARG;
  return moe::launch_regroup_128x1(src, src_rows, rows, cols, offsets, pad, G, kcap / 128, kcap,
                                   qT, sT, dev_status, as_stream(stream));
}

int moe_swiglu_bwd_fp8(const uint8_t* guq, const float* sgu, const uint16_t* dh, int rows, int f,
                       const int32_t* offsets, const int32_t* pad, int G, int kcap,
                       uint8_t* dguq, float* sdgu, uint8_t* hT, float* shT, uint8_t* dguT,
                       float* sdguT, void* stream) {
  if (rows < 0 || f <= 0 || f % 128 != 0 || G < 1 || kcap < 0 || kcap % 128 != 0)
    return MOE_ERR_INVALID_ARG;
  if (G > 1024 || f / 128 > 65535) return MOE_ERR_UNSUPPORTED;
  if (rows == 0 || kcap == 0) return MOE_OK;
  if (!guq || !sgu || !dh || !offsets || !pad || !dguq || !sdgu || !hT || !shT || !dguT || !sdguT)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(guq) || !aligned16(dh) || !aligned16(hT) || !aligned16(dguT))
    return MOE_ERR_INVALID_ARG;
  return moe::launch_swiglu_bwd(guq, sgu, dh, rows, f, offsets, pad, G, kcap / 128, kcap, dguq,
                                sdgu, hT, shT, dguT, sdguT, as_stream(stream));
}

int fp8_wgrad_grouped_gemm(const uint8_t* aT, const float* saT, const uint8_t* bT,
                           const float* sbT, const int32_t* pad, int G, int I, int J, int kcap,
                           float* dW, int32_t* dev_status, void* stream) {
  if (G < 1 || I <= 0 || J <= 0 || kcap <= 0 || I % 128 != 0 || J % 128 != 0 || kcap % 128 != 0)
    return MOE_ERR_INVALID_ARG;
  if (G > 1024 || static_cast<long long>(G) * (I / 128) * ((J + 255) / 256) > INT32_MAX)
    return MOE_ERR_UNSUPPORTED;
  if (!aT || !saT || !bT || !sbT || !pad || !dW || !aligned16(aT) || !aligned16(bT) ||
      !aligned16(dW))
    return MOE_ERR_INVALID_ARG;
  return moe::launch_wgrad_gemm(aT, saT, bT, sbT, pad, G, I, J, kcap, dW, dev_status,
                                as_stream(stream));
}

// ---- combine, bias update, workspace -------------------------------------------------

int moe_combine(const uint16_t* y_rows, int n_rows, const int32_t* row_of, const float* gate,
                int T, int K, int d, int shared_row_base, uint16_t* y, int32_t* dev_status,
                void* stream) {
  if (T < 0 || K < 1 || d <= 0 || d % 8 != 0 || n_rows < 0) return MOE_ERR_INVALID_ARG;
  if (K > 32) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!y_rows || !row_of || !gate || !y || !aligned16(y_rows) || !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  return moe::launch_combine(y_rows, n_rows, row_of, gate, T, K, d, shared_row_base, y,
                             dev_status, as_stream(stream));
}

int moe_bias_update(float* bias, const int32_t* counts, int E, int T, int K, float gamma,
                    void* stream) {
  if (E < 1 || T < 0 || K < 1) return MOE_ERR_INVALID_ARG;
  if (!bias || !counts) return MOE_ERR_INVALID_ARG;
  return moe::launch_bias_update(bias, counts, E, T, K, gamma, as_stream(stream));
}

size_t moe_seq_balance_stats_ws_bytes(int T, int E, int seq_len) {
  if (T <= 0 || E <= 0 || seq_len <= 0 || T % seq_len != 0) return 0;
  return moe::seq_balance_ws_bytes(T, E, seq_len);
}

int moe_seq_balance_stats(const float* scores, int scores_are_affinities, int T, int E, int K,
                          int seq_len, float alpha, float* f, float* P, float* loss, void* ws,
                          size_t ws_bytes, void* stream) {
  if (T < 0 || E < 1 || K < 1 || K > E || seq_len < 1 || T % seq_len != 0)
    return MOE_ERR_INVALID_ARG;
  if (E > 1024 || K > 32 || T / seq_len > 65535) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!scores || !f || !P || !loss) return MOE_ERR_INVALID_ARG;
  const size_t need = moe::seq_balance_ws_bytes(T, E, seq_len);
  if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
  return moe::launch_seq_balance(scores, scores_are_affinities, T, E, K, seq_len, alpha, f, P,
                                 loss, ws, as_stream(stream));
}

size_t moe_workspace_bytes(int T, int K, int E, int d, int f) {
  (void)f;
  if (T <= 0 || K <= 0 || E <= 0 || d <= 0) return 0;
  const long long rows = static_cast<long long>(T) * (K + 1);
  size_t need = moe::permute_ws_bytes(T, K, E);
  const size_t sw = gathered_bytes(rows, d);
  if (sw > need) need = sw;
  const size_t rl = moe::router_logits_ws_bytes(T, d, E);
  if (rl > need) need = rl;
  return need;
}

}  // extern "C"
