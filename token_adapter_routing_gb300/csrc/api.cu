// api.cu -- the C ABI declared in include/molora.h: host-side argument validation, then
// kernel selection and launch.  Nothing here allocates, frees or synchronises.
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace molora {

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool valid_dtype(molora_dtype d) { return d == MOLORA_F32 || d == MOLORA_BF16; }
static molora_status launched(cudaError_t e) { return e == cudaSuccess ? MOLORA_OK : MOLORA_ERR_CUDA; }

// Smallest slot count (N*k) at which the grouped tensor-core apply beats the scalar apply,
// measured on GB300 with the decode sweep (d = 4096, top-1, batch 1..2048, K = 4..64 hot-set
// adapters drawn uniformly and Zipf(1.1); vocabulary routing -> scalar apply against routing with
// dispatch -> grouped apply; calls back to back in one CUDA graph, the decode steady state with
// the hot set in L2).  The scalar path re-reads its token's A_a and B_a (d_in r + r d_out
// elements) from L2 for every token, so the crossover falls as the rank grows:
//   r <= 16: 768 tokens up to 8 adapters, 1024 with 16, 2048 with 32; scalar at every batch
//            measured with 64;
//   r = 32:  768 up to 16 adapters, 1536 with 32 (768 under uniform draws, 1536 under Zipf),
//            2048 with 64;
//   r = 64:  160 up to 8 adapters (Figures 5 and 9 put it near batch 160 for 8 adapters of rank
//            64), 512 with 16, 768 with 32, 1024 with 64.
static int64_t crossover_tokens(int32_t K, int32_t r) {
  if (r >= 64) {
    if (K <= 8) return 160;
    if (K <= 16) return 512;
    if (K <= 32) return 768;
    return 1024;
  }
  if (r >= 32) {
    if (K <= 16) return 768;
    if (K <= 32) return 1536;
    return 2048;
  }
  if (K <= 8) return 768;
  if (K <= 16) return 1024;
  if (K <= 32) return 2048;
  return 4096;
}

static molora_status check_apply_sizes(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K,
                                       int32_t r, int32_t k) {
  if (!valid_dtype(dtype) || N < 0 || d_in < 1 || d_out < 1 || K < 1 || K > kMaxAdapters || k < 1 || k > K)
    return MOLORA_ERR_INVALID_ARG;
  if (!(r == 8 || r == 16 || r == 32 || r == 64)) return MOLORA_ERR_INVALID_ARG;
  if (N > INT32_MAX || N * (int64_t)k > INT32_MAX) return MOLORA_ERR_INVALID_ARG;
  return MOLORA_OK;
}

static molora_status check_apply_args(const void* x, molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out,
                                      const void* A, const void* B, int32_t K, int32_t r, const int32_t* ids,
                                      int32_t k, const void* y) {
  const molora_status st = check_apply_sizes(dtype, N, d_in, d_out, K, r, k);
  if (st != MOLORA_OK || N == 0) return st;
  if (!x || !A || !B || !ids || !y) return MOLORA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(A) || !aligned16(B) || !aligned16(y)) return MOLORA_ERR_INVALID_ARG;
  return MOLORA_OK;
}

// The best path that needs no workspace (AUTO without one, or with the adapter table of the
// indirect layout, which only the scalar and grouped kernels read).
static molora_path select_without_ws(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K,
                                     int32_t r, int32_t k, bool table) {
  if (!table && k >= 2 && dense_preferred(dtype, N, d_in, d_out, K, r)) return MOLORA_PATH_DENSE;
  if (!grouped_supported(dtype, N, d_in, d_out, K, r, k)) return MOLORA_PATH_SCALAR;
  return N * (int64_t)k >= crossover_tokens(K, r) ? MOLORA_PATH_GROUPED : MOLORA_PATH_SCALAR;
}

// Workspace convention (include/molora.h): ws_bytes == NULL -> none; ws == NULL -> query;
// else a buffer of *ws_bytes bytes.  `need` is what the chosen path needs.
static molora_status check_ws(void* ws, size_t* ws_bytes, size_t need, bool* query) {
  *query = ws_bytes != nullptr && ws == nullptr;
  if (*query) {
    *ws_bytes = need;
    return MOLORA_OK;
  }
  if (need == 0) return MOLORA_OK;
  if (!ws || !ws_bytes || *ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOLORA_ERR_INVALID_ARG;
  return MOLORA_OK;
}

static molora_status apply_impl(const void* x, molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out,
                                const void* A, const void* B, int32_t K, int32_t r, const int32_t* ids, const float* w,
                                int32_t k, const int32_t* counts, const int32_t* offsets, const int32_t* perm,
                                float scale, void* y, bool y_bf16, int32_t* err_word, molora_path path,
                                cudaStream_t stream, const AdapterTable* table = nullptr, void* ws = nullptr,
                                size_t* ws_bytes = nullptr) {
  const bool have_ws = ws_bytes != nullptr;
  const bool query = have_ws && ws == nullptr;  // sizes only: no pointer is looked at
  const molora_status st = query ? check_apply_sizes(dtype, N, d_in, d_out, K, r, k)
                                 : check_apply_args(x, dtype, N, d_in, d_out, A, B, K, r, ids, k, y);
  if (st != MOLORA_OK) return st;
  if (path == MOLORA_PATH_AUTO) {
    if (table) {
      // the adapter table is read by the scalar and grouped kernels only: choose between them
      path = select_without_ws(dtype, N, d_in, d_out, K, r, k, true);
    } else {
      path = molora_select_path(dtype, N, d_in, d_out, K, r, k);
      if (path == MOLORA_PATH_STACKED && (!have_ws || y_bf16 || !stacked_supported(dtype, N, d_in, d_out, K, r, false)))
        path = select_without_ws(dtype, N, d_in, d_out, K, r, k, false);
    }
    // AUTO takes the grouped path only with the dispatch outputs it reads; without them, the
    // fastest path that needs none (the stacked pair if its workspace was given)
    if (path == MOLORA_PATH_GROUPED && !query && (!counts || !offsets || !perm)) {
      const bool ws_fits = have_ws && ws != nullptr && *ws_bytes >= stacked_workspace_bytes(N, K, r);
      if (!table && !y_bf16 && ws_fits && stacked_supported(dtype, N, d_in, d_out, K, r, false))
        path = MOLORA_PATH_STACKED;
      else if (!table && k >= 2 && dense_supported(dtype, N, d_in, d_out, K, r))
        path = MOLORA_PATH_DENSE;
      else
        path = MOLORA_PATH_SCALAR;
    }
  }
  if (path == MOLORA_PATH_STACKED) {
    if (!have_ws) return N == 0 ? MOLORA_OK : MOLORA_ERR_INVALID_ARG;
    if (table || y_bf16 || !stacked_supported(dtype, N, d_in, d_out, K, r, false)) return MOLORA_ERR_UNSUPPORTED;
    bool is_query = false;
    const molora_status ws_st = check_ws(ws, ws_bytes, stacked_workspace_bytes(N, K, r), &is_query);
    if (ws_st != MOLORA_OK || is_query || N == 0) return ws_st;
    return launched(launch_lora_stacked(x, N, d_in, d_out, A, B, K, r, ids, w, k, scale, static_cast<float*>(y), ws,
                                        err_word, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                        stream));
  }
  if (path < MOLORA_PATH_AUTO || path > MOLORA_PATH_STACKED) return MOLORA_ERR_INVALID_ARG;
  if (query) {  // the other paths need no workspace
    *ws_bytes = 0;
    return MOLORA_OK;
  }
  if (N == 0) return MOLORA_OK;
  if (path == MOLORA_PATH_SCALAR)
    return launched(launch_lora_scalar(x, dtype, N, d_in, d_out, A, B, K, r, ids, w, k, scale, y, y_bf16, -1,
                                       err_word, stream, table));
  if (path == MOLORA_PATH_DENSE) {
    if (table || !dense_supported(dtype, N, d_in, d_out, K, r)) return MOLORA_ERR_UNSUPPORTED;
    return launched(launch_lora_dense(x, N, d_in, d_out, A, B, K, r, ids, w, k, scale, y, y_bf16, err_word, stream));
  }
  if (path != MOLORA_PATH_GROUPED) return MOLORA_ERR_INVALID_ARG;
  if (!grouped_supported(dtype, N, d_in, d_out, K, r, k)) return MOLORA_ERR_UNSUPPORTED;
  if (!counts || !offsets || !perm) return MOLORA_ERR_INVALID_ARG;
  return launched(launch_lora_grouped(x, N, d_in, d_out, A, B, K, r, ids, w, k, counts, offsets, perm, scale, y,
                                      y_bf16, -1, err_word, stream, table));
}

}  // namespace molora

using namespace molora;

extern "C" {

molora_status molora_route_vocab_ex(const int32_t* tok, int64_t N, const int32_t* starts, int32_t K,
                                    int32_t* adapter, int32_t* err_word, uint32_t flags, cudaStream_t stream) {
  if (flags & ~(uint32_t)MOLORA_INPUTS_READY) return MOLORA_ERR_INVALID_ARG;
  if (N < 0 || K < 1 || K > kMaxAdapters) return MOLORA_ERR_INVALID_ARG;
  if (N == 0) return MOLORA_OK;
  if (!tok || !starts || !adapter) return MOLORA_ERR_INVALID_ARG;
  const int early = (flags & MOLORA_INPUTS_READY) ? 1 : 0;
  return launched(launch_route_vocab(tok, N, starts, K, adapter, err_word, early, stream));
}

molora_status molora_route_vocab(const int32_t* tok, int64_t N, const int32_t* starts, int32_t K, int32_t* adapter,
                                 int32_t* err_word, cudaStream_t stream) {
  return molora_route_vocab_ex(tok, N, starts, K, adapter, err_word, 0u, stream);
}

molora_status molora_router_topk(const void* x, molora_dtype dtype, int64_t N, int32_t d_in, const void* W1,
                                 const float* b1, const void* W2, const float* b2, int32_t K, int32_t k,
                                 float* logits, int32_t* ids, float* w, cudaStream_t stream) {
  if (!valid_dtype(dtype) || N < 0 || d_in < 1 || K < 1 || K > kMaxAdapters || k < 1 || k > K)
    return MOLORA_ERR_INVALID_ARG;
  if (N > INT32_MAX || N * (int64_t)K > INT32_MAX) return MOLORA_ERR_INVALID_ARG;
  if (N == 0) return MOLORA_OK;
  if (!x || !W1 || !W2 || !ids || !w) return MOLORA_ERR_INVALID_ARG;
  if (router_tc_supported(dtype, N, d_in, K, k)) {
    if (!aligned16(x) || !aligned16(W1)) return MOLORA_ERR_INVALID_ARG;
    return launched(launch_router_tc(x, N, d_in, W1, b1, W2, b2, K, k, logits, ids, w, stream));
  }
  return launched(launch_router_scalar(x, dtype, N, d_in, W1, b1, W2, b2, K, k, logits, ids, w, stream));
}

molora_status molora_dispatch(const int32_t* ids, int64_t N, int32_t k, int32_t K, int32_t* counts, int32_t* offsets,
                              int32_t* perm, int32_t* err_word, cudaStream_t stream) {
  if (N < 0 || k < 1 || K < 1 || K > kMaxAdapters || k > K) return MOLORA_ERR_INVALID_ARG;
  if (N * (int64_t)k > INT32_MAX) return MOLORA_ERR_INVALID_ARG;
  if (!counts || !offsets || (N > 0 && (!ids || !perm))) return MOLORA_ERR_INVALID_ARG;
  return launched(launch_dispatch(ids, N, k, K, counts, offsets, perm, err_word, stream));
}

molora_status molora_route_vocab_dispatch(const int32_t* tok, int64_t N, const int32_t* starts, int32_t K,
                                          int32_t* adapter, int32_t* counts, int32_t* offsets, int32_t* perm,
                                          int32_t* err_word, cudaStream_t stream) {
  if (N < 0 || K < 1 || K > kMaxAdapters || N > INT32_MAX) return MOLORA_ERR_INVALID_ARG;
  if (!starts || !counts || !offsets || (N > 0 && (!tok || !adapter || !perm))) return MOLORA_ERR_INVALID_ARG;
  return launched(launch_route_vocab_dispatch(tok, N, starts, K, adapter, counts, offsets, perm, err_word, 0, stream));
}

molora_status molora_route_vocab_dispatch_ex(const int32_t* tok, int64_t N, const int32_t* starts, int32_t K,
                                             int32_t* adapter, int32_t* counts, int32_t* offsets, int32_t* perm,
                                             int32_t* err_word, uint32_t flags, cudaStream_t stream) {
  if (flags & ~(uint32_t)MOLORA_INPUTS_READY) return MOLORA_ERR_INVALID_ARG;
  if (N < 0 || K < 1 || K > kMaxAdapters || N > INT32_MAX) return MOLORA_ERR_INVALID_ARG;
  if (!starts || !counts || !offsets || (N > 0 && (!tok || !adapter || !perm))) return MOLORA_ERR_INVALID_ARG;
  const int early = (flags & MOLORA_INPUTS_READY) ? 1 : 0;
  return launched(launch_route_vocab_dispatch(tok, N, starts, K, adapter, counts, offsets, perm, err_word, early, stream));
}

molora_status molora_route_vocab_lora_apply_ex(const int32_t* tok, int64_t N, const int32_t* starts, int32_t K,
                                               const void* x, molora_dtype dtype, int32_t d_in, int32_t d_out,
                                               const void* A, const void* B, int32_t r, float scale, void* y,
                                               int32_t y_bf16, int32_t* adapter, int32_t* counts, int32_t* offsets,
                                               int32_t* perm, int32_t* err_word, uint32_t flags, cudaStream_t stream) {
  if (flags & ~(uint32_t)MOLORA_INPUTS_READY) return MOLORA_ERR_INVALID_ARG;
  const molora_status st = check_apply_args(x, dtype, N, d_in, d_out, A, B, K, r, tok, 1, y);
  if (st != MOLORA_OK) return st;
  if (!starts || !counts || !offsets || (N > 0 && (!adapter || !perm))) return MOLORA_ERR_INVALID_ARG;
  const int early = (flags & MOLORA_INPUTS_READY) ? 1 : 0;
  if (N == 0)  // the empty histogram, as molora_route_vocab_dispatch writes it
    return launched(launch_route_vocab_dispatch(tok, 0, starts, K, adapter, counts, offsets, perm, err_word, early,
                                                stream));
  const molora_path path = select_without_ws(dtype, N, d_in, d_out, K, r, 1, false);
  if (launch_route_vocab_dispatch(tok, N, starts, K, adapter, counts, offsets, perm, err_word, early, stream) !=
      cudaSuccess)
    return MOLORA_ERR_CUDA;
  return apply_impl(x, dtype, N, d_in, d_out, A, B, K, r, adapter, nullptr, 1, counts, offsets, perm, scale, y,
                    y_bf16 != 0, err_word, path, stream);
}

molora_status molora_route_vocab_lora_apply(const int32_t* tok, int64_t N, const int32_t* starts, int32_t K,
                                            const void* x, molora_dtype dtype, int32_t d_in, int32_t d_out,
                                            const void* A, const void* B, int32_t r, float scale, void* y,
                                            int32_t y_bf16, int32_t* adapter, int32_t* counts, int32_t* offsets,
                                            int32_t* perm, int32_t* err_word, cudaStream_t stream) {
  return molora_route_vocab_lora_apply_ex(tok, N, starts, K, x, dtype, d_in, d_out, A, B, r, scale, y, y_bf16,
                                          adapter, counts, offsets, perm, err_word, 0u, stream);
}

molora_path molora_select_path(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r,
                               int32_t k) {
  if (stacked_preferred(dtype, N, d_in, d_out, K, r, k, false)) return MOLORA_PATH_STACKED;
  return select_without_ws(dtype, N, d_in, d_out, K, r, k, false);
}

molora_status molora_lora_apply_ex(const void* x, molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out,
                                   const void* A, const void* B, int32_t K, int32_t r, const int32_t* ids,
                                   const float* w, int32_t k, const int32_t* counts, const int32_t* offsets,
                                   const int32_t* perm, float scale, float* y, void* ws, size_t* ws_bytes,
                                   int32_t* err_word, molora_path path, cudaStream_t stream) {
  return molora::apply_impl(x, dtype, N, d_in, d_out, A, B, K, r, ids, w, k, counts, offsets, perm, scale, y, false,
                            err_word, path, stream, nullptr, ws, ws_bytes);
}

molora_status molora_lora_apply_bf16y(const void* x, molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out,
                                      const void* A, const void* B, int32_t K, int32_t r, const int32_t* ids,
                                      const float* w, int32_t k, const int32_t* counts, const int32_t* offsets,
                                      const int32_t* perm, float scale, void* y, int32_t* err_word,
                                      molora_path path, cudaStream_t stream) {
  return molora::apply_impl(x, dtype, N, d_in, d_out, A, B, K, r, ids, w, k, counts, offsets, perm, scale, y, true,
                            err_word, path, stream);
}

molora_status molora_lora_apply_indirect(const void* x, molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out,
                                         const void* const* A_ptrs, const void* const* B_ptrs, int32_t K, int32_t r,
                                         const int32_t* ids, const float* w, int32_t k, const int32_t* counts,
                                         const int32_t* offsets, const int32_t* perm, float scale, void* y,
                                         int32_t y_bf16, int32_t* err_word, molora_path path, cudaStream_t stream) {
  if (!A_ptrs || !B_ptrs || K < 1 || K > kMaxAdapters) return MOLORA_ERR_INVALID_ARG;
  molora::AdapterTable table;
  for (int i = 0; i < kMaxAdapters; ++i) table.a[i] = table.b[i] = nullptr;
  for (int32_t i = 0; i < K; ++i) {
    if (!A_ptrs[i] || !B_ptrs[i] || !aligned16(A_ptrs[i]) || !aligned16(B_ptrs[i])) return MOLORA_ERR_INVALID_ARG;
    table.a[i] = A_ptrs[i];
    table.b[i] = B_ptrs[i];
  }
  return molora::apply_impl(x, dtype, N, d_in, d_out, A_ptrs[0], B_ptrs[0], K, r, ids, w, k, counts, offsets, perm,
                            scale, y, y_bf16 != 0, err_word, path, stream, &table);
}

molora_status molora_router_lora_apply(const void* x, molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out,
                                       const void* W1, const float* b1, const void* W2, const float* b2,
                                       const void* A, const void* B, int32_t K, int32_t r, int32_t k, float scale,
                                       float* logits, int32_t* ids, float* w, void* y, int32_t y_bf16, void* ws,
                                       size_t* ws_bytes, int32_t* err_word, cudaStream_t stream) {
  const bool query = ws_bytes != nullptr && ws == nullptr;  // sizes only: no pointer is looked at
  const molora_status st = query ? check_apply_sizes(dtype, N, d_in, d_out, K, r, k)
                                 : check_apply_args(x, dtype, N, d_in, d_out, A, B, K, r, ids, k, y);
  if (st != MOLORA_OK) return st;
  if (N * (int64_t)K > INT32_MAX) return MOLORA_ERR_INVALID_ARG;
  if (!query && N > 0 && (!W1 || !W2 || !w || !aligned16(W1))) return MOLORA_ERR_INVALID_ARG;
  // A query sizes the preferred family: the stacked pair where it applies and either wins or is
  // the only one.  A call given a buffer runs the stacked pair wherever it applies.
  const bool one_kernel = router_dense_supported(dtype, N, d_in, d_out, K, r);
  const bool stacked_ok = y_bf16 == 0 && stacked_supported(dtype, N, d_in, d_out, K, r, true);
  const bool stacked = stacked_ok && ws_bytes != nullptr &&
                       (query ? !one_kernel || stacked_preferred(dtype, N, d_in, d_out, K, r, k, true) : true);
  if (stacked) {
    bool is_query = false;
    const molora_status ws_st = check_ws(ws, ws_bytes, stacked_workspace_bytes(N, K, r), &is_query);
    if (ws_st != MOLORA_OK || is_query || N == 0) return ws_st;
    return launched(launch_lora_stacked(x, N, d_in, d_out, A, B, K, r, nullptr, nullptr, k, scale,
                                        static_cast<float*>(y), ws, err_word, W1, b1, W2, b2, logits, ids, w, stream));
  }
  if (query) {  // the one-kernel path needs no workspace
    *ws_bytes = 0;
    return one_kernel || N == 0 ? MOLORA_OK : MOLORA_ERR_UNSUPPORTED;
  }
  if (N == 0) return MOLORA_OK;
  if (!one_kernel) return MOLORA_ERR_UNSUPPORTED;
  return launched(launch_router_lora_dense(x, N, d_in, d_out, W1, b1, W2, b2, A, B, K, r, k, scale, logits, ids, w, y,
                                           y_bf16 != 0, err_word, stream));
}

molora_status molora_lora_apply(const void* x, molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out,
                                const void* A, const void* B, int32_t K, int32_t r, const int32_t* ids, const float* w,
                                int32_t k, const int32_t* counts, const int32_t* offsets, const int32_t* perm,
                                float scale, float* y, void* ws, size_t* ws_bytes, int32_t* err_word,
                                cudaStream_t stream) {
  return molora_lora_apply_ex(x, dtype, N, d_in, d_out, A, B, K, r, ids, w, k, counts, offsets, perm, scale, y, ws,
                              ws_bytes, err_word, MOLORA_PATH_AUTO, stream);
}

molora_status molora_lora_apply_masked_pass(const void* x, molora_dtype dtype, int64_t N, int32_t d_in,
                                            int32_t d_out, const void* A, const void* B, int32_t K, int32_t r,
                                            const int32_t* adapter_of, int32_t a, float scale, float* y,
                                            int32_t* err_word, molora_path path, cudaStream_t stream) {
  const molora_status st = check_apply_args(x, dtype, N, d_in, d_out, A, B, K, r, adapter_of, 1, y);
  if (st != MOLORA_OK) return st;
  if (a < 0 || a >= K) return MOLORA_ERR_INVALID_ARG;
  if (N == 0) return MOLORA_OK;
  // a masked pass takes no workspace: AUTO chooses between the scalar and grouped kernels
  if (path == MOLORA_PATH_AUTO) path = select_without_ws(dtype, N, d_in, d_out, K, r, 1, false);
  if (path == MOLORA_PATH_SCALAR)
    return launched(launch_lora_scalar(x, dtype, N, d_in, d_out, A, B, K, r, adapter_of, nullptr, 1, scale, y, false,
                                       a, err_word, stream));
  if (path != MOLORA_PATH_GROUPED) return MOLORA_ERR_INVALID_ARG;
  if (!grouped_supported(dtype, N, d_in, d_out, K, r, 1)) return MOLORA_ERR_UNSUPPORTED;
  return launched(launch_lora_grouped(x, N, d_in, d_out, A, B, K, r, adapter_of, nullptr, 1, nullptr, nullptr,
                                      nullptr, scale, y, false, a, err_word, stream));
}

molora_status molora_lora_apply_static_ws(const void* x, molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out,
                                          const void* A, const void* B, int32_t K, int32_t r, const int32_t* ids,
                                          const float* w, int32_t k, float scale, float* y, int32_t* err_word,
                                          cudaStream_t stream) {
  const molora_status st = check_apply_args(x, dtype, N, d_in, d_out, A, B, K, r, ids, k, y);
  if (st != MOLORA_OK || N == 0) return st;
  if (!stacked_supported(dtype, N, d_in, d_out, K, r, false)) return MOLORA_ERR_UNSUPPORTED;
  const size_t need = stacked_workspace_bytes(N, K, r);
  if (need > stacked_static_scratch_bytes() || stacked_static_scratch_bytes() != MOLORA_STATIC_SCRATCH_BYTES)
    return MOLORA_ERR_SCRATCH_TOO_SMALL;
  void* scratch = nullptr;
  if (stacked_static_scratch(&scratch) != cudaSuccess) return MOLORA_ERR_CUDA;
  return launched(launch_lora_stacked(x, N, d_in, d_out, A, B, K, r, ids, w, k, scale, y, scratch, err_word, nullptr,
                                      nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, stream));
}

const char* molora_status_string(molora_status status) {
  switch (status) {
    case MOLORA_OK:
      return "ok";
    case MOLORA_ERR_INVALID_ARG:
      return "invalid argument";
    case MOLORA_ERR_UNSUPPORTED:
      return "unsupported shape for this path";
    case MOLORA_ERR_CUDA:
      return "CUDA launch error";
    case MOLORA_ERR_SCRATCH_TOO_SMALL:
      return "problem too large for the fixed scratch buffer (N * K * r too large)";
  }
  return "unknown status";
}

int32_t molora_version(void) { return 100; }

molora_status molora_selftest_bounded_wait(uint32_t limit_us, int32_t* err_word, cudaStream_t stream) {
  if (!err_word || limit_us == 0 || limit_us > 1000000u) return MOLORA_ERR_INVALID_ARG;
  return launched(launch_bounded_wait_selftest((uint64_t)limit_us * 1000ull, err_word, stream));
}

}  // extern "C"
