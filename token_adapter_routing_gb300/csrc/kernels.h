// kernels.h -- host-side launchers of the library's kernels (internal; the public surface
// is include/molora.h).  Each launcher assumes its arguments were validated by api.cu and
// returns the launch's cudaError_t.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "molora.h"

namespace molora {

// Per-adapter base addresses for the indirect layout (adapters anywhere in memory): a[i] is
// adapter i's A [d_in x r], b[i] its B [r x d_out].  Passed to kernels by value.
struct AdapterTable {
  const void* a[MOLORA_MAX_ADAPTERS];
  const void* b[MOLORA_MAX_ADAPTERS];
};

// early != 0: tok and starts are not written by the preceding kernel (see route_vocab_kernel).
cudaError_t launch_route_vocab(const int32_t* tok, int64_t N, const int32_t* starts, int32_t K,
                               int32_t* adapter, int32_t* err_word, int early, cudaStream_t stream);

cudaError_t launch_dispatch(const int32_t* ids, int64_t N, int32_t k, int32_t K, int32_t* counts,
                            int32_t* offsets, int32_t* perm, int32_t* err_word, cudaStream_t stream);
// Vocabulary routing and dispatch in one single-CTA kernel (k = 1).  early != 0: tok and starts
// are not written by the preceding kernel, so they are read before waiting on it.
cudaError_t launch_route_vocab_dispatch(const int32_t* tok, int64_t N, const int32_t* starts, int32_t K,
                                        int32_t* adapter, int32_t* counts, int32_t* offsets, int32_t* perm,
                                        int32_t* err_word, int early, cudaStream_t stream);

// Token-major CUDA-core apply.  mask_adapter >= 0 turns it into one masked per-sequence pass:
// adapter mask_adapter for every token, weight [ids[t] == mask_adapter] (k must be 1).
cudaError_t launch_lora_scalar(const void* x, molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out,
                               const void* A, const void* B, int32_t K, int32_t r, const int32_t* ids,
                               const float* w, int32_t k, float scale, void* y, bool y_bf16, int32_t mask_adapter,
                               int32_t* err_word, cudaStream_t stream, const AdapterTable* table = nullptr);

// Token-major tcgen05 apply over all K adapters (K*r = 64 or 128; weight 0 for the unselected).
bool dense_supported(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r);
// True where AUTO takes the dense path (measured faster than the grouped one).
bool dense_preferred(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r);
cudaError_t launch_lora_dense(const void* x, int64_t N, int32_t d_in, int32_t d_out, const void* A, const void* B,
                              int32_t K, int32_t r, const int32_t* ids, const float* w, int32_t k, float scale,
                              void* y, bool y_bf16, int32_t* err_word, cudaStream_t stream);
// The learned router and the dense apply in one kernel: x is read once for both.
bool router_dense_supported(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r);
cudaError_t launch_router_lora_dense(const void* x, int64_t N, int32_t d_in, int32_t d_out, const void* W1,
                                     const float* b1, const void* W2, const float* b2, const void* A, const void* B,
                                     int32_t K, int32_t r, int32_t k, float scale, float* logits, int32_t* ids,
                                     float* w, void* y, bool y_bf16, int32_t* err_word, cudaStream_t stream);

// Stacked two-kernel tcgen05 apply (K*r up to 1024): shrink (optionally with the learned
// router) into a workspace of stacked_workspace_bytes, then a persistent expand GEMM into y.
bool stacked_supported(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r,
                       bool router);
// True where AUTO takes the stacked path (measured faster than the paths needing no workspace).
bool stacked_preferred(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r,
                       int32_t k, bool router);
size_t stacked_workspace_bytes(int64_t N, int32_t K, int32_t r);
// W1 == nullptr: ids and w are given.  Otherwise the router (W1, b1, W2, b2) runs in the shrink
// kernel and writes logits (if non-null), ids_out and w_out.
cudaError_t launch_lora_stacked(const void* x, int64_t N, int32_t d_in, int32_t d_out, const void* A, const void* B,
                                int32_t K, int32_t r, const int32_t* ids, const float* w, int32_t k, float scale,
                                float* y, void* ws, int32_t* err_word, const void* W1, const float* b1,
                                const void* W2, const float* b2, float* logits, int32_t* ids_out, float* w_out,
                                cudaStream_t stream);

// The fixed scratch of molora_lora_apply_static_ws: its size, and its device address on the
// current device (looked up on the first call per device).
size_t stacked_static_scratch_bytes();
cudaError_t stacked_static_scratch(void** ptr);

// CUDA-core learned router (any dtype / shape).
cudaError_t launch_router_scalar(const void* x, molora_dtype dtype, int64_t N, int32_t d_in, const void* W1,
                                 const float* b1, const void* W2, const float* b2, int32_t K, int32_t k,
                                 float* logits, int32_t* ids, float* w, cudaStream_t stream);

// Grouped tcgen05 apply: true if this shape is supported.
bool grouped_supported(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r,
                       int32_t k);
// Grouped tcgen05 apply.  With mask_adapter >= 0 the tiles cover tokens 0..N-1 in order with
// adapter mask_adapter and weight [ids[t] == mask_adapter] (one masked per-sequence pass);
// counts/offsets/perm are then unused.
cudaError_t launch_lora_grouped(const void* x, int64_t N, int32_t d_in, int32_t d_out, const void* A,
                                const void* B, int32_t K, int32_t r, const int32_t* ids, const float* w,
                                int32_t k, const int32_t* counts, const int32_t* offsets, const int32_t* perm,
                                float scale, void* y, bool y_bf16, int32_t mask_adapter, int32_t* err_word,
                                cudaStream_t stream, const AdapterTable* table = nullptr);

// tcgen05 learned router: true if this shape is supported.
bool router_tc_supported(molora_dtype dtype, int64_t N, int32_t d_in, int32_t K, int32_t k);
cudaError_t launch_router_tc(const void* x, int64_t N, int32_t d_in, const void* W1, const float* b1,
                             const void* W2, const float* b2, int32_t K, int32_t k, float* logits,
                             int32_t* ids, float* w, cudaStream_t stream);

int num_sms();

cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, int32_t* err_word, cudaStream_t stream);

// Launches `kernel` with programmatic stream serialization (see pdl_wait in common.cuh) and,
// when cluster >= 1, an explicit 1-D thread-block cluster of that size.  Kernels that use
// cluster-scope instructions (mapa, st.async, barrier.cluster) must pass their cluster size,
// 1 included; others pass 0.  Clears the runtime's error state.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster >= 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  const cudaError_t last = cudaGetLastError();
  return e != cudaSuccess ? e : last;
}

}  // namespace molora
