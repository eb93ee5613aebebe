// route_dispatch.cu -- vocabulary routing and the dispatch step (histogram, exclusive scan,
// stable permutation) of "MoLoRA: Composable Specialization via Per-Token Adapter Routing"
// (Table 1: R_vocab(v), histogram computation, pointer arrays; Figure 2 right: tokens
// grouped by their selected adapter).
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace molora {

// One thread per token; the K+1 range starts sit in shared memory and each token does a
// binary search for the last start <= its id.  With `early` (the ids and ranges are not written
// by the kernel before this one, and one pass of the grid covers N), each thread routes its
// token before waiting on that kernel and stores the result, and any error bit, after it: the
// kernel before may still read `adapter` (the previous step's routing).
__global__ void __launch_bounds__(256) route_vocab_kernel(const int32_t* __restrict__ tok, int64_t N,
                                                          const int32_t* __restrict__ starts, int32_t K,
                                                          int32_t* __restrict__ adapter, int32_t* err_word,
                                                          int early) {
  __shared__ int32_t s_starts[kMaxAdapters + 1];
  const int64_t t0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  const bool read_early = early && step >= N;
  if (!read_early) pdl_wait();
  pdl_launch_dependents();
  for (int i = threadIdx.x; i <= K; i += blockDim.x) s_starts[i] = starts[i];
  __syncthreads();
  bool bad_ranges = false;
  if (blockIdx.x == 0 && threadIdx.x == 0)
    for (int a = 0; a < K; ++a)
      if (s_starts[a] >= s_starts[a + 1]) {
        bad_ranges = true;
        break;
      }
  auto route = [&](int64_t t, bool& outside) {
    const int32_t v = tok[t];
    int32_t a = -1;
    if (v >= s_starts[0] && v < s_starts[K]) {
      int lo = 0, hi = K;  // s_starts[lo] <= v < s_starts[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_starts[mid] <= v)
          lo = mid;
        else
          hi = mid;
      }
      a = lo;
    } else {
      outside = true;
    }
    return a;
  };
  bool outside = false;
  if (read_early) {
    const int32_t a = t0 < N ? route(t0, outside) : -1;
    pdl_wait();
    if (t0 < N) adapter[t0] = a;
  } else {
    for (int64_t t = t0; t < N; t += step) adapter[t] = route(t, outside);
  }
  if (bad_ranges) report(err_word, MOLORA_DEV_BAD_RANGES);
  if (__any_sync(0xffffffffu, outside) && (threadIdx.x & 31) == 0) report(err_word, MOLORA_DEV_TOKEN_OUTSIDE_RANGES);
}

cudaError_t launch_route_vocab(const int32_t* tok, int64_t N, const int32_t* starts, int32_t K, int32_t* adapter,
                               int32_t* err_word, int early, cudaStream_t stream) {
  const int64_t blocks = (N + 255) / 256;
  const int grid = (int)(blocks < 8 * num_sms() ? blocks : 8 * num_sms());
  return launch_kernel(route_vocab_kernel, dim3(grid > 0 ? grid : 1), dim3(256), 0, stream, 0, tok, N, starts, K,
                       adapter, err_word, early);
}

// ---------------------------------------------------------------------------------------
// Dispatch: a single CTA of 32 warps.  Every slot's id is read once (with coalesced loads)
// and, up to kStageSlots slots, kept in shared memory for the two passes below.  Warp w owns
// a contiguous run of slots; it walks the run 32 slots at a time, and __match_any_sync
// groups the lanes that carry the same adapter id.  Pass 1 counts slots per (warp, adapter).
// The counts, read adapter-major, give each (adapter, warp) the first output position of
// its slots (the exclusive scan).  Pass 2 repeats the walk and writes each slot at base +
// its rank among equal lanes of lower index, so the permutation is stable: within an
// adapter, slots appear in ascending order.  No atomics whose order could change a result;
// no inter-CTA waiting.
//
// kVocab: the slots are tokens (k = 1) and their ids come from vocabulary routing done in
// the same pass (the routed ids are also written to `adapter`), which saves the separate
// routing kernel and its round trip through global memory.
constexpr int kDispatchWarps = 32;
constexpr int64_t kStageSlots = 40960;  // 160 KB of shared memory

__device__ __forceinline__ int32_t vocab_range(const int32_t* s_starts, int32_t K, int32_t v) {
  if (v < s_starts[0] || v >= s_starts[K]) return -1;
  int lo = 0, hi = K;  // s_starts[lo] <= v < s_starts[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_starts[mid] <= v)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

template <bool kVocab>
__global__ void __launch_bounds__(kDispatchWarps * 32, 1)
    dispatch_kernel(const int32_t* __restrict__ src, const int32_t* __restrict__ starts, int64_t S, int32_t K,
                    int32_t* adapter, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                    int32_t* __restrict__ perm, int32_t* err_word, int early) {
  extern __shared__ int32_t s_ids[];  // [S] when S <= kStageSlots
  __shared__ int32_t cnt[kDispatchWarps][kMaxAdapters];
  __shared__ int32_t s_total[kMaxAdapters];
  __shared__ int32_t s_off[kMaxAdapters + 1];
  __shared__ int32_t s_starts[kMaxAdapters + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool staged = S <= kStageSlots;
  // With `early`, the token ids and ranges are not written by the kernel before this one, so
  // reading them, the histogram, the scan and the ranks run before waiting on that kernel
  // (which may still be reading this call's output buffers); every store comes after the wait.
  // The ids must stay in shared memory for that, so only staged sizes read early.  The next
  // kernel may start at once: it waits for this one to finish before it reads what it wrote.
  const bool read_early = kVocab && early && staged;
  for (int i = threadIdx.x; i < kDispatchWarps * kMaxAdapters; i += blockDim.x) (&cnt[0][0])[i] = 0;
  if (!read_early) pdl_wait();
  pdl_launch_dependents();
  // this thread's slots' ids (up to kPre per thread), loaded before the ranges so that the two
  // global loads are in flight together rather than one after the other
  constexpr int kPre = 4;
  const bool pre_ok = S <= (int64_t)kPre * blockDim.x;
  int32_t pre[kPre];
#pragma unroll
  for (int q = 0; q < kPre; ++q) {
    const int64_t s = threadIdx.x + (int64_t)q * blockDim.x;
    pre[q] = pre_ok && s < S ? src[s] : 0;
  }
  if (kVocab) {
    for (int i = threadIdx.x; i <= K; i += blockDim.x) s_starts[i] = starts[i];
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int a = 0; a < K; ++a)
        if (s_starts[a] >= s_starts[a + 1]) {
          report(err_word, MOLORA_DEV_BAD_RANGES);
          break;
        }
    }
  }

  // every slot's id, read once; invalid ids become -1
  bool bad = false, outside = false;
  for (int64_t s = threadIdx.x, q = 0; s < S; s += blockDim.x, ++q) {
    int32_t v = 0;
    if (pre_ok) {
#pragma unroll
      for (int i = 0; i < kPre; ++i)
        if (i == q) v = pre[i];
    } else {
      v = src[s];
    }
    int32_t a;
    if (kVocab) {
      a = vocab_range(s_starts, K, v);
      outside |= a < 0;
      if (!read_early) adapter[s] = a;  // (read_early: stored from s_ids after the wait)
    } else {
      a = v;
    }
    if (a < 0 || a >= K) {
      bad = true;
      a = -1;
    }
    if (staged) s_ids[s] = a;
  }
  __syncthreads();  // also orders the adapter[] stores above before the re-reads below
  auto id_of = [&](int64_t s) -> int32_t {
    if (staged) return s_ids[s];
    const int32_t a = kVocab ? adapter[s] : src[s];
    return (a < 0 || a >= K) ? -1 : a;
  };

  const int64_t per_warp = ((S + kDispatchWarps * 32 - 1) / (kDispatchWarps * 32)) * 32;
  const int64_t beg = min(S, (int64_t)warp * per_warp);
  const int64_t end = min(S, beg + per_warp);
  const unsigned lanes_below = (1u << lane) - 1u;

  for (int64_t base = beg; base < end; base += 32) {
    const int64_t s = base + lane;
    const int32_t a = s < end ? id_of(s) : -1;
    const unsigned m = __match_any_sync(0xffffffffu, a);
    if (a >= 0 && lane == __ffs(m) - 1) cnt[warp][a] += __popc(m);
  }
  __syncthreads();

  if (threadIdx.x < K) {
    int32_t sum = 0;
    for (int w = 0; w < kDispatchWarps; ++w) sum += cnt[w][threadIdx.x];
    s_total[threadIdx.x] = sum;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t run = 0;
    for (int a = 0; a < K; ++a) {
      s_off[a] = run;
      run += s_total[a];
    }
    s_off[K] = run;
  }
  __syncthreads();
  if (read_early) {
    pdl_wait();
    for (int64_t s = threadIdx.x; s < S; s += blockDim.x) adapter[s] = s_ids[s];
  }
  if (threadIdx.x < K) {
    const int a = threadIdx.x;
    int32_t run = s_off[a];
    for (int w = 0; w < kDispatchWarps; ++w) {
      const int32_t c = cnt[w][a];
      cnt[w][a] = run;  // first output position of warp w's slots of adapter a
      run += c;
    }
    counts[a] = s_total[a];
  }
  if (threadIdx.x <= K) offsets[threadIdx.x] = s_off[threadIdx.x];
  __syncthreads();

  for (int64_t base = beg; base < end; base += 32) {
    const int64_t s = base + lane;
    const int32_t a = s < end ? id_of(s) : -1;
    const unsigned m = __match_any_sync(0xffffffffu, a);
    if (a >= 0) perm[cnt[warp][a] + __popc(m & lanes_below)] = (int32_t)s;
    __syncwarp();
    if (a >= 0 && lane == __ffs(m) - 1) cnt[warp][a] += __popc(m);
    __syncwarp();
  }
  for (int64_t i = s_off[K] + threadIdx.x; i < S; i += blockDim.x) perm[i] = -1;
  if (__any_sync(0xffffffffu, bad) && lane == 0) report(err_word, MOLORA_DEV_BAD_ADAPTER_ID);
  if (kVocab && __any_sync(0xffffffffu, outside) && lane == 0) report(err_word, MOLORA_DEV_TOKEN_OUTSIDE_RANGES);
}

template <bool kVocab>
static cudaError_t launch_dispatch_impl(const int32_t* src, const int32_t* starts, int64_t S, int32_t K,
                                        int32_t* adapter, int32_t* counts, int32_t* offsets, int32_t* perm,
                                        int32_t* err_word, int early, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(dispatch_kernel<kVocab>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(kStageSlots * 4));
    if (attr != cudaSuccess) cudaGetLastError();
  });
  if (attr != cudaSuccess) return attr;
  const size_t smem = S <= kStageSlots ? (size_t)S * 4 : 0;
  return launch_kernel(dispatch_kernel<kVocab>, dim3(1), dim3(kDispatchWarps * 32), smem, stream, 0, src, starts, S,
                       K, adapter, counts, offsets, perm, err_word, early);
}

cudaError_t launch_dispatch(const int32_t* ids, int64_t N, int32_t k, int32_t K, int32_t* counts, int32_t* offsets,
                            int32_t* perm, int32_t* err_word, cudaStream_t stream) {
  return launch_dispatch_impl<false>(ids, nullptr, N * (int64_t)k, K, nullptr, counts, offsets, perm, err_word, 0,
                                     stream);
}

cudaError_t launch_route_vocab_dispatch(const int32_t* tok, int64_t N, const int32_t* starts, int32_t K,
                                        int32_t* adapter, int32_t* counts, int32_t* offsets, int32_t* perm,
                                        int32_t* err_word, int early, cudaStream_t stream) {
  return launch_dispatch_impl<true>(tok, starts, N, K, adapter, counts, offsets, perm, err_word, early, stream);
}

// ---------------------------------------------------------------------------------------
// Self-test of the bounded waits every kernel uses: one CTA waits on an mbarrier whose phase
// nothing completes (armed for one arrival that never comes), gives up after `limit_ns`,
// reports MOLORA_DEV_WAIT_TIMEOUT and returns normally.
__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns, int32_t* err_word) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
}

cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, int32_t* err_word, cudaStream_t stream) {
  return launch_kernel(bounded_wait_selftest_kernel, dim3(1), dim3(32), 0, stream, 0, limit_ns, err_word);
}

}  // namespace molora
