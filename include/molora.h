/*
 * molora.h -- C ABI of the GB300 (sm_103a) per-token adapter routing library.
 *
 * The method is "MoLoRA: Composable Specialization via Per-Token Adapter Routing"
 * (Shah & Wagle).  Its pages define the path this library runs:
 *   - Table 1: two routing decisions, vocabulary ranges R_vocab(v) (O(1) per token) and a
 *     learned router TopK(g(x)) (O(64d + 64K) per token), followed by infrastructure both
 *     share: histogram computation, pointer arrays, grouped GEMM dispatch.
 *   - Figure 2: the top-k selected adapters are combined by a weighted sum; in execution,
 *     tokens are grouped by their selected adapter and the groups run as grouped GEMMs.
 *   - Table 10: adapter weight shapes A: (K, d, r) and B: (K, r, d).
 *   - Figure 4: adapters live in a GPU-resident hot set at fixed addresses, so the whole
 *     sequence can be captured in one CUDA graph.
 *   - Tables 3 and 7: the per-sequence alternative runs K masked passes (K*N token-work
 *     against N for per-token routing).
 *
 * Workspace (ws, ws_bytes), for the calls that take it (Table 1's shared dispatch
 * infrastructure needs none; only MOLORA_PATH_STACKED does):
 *   - ws_bytes == NULL: no workspace.  AUTO chooses among the paths that need none, and an
 *     explicit MOLORA_PATH_STACKED returns MOLORA_ERR_INVALID_ARG.
 *   - ws == NULL, ws_bytes != NULL: a query.  *ws_bytes is set to the bytes the call would
 *     need (0 if its path needs none); nothing is launched.
 *   - ws != NULL: a caller-owned device buffer of *ws_bytes bytes, 256-byte aligned, at least
 *     the queried size (else MOLORA_ERR_INVALID_ARG).  The call overwrites it; it must not be
 *     shared with work that may run concurrently.  Its contents after the call are unspecified.
 *
 * Conventions for every call:
 *   - All array pointers are DEVICE pointers owned by the caller (for example torch tensors).
 *     The library never allocates, frees or synchronises inside a call: each call only
 *     enqueues kernels on `stream`, so a sequence of calls can be captured in a CUDA graph.
 *     Pointers must stay valid until the enqueued work completes.
 *   - All arrays are dense and row-major; slot s = t*k + j is token t's j-th choice.
 *   - Sizes are validated on the host before anything is launched; a bad argument returns
 *     MOLORA_ERR_INVALID_ARG (or MOLORA_ERR_UNSUPPORTED for a valid but unimplemented
 *     shape) and launches nothing.  MOLORA_ERR_CUDA means a launch failed; call
 *     cudaGetLastError() for the detail.
 *   - Conditions only the device can see (an id outside [0, K), a token outside every
 *     vocabulary range, ranges that do not increase, an inconsistent permutation, a wait
 *     that ran out of time) are OR-ed into *err_word (a device int32 the caller zeroes; may
 *     be NULL to ignore them) with the MOLORA_DEV_* bits below.  The offending slot or
 *     token is skipped; no kernel traps or aborts.
 *   - Empty inputs (N == 0) are valid and launch nothing (apart from writing the empty
 *     histogram in molora_dispatch).
 */
#ifndef MOLORA_H_
#define MOLORA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define MOLORA_API __attribute__((visibility("default")))
#else
#define MOLORA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOLORA_OK = 0,
  MOLORA_ERR_INVALID_ARG = 1,
  MOLORA_ERR_UNSUPPORTED = 2,
  MOLORA_ERR_CUDA = 3,
  MOLORA_ERR_SCRATCH_TOO_SMALL = 4  /* molora_lora_apply_static_ws: the problem needs more than
                                       its fixed scratch holds */
} molora_status;

typedef enum { MOLORA_F32 = 0, MOLORA_BF16 = 1 } molora_dtype;

/* Which kernel family molora_lora_apply_ex uses.  AUTO, given a workspace, picks the stacked
 * path where it measured faster than dispatch + grouped (a stacked rank K*r of at least 256,
 * few adapters per selected one, enough tokens); else the dense path for k >= 2 when it
 * applies and is measured faster; else the scalar or grouped path by their crossover, measured
 * on GB300 by rank and hot-set size: from 160 tokens for 8 adapters of rank 64 (where Figures 5
 * and 9 put it, near batch 160), 768-2048 at rank 32, 768-2048 at rank 16 (scalar only beyond
 * 32 adapters of rank 16).  AUTO takes the grouped path only when the dispatch outputs are
 * given. */
typedef enum {
  MOLORA_PATH_AUTO = 0,
  MOLORA_PATH_SCALAR = 1,  /* CUDA-core, token-major, one CTA per token (the memory-bound regime) */
  MOLORA_PATH_GROUPED = 2, /* grouped tcgen05 shrink + expand over the dispatch permutation */
  MOLORA_PATH_DENSE = 3,   /* tcgen05 over all K adapters per token, weight 0 for the unselected
                              (K*r = 64 or 128, bf16); needs no dispatch; one y update per token */
  MOLORA_PATH_STACKED = 4  /* the same sum as DENSE for a stacked rank K*r up to 1024 (bf16, fp32 y,
                              d_in a multiple of 64): a shrink kernel writes scale * c[t,a] (x A_a) for
                              every adapter to a caller workspace, then a persistent tcgen05 GEMM adds
                              it times [B_0; ...; B_{K-1}] into y; no dispatch; one y update per token */
} molora_path;

/* Device-side error bits OR-ed into *err_word. */
#define MOLORA_DEV_TOKEN_OUTSIDE_RANGES 0x1 /* route_vocab: token in no range; adapter = -1 */
#define MOLORA_DEV_BAD_RANGES 0x2           /* route_vocab: starts not strictly increasing */
#define MOLORA_DEV_BAD_ADAPTER_ID 0x4       /* dispatch / apply: id outside [0, K); slot skipped */
#define MOLORA_DEV_BAD_PERMUTATION 0x8      /* apply: offsets or perm inconsistent; entry skipped */
#define MOLORA_DEV_WAIT_TIMEOUT 0x10        /* a bounded on-chip wait ran out; work abandoned */

#define MOLORA_MAX_ADAPTERS 64   /* K: hot-set size limit (the decode sweep goes to 64) */

/* Flags of the *_ex routing calls (molora_route_vocab_ex, molora_route_vocab_dispatch_ex,
 * molora_route_vocab_lora_apply_ex): see molora_route_vocab_dispatch_ex for the promise. */
#define MOLORA_INPUTS_READY 1u
#define MOLORA_ROUTER_HIDDEN 64  /* hidden width of the learned router (Table 1 cost term 64d) */

/*
 * molora_route_vocab -- vocabulary routing R_vocab(v) (Table 1; Table 12 "disjoint vocab").
 *
 *   adapter[t] = a   where starts[a] <= tok[t] < starts[a+1]
 *   adapter[t] = -1  if tok[t] lies in no range (sets MOLORA_DEV_TOKEN_OUTSIDE_RANGES)
 *
 * tok     int32 [N]     token ids
 * starts  int32 [K+1]   strictly increasing range starts; adapter a owns [starts[a], starts[a+1])
 * K       1..MOLORA_MAX_ADAPTERS
 * adapter int32 [N]     output
 */
MOLORA_API molora_status molora_route_vocab(const int32_t* tok, int64_t N, const int32_t* starts, int32_t K,
                                 int32_t* adapter, int32_t* err_word, cudaStream_t stream);

/*
 * molora_route_vocab_ex -- molora_route_vocab with flags; flags == 0 is exactly
 * molora_route_vocab, and the outputs are identical with and without flags.
 * MOLORA_INPUTS_READY (above; described with molora_route_vocab_dispatch_ex) is the same promise
 * about tok and starts.  Each thread then routes its token before the kernel waits for the one
 * enqueued before it (which may still read `adapter`: the previous step's routing, in a decode
 * loop) and stores after; the next kernel may start at once.  Applies while N <= 256 * 8 * the
 * SM count (one pass of the grid); larger N runs as flags == 0.  Any other bit:
 * MOLORA_ERR_INVALID_ARG.
 */
MOLORA_API molora_status molora_route_vocab_ex(const int32_t* tok, int64_t N, const int32_t* starts, int32_t K,
                                    int32_t* adapter, int32_t* err_word, uint32_t flags,
                                    cudaStream_t stream);

/*
 * molora_router_topk -- learned router TopK(g(x)) (Table 1; Figure 2 with k = 2;
 * Table 10's softmax(Wx + b) gating), hidden width 64:
 *
 *   hidden = ReLU(x W1 + b1)                       [N x 64], fp32 accumulation
 *   logits = hidden W2 + b2                        [N x K], fp32
 *   ids[t] = the k adapters with the largest logits, ordered by logit descending;
 *            equal logits order by the lower index first
 *   w[t,j] = exp(logits[t,ids[t,j]] - m) / sum over the k selected of exp(logit - m),
 *            m = the largest selected logit (the softmax renormalised over the top k)
 *
 * x       [N x d_in]  dtype (MOLORA_BF16 or MOLORA_F32), row-major
 * W1      [d_in x 64] same dtype;   b1 fp32 [64] or NULL (zero)
 * W2      [64 x K]    same dtype;   b2 fp32 [K]  or NULL (zero)
 * K       1..MOLORA_MAX_ADAPTERS;   k  1..K
 * logits  fp32 [N x K] output, or NULL to skip storing it
 * ids     int32 [N x k] output;  w  fp32 [N x k] output
 * bf16 x with d_in a multiple of 64 runs on the tcgen05 tensor cores; other shapes and fp32
 * run on CUDA cores.
 */
MOLORA_API molora_status molora_router_topk(const void* x, molora_dtype dtype, int64_t N, int32_t d_in,
                                 const void* W1, const float* b1, const void* W2, const float* b2,
                                 int32_t K, int32_t k, float* logits, int32_t* ids, float* w,
                                 cudaStream_t stream);

/*
 * molora_dispatch -- histogram, pointer arrays and grouping (Table 1 rows "Histogram
 * computation" and "Pointer arrays"; Figure 2 right "tokens are grouped by their selected
 * adapter").  Over the S = N*k slots:
 *
 *   counts[a]   = number of slots s with ids[s] == a
 *   offsets[0]  = 0,  offsets[a+1] = offsets[a] + counts[a]
 *   perm[offsets[a] + q] = the q-th slot, in ascending s, whose id is a   (stable)
 *   perm[offsets[K] .. S-1] = -1
 *
 * Slots with an id outside [0, K) are left out and set MOLORA_DEV_BAD_ADAPTER_ID.
 * Deterministic and bit-exact: one CTA, no atomics whose order matters.
 * ids int32 [N x k];  counts int32 [K];  offsets int32 [K+1];  perm int32 [N*k]
 */
MOLORA_API molora_status molora_dispatch(const int32_t* ids, int64_t N, int32_t k, int32_t K, int32_t* counts,
                              int32_t* offsets, int32_t* perm, int32_t* err_word,
                              cudaStream_t stream);

/*
 * molora_route_vocab_dispatch -- molora_route_vocab followed by molora_dispatch with k = 1,
 * as one kernel (Table 1: vocabulary routing, then the histogram and pointer arrays both
 * routing decisions share).  Every output, and every bit set in *err_word, equals what the
 * two calls in sequence produce:
 *
 *   adapter[t] as molora_route_vocab;  counts, offsets, perm as molora_dispatch(adapter, N, 1, K)
 *
 * tok int32 [N];  starts int32 [K+1];  adapter int32 [N];  counts int32 [K];
 * offsets int32 [K+1];  perm int32 [N].  N == 0 writes the empty histogram.
 */
MOLORA_API molora_status molora_route_vocab_dispatch(const int32_t* tok, int64_t N, const int32_t* starts,
                                          int32_t K, int32_t* adapter, int32_t* counts, int32_t* offsets,
                                          int32_t* perm, int32_t* err_word, cudaStream_t stream);

/*
 * molora_route_vocab_dispatch_ex -- molora_route_vocab_dispatch with flags; flags == 0 is
 * exactly molora_route_vocab_dispatch.  Outputs are identical with and without flags.
 *
 * MOLORA_INPUTS_READY: the caller promises that tok and starts are not written by any kernel
 * that may still run when this call's kernel starts.  Examples: the ids were copied in from
 * the host, or written by an earlier step.  That kernel starts once the kernel enqueued just
 * before it lets it start:
 *   - Every other call of this library lets its successor start only after everything before
 *     it has finished. Enqueued after one of them, the promise concerns only the kernel just
 *     before this call.
 *   - A call made with this flag lets its successor start at once.  After a chain of such
 *     calls, the promise extends to the kernel before the chain.
 *   - The kernel then starts while the preceding kernel still runs.  It reads tok and starts
 *     and builds the histogram, offsets and permutation in shared memory.
 *   - It waits for the preceding kernel to finish only before its first store, because that
 *     kernel may still read the buffers this call writes (the previous step's adapter,
 *     counts, offsets or perm).
 *   - This moves the routing of step i+1 under the apply of step i when both are enqueued back
 *     to back; programmatic dependent launch, Figure 4's one captured graph per step.
 *   - Applies up to N = 40960 tokens, the sizes held in shared memory. Larger N runs as
 *     flags == 0.
 * Any other bit set in flags: MOLORA_ERR_INVALID_ARG, nothing launched.
 */
MOLORA_API molora_status molora_route_vocab_dispatch_ex(const int32_t* tok, int64_t N, const int32_t* starts,
                                             int32_t K, int32_t* adapter, int32_t* counts, int32_t* offsets,
                                             int32_t* perm, int32_t* err_word, uint32_t flags,
                                             cudaStream_t stream);

/*
 * molora_route_vocab_lora_apply -- the whole vocabulary-routed step: molora_route_vocab_dispatch
 * followed by molora_lora_apply on its outputs (k = 1, weights 1), with the same results:
 *
 *   adapter, counts, offsets, perm   as molora_route_vocab_dispatch(tok, N, starts, K)
 *   y[t,:] += scale * (x[t,:] A_{adapter[t]}) B_{adapter[t]}   for every routed token
 *
 * Two kernels, enqueued back to back on `stream`: the routing + dispatch kernel, then the
 * apply on the path molora_lora_apply would choose.  (Routing inside the apply, every CTA
 * routing all N tokens for its own tile, measured slower on GB300 at 2048 tokens: the
 * redundant routing costs more than the launch it saves.)
 *
 * tok int32 [N];  starts int32 [K+1];  x, A, B, r, d_in, d_out, scale as molora_lora_apply;
 * y fp32 (y_bf16 = 0) or bf16 (y_bf16 = 1) [N x d_out], updated in place;
 * adapter int32 [N], counts int32 [K], offsets int32 [K+1], perm int32 [N]: outputs, all
 * required.  Error bits as the two calls.
 */
MOLORA_API molora_status molora_route_vocab_lora_apply(const int32_t* tok, int64_t N, const int32_t* starts,
                                            int32_t K, const void* x, molora_dtype dtype, int32_t d_in,
                                            int32_t d_out, const void* A, const void* B, int32_t r,
                                            float scale, void* y, int32_t y_bf16, int32_t* adapter,
                                            int32_t* counts, int32_t* offsets, int32_t* perm,
                                            int32_t* err_word, cudaStream_t stream);

/*
 * molora_route_vocab_lora_apply_ex -- molora_route_vocab_lora_apply with flags; flags == 0 is
 * exactly molora_route_vocab_lora_apply, and results are identical with and without flags.
 * MOLORA_INPUTS_READY means what it means for molora_route_vocab_dispatch_ex: the caller's
 * promise about tok and starts, which lets this step's routing kernel run under the kernel
 * enqueued before it, for example the previous step's apply.  Any other bit:
 * MOLORA_ERR_INVALID_ARG, nothing launched.
 */
MOLORA_API molora_status molora_route_vocab_lora_apply_ex(const int32_t* tok, int64_t N, const int32_t* starts,
                                               int32_t K, const void* x, molora_dtype dtype, int32_t d_in,
                                               int32_t d_out, const void* A, const void* B, int32_t r,
                                               float scale, void* y, int32_t y_bf16, int32_t* adapter,
                                               int32_t* counts, int32_t* offsets, int32_t* perm,
                                               int32_t* err_word, uint32_t flags, cudaStream_t stream);

/*
 * molora_lora_apply -- batched per-token LoRA apply over the hot set (Figure 2; Table 10
 * shapes; Figure 4 hot set):
 *
 *   y[t,:] += scale * sum_j w[t,j] * (x[t,:] A_{ids[t,j]}) B_{ids[t,j]}
 *
 * x       [N x d_in]      dtype, row-major
 * A       [K x d_in x r]  dtype, the hot set's down-projections, contiguous, fixed address
 * B       [K x r x d_out] dtype, the hot set's up-projections, contiguous, fixed address
 * r       8, 16, 32 or 64
 * ids     int32 [N x k]   adapter per slot (from molora_route_vocab with k = 1, or
 *                         molora_router_topk)
 * w       fp32 [N x k]    slot weights, or NULL for all ones
 * counts, offsets, perm   molora_dispatch's outputs for these ids (read by the grouped
 *                         path; the scalar path reads ids directly and ignores them).  AUTO
 *                         takes the grouped path only when all three are given
 * y       fp32 [N x d_out], updated in place (read-modify-write)
 *
 * ws, ws_bytes  workspace (see the convention above); the stacked path needs
 *               2 * roundup256(N * K * r * 2) bytes, every other path none
 *
 * Accumulation is fp32 (tensor cores or FMA); x, A, B are read as given.  The grouped path
 * needs bf16 and r >= 16; anything else runs on the scalar path.  With k > 1 the grouped
 * path adds each slot's contribution to y with an fp32 reduction in L2, so the order of the
 * k additions (and therefore the last bits of y) may vary from run to run; with k = 1, and
 * on the scalar, dense and stacked paths for any k, every element of y receives one
 * addition and results are reproducible bit for bit.
 */
MOLORA_API molora_status molora_lora_apply(const void* x, molora_dtype dtype, int64_t N, int32_t d_in,
                                int32_t d_out, const void* A, const void* B, int32_t K, int32_t r,
                                const int32_t* ids, const float* w, int32_t k,
                                const int32_t* counts, const int32_t* offsets,
                                const int32_t* perm, float scale, float* y, void* ws,
                                size_t* ws_bytes, int32_t* err_word, cudaStream_t stream);

/* molora_lora_apply with an explicit kernel family (used to measure the crossover).
 * A path that does not support the shape returns MOLORA_ERR_UNSUPPORTED. */
MOLORA_API molora_status molora_lora_apply_ex(const void* x, molora_dtype dtype, int64_t N, int32_t d_in,
                                   int32_t d_out, const void* A, const void* B, int32_t K,
                                   int32_t r, const int32_t* ids, const float* w, int32_t k,
                                   const int32_t* counts, const int32_t* offsets,
                                   const int32_t* perm, float scale, float* y, void* ws,
                                   size_t* ws_bytes, int32_t* err_word, molora_path path,
                                   cudaStream_t stream);

/*
 * molora_lora_apply_bf16y -- molora_lora_apply_ex with y held in bf16 (the output dtype a
 * bf16 model keeps its activations in; the pages leave y's dtype open).  Same arguments,
 * except y: bf16 [N x d_out], updated in place.
 *
 * Rounding: the contributions are formed in fp32 as in molora_lora_apply.  The scalar path
 * adds a token's whole fp32 sum to y and rounds once to bf16 (nearest even).  The grouped
 * path rounds each slot's contribution to bf16 and adds it into y with a bf16 bulk
 * reduction in L2 (one more rounding per slot), so it may differ from the once-rounded
 * result by about one bf16 unit in the last place per slot.
 */
MOLORA_API molora_status molora_lora_apply_bf16y(const void* x, molora_dtype dtype, int64_t N, int32_t d_in,
                                      int32_t d_out, const void* A, const void* B, int32_t K, int32_t r,
                                      const int32_t* ids, const float* w, int32_t k,
                                      const int32_t* counts, const int32_t* offsets,
                                      const int32_t* perm, float scale, void* y, int32_t* err_word,
                                      molora_path path, cudaStream_t stream);

/*
 * molora_lora_apply_indirect -- the apply with the hot set given adapter by adapter
 * instead of as two contiguous slabs (Table 2: indirect, pointer-array adapter addressing).
 *
 * A_ptrs[i]  device address of adapter i's A, [d_in x r] of dtype, row-major, 16-byte aligned
 * B_ptrs[i]  device address of adapter i's B, [r x d_out], 16-byte aligned
 * A_ptrs and B_ptrs are HOST arrays of K entries.  Their values are read when the call is
 * made (a CUDA graph captures them by value), so the adapters must stay at those addresses
 * while enqueued work and captured graphs use them.  y is fp32 (y_bf16 = 0) or bf16
 * (y_bf16 = 1, rounding as molora_lora_apply_bf16y).  Every other argument, the path choice
 * and the results are those of molora_lora_apply_ex on the same adapters held in slabs.
 */
MOLORA_API molora_status molora_lora_apply_indirect(const void* x, molora_dtype dtype, int64_t N,
                                         int32_t d_in, int32_t d_out, const void* const* A_ptrs,
                                         const void* const* B_ptrs, int32_t K, int32_t r,
                                         const int32_t* ids, const float* w, int32_t k,
                                         const int32_t* counts, const int32_t* offsets,
                                         const int32_t* perm, float scale, void* y, int32_t y_bf16,
                                         int32_t* err_word, molora_path path, cudaStream_t stream);

/*
 * molora_router_lora_apply -- the learned router and the top-k apply in one pass over x
 * (Table 1: routing cost O(64d + 64K) on top of the apply; Figure 2: top-k adapters combined
 * by a weighted sum).  It computes molora_router_topk followed by molora_lora_apply on the
 * dense path (MOLORA_PATH_DENSE) in one kernel that reads each x row once for both: the
 * router's x W1 is 64 more columns of the apply's shrink x [A_0 | ... | A_{K-1}].
 *
 *   logits, ids, w   as molora_router_topk (same hidden width 64, same top-k and softmax rule)
 *   y[t,:] += scale * sum_j w[t,j] * (x[t,:] A_{ids[t,j]}) B_{ids[t,j]}
 *
 * x [N x d_in] bf16;  W1 [d_in x 64] bf16;  b1 fp32 [64] or NULL;  W2 [64 x K] bf16;
 * b2 fp32 [K] or NULL;  A [K x d_in x r] and B [K x r x d_out] bf16 slabs;  1 <= k <= K;
 * logits fp32 [N x K] output or NULL;  ids int32 [N x k] and w fp32 [N x k] outputs;
 * y fp32 (y_bf16 = 0) or bf16 (y_bf16 = 1) [N x d_out], updated in place.
 * ws, ws_bytes: workspace (see the convention above).
 * Every y element receives one addition, so results are reproducible for any k.
 * Two kernel families:
 *   - one kernel, K*r = 64 or 128, y fp32 or bf16, d_in and d_out multiples of 64 that split
 *     evenly over its cluster.  Its logits, ids, w and y equal molora_router_topk followed by
 *     the dense molora_lora_apply bit for bit whenever both split d_in over the same number
 *     of CTAs (each takes the widest cluster whose CTAs fit one wave: 64-token tiles here,
 *     128-token tiles in molora_router_topk; with 152 SMs both split 8 ways up to 2432
 *     tokens).  Otherwise the hidden units' partial sums group differently and the logits
 *     may differ in the last bits.  Used without a workspace (ws_bytes == NULL);
 *   - the stacked pair (the shrink with the router, then the expand GEMM), K*r up to 1024,
 *     fp32 y, d_in a multiple of 64.  Its router sums the 64 hidden units in order for each
 *     logit, so its logits may differ from molora_router_topk's in the last bits.  Used
 *     whenever a buffer is passed (ws != NULL) and it applies.
 * A query (ws == NULL, ws_bytes != NULL) returns the stacked pair's size where it applies and
 * the one kernel does not or is measured slower, else 0.
 * The stacked pair evaluates all K adapters for every token.  With many adapters per selected
 * one and few tokens, molora_router_topk then molora_dispatch and the grouped apply (the
 * separate calls) measured faster on GB300 at d = 4096, by the rule molora_lora_apply's AUTO
 * uses for its own workspace path: e.g. top-1 over 16 adapters of rank 16, or top-2 over 64.
 * Other shapes return MOLORA_ERR_UNSUPPORTED (use the separate calls).  dtype must be
 * MOLORA_BF16; x, W1, A, B and y must be 16-byte aligned.
 */
MOLORA_API molora_status molora_router_lora_apply(const void* x, molora_dtype dtype, int64_t N, int32_t d_in,
                                       int32_t d_out, const void* W1, const float* b1, const void* W2,
                                       const float* b2, const void* A, const void* B, int32_t K, int32_t r,
                                       int32_t k, float scale, float* logits, int32_t* ids, float* w,
                                       void* y, int32_t y_bf16, void* ws, size_t* ws_bytes,
                                       int32_t* err_word, cudaStream_t stream);

/*
 * molora_lora_apply_static_ws -- molora_lora_apply on the stacked path (MOLORA_PATH_STACKED)
 * for callers that cannot allocate device memory.  The paper has no counterpart: this is a
 * convenience of this library.
 *
 * Who needs it: code that runs where cudaMalloc is not an option -- a process whose device
 * memory is entirely reserved by another allocator (a serving framework's pool), a latency
 * path that may not call cudaMalloc or cudaFree because they can synchronise the device, or a
 * caller that holds only raw pointers and a stream and has no allocator at all.  Instead of a
 * caller-provided workspace it uses a fixed scratch buffer compiled into the library (a
 * file-scope device array of MOLORA_STATIC_SCRATCH_BYTES, held by every GPU that loads the
 * library until the process exits).  The call itself allocates nothing.
 *
 * Arguments and results: those of molora_lora_apply (y fp32, bf16 x/A/B, d_in a multiple of
 * 64); the results equal molora_lora_apply_ex with MOLORA_PATH_STACKED.
 * Limit: 2 * roundup256(N * K * r * 2) <= MOLORA_STATIC_SCRATCH_BYTES (N * K * r up to 4M,
 * e.g. N = 8192 tokens at K*r = 512); larger problems return MOLORA_ERR_SCRATCH_TOO_SMALL
 * before anything is launched.  Shapes the stacked path does not support return
 * MOLORA_ERR_UNSUPPORTED.
 * Sharing: every call on a device uses the same buffer, which keeps the last call's contents
 * (nothing in it needs to start at zero).  Calls whose work can overlap on the GPU -- on
 * different streams, or from several threads -- race on it and must be serialised by the
 * caller.
 * Set-up: the first call on each device looks up the buffer's device address (with that
 * device current); make that first call before any stream capture begins.
 */
#define MOLORA_STATIC_SCRATCH_BYTES (16u << 20)
MOLORA_API molora_status molora_lora_apply_static_ws(const void* x, molora_dtype dtype, int64_t N, int32_t d_in,
                                          int32_t d_out, const void* A, const void* B, int32_t K, int32_t r,
                                          const int32_t* ids, const float* w, int32_t k, float scale,
                                          float* y, int32_t* err_word, cudaStream_t stream);

/*
 * molora_lora_apply_masked_pass -- one pass of the per-sequence baseline (Tables 3 and 7:
 * per-sequence routing needs K passes for a K-modality batch).  Adapter `a` is evaluated
 * for EVERY token; the result is multiplied by the 0/1 mask [adapter_of[t] == a]:
 *
 *   y[t,:] += [adapter_of[t] == a] * scale * (x[t,:] A_a) B_a
 *
 * Running it for a = 0..K-1 reproduces molora_lora_apply with k = 1 at K times the work.
 * It exists only as the comparison baseline.  adapter_of int32 [N]; 0 <= a < K.
 */
MOLORA_API molora_status molora_lora_apply_masked_pass(const void* x, molora_dtype dtype, int64_t N,
                                            int32_t d_in, int32_t d_out, const void* A,
                                            const void* B, int32_t K, int32_t r,
                                            const int32_t* adapter_of, int32_t a, float scale,
                                            float* y, int32_t* err_word, molora_path path,
                                            cudaStream_t stream);

/* The kernel family molora_lora_apply would choose for this shape when given a workspace
 * (never AUTO; without one, a STACKED choice becomes the best path that needs none). */
MOLORA_API molora_path molora_select_path(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out,
                               int32_t K, int32_t r, int32_t k);

/*
 * molora_selftest_bounded_wait -- checks the bounded on-chip waits every kernel here relies
 * on: one CTA waits on an mbarrier phase that nothing completes, gives up after `limit_us`
 * microseconds (1 .. 1e6), ORs MOLORA_DEV_WAIT_TIMEOUT into *err_word (a device int32,
 * required) and exits normally, leaving the context usable.  Not part of the method.
 */
MOLORA_API molora_status molora_selftest_bounded_wait(uint32_t limit_us, int32_t* err_word, cudaStream_t stream);

/* Short text for a status code (static storage). */
MOLORA_API const char* molora_status_string(molora_status status);

/* Library version as major*10000 + minor*100 + patch. */
MOLORA_API int32_t molora_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOLORA_H_ */
