// lora_scalar.cu -- the CUDA-core paths of "MoLoRA: Composable Specialization via Per-Token
// Adapter Routing":
//   * the token-major LoRA apply for the memory-bound small-batch regime (Figures 5 and 9:
//     below the crossover a scalar per-token kernel beats the tensor-core kernel), which
//     also serves fp32 inputs, rank 8 and shapes the grouped tcgen05 path does not take;
//   * a CUDA-core learned router TopK(g(x)) (Table 1) for fp32 or odd shapes.
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace molora {

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

// 16 bytes of T unpacked to floats.
template <typename T>
struct Chunk16;
template <>
struct Chunk16<float> {
  static constexpr int kVec = 4;
  __device__ __forceinline__ static void load(const float* p, float (&v)[4]) {
    const float4 q = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = q.x, v[1] = q.y, v[2] = q.z, v[3] = q.w;
  }
};
template <>
struct Chunk16<__nv_bfloat16> {
  static constexpr int kVec = 8;
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(u[i] << 16);
      v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
  }
};

// Four consecutive elements of T as floats (8 bytes of bf16 or 16 bytes of fp32).
__device__ __forceinline__ void load4(const float* p, float (&v)[4]) {
  const float4 q = __ldg(reinterpret_cast<const float4*>(p));
  v[0] = q.x, v[1] = q.y, v[2] = q.z, v[3] = q.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
  v[0] = __uint_as_float(q.x << 16), v[1] = __uint_as_float(q.x & 0xFFFF0000u);
  v[2] = __uint_as_float(q.y << 16), v[3] = __uint_as_float(q.y & 0xFFFF0000u);
}

constexpr int kScalarThreads = 256;
// Small batches split each token over a cluster of C CTAs (see lora_scalar_kernel): the widest
// C in {8, 4, 2} with N * C <= this many CTAs.  Measured on GB300, routing + scalar apply at
// d = 4096, r = 16, K = 16: the fastest width at each batch kept the grid near 256-384 CTAs
// (C = 8 at 1-32 tokens: 6.3 -> 3.8 us at 1; C = 4 at 96: 7.9 -> 5.7; C = 2 at 128 and 160:
// 9.0 -> 7.1 and 7.9), and from 256 tokens no split was fastest.
constexpr int64_t kScalarSplitCtas = 384;

// y element access: fp32, or bf16 (the fp32 sum rounded to nearest even once per update).
__device__ __forceinline__ void y_add4(float* p, const float (&a)[4]) {
  float4 v = *reinterpret_cast<float4*>(p);
  v.x += a[0], v.y += a[1], v.z += a[2], v.w += a[3];
  *reinterpret_cast<float4*>(p) = v;
}
__device__ __forceinline__ void y_add4(__nv_bfloat16* p, const float (&a)[4]) {
  uint2 q = *reinterpret_cast<uint2*>(p);
  const __nv_bfloat162 lo = __floats2bfloat162_rn(__uint_as_float(q.x << 16) + a[0],
                                                  __uint_as_float(q.x & 0xFFFF0000u) + a[1]);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(__uint_as_float(q.y << 16) + a[2],
                                                  __uint_as_float(q.y & 0xFFFF0000u) + a[3]);
  q.x = *reinterpret_cast<const uint32_t*>(&lo);
  q.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = q;
}
__device__ __forceinline__ void y_add1(float* p, float a) { *p += a; }
__device__ __forceinline__ void y_add1(__nv_bfloat16* p, float a) {
  *p = __float2bfloat16_rn(__bfloat162float(*p) + a);
}

// One CTA per (token, column split).  Phase 1: for each of the token's k slots the CTA
// reduces h = x[t] A_a over d_in (each thread streams 16-byte chunks of A_a, which is
// row-major [d_in x R], so a warp reads 512 contiguous bytes per step) and stores
// g_j = scale * w_j * h.  Phase 2: each thread owns 4 output columns and accumulates
// sum_j sum_q g_j[q] B_a[q, c..c+3] in registers, then updates y once.  Every y element is
// read and written exactly once whatever k is, so the result is deterministic.
//
// kSplit (small batches): a cluster of `split` CTAs per token instead, CTA c taking the rows
// [c d_in / split, (c+1) d_in / split) of the shrink and the columns [c d_out / split, ...) of
// the expand.  Each CTA stores its partial h into slot c of every CTA of the cluster (after a
// cluster barrier that every CTA has started), and after a second one adds the slots in rank
// order, so all agree bit for bit.  A token's shrink chain is then `split` times shorter,
// which is what a decode step at small batch waits on.
template <typename T, typename YT, int R, bool kSplit>
__global__ void __launch_bounds__(kScalarThreads)
    lora_scalar_kernel(const T* __restrict__ x, int32_t d_in, int32_t d_out, const T* __restrict__ A,
                       const T* __restrict__ B, int32_t K, const int32_t* __restrict__ ids,
                       const float* __restrict__ w, int32_t k, float scale, YT* __restrict__ y,
                       int32_t split_param, int32_t mask_adapter, int32_t* err_word, int32_t indirect,
                       const __grid_constant__ AdapterTable table) {
  using C16 = Chunk16<T>;
  constexpr int VEC = C16::kVec;
  constexpr int CPR = R / VEC;  // 16-byte chunks per row of A_a
  static_assert(R % VEC == 0 && (kScalarThreads % CPR) == 0, "chunking");
  extern __shared__ float smem[];
  float* g = smem;                 // [k][R]
  float* red = smem + k * R;       // [8 warps][R]
  // kSplit: split_param CTAs per token, their partials [split][k][R]; else the columns per CTA
  const int csplit = kSplit ? split_param : 1;
  float* part = red + (kScalarThreads / 32) * R;
  int32_t* s_adapter = reinterpret_cast<int32_t*>(kSplit ? part + csplit * k * R : part);  // [k]

  const int64_t t = kSplit ? (int64_t)(blockIdx.x / (unsigned)csplit) : (int64_t)blockIdx.x;
  const int crank = kSplit ? (int)(blockIdx.x % (unsigned)csplit) : 0;  // == %cluster_ctarank
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t r_begin = kSplit ? (int32_t)((int64_t)d_in * crank / csplit) : 0;
  const int32_t r_end = kSplit ? (int32_t)((int64_t)d_in * (crank + 1) / csplit) : d_in;
  const T* xr = x + t * (int64_t)d_in;
  if constexpr (kSplit) cluster_arrive();  // a peer's shared memory is written only once all have started
  pdl_wait();
  pdl_launch_dependents();
  if constexpr (kSplit) cluster_wait();

  for (int j = 0; j < k; ++j) {
    int32_t a;
    float wj;
    if (mask_adapter >= 0) {
      a = mask_adapter;
      wj = (ids[t] == mask_adapter) ? 1.f : 0.f;
    } else {
      a = ids[t * k + j];
      wj = w ? w[t * k + j] : 1.f;
      if (a < 0 || a >= K) {
        if (tid == 0) report(err_word, MOLORA_DEV_BAD_ADAPTER_ID);
        a = -1;
      }
    }
    if (a < 0) {  // uniform over the CTA
      if (tid == 0) s_adapter[j] = -1;
      continue;
    }
    float acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v) acc[v] = 0.f;
    const T* Aa = indirect ? static_cast<const T*>(table.a[a]) : A + (int64_t)a * d_in * R;
    const int64_t nchunks = (int64_t)r_end * CPR;
#pragma unroll 4
    for (int64_t c = (int64_t)r_begin * CPR + tid; c < nchunks; c += kScalarThreads) {
      const float xv = to_f(xr[c / CPR]);
      float av[VEC];
      C16::load(Aa + c * VEC, av);
#pragma unroll
      for (int v = 0; v < VEC; ++v) acc[v] = fmaf(xv, av[v], acc[v]);
    }
    // lanes with equal (lane % CPR) hold the same columns q0..q0+VEC-1
#pragma unroll
    for (int off = 16; off >= CPR; off >>= 1)
#pragma unroll
      for (int v = 0; v < VEC; ++v) acc[v] += __shfl_xor_sync(0xffffffffu, acc[v], off);
    if (lane < CPR)
#pragma unroll
      for (int v = 0; v < VEC; ++v) red[warp * R + lane * VEC + v] = acc[v];
    __syncthreads();
    if (tid < R) {
      float h = 0.f;
#pragma unroll
      for (int q = 0; q < kScalarThreads / 32; ++q) h += red[q * R + tid];
      if constexpr (kSplit) {
        // this rank's partial sum, into slot crank of every CTA of the cluster
        const uint32_t local = smem_u32(part + (crank * k + j) * R + tid);
        for (int p = 0; p < csplit; ++p) st_cluster_f32(dsmem_addr(local, (uint32_t)p), h);
        g[j * R + tid] = scale * wj;  // the weight, until the partials are in
      } else {
        g[j * R + tid] = scale * wj * h;
      }
    }
    if (tid == 0) s_adapter[j] = a;
    __syncthreads();
  }
  if constexpr (kSplit) {
    // every rank's partials are in every CTA (the barrier orders the remote stores); nothing is
    // read or written remotely after it, so a CTA may leave whenever it is done
    cluster_sync();
    for (int i = tid; i < k * R; i += kScalarThreads) {
      if (s_adapter[i / R] < 0) continue;
      float h = 0.f;
      for (int p = 0; p < csplit; ++p) h += part[p * k * R + i];
      g[i] *= h;
    }
  }
  __syncthreads();

  const int32_t c_begin = kSplit ? (int32_t)((int64_t)d_out * crank / csplit) : (int32_t)blockIdx.y * split_param;
  const int32_t c_end = kSplit ? (int32_t)((int64_t)d_out * (crank + 1) / csplit) : min(d_out, c_begin + split_param);
  YT* yr = y + t * (int64_t)d_out;
  if ((d_out & 3) == 0) {
    for (int32_t c = c_begin + 4 * tid; c < c_end; c += 4 * kScalarThreads) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int j = 0; j < k; ++j) {
        const int32_t a = s_adapter[j];
        if (a < 0) continue;
        const T* Bq = (indirect ? static_cast<const T*>(table.b[a]) : B + (int64_t)a * R * d_out) + c;
        const float* gj = g + j * R;
#pragma unroll
        for (int q = 0; q < R; ++q) {
          float b[4];
          load4(Bq + (int64_t)q * d_out, b);
          const float gq = gj[q];
#pragma unroll
          for (int v = 0; v < 4; ++v) acc[v] = fmaf(gq, b[v], acc[v]);
        }
      }
      y_add4(yr + c, acc);
    }
  } else {
    for (int32_t c = c_begin + tid; c < c_end; c += kScalarThreads) {
      float acc = 0.f;
      for (int j = 0; j < k; ++j) {
        const int32_t a = s_adapter[j];
        if (a < 0) continue;
        const T* Bq = (indirect ? static_cast<const T*>(table.b[a]) : B + (int64_t)a * R * d_out) + c;
        for (int q = 0; q < R; ++q) acc = fmaf(g[j * R + q], to_f(Bq[(int64_t)q * d_out]), acc);
      }
      y_add1(yr + c, acc);
    }
  }
}

template <typename T, typename YT, int R>
static cudaError_t launch_scalar_r(dim3 grid, size_t smem, int cluster, bool split, cudaStream_t stream,
                                   const T* xp, int32_t d_in, int32_t d_out, const T* Ap, const T* Bp, int32_t K,
                                   const int32_t* ids, const float* w, int32_t k, float scale, YT* yp,
                                   int32_t split_param, int32_t mask_adapter, int32_t* err_word, int32_t ind,
                                   const AdapterTable& tab) {
  if (split)
    return launch_kernel(lora_scalar_kernel<T, YT, R, true>, grid, dim3(kScalarThreads), smem, stream, cluster, xp,
                         d_in, d_out, Ap, Bp, K, ids, w, k, scale, yp, split_param, mask_adapter, err_word, ind, tab);
  return launch_kernel(lora_scalar_kernel<T, YT, R, false>, grid, dim3(kScalarThreads), smem, stream, 0, xp, d_in,
                       d_out, Ap, Bp, K, ids, w, k, scale, yp, split_param, mask_adapter, err_word, ind, tab);
}

template <typename T, typename YT>
static cudaError_t launch_scalar_t(const void* x, int64_t N, int32_t d_in, int32_t d_out, const void* A,
                                   const void* B, int32_t K, int32_t r, const int32_t* ids, const float* w,
                                   int32_t k, float scale, void* y, int32_t mask_adapter, int32_t* err_word,
                                   cudaStream_t stream, const AdapterTable* table) {
  const size_t base_smem = sizeof(float) * ((size_t)k * r + (kScalarThreads / 32) * r) + sizeof(int32_t) * k;
  // Small batches: a cluster of C CTAs per token splits d_in for the shrink (C times shorter a
  // chain) and d_out for the expand.  The widest C within the CTA budget, with row and column
  // splits that keep 4-column groups aligned, at least 256 rows and columns per CTA, and the
  // shared memory within 48 KB.
  int64_t split_ctas = kScalarSplitCtas;
#ifdef MOLORA_TUNING_ENV
  if (const char* e = getenv("MOLORA_SCALAR_SPLIT_CTAS")) split_ctas = atoi(e);
#endif
  int csplit = 1;
  int only_c = 0;
#ifdef MOLORA_TUNING_ENV
  if (const char* e = getenv("MOLORA_SCALAR_SPLIT_C")) only_c = atoi(e);
#endif
  for (int c : {8, 4, 2}) {
    if (only_c && c != only_c) continue;
    if (N * c <= split_ctas && d_in % c == 0 && d_out % (4 * c) == 0 && d_in / c >= 256 && d_out / c >= 256 &&
        base_smem + sizeof(float) * (size_t)c * k * r <= 48 * 1024) {
      csplit = c;
      break;
    }
  }
  dim3 grid;
  size_t smem = base_smem;
  int32_t split_param;
  if (csplit > 1) {
    grid = dim3((unsigned)(N * csplit));
    smem += sizeof(float) * (size_t)csplit * k * r;
    split_param = csplit;
  } else {
    // Enough CTAs to cover the GPU twice: other batches split the output columns (each split
    // recomputes the token's shrink).
    const int64_t want = 2 * (int64_t)num_sms();
    int64_t splits = N >= want ? 1 : (want + N - 1) / N;
    const int64_t max_splits = d_out >= 512 ? d_out / 512 : 1;
    if (splits > max_splits) splits = max_splits;
    int32_t cols = (int32_t)((d_out + splits - 1) / splits);
    cols = (cols + 3) & ~3;
    splits = (d_out + cols - 1) / cols;
    grid = dim3((unsigned)N, (unsigned)splits);
    split_param = cols;
  }
  const T* xp = static_cast<const T*>(x);
  const T* Ap = static_cast<const T*>(A);
  const T* Bp = static_cast<const T*>(B);
  YT* yp = static_cast<YT*>(y);
  AdapterTable tab;
  memset(&tab, 0, sizeof(tab));
  if (table) tab = *table;
  const int32_t ind = table ? 1 : 0;
  const bool split = csplit > 1;
  switch (r) {
    case 8:
      return launch_scalar_r<T, YT, 8>(grid, smem, csplit, split, stream, xp, d_in, d_out, Ap, Bp, K, ids, w, k, scale,
                                       yp, split_param, mask_adapter, err_word, ind, tab);
    case 16:
      return launch_scalar_r<T, YT, 16>(grid, smem, csplit, split, stream, xp, d_in, d_out, Ap, Bp, K, ids, w, k,
                                        scale, yp, split_param, mask_adapter, err_word, ind, tab);
    case 32:
      return launch_scalar_r<T, YT, 32>(grid, smem, csplit, split, stream, xp, d_in, d_out, Ap, Bp, K, ids, w, k,
                                        scale, yp, split_param, mask_adapter, err_word, ind, tab);
    case 64:
      return launch_scalar_r<T, YT, 64>(grid, smem, csplit, split, stream, xp, d_in, d_out, Ap, Bp, K, ids, w, k,
                                        scale, yp, split_param, mask_adapter, err_word, ind, tab);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_lora_scalar(const void* x, molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out,
                               const void* A, const void* B, int32_t K, int32_t r, const int32_t* ids,
                               const float* w, int32_t k, float scale, void* y, bool y_bf16, int32_t mask_adapter,
                               int32_t* err_word, cudaStream_t stream, const AdapterTable* table) {
  if (dtype == MOLORA_BF16)
    return y_bf16 ? launch_scalar_t<__nv_bfloat16, __nv_bfloat16>(x, N, d_in, d_out, A, B, K, r, ids, w, k, scale, y,
                                                                   mask_adapter, err_word, stream, table)
                  : launch_scalar_t<__nv_bfloat16, float>(x, N, d_in, d_out, A, B, K, r, ids, w, k, scale, y,
                                                          mask_adapter, err_word, stream, table);
  return y_bf16 ? launch_scalar_t<float, __nv_bfloat16>(x, N, d_in, d_out, A, B, K, r, ids, w, k, scale, y,
                                                         mask_adapter, err_word, stream, table)
                : launch_scalar_t<float, float>(x, N, d_in, d_out, A, B, K, r, ids, w, k, scale, y, mask_adapter,
                                                err_word, stream, table);
}

// ---------------------------------------------------------------------------------------
// CUDA-core router (fp32 x, or shapes the tensor-core router does not take).  A CTA owns 32
// tokens and all 64 hidden units: d_in is walked in chunks of 32, each chunk of x (token-major,
// [32 tokens][32 inputs], rows padded to 36 floats) and of W1 ([32 inputs][64 units]) staged in
// shared memory (two buffers; the next chunk's global loads are in flight in registers while the
// current one is multiplied).  Thread (tq, tu) accumulates tokens tq, tq+8, tq+16, tq+24 and
// hidden units 4tu..4tu+3, in order over d_in.  A warp spans 4 consecutive tq and 8 consecutive
// tu, so per 4 inputs it reads 4 float4 of x (rows 36 floats apart: distinct banks) and 4 float4
// of W1 (128 contiguous bytes): two shared-memory wavefronts per 16 FMAs of each thread.  Then
// ReLU, the 64 x K second layer, and one thread per token selects the top k (strictly greater
// wins, so equal logits keep the lower index) and renormalises the softmax over the selected k.
constexpr int kRouterTok = 32;
constexpr int kRouterChunk = 32;
constexpr int kRouterThreads = 128;
constexpr int kRouterXPad = kRouterChunk + 4;  // x rows: float4-aligned, 4 banks apart
// kSplit: a cluster of kRouterSplit CTAs per 32-token tile, CTA c taking a contiguous quarter
// of d_in (in whole chunks).  CTA j owns tokens 8j..8j+7 of the tile -- the tokens tq + 8j of
// every thread -- and the others push their partial hidden sums for those tokens into its slots
// in distributed shared memory; after one cluster barrier the owner adds the slots in rank order
// (so the result does not depend on timing), then runs the second layer and the top k for its
// tokens.  Four times the CTAs of the unsplit kernel, for the occupancy a 32-token tile alone
// cannot give.
constexpr int kRouterSplit = 4;
constexpr int kRouterOwn = kRouterTok / kRouterSplit;  // tokens each CTA of a cluster finishes

// 4 consecutive elements of T as floats: one 16-byte (fp32) or 8-byte (bf16) load when vec (the
// caller has checked alignment and that all 4 lie inside the row), else element by element up
// to n (zero past it).
__device__ __forceinline__ float4 load4(const float* p, bool vec, int n) {
  if (vec) return __ldg(reinterpret_cast<const float4*>(p));
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (n > 0) v.x = p[0];
  if (n > 1) v.y = p[1];
  if (n > 2) v.z = p[2];
  if (n > 3) v.w = p[3];
  return v;
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p, bool vec, int n) {
  if (vec) {
    const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
    return make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xFFFF0000u), __uint_as_float(q.y << 16),
                       __uint_as_float(q.y & 0xFFFF0000u));
  }
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (n > 0) v.x = to_f(p[0]);
  if (n > 1) v.y = to_f(p[1]);
  if (n > 2) v.z = to_f(p[2]);
  if (n > 3) v.w = to_f(p[3]);
  return v;
}

template <typename T, bool kSplit>
__global__ void __launch_bounds__(kRouterThreads)
    router_scalar_kernel(const T* __restrict__ x, int64_t N, int32_t d_in, const T* __restrict__ W1,
                         const float* __restrict__ b1, const T* __restrict__ W2, const float* __restrict__ b2,
                         int32_t K, int32_t k, float* __restrict__ logits, int32_t* __restrict__ ids,
                         float* __restrict__ w, int vec) {
  __shared__ __align__(16) float xs[2][kRouterTok][kRouterXPad];
  __shared__ __align__(16) float ws[2][kRouterChunk][kRouterHidden];
  // the hidden units and logits of the tokens this CTA finishes (all 32, or its block of 8)
  __shared__ float hid[kSplit ? kRouterOwn : kRouterTok][kRouterHidden + 1];
  __shared__ float lg[kSplit ? kRouterOwn : kRouterTok][kMaxAdapters];
  // kSplit: slots[rank][token of this CTA's block][hidden unit] (kRouterSplit x 8 x 65 floats).
  // Not aliased with the staging buffers: a peer may push while this CTA still multiplies.
  __shared__ float slots[kSplit ? kRouterSplit : 1][kRouterOwn][kRouterHidden + 1];
  constexpr int kXG = kRouterChunk / 4, kWG = kRouterHidden / 4;      // float4 groups per row
  constexpr int kXPer = kRouterTok * kXG / kRouterThreads;            // 2 groups of x per thread
  constexpr int kWPer = kRouterChunk * kWG / kRouterThreads;          // 4 groups of W1 per thread
  const int crank = kSplit ? (int)(blockIdx.x % (unsigned)kRouterSplit) : 0;  // == %cluster_ctarank
  const int64_t t0 = (int64_t)(kSplit ? blockIdx.x / (unsigned)kRouterSplit : blockIdx.x) * kRouterTok;
  const int tid = threadIdx.x, lane = tid & 31, wi = tid >> 5;
  const int tq = (wi & 1) * 4 + (lane >> 3), tu = (wi >> 1) * 8 + (lane & 7);
  // this CTA's rows of d_in: whole chunks, a contiguous share per rank
  const int nch_all = (d_in + kRouterChunk - 1) / kRouterChunk;
  const int per_rank = (nch_all + kRouterSplit - 1) / kRouterSplit;
  const int c_lo = kSplit ? min(nch_all, crank * per_rank) : 0;
  const int c_hi = kSplit ? min(nch_all, c_lo + per_rank) : nch_all;
  const bool v4 = vec != 0;
  if constexpr (kSplit) cluster_arrive();  // a peer's shared memory is written only once all have started
  pdl_wait();
  pdl_launch_dependents();
  if constexpr (kSplit) cluster_wait();
  float4 rx[kXPer], rw[kWPer];
  auto gload = [&](int c) {  // chunk c of x and W1 into registers (zero past the ends)
    const int i0 = c * kRouterChunk;
#pragma unroll
    for (int e = 0; e < kXPer; ++e) {
      const int idx = tid + e * kRouterThreads, q = idx / kXG, i = i0 + 4 * (idx % kXG);
      rx[e] = (t0 + q < N && i < d_in) ? load4(x + (t0 + q) * d_in + i, v4, d_in - i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int e = 0; e < kWPer; ++e) {
      const int idx = tid + e * kRouterThreads, ii = idx / kWG, u = 4 * (idx % kWG);
      rw[e] = i0 + ii < d_in ? load4(W1 + (int64_t)(i0 + ii) * kRouterHidden + u, v4, 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto sstore = [&](int b) {
#pragma unroll
    for (int e = 0; e < kXPer; ++e) {
      const int idx = tid + e * kRouterThreads;
      *reinterpret_cast<float4*>(&xs[b][idx / kXG][4 * (idx % kXG)]) = rx[e];
    }
#pragma unroll
    for (int e = 0; e < kWPer; ++e) {
      const int idx = tid + e * kRouterThreads;
      *reinterpret_cast<float4*>(&ws[b][idx / kWG][4 * (idx % kWG)]) = rw[e];
    }
  };
  float acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  if (c_lo < c_hi) {
    gload(c_lo);
    sstore(0);
  }
  __syncthreads();
  for (int c = c_lo; c < c_hi; ++c) {
    const int b = (c - c_lo) & 1;
    if (c + 1 < c_hi) gload(c + 1);
#pragma unroll 2
    for (int ii = 0; ii < kRouterChunk; ii += 4) {
      float4 xv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) xv[j] = *reinterpret_cast<const float4*>(&xs[b][tq + 8 * j][ii]);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const float4 wv = *reinterpret_cast<const float4*>(&ws[b][ii + s][4 * tu]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float a = s == 0 ? xv[j].x : s == 1 ? xv[j].y : s == 2 ? xv[j].z : xv[j].w;
          acc[j][0] = fmaf(a, wv.x, acc[j][0]);
          acc[j][1] = fmaf(a, wv.y, acc[j][1]);
          acc[j][2] = fmaf(a, wv.z, acc[j][2]);
          acc[j][3] = fmaf(a, wv.w, acc[j][3]);
        }
      }
    }
    if (c + 1 < c_hi) sstore(b ^ 1);  // buffer b^1 was last read before the previous barrier
    __syncthreads();
  }
  // tokens this CTA finishes: all 32, or its block of kRouterOwn within the cluster's tile
  const int q_lo = kSplit ? crank * kRouterOwn : 0;
  const int q_n = kSplit ? kRouterOwn : kRouterTok;
  if constexpr (kSplit) {
#pragma unroll
    for (int j = 0; j < 4; ++j)  // token tq + 8j of the tile is row tq of rank j's block
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const uint32_t local = smem_u32(&slots[crank][tq][4 * tu + jj]);
        st_cluster_f32(dsmem_addr(local, (uint32_t)j), acc[j][jj]);
      }
    cluster_sync();  // every rank's partials have landed; nothing remote after this
    for (int idx = tid; idx < kRouterOwn * kRouterHidden; idx += kRouterThreads) {
      const int ql = idx / kRouterHidden, u = idx % kRouterHidden;
      float h = 0.f;
#pragma unroll
      for (int p = 0; p < kRouterSplit; ++p) h += slots[p][ql][u];
      h += b1 ? b1[u] : 0.f;
      hid[ql][u] = h > 0.f ? h : 0.f;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const float h = acc[j][jj] + (b1 ? b1[4 * tu + jj] : 0.f);
        hid[tq + 8 * j][4 * tu + jj] = h > 0.f ? h : 0.f;
      }
  }
  __syncthreads();
  // hid rows 0..q_n-1 are tokens t0 + q_lo + 0..q_n-1
  const int64_t tb = t0 + q_lo;
  for (int idx = tid; idx < q_n * K; idx += kRouterThreads) {
    const int q = idx / K, a = idx % K;
    float s = 0.f;
    for (int jj = 0; jj < kRouterHidden; ++jj) s = fmaf(hid[q][jj], to_f(W2[jj * K + a]), s);
    if (b2) s += b2[a];
    lg[q][a] = s;
    if (logits && tb + q < N) logits[(tb + q) * K + a] = s;
  }
  __syncthreads();
  if (tid < q_n && tb + tid < N) {
    const int q = tid;
    const int64_t t = tb + q;
    uint64_t used = 0;
    float m = 0.f, denom = 0.f;
    for (int js = 0; js < k; ++js) {
      int best = -1;
      for (int a = 0; a < K; ++a)
        if (!((used >> a) & 1ull) && (best < 0 || lg[q][a] > lg[q][best])) best = a;
      used |= 1ull << best;
      ids[t * k + js] = best;
      if (js == 0) m = lg[q][best];
      const float e = expf(lg[q][best] - m);
      w[t * k + js] = e;
      denom += e;
    }
    const float inv = 1.f / denom;
    for (int js = 0; js < k; ++js) w[t * k + js] *= inv;
  }
}

cudaError_t launch_router_scalar(const void* x, molora_dtype dtype, int64_t N, int32_t d_in, const void* W1,
                                 const float* b1, const void* W2, const float* b2, int32_t K, int32_t k,
                                 float* logits, int32_t* ids, float* w, cudaStream_t stream) {
  const int64_t tiles = (N + kRouterTok - 1) / kRouterTok;
  // A cluster per tile where it pays (measured over N = 64..32768, d_in = 256..4096): a long d_in
  // (16+ chunks per rank), a grid of fewer tiles than SMs with 8+ chunks per rank, or tiles for
  // at most half the SMs.  Otherwise one CTA per tile: with 4-8 chunks per rank and the SMs
  // already busy, the cluster's exchange costs more than the CTAs it adds.
  const int64_t sms = num_sms();
  bool split = d_in >= kRouterSplit * kRouterChunk &&
               (d_in >= 2048 || (d_in >= 1024 && tiles < sms) || 2 * tiles <= sms);
#ifdef MOLORA_TUNING_ENV
  if (const char* e = getenv("MOLORA_ROUTER_SCALAR_SPLIT")) split = split && atoi(e) != 0;
#endif
  const unsigned grid = (unsigned)(tiles * (split ? kRouterSplit : 1));
  // whole 4-element groups of x rows and W1 rows, 16-byte (fp32) or 8-byte (bf16) aligned
  const uintptr_t align = dtype == MOLORA_BF16 ? 8 : 16;
  const int vec = d_in % 4 == 0 && (uintptr_t)x % align == 0 && (uintptr_t)W1 % align == 0;
  const int cluster = split ? kRouterSplit : 0;
  if (dtype == MOLORA_BF16) {
    const auto* xp = static_cast<const __nv_bfloat16*>(x);
    const auto* w1 = static_cast<const __nv_bfloat16*>(W1);
    const auto* w2 = static_cast<const __nv_bfloat16*>(W2);
    return split ? launch_kernel(router_scalar_kernel<__nv_bfloat16, true>, dim3(grid), dim3(kRouterThreads), 0, stream,
                                 cluster, xp, N, d_in, w1, b1, w2, b2, K, k, logits, ids, w, vec)
                 : launch_kernel(router_scalar_kernel<__nv_bfloat16, false>, dim3(grid), dim3(kRouterThreads), 0, stream,
                                 0, xp, N, d_in, w1, b1, w2, b2, K, k, logits, ids, w, vec);
  }
  const auto* xp = static_cast<const float*>(x);
  const auto* w1 = static_cast<const float*>(W1);
  const auto* w2 = static_cast<const float*>(W2);
  return split ? launch_kernel(router_scalar_kernel<float, true>, dim3(grid), dim3(kRouterThreads), 0, stream, cluster,
                               xp, N, d_in, w1, b1, w2, b2, K, k, logits, ids, w, vec)
               : launch_kernel(router_scalar_kernel<float, false>, dim3(grid), dim3(kRouterThreads), 0, stream, 0, xp,
                               N, d_in, w1, b1, w2, b2, K, k, logits, ids, w, vec);
}

}  // namespace molora
