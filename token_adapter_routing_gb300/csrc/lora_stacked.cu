// lora_stacked.cu -- the top-k LoRA apply of "MoLoRA: Composable Specialization via
// Per-Token Adapter Routing" for a large stacked rank K*r (up to 1024 columns), token-major,
// in two tcgen05 kernels around a workspace (Figure 2: a token's output is the weighted sum
// over its top-k adapters; Table 10's shapes; Table 16: the cost of raising k):
//
//   y[t,:] += sum_a G[t, a*r:(a+1)*r] B_a,   G[t, a*r + j] = scale * c[t,a] * (x[t,:] A_a)[j],
//   c[t,a] = sum_j [ids[t,j] == a] w[t,j]   (zero for the adapters a token did not select)
//
// i.e. the pages' sum written over all K adapters.  It costs K/k times the tensor work of
// grouping slots by adapter, and in exchange x is read once per token and every y element
// receives exactly one addition whatever k is, so the result is reproducible run to run.
//
// stacked_shrink_kernel: a 128-token tile is split over C CTAs by columns of the stacked
//   operand [A_0 | ... | A_{K-1}] (CTA c: adapters [c*K/C, (c+1)*K/C)).  A TMA producer warp
//   streams the tile's x K-blocks and the matching A rows through a ring of stages, one
//   thread issues tcgen05.mma (M = 128, N = the CTA's K*r/C columns) into TMEM.  With the
//   learned router (kRouter), W1's 64 columns ride along, 64/C per CTA, as a second MMA per
//   K step issued by a second thread (warp 6), so the two MMA streams are issued in parallel
//   and a stage is released by both threads' commits; the CTAs of a tile exchange their ReLU'd hidden units through distributed shared
//   memory, and every CTA evaluates the router's second stage for all 128 rows in the same
//   order (so all agree on ids and weights) and keeps the coefficients of its own adapters.
//   The epilogue scales each adapter's r columns by scale * c[t,a] and writes G as two bf16
//   terms G_hi + G_lo (relative error 2^-17) to the workspace.
// stacked_expand_kernel: a persistent tcgen05 GEMM y[N x d_out] += [G_hi | G_lo] B over
//   tiles of 128 rows x BN columns: a TMA producer warp fills a ring of (G_hi, G_lo, B)
//   K-blocks, one thread issues the MMAs into one of two TMEM accumulators, and four epilogue
//   warps drain the other: TMEM -> registers -> a swizzled staging box -> a TMA tensor
//   reduce-add into y (the fp32 addition happens in L2).  Each CTA prefetches the y rows of
//   its next tile into L2 while it works on the current one.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#ifdef MOLORA_TUNING_ENV
#include <cstdlib>
#endif

#include "common.cuh"
#include "kernels.h"

namespace molora {

namespace {

constexpr int kRows = 128;      // tile rows = TMEM lanes = MMA M
constexpr int kKBlock = 64;     // K elements per stage (one 128-byte swizzle row of bf16)
constexpr int kEpiThreads = 128;
constexpr int kThreads = kEpiThreads + 64;  // + TMA producer warp (4) + MMA warp (5)
constexpr int kShrThreads = kThreads + 32;  // shrink: + a second MMA warp (6) for the router's W1
constexpr size_t kMaxSmem = 227 * 1024;
constexpr size_t kSmemSlack = 1024;         // alignment of the dynamic smem base to 1024 B
constexpr int kMaxStages = 6;
constexpr int kHidStride = kRouterHidden + 4;  // floats per row of hidden units: conflict-free float4 rows

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---------------------------------------------------------------------------------------------
// shrink plan
struct ShrinkPlan {
  int C;                 // CTAs per tile (split of the stacked columns)
  int KC;                // adapters per CTA
  int NA;                // KC * r: adapter columns per CTA (MMA N, <= 256)
  int NH;                // router hidden columns per CTA (64 / C; 0 without the router)
  int S;                 // stages in the ring
  int PF;                // x K-blocks prefetched into L2 ahead of the TMA loads (0: none)
  uint32_t stage_bytes;  // x block, then the KC adapter blocks, then the W1 block
  uint32_t off_a, off_w1;
  uint32_t off_recv;     // router: all 64 hidden units of the 128 rows, fp32 [128][kHidStride], in
                         // the stage ring (free once every MMA of the tile's CTAs is done)
  uint32_t off_lg;       // router: the rows' logits fp32 [K][128 + 1] (transposed)
  uint32_t off_gst;      // G staging, 4 warps x (hi, lo) x [32 rows x 128 B], after those
  uint32_t off_par;      // router: W2 fp32 [64][K], b1 [64], b2 [K]; then coef fp32 [128][KC]
  uint32_t off_coef;
  uint32_t off_ctrl;
  uint32_t tmem_cols;
  uint32_t smem;
};

bool shrink_layout(int32_t K, int32_t r, int C, bool router, ShrinkPlan* s, int max_stages = kMaxStages) {
  if (K % C) return false;
  s->C = C;
  s->KC = K / C;
  s->NA = s->KC * r;
  s->NH = router ? kRouterHidden / C : 0;
  if (s->NA > 256 || s->NA % 16 || (router && s->NH < 16)) return false;
  s->off_a = (uint32_t)(kRows * kKBlock * 2);
  s->off_w1 = s->off_a + (uint32_t)(s->NA * kKBlock * 2);
  s->stage_bytes = (uint32_t)align_up(s->off_w1 + (size_t)s->NH * kKBlock * 2, 1024);
  const size_t recv = router ? (size_t)kRows * kHidStride * 4 : 0;
  const size_t lg = router ? (size_t)(kRows + 1) * K * 4 : 0;
  const size_t par = router ? sizeof(float) * ((size_t)kRouterHidden * K + kRouterHidden + K) : 0;
  const size_t coef = sizeof(float) * (size_t)kRows * s->KC;
  const size_t ctrl = 256 + 16 * kMaxStages;
  const uint32_t cols = (uint32_t)(s->NA + s->NH);
  s->tmem_cols = cols <= 32 ? 32 : cols <= 64 ? 64 : cols <= 128 ? 128 : cols <= 256 ? 256 : 512;
  s->PF = 8;
  s->off_recv = 0;
  s->off_lg = (uint32_t)recv;
  s->off_gst = (uint32_t)align_up(recv + lg, 1024);
  const size_t gst = (size_t)4 * 2 * 32 * 128;
  for (int S = max_stages; S >= 2; --S) {
    const size_t base = (size_t)S * s->stage_bytes;
    if (base < s->off_gst + gst) break;  // the epilogue's rows live in the ring after the MMAs
    const size_t off_par = base;
    const size_t off_coef = align_up(off_par + par, 16);
    const size_t off_ctrl = align_up(off_coef + coef, 64);
    size_t total = off_ctrl + ctrl + kSmemSlack;
    // all 512 TMEM columns: keep the CTA alone on its SM, so an allocation never waits
    if (s->tmem_cols > 256 && total < 116 * 1024) total = 116 * 1024;
    if (total <= kMaxSmem) {
      s->S = S;
      s->off_par = (uint32_t)off_par;
      s->off_coef = (uint32_t)off_coef;
      s->off_ctrl = (uint32_t)off_ctrl;
      s->smem = (uint32_t)total;
      return true;
    }
  }
  return false;
}

// The fewest column splits that fit (a CTA's MMA covers at most 256 columns), then more while
// the grid still fits the SMs twice over: a tile's CTAs run side by side.
bool shrink_choose(int64_t N, int32_t K, int32_t r, bool router, ShrinkPlan* s) {
  const int64_t tiles = (N + kRows - 1) / kRows;
  int max_stages = kMaxStages;
#ifdef MOLORA_TUNING_ENV
  if (const char* e = getenv("MOLORA_SHR_S")) max_stages = atoi(e);
#endif
  bool found = false;
  for (int C : {1, 2, 4}) {
    ShrinkPlan t;
    if (!shrink_layout(K, r, C, router, &t, max_stages)) continue;
    if (!found) {
      *s = t;
      found = true;
    } else if (tiles * C <= (int64_t)num_sms()) {
      *s = t;
    }
  }
#ifdef MOLORA_TUNING_ENV
  if (const char* e = getenv("MOLORA_SHR_PF")) s->PF = atoi(e);
#endif
  return found;
}

// ---------------------------------------------------------------------------------------------
// expand plan
struct ExpandPlan {
  int BN;                // output columns per tile (MMA N; two TMEM accumulators of BN columns)
  int S;                 // stages in the ring
  int nkb;               // K-blocks per tile: ceil(KR / 64)
  int nstg;              // epilogue staging buffers per warp (reductions in flight per warp)
  uint32_t stage_bytes;  // G_hi block, G_lo block, BN/64 B boxes
  uint32_t off_glo, off_b;
  uint32_t off_stage;    // epilogue staging: 4 warps x nstg buffers x [32 rows x 128 B]
  uint32_t off_ctrl;
  uint32_t smem;
};

bool expand_layout(int32_t KR, int BN, int nstg, int max_stages, ExpandPlan* s) {
  s->BN = BN;
  s->nkb = (KR + kKBlock - 1) / kKBlock;
  s->nstg = nstg;
  s->off_glo = (uint32_t)(kRows * kKBlock * 2);
  s->off_b = 2 * s->off_glo;
  s->stage_bytes = s->off_b + (uint32_t)(BN * kKBlock * 2);
  const size_t staging = (size_t)4 * nstg * 32 * 128;
  const size_t ctrl = 256 + 16 * kMaxStages;
  for (int S = max_stages; S >= 2; --S) {
    const size_t off_stage = (size_t)S * s->stage_bytes;
    const size_t off_ctrl = off_stage + staging;
    const size_t total = off_ctrl + ctrl + kSmemSlack;
    if (total <= kMaxSmem) {
      s->S = S;
      s->off_stage = (uint32_t)off_stage;
      s->off_ctrl = (uint32_t)off_ctrl;
      s->smem = (uint32_t)total;
      return true;
    }
  }
  return false;
}

// 256-column tiles halve the re-reads of G (narrow outputs take 128).  Measured on GB300 (top-k
// scaling workload, N = 8192, K*r = 512): three operand stages of 64 KB with two staging
// buffers per epilogue warp beat two stages with four or six buffers (121 vs 129 us for the
// router + apply), and 128-column tiles lose (136-146 us).
bool expand_choose(int32_t KR, int32_t d_out, ExpandPlan* s) {
  int only_bn = 0, nstg = 2, max_stages = kMaxStages;
#ifdef MOLORA_TUNING_ENV
  if (const char* e = getenv("MOLORA_EXP_BN")) only_bn = atoi(e);
  if (const char* e = getenv("MOLORA_EXP_NSTG")) nstg = atoi(e);
  if (const char* e = getenv("MOLORA_EXP_S")) max_stages = atoi(e);
#endif
  for (int BN : {256, 128}) {
    if (only_bn && BN != only_bn) continue;
    if (BN == 256 && d_out < 256) continue;
    for (int n = nstg; n >= 2; n -= 2)
      if (expand_layout(KR, BN, n, max_stages, s)) return true;
  }
  return false;
}

struct __align__(8) SCtrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t mma_done;
  uint64_t recv;
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint32_t tmem_base;
  int32_t abort;
};

__device__ __forceinline__ SmemLayout swizzle_for_row_bytes(uint32_t row_bytes) {
  return row_bytes == 32 ? kSwizzle32B : (row_bytes == 64 ? kSwizzle64B : kSwizzle128B);
}

}  // namespace

// The learned router's parameters and outputs for the fused variant.
struct StackRouterIo {
  const __nv_bfloat16* W2;  // [64 x K]
  const float* b1;          // [64] or null
  const float* b2;          // [K] or null
  float* logits;            // [N x K] or null
  int32_t* ids;             // [N x k]
  float* w;                 // [N x k]
};

template <bool kRouter>
__global__ void __launch_bounds__(kShrThreads, 1)
    stacked_shrink_kernel(int64_t N, int32_t d_in, int32_t K, int32_t r, int32_t k, const int32_t* __restrict__ ids,
                          const float* __restrict__ w, float scale, __nv_bfloat16* __restrict__ g_hi,
                          __nv_bfloat16* __restrict__ g_lo, int32_t* err_word, const StackRouterIo rio,
                          const ShrinkPlan P, const __grid_constant__ CUtensorMap map_x,
                          const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SCtrl* ctrl = reinterpret_cast<SCtrl*>(sm + P.off_ctrl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = P.C, KC = P.KC, NA = P.NA, NH = P.NH, S = P.S;
  const int crank = (int)(blockIdx.x % (unsigned)C);  // == %cluster_ctarank for the router's clusters of C
  const bool exchange = kRouter && C > 1;
  const int64_t t0 = (int64_t)(blockIdx.x / (unsigned)C) * kRows;
  const int a0 = crank * KC;
  const int KR = K * r;
  const int nkb = d_in / kKBlock;
  float* recv = reinterpret_cast<float*>(sm + P.off_recv);  // [128][kHidStride] hidden units (router), in the ring
  float* w2T = reinterpret_cast<float*>(sm + P.off_par);    // [K][64]: W2 transposed
  float* b1s = w2T + kRouterHidden * K;
  float* b2s = b1s + kRouterHidden;
  float* coef = reinterpret_cast<float*>(sm + P.off_coef);  // [128][KC] (coefficients given by ids / w)
  float* lg = reinterpret_cast<float*>(sm + P.off_lg);      // router: [K][128 + 1] logits, in the ring
  volatile int32_t* abort = &ctrl->abort;

  if (warp == 5) {
    tmem_alloc(&ctrl->tmem_base, P.tmem_cols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&ctrl->full[s], 1);
      mbar_init(&ctrl->empty[s], kRouter ? 2 : 1);
    }
    mbar_init(&ctrl->mma_done, kRouter ? 2 : 1);
    mbar_init(&ctrl->recv, 1);
    ctrl->abort = 0;
    mbar_fence_init();
    // the other CTAs' hidden units of all 128 rows
    if (exchange) mbar_arrive_expect_tx(&ctrl->recv, (uint32_t)kRows * (uint32_t)(kRouterHidden - NH) * 4u);
    tma_prefetch_desc(&map_x);
    tma_prefetch_desc(&map_a);
    if (kRouter) tma_prefetch_desc(&map_w1);
  }
  pdl_wait();  // x, ids and w may come from the previous kernel
  pdl_launch_dependents();
  if (warp < 4) {
    if (kRouter) {
      for (int i = tid; i < kRouterHidden * K; i += kEpiThreads) {
        const int u = i / K, a = i - u * K;
        w2T[a * kRouterHidden + u] = __bfloat162float(rio.W2[i]);
      }
      if (tid < kRouterHidden) b1s[tid] = rio.b1 ? rio.b1[tid] : 0.f;
      for (int i = tid; i < K; i += kEpiThreads) b2s[i] = rio.b2 ? rio.b2[i] : 0.f;
    } else {
      // this row's coefficient for each of the CTA's adapters: sum of the weights of the
      // slots that chose it (invalid ids are skipped and reported once per tile)
      const int64_t t = t0 + tid;
      for (int j = 0; j < KC; ++j) coef[tid * KC + j] = 0.f;
      if (t < N) {
        for (int j = 0; j < k; ++j) {
          const int32_t id = ids[t * k + j];
          if (id >= a0 && id < a0 + KC) coef[tid * KC + (id - a0)] += w ? w[t * k + j] : 1.f;
          if ((id < 0 || id >= K) && crank == 0) report(err_word, MOLORA_DEV_BAD_ADAPTER_ID);
        }
      }
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  if (exchange) cluster_arrive();  // every CTA's receive barrier is armed before any remote store

  if (warp == 4) {
    // ---- TMA producer: x K-block, the CTA's adapter rows of it, W1's columns of it
    if (lane == 0) {
      const uint32_t bytes = (uint32_t)(kRows + NA + NH) * kKBlock * 2u;
      // x streams from DRAM once per tile: the tile's first CTA asks L2 for its K-blocks PF
      // stages ahead of the loads, so the loads see L2 latency, not DRAM latency
      const bool prefetcher = crank == 0 && P.PF > 0;
      if (prefetcher)
        for (int kb = 0; kb < P.PF && kb < nkb; ++kb) tma_prefetch_l2_2d(&map_x, kb * kKBlock, (int32_t)t0);
      int issued = 0;
      for (int kb = 0; kb < nkb; ++kb, ++issued) {
        const int s = kb % S, use = kb / S;
        if (prefetcher && kb + P.PF < nkb) tma_prefetch_l2_2d(&map_x, (kb + P.PF) * kKBlock, (int32_t)t0);
        if (use > 0 && !mbar_wait_or_abort(&ctrl->empty[s], (uint32_t)(use - 1) & 1u, abort)) break;
        uint8_t* st = sm + (size_t)s * P.stage_bytes;
        mbar_arrive_expect_tx(&ctrl->full[s], bytes);
        tma_load_2d(smem_u32(st), &map_x, kb * kKBlock, (int32_t)t0, &ctrl->full[s]);
        for (int j = 0; j < KC; ++j)
          tma_load_2d(smem_u32(st + P.off_a + (size_t)j * kKBlock * r * 2), &map_a, 0,
                      (a0 + j) * d_in + kb * kKBlock, &ctrl->full[s]);
        if (kRouter) tma_load_2d(smem_u32(st + P.off_w1), &map_w1, crank * NH, kb * kKBlock, &ctrl->full[s]);
      }
      // nothing may land in shared memory after the CTA has left: wait for the last loads
      for (int s = 0; s < S && s < issued; ++s) {
        const int last = (issued - 1 - s) / S;  // last use of stage s
        mbar_wait(&ctrl->full[s], (uint32_t)last & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_a = idesc_bf16_f32(kRows, (uint32_t)NA, false, true);
      const SmemLayout swa = swizzle_for_row_bytes((uint32_t)r * 2u);
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int s = kb % S;
        ok = mbar_wait_or_abort(&ctrl->full[s], (uint32_t)(kb / S) & 1u, abort);
        if (!ok) break;
        tc_fence_after();
        const uint8_t* st = sm + (size_t)s * P.stage_bytes;
        for (int ks = 0; ks < kKBlock / 16; ++ks) {
          const uint64_t dx = smem_desc(smem_u32(st + ks * 32), 16, 1024, kSwizzle128B);
          // the CTA's adapters stacked along N: one box of 64 rows x r per adapter
          const uint64_t da = smem_desc(smem_u32(st + P.off_a + (size_t)ks * 16 * r * 2), (uint32_t)kKBlock * r * 2,
                                        8u * r * 2, swa);
          umma_f16(tmem, dx, da, idesc_a, (kb | ks) != 0);
        }
        umma_commit(&ctrl->empty[s]);  // the stage is free once these MMAs have read it
      }
      if (ok) {
        umma_commit(&ctrl->mma_done);
      } else {
        report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
        umma_commit(&ctrl->mma_done);  // still arrives once every MMA issued above has finished
      }
    }
    __syncwarp();
  } else if (kRouter && warp == 6) {
    // ---- the router's W1 MMAs, issued in parallel with the adapters' by a second thread
    if (lane == 0) {
      const uint32_t idesc_h = idesc_bf16_f32(kRows, (uint32_t)NH, false, true);
      const SmemLayout swh = swizzle_for_row_bytes((uint32_t)NH * 2u);
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int s = kb % S;
        ok = mbar_wait_or_abort(&ctrl->full[s], (uint32_t)(kb / S) & 1u, abort);
        if (!ok) break;
        tc_fence_after();
        const uint8_t* st = sm + (size_t)s * P.stage_bytes;
        for (int ks = 0; ks < kKBlock / 16; ++ks) {
          const uint64_t dx = smem_desc(smem_u32(st + ks * 32), 16, 1024, kSwizzle128B);
          const uint64_t dh =
              smem_desc(smem_u32(st + P.off_w1 + (size_t)ks * 16 * NH * 2), (uint32_t)kKBlock * NH * 2, 8u * NH * 2, swh);
          umma_f16(tmem + (uint32_t)NA, dx, dh, idesc_h, (kb | ks) != 0);
        }
        umma_commit(&ctrl->empty[s]);
      }
      if (!ok) report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
      umma_commit(&ctrl->mma_done);
    }
    __syncwarp();
  }

  // ---- epilogue (warps 0-3, one token row per thread)
  const int row = tid;
  const int64_t t = t0 + row;
  const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  bool have = false;
  float hid_own[kRouterHidden];  // this CTA's hidden units of the row (the first NH are used)
  if (warp < 4) {
    // warp-uniform: every lane of a warp must take the same branch around tcgen05.ld (.aligned)
    have = __all_sync(0xffffffffu, mbar_wait_or_abort(&ctrl->mma_done, 0, abort) && !*abort);
    tc_fence_after();
    if (kRouter) {
      // this CTA's sums x W1 for its hidden units, held in registers until the ring is free
#pragma unroll
      for (int c0 = 0; c0 < kRouterHidden; c0 += 16) {
        if (c0 < NH) {
          float v[16];
          if (have)
            tmem_ld16(lane_base + (uint32_t)(NA + c0), v);
          else
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) hid_own[c0 + i] = v[i];
        }
      }
    }
  }
  if (exchange) {
    __syncwarp();
    cluster_wait();  // every CTA's barriers are armed
    // the receive rows live in the stage ring: nobody writes them until every CTA of the tile
    // has finished its MMAs (its epilogue warps arrive here only after its mma_done)
    cluster_arrive();
    cluster_wait();
  }
  if (kRouter && warp < 4) {
    float* dst = recv + (size_t)row * kHidStride + crank * NH;
#pragma unroll
    for (int c0 = 0; c0 < kRouterHidden; c0 += 4)
      if (c0 < NH)
        reinterpret_cast<float4*>(dst)[c0 / 4] = make_float4(hid_own[c0], hid_own[c0 + 1], hid_own[c0 + 2], hid_own[c0 + 3]);
  }
  if (exchange) {
    if (warp < 4) {
      const uint32_t src = smem_u32(recv + (size_t)row * kHidStride + crank * NH);
      for (int d = 1; d < C; ++d) {
        const uint32_t peer = (uint32_t)((crank + d) % C);
        const uint32_t dst = dsmem_addr(src, peer);
        const uint32_t bar = dsmem_addr(smem_u32(&ctrl->recv), peer);
        for (int c = 0; c < NH; c += 4) {
          const float4 v = *reinterpret_cast<const float4*>(recv + (size_t)row * kHidStride + crank * NH + c);
          st_async_v4(dst + (uint32_t)c * 4u,
                      make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w)),
                      bar);
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&ctrl->recv, 0))) {
        have = false;
        if (lane == 0) report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
      }
    }
  }
  if (warp < 4) {
    if (kRouter) {
      // the router's second stage for this row, identical in every CTA of the tile so all agree
      // on ids and weights: hidden = ReLU(sum + b1); each logit is 8 group partials (an fmaf
      // chain over the group's 8 hidden units, chains independent) added in group order, then
      // b2; top k by logit (strictly greater wins, so equal logits keep the lower index);
      // softmax over the k, shifted by the largest.  The logits are kept transposed,
      // lgT[a][row], so a warp's accesses fall in distinct banks.  CTA 0 stores logits, ids
      // and w; every CTA keeps the coefficients of its own adapters.
      float* lgT = lg;  // [K][kRows + 1], used when K > 16
      float h[kRouterHidden];
#pragma unroll
      for (int i = 0; i < kRouterHidden / 4; ++i) {
        const float4 v = reinterpret_cast<const float4*>(recv + (size_t)row * kHidStride)[i];
        h[4 * i] = fmaxf(v.x + b1s[4 * i], 0.f);
        h[4 * i + 1] = fmaxf(v.y + b1s[4 * i + 1], 0.f);
        h[4 * i + 2] = fmaxf(v.z + b1s[4 * i + 2], 0.f);
        h[4 * i + 3] = fmaxf(v.w + b1s[4 * i + 3], 0.f);
      }
      auto logit = [&](int a) {  // 8 independent group chains, added in group order, then b2
        const float4* wr = reinterpret_cast<const float4*>(w2T + a * kRouterHidden);
        float p8[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float4 w0 = wr[2 * g], w1 = wr[2 * g + 1];
          float sg = 0.f;
          sg = fmaf(h[g * 8 + 0], w0.x, sg);
          sg = fmaf(h[g * 8 + 1], w0.y, sg);
          sg = fmaf(h[g * 8 + 2], w0.z, sg);
          sg = fmaf(h[g * 8 + 3], w0.w, sg);
          sg = fmaf(h[g * 8 + 4], w1.x, sg);
          sg = fmaf(h[g * 8 + 5], w1.y, sg);
          sg = fmaf(h[g * 8 + 6], w1.z, sg);
          sg = fmaf(h[g * 8 + 7], w1.w, sg);
          p8[g] = sg;
        }
        float acc = p8[0];
#pragma unroll
        for (int g = 1; g < 8; ++g) acc += p8[g];
        return acc + b2s[a];
      };
      for (int j = 0; j < KC; ++j) coef[row * KC + j] = 0.f;
      const bool writer = crank == 0 && t < N && have;
      // top k by logit (strictly greater wins, so equal logits keep the lower index), softmax
      // over the k shifted by the largest; run twice (denominator, then weights)
      auto select = [&](auto get) {
        float m = 0.f, denom = 0.f;
        for (int pass = 0; pass < 2; ++pass) {
          const float inv = pass ? 1.f / denom : 0.f;
          uint64_t used = 0;
          for (int js = 0; js < k; ++js) {
            int best = -1;
            float bl = 0.f;
            get(used, best, bl);
            used |= 1ull << best;
            if (js == 0) m = bl;
            const float e = expf(bl - m);
            if (pass == 0) {
              denom += e;
            } else {
              const float wj = e * inv;
              if (writer) {
                rio.ids[t * k + js] = best;
                rio.w[t * k + js] = wj;
              }
              if (best >= a0 && best < a0 + KC) coef[row * KC + (best - a0)] = wj;
            }
          }
        }
      };
      if (K <= 16) {  // the row's logits stay in registers
        float lr[16];
#pragma unroll
        for (int a = 0; a < 16; ++a) lr[a] = a < K ? logit(a) : 0.f;
        if (writer && rio.logits)
#pragma unroll
          for (int a = 0; a < 16; ++a)
            if (a < K) rio.logits[t * K + a] = lr[a];
        select([&](uint64_t used, int& best, float& bl) {
#pragma unroll
          for (int a = 0; a < 16; ++a)
            if (a < K && !((used >> a) & 1ull) && (best < 0 || lr[a] > bl)) best = a, bl = lr[a];
        });
      } else {  // kept transposed in shared memory, one column per row: distinct banks
        for (int a = 0; a < K; ++a) lgT[a * (kRows + 1) + row] = logit(a);
        if (writer && rio.logits)
          for (int a = 0; a < K; ++a) rio.logits[t * K + a] = lgT[a * (kRows + 1) + row];
        select([&](uint64_t used, int& best, float& bl) {
          for (int a = 0; a < K; ++a) {
            const float la = lgT[a * (kRows + 1) + row];
            if (!((used >> a) & 1ull) && (best < 0 || la > bl)) best = a, bl = la;
          }
        });
      }
    }
    // G = scale * c[t,a] * (x A_a), split into bf16 hi + lo, to the workspace rows, 64
    // columns at a time: each lane (a row) forms its values from TMEM into a swizzled staging
    // box [32 rows x 128 B] per term, then the warp writes them back row-wise, eight lanes to a
    // 128-byte row piece, so every store instruction covers four whole row pieces.  Every lane
    // loads TMEM (a warp-collective instruction); rows past N store nothing.
    if (have) {
      uint8_t* gst_hi = sm + P.off_gst + (size_t)warp * 2 * 4096;
      uint8_t* gst_lo = gst_hi + 4096;
      const int sub = lane >> 3, q = lane & 7;
      for (int c64 = 0; c64 < NA; c64 += 64) {
        const int wc = min(64, NA - c64);
        // both 32-column loads in flight, one wait (columns read past NA stay inside the
        // allocation, a power of two >= NA + the router's columns, and are not used)
        uint32_t ra[32], rb[32];
        tmem_ld32_start(lane_base + (uint32_t)c64, ra);
        if (wc > 32) tmem_ld32_start(lane_base + (uint32_t)(c64 + 32), rb);
        tmem_ld_wait(ra);
        tmem_ld_bind(rb);
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
          const int c16 = pc * 16;
          if (c16 >= wc) continue;
          const int j = (c64 + c16) / r;  // a 16-column piece never straddles two adapters (r >= 16)
          const float cf = scale * coef[row * KC + j];
          uint32_t hi[8], lo[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t u0 = pc < 2 ? ra[(pc & 1) * 16 + 2 * i] : rb[(pc & 1) * 16 + 2 * i];
            const uint32_t u1 = pc < 2 ? ra[(pc & 1) * 16 + 2 * i + 1] : rb[(pc & 1) * 16 + 2 * i + 1];
            const float g0 = cf * __uint_as_float(u0), g1 = cf * __uint_as_float(u1);
            const __nv_bfloat16 h0 = __float2bfloat16_rn(g0), h1 = __float2bfloat16_rn(g1);
            const __nv_bfloat16 l0 = __float2bfloat16_rn(g0 - __bfloat162float(h0));
            const __nv_bfloat16 l1 = __float2bfloat16_rn(g1 - __bfloat162float(h1));
            hi[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
            lo[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
          }
          const uint32_t cc = (uint32_t)c16 / 8u;  // 16-byte chunk of the 128-byte staging row
          *reinterpret_cast<uint4*>(gst_hi + sw128_offset((uint32_t)lane, cc)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(gst_hi + sw128_offset((uint32_t)lane, cc + 1)) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
          *reinterpret_cast<uint4*>(gst_lo + sw128_offset((uint32_t)lane, cc)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          *reinterpret_cast<uint4*>(gst_lo + sw128_offset((uint32_t)lane, cc + 1)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
        }
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int rr = it * 4 + sub;
          const int64_t t_rr = t0 + warp * 32 + rr;
          if (q * 8 < wc && t_rr < N) {
            const int64_t off = t_rr * KR + (int64_t)a0 * r + c64 + q * 8;
            *reinterpret_cast<uint4*>(g_hi + off) = *reinterpret_cast<const uint4*>(gst_hi + sw128_offset((uint32_t)rr, (uint32_t)q));
            *reinterpret_cast<uint4*>(g_lo + off) = *reinterpret_cast<const uint4*>(gst_lo + sw128_offset((uint32_t)rr, (uint32_t)q));
          }
        }
        __syncwarp();
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (exchange) {
    cluster_arrive();
    cluster_wait();  // no CTA leaves while a peer may still store into its shared memory
  }
  if (warp == 5) {
    if (lane == 0) mbar_wait(&ctrl->mma_done, 0);  // (already complete unless a wait gave up)
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, P.tmem_cols);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    stacked_expand_kernel(int64_t N, int32_t d_out, float* __restrict__ y, int32_t* err_word, const ExpandPlan P,
                          const __grid_constant__ CUtensorMap map_ghi, const __grid_constant__ CUtensorMap map_glo,
                          const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_y) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  SCtrl* ctrl = reinterpret_cast<SCtrl*>(sm + P.off_ctrl);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BN = P.BN, S = P.S, nkb = P.nkb;
  const int64_t m_tiles = (N + kRows - 1) / kRows;
  const int n_tiles = (d_out + BN - 1) / BN;
  // A cluster of two CTAs takes pairs of tiles: the same columns, consecutive 128-row blocks
  // (rank 0 the even block, rank 1 the odd one).  Both need the same B blocks, so each loads
  // half of every B block and multicasts it to both.  A rank-1 tile past the last row block
  // reads G as zeros (out of bounds) and writes nothing.
  const int rank = (int)cluster_ctarank();
  const int64_t ptiles = (m_tiles + 1) / 2 * n_tiles;  // tile pairs
  const int64_t cl = blockIdx.x / 2, ncl = gridDim.x / 2;
  auto tile_m0 = [&](int64_t pt) { return (int32_t)(((pt / n_tiles) * 2 + rank) * kRows); };
  auto tile_n0 = [&](int64_t pt) { return (int32_t)((pt % n_tiles) * BN); };
  volatile int32_t* abort = &ctrl->abort;
  // this thread's row segment of a tile, prefetched into L2 one tile ahead
  auto prefetch_y = [&](int64_t pt) {
    if (pt >= ptiles) return;
    const int64_t t = (int64_t)tile_m0(pt) + tid;
    const int n0 = tile_n0(pt);
    const int cols = min(BN, d_out - n0);
    if (t < N && cols > 0) prefetch_l2_bulk(y + t * d_out + n0, (uint32_t)cols * 4u);
  };

  if (warp == 5) {
    tmem_alloc(&ctrl->tmem_base, 2u * (uint32_t)BN);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&ctrl->full[s], 1);
      mbar_init(&ctrl->empty[s], 2);  // released by both CTAs' MMAs (B lands in both)
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctrl->tfull[b], 1);
      mbar_init(&ctrl->tempty[b], kEpiThreads);
    }
    mbar_init(&ctrl->mma_done, 1);
    ctrl->abort = 0;
    mbar_fence_init();
    tma_prefetch_desc(&map_ghi);
    tma_prefetch_desc(&map_glo);
    tma_prefetch_desc(&map_b);
    tma_prefetch_desc(&map_y);
  }
  // y is not written by the kernel this one may overlap; a prefetch only moves lines into L2
  if (warp < 4) prefetch_y(cl);
  pdl_wait();  // G comes from the previous kernel
  pdl_launch_dependents();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  cluster_arrive();
  cluster_wait();  // the partner's barriers are initialised before any multicast reaches them

  if (warp == 4) {
    // ---- TMA producer: per tile, nkb K-blocks of G_hi, G_lo and B
    if (lane == 0) {
      const uint32_t bytes = P.stage_bytes;
      int64_t it = 0;
      bool ok = true;
      for (int64_t pt = cl; pt < ptiles && ok; pt += ncl) {
        const int32_t m0 = tile_m0(pt);
        const int32_t n0 = tile_n0(pt);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = (int)(it % S);
          const int64_t use = it / S;
          if (use > 0 && !mbar_wait_or_abort(&ctrl->empty[s], (uint32_t)(use - 1) & 1u, abort)) {
            ok = false;
            break;
          }
          uint8_t* st = sm + (size_t)s * P.stage_bytes;
          mbar_arrive_expect_tx(&ctrl->full[s], bytes);
          tma_load_2d(smem_u32(st), &map_ghi, kb * kKBlock, m0, &ctrl->full[s]);
          tma_load_2d(smem_u32(st + P.off_glo), &map_glo, kb * kKBlock, m0, &ctrl->full[s]);
          // this CTA's half of the B boxes, into both CTAs (each counts all of B on its own full[s])
          for (int q = rank; q < BN / 64; q += 2)
            tma_load_2d_multicast(smem_u32(st + P.off_b + (size_t)q * kKBlock * 128), &map_b, n0 + q * 64,
                                  kb * kKBlock, &ctrl->full[s], (uint16_t)0x3);
        }
      }
      // nothing may land in shared memory after the CTA has left: the last fill of every stage
      // (the partner's multicast halves included) and both CTAs' last releases of it
      const int64_t issued = it;
      for (int s = 0; s < S && s < issued; ++s) {
        const int64_t last = (issued - 1 - s) / S;
        mbar_wait(&ctrl->full[s], (uint32_t)last & 1u);
        mbar_wait(&ctrl->empty[s], (uint32_t)last & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---- MMA issuer: D[buf] = G_hi B + G_lo B over the tile's K-blocks
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kRows, (uint32_t)BN, false, true);
      int64_t it = 0, tc = 0;
      bool ok = true;
      for (int64_t pt = cl; pt < ptiles && ok; pt += ncl, ++tc) {
        const int buf = (int)(tc & 1);
        const int64_t use = tc >> 1;
        if (use > 0 && !mbar_wait_or_abort(&ctrl->tempty[buf], (uint32_t)(use - 1) & 1u, abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * BN);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = (int)(it % S);
          if (!mbar_wait_or_abort(&ctrl->full[s], (uint32_t)(it / S) & 1u, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* st = sm + (size_t)s * P.stage_bytes;
          for (int ks = 0; ks < kKBlock / 16; ++ks) {
            // B: BN/64 boxes of [64 K-rows x 128 B], MN-major; 16 K-rows per step
            const uint64_t db = smem_desc(smem_u32(st + P.off_b + ks * 2048), kKBlock * 128, 1024, kSwizzle128B);
            const uint64_t dh = smem_desc(smem_u32(st + ks * 32), 16, 1024, kSwizzle128B);
            const uint64_t dl = smem_desc(smem_u32(st + P.off_glo + ks * 32), 16, 1024, kSwizzle128B);
            umma_f16(d, dh, db, idesc, (kb | ks) != 0);
            umma_f16(d, dl, db, idesc, 1);
          }
          umma_commit_multicast(&ctrl->empty[s], (uint16_t)0x3);  // the stage is free in both CTAs' eyes
        }
        if (!ok) break;
        umma_commit(&ctrl->tfull[buf]);
      }
      if (!ok) report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
      // TMEM is freed below only once every MMA issued here has completed
      umma_commit(&ctrl->mma_done);
    }
    __syncwarp();
  } else {
    // ---- epilogue: TMEM -> registers -> swizzled [32 rows x 32 cols] box -> TMA reduce-add into y
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const int nstg = P.nstg;
    uint8_t* stg = sm + P.off_stage + (size_t)warp * nstg * 4096;
    int sb = 0;
    int64_t tc = 0;
    for (int64_t pt = cl; pt < ptiles; pt += ncl, ++tc) {
      const int buf = (int)(tc & 1);
      prefetch_y(pt + ncl);
      // warp-uniform, since the TMEM loads below are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait_or_abort(&ctrl->tfull[buf], (uint32_t)(tc >> 1) & 1u, abort))) break;
      tc_fence_after();
      const int32_t m0 = tile_m0(pt) + warp * 32;
      const int32_t n0 = tile_n0(pt);
      // boxes that start past the last row or column hold nothing of y: skipped outright
      // (warp-uniform), so that the staging buffers are taken strictly in turn by issued
      // reductions and the wait below always covers the buffer about to be rewritten
      const int cmax = m0 < N ? min(BN / 32, (d_out - n0 + 31) / 32) : 0;
      auto emit = [&](const uint32_t(&v)[32], int c) {
        uint8_t* box = stg + (size_t)sb * 4096;
        if (lane == 0) bulk_wait_read_upto(nstg - 1);  // the reduction last issued from this buffer has read it
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<uint4*>(box + sw128_offset((uint32_t)lane, (uint32_t)i)) =
              make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_2d(&map_y, smem_u32(box), n0 + c * 32, m0);
          bulk_commit();
        }
        sb = sb + 1 == nstg ? 0 : sb + 1;
      };
      // TMEM loads one chunk ahead: the next 32 columns are in flight while this chunk is
      // staged and handed to the TMA unit
      const uint32_t cbase = lane_base + (uint32_t)(buf * BN);
      uint32_t va[32], vb[32];
      if (cmax > 0) tmem_ld32_start(cbase, va);
      for (int c = 0; c < cmax; c += 2) {
        tmem_ld_wait(va);
        if (c + 1 < cmax) tmem_ld32_start(cbase + (uint32_t)((c + 1) * 32), vb);
        emit(va, c);
        if (c + 1 < cmax) {
          tmem_ld_wait(vb);
          if (c + 2 < cmax) tmem_ld32_start(cbase + (uint32_t)((c + 2) * 32), va);
          emit(vb, c + 1);
        }
      }
      tc_fence_before();
      mbar_arrive(&ctrl->tempty[buf]);
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  __syncthreads();
  if (warp == 5) mbar_wait(&ctrl->mma_done, 0);
  __syncwarp();
  cluster_arrive();
  cluster_wait();  // neither CTA leaves while the other may still write or arrive into it
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 2u * (uint32_t)BN);
  }
}

// ---------------------------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 stacked_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// 2-D tensor map over a row-major [rows x cols] array of `esize`-byte elements.
bool stacked_map(CUtensorMap* m, CUtensorMapDataType type, uint32_t esize, const void* base, uint64_t rows,
                 uint64_t cols, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
  auto enc = stacked_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * esize};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, type, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

CUtensorMapSwizzle swizzle_for(uint32_t row_bytes) {
  return row_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                         : (row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
}

size_t g_bytes(int64_t N, int32_t KR) { return align_up((size_t)N * (size_t)KR * 2u, 256); }

}  // namespace

bool stacked_supported(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r,
                       bool router) {
  if (dtype != MOLORA_BF16 || !(r == 16 || r == 32 || r == 64) || d_in % kKBlock || d_out % 8) return false;
  ShrinkPlan sp;
  ExpandPlan ep;
  return shrink_choose(N, K, r, router, &sp) && expand_choose(K * r, d_out, &ep) && stacked_encoder() != nullptr;
}

size_t stacked_workspace_bytes(int64_t N, int32_t K, int32_t r) { return 2 * g_bytes(N, K * r); }

// Where AUTO takes the stacked pair rather than dispatch + grouped apply: a stacked rank of at
// least 256 columns (beyond the one-kernel dense path), few enough adapters per selected one
// (the pair does K/k times the grouped path's tensor work) and enough tokens for its tiles to
// fill the GPU.  Measured on GB300 at d = 4096 (bench.py --mode crossover_stacked: K*r of 256,
// 512 and 1024 with r = 16 and 64, k = 1, 2, 4, 1024..8192 tokens); this rule picks the faster
// path at 71 of the 72 points (the miss: a tie within 1%).  With k = 1 the grouped path gathers
// and reduces each token once, which is why it keeps small batches even at K/k = 4, and 2048
// tokens at K/k = 8 (8 adapters of rank 64: 46.3 vs 49.9 us, since the grouped plan counts
// waves of resident clusters at that rank).
bool stacked_preferred(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r, int32_t k,
                       bool router) {
  if (K * r < 256 || k < 1) return false;
  const int32_t per_pick = (K + k - 1) / k;
  const bool wins = (per_pick <= 4 && N >= 1024 && !(k == 1 && N < 2048)) ||
                    (per_pick <= 8 && N >= (k == 1 ? 4096 : 2048)) ||
                    (per_pick <= 16 && k >= 2 && N >= (k >= 4 ? 2048 : 4096));
  return wins && stacked_supported(dtype, N, d_in, d_out, K, r, router);
}

cudaError_t launch_lora_stacked(const void* x, int64_t N, int32_t d_in, int32_t d_out, const void* A, const void* B,
                                int32_t K, int32_t r, const int32_t* ids, const float* w, int32_t k, float scale,
                                float* y, void* ws, int32_t* err_word, const void* W1, const float* b1,
                                const void* W2, const float* b2, float* logits, int32_t* ids_out, float* w_out,
                                cudaStream_t stream) {
  const bool router = W1 != nullptr;
  const int32_t KR = K * r;
  ShrinkPlan sp;
  ExpandPlan ep;
  if (!shrink_choose(N, K, r, router, &sp) || !expand_choose(KR, d_out, &ep)) return cudaErrorNotSupported;
  __nv_bfloat16* g_hi = static_cast<__nv_bfloat16*>(ws);
  __nv_bfloat16* g_lo = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(ws) + g_bytes(N, KR));
  CUtensorMap map_x, map_a, map_w1, map_ghi, map_glo, map_b, map_y;
  const auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // x [N x d_in]: boxes of 128 rows x 64 columns (K-major, 128-byte swizzle)
  if (!stacked_map(&map_x, BF, 2, x, (uint64_t)N, (uint64_t)d_in, kKBlock, kRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // A seen as [K*d_in x r]: boxes of 64 rows of one adapter, swizzle matching r (MN-major)
  if (!stacked_map(&map_a, BF, 2, A, (uint64_t)K * d_in, (uint64_t)r, (uint32_t)r, kKBlock, swizzle_for((uint32_t)r * 2)))
    return cudaErrorInvalidValue;
  if (router) {
    // W1 [d_in x 64]: boxes of 64 rows x the CTA's 64/C columns
    if (!stacked_map(&map_w1, BF, 2, W1, (uint64_t)d_in, kRouterHidden, (uint32_t)sp.NH, kKBlock,
                     swizzle_for((uint32_t)sp.NH * 2)))
      return cudaErrorInvalidValue;
  } else {
    std::memset(&map_w1, 0, sizeof(map_w1));
  }
  // G_hi, G_lo [N x K*r]: boxes of 128 rows x 64 columns (K-major); columns past K*r read as 0
  if (!stacked_map(&map_ghi, BF, 2, g_hi, (uint64_t)N, (uint64_t)KR, kKBlock, kRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !stacked_map(&map_glo, BF, 2, g_lo, (uint64_t)N, (uint64_t)KR, kKBlock, kRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // B seen as [K*r x d_out]: boxes of 64 rows x 64 columns (MN-major); rows past K*r read as 0
  if (!stacked_map(&map_b, BF, 2, B, (uint64_t)KR, (uint64_t)d_out, 64, kKBlock, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // y [N x d_out] fp32: reduce boxes of 32 rows x 32 columns (128-byte swizzle)
  if (!stacked_map(&map_y, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, y, (uint64_t)N, (uint64_t)d_out, 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;

  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(stacked_shrink_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kMaxSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(stacked_shrink_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kMaxSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(stacked_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kMaxSmem);
    if (attr_err != cudaSuccess) cudaGetLastError();
  });
  if (attr_err != cudaSuccess) return attr_err;

  const StackRouterIo rio = {static_cast<const __nv_bfloat16*>(W2), b1, b2, logits, ids_out, w_out};
  const int64_t tiles = (N + kRows - 1) / kRows;
  // the router variant exchanges hidden units within a tile's CTAs: a cluster of C
  const int cluster = router && sp.C > 1 ? sp.C : 0;
  cudaError_t e = launch_kernel(router ? stacked_shrink_kernel<true> : stacked_shrink_kernel<false>,
                                dim3((unsigned)(tiles * sp.C)), dim3(kShrThreads), sp.smem, stream, cluster, N, d_in, K,
                                r, k, ids, w, scale, g_hi, g_lo, err_word, rio, sp, map_x, map_a, map_w1);
  if (e != cudaSuccess) return e;
  // persistent clusters of two CTAs over pairs of tiles (see stacked_expand_kernel)
  const int64_t exp_pairs = (tiles + 1) / 2 * ((d_out + ep.BN - 1) / ep.BN);
  const int64_t max_clusters = num_sms() / 2;
  const int grid = 2 * (int)(exp_pairs < max_clusters ? exp_pairs : max_clusters);
  return launch_kernel(stacked_expand_kernel, dim3((unsigned)grid), dim3(kThreads), ep.smem, stream, 2, N, d_out, y,
                       err_word, ep, map_ghi, map_glo, map_b, map_y);
}


// ---------------------------------------------------------------------------------------------
// Fixed scratch for molora_lora_apply_static_ws: a caller that cannot allocate device memory
// (see include/molora.h) gets the stacked path's workspace from this file-scope array instead.
// Every GPU that loads the library holds it until the process exits.  All calls on a device
// share it, so calls that may run at the same time on the GPU (different streams, or graphs
// replayed concurrently) race on it; nothing in it has to start at zero, because the shrink
// writes every row of G that the expand reads (rows past N come from the tensor map's
// out-of-bounds zero fill, not from memory).
namespace {
constexpr size_t kStaticScratchBytes = 16u << 20;
constexpr int kMaxDevices = 64;
}  // namespace
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

size_t stacked_static_scratch_bytes() { return kStaticScratchBytes; }

// The device address of g_static_scratch on the current device.  In host code the array's
// name only stands for the device symbol, so the address is looked up once per device (with
// that device current) and cached; the first call on a device does this.
cudaError_t stacked_static_scratch(void** ptr) {
  static void* addr[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
    }
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

}  // namespace molora
