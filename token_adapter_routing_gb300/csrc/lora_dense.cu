// lora_dense.cu -- the top-k LoRA apply of "MoLoRA: Composable Specialization via
// Per-Token Adapter Routing" computed token-major over the whole hot set (Figure 2: a
// token's output is the weighted sum over its top-k adapters; Table 10's shapes):
//
//   y[t,:] += scale * sum_a c[t,a] (x[t,:] A_a) B_a,   c[t,a] = sum_j [ids[t,j] == a] w[t,j]
//
// which is the pages' sum written over all K adapters, with weight zero for the ones a
// token did not select.  When K*r is small (the hot set's ranks stacked: 64 or 128
// columns) this evaluates every adapter for every token on the tensor cores instead of
// grouping slots by adapter, and in exchange reads each token's x row once and adds into
// each y row once, whatever k is -- the grouped path reads x and reduces into y once per
// slot, k times per token.  No dispatch is needed.
//
// A tile is 64 consecutive tokens, handled by a cluster of C CTAs:
//   1. shrink, split over d_in: CTA c gathers x[t0:t0+64, c*KS:(c+1)*KS) and the K-slices
//      of all K adapters' A with 16-byte cp.async, the latter stacked into one MN-major
//      operand [A_0 | ... | A_{K-1}] (K*r = 64 or 128 columns), and accumulates
//      H = x [A_0 | ... | A_{K-1}] (fp32) in TMEM with one tcgen05.mma per 16-element K step
//      (M = 128: rows past 64 are unused; N = K*r, so x is read from shared memory once per
//      step rather than once per adapter).  The K-slice comes in one round, or in two through
//      one buffer where one round would not fit two CTAs per SM; the tile's coefficients
//      c[t,a] are read while the gather is in flight;
//   2. the C partial H are summed through distributed shared memory in rank order
//      (deterministic), each adapter's r columns are scaled by scale * c[t,a], and the
//      result G is split into bf16 hi + lo and sent to every CTA of the cluster;
//   3. expand, split over d_out: D = G [B_0; ...; B_{K-1}] -- the B slab seen as
//      [K*r x d_out] is exactly the stacked operand -- in double-buffered passes of 128
//      columns whose B tiles stream in by TMA, two buffers deep;
//   4. epilogue: D goes TMEM -> registers -> shared memory -> one bulk fp32 (or bf16) add
//      per row segment into y, performed by the TMA unit in L2.  Every y element receives
//      one addition, so results are reproducible for any k.
// The router variant (kRouter) adds the learned router's W1 as one more 64-column block of
// the stacked shrink operand, so one pass over x feeds both; the owner CTA of each row runs
// the router's second stage (ReLU, logits, top k, softmax) on the reduced hidden partials and
// uses the resulting weights as c[t,a].
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

constexpr int kTileRows = 64;  // tokens per tile; the MMA has M = 128
constexpr int kMmaM = 128;
constexpr int kKBlock = 64;
constexpr int kPassW = 128;    // expand pass width (TMEM columns per buffer)
constexpr int kPiece = 128;    // y columns per bulk reduction
constexpr int kEpilogueThreads = 128;
constexpr int kThreads = kEpilogueThreads + 32;
constexpr uint32_t kTmemCols = 256;
constexpr size_t kMaxSmem = 227 * 1024;
constexpr size_t kTwoPerSm = 113 * 1024;
constexpr size_t kCtrlBytes = 1024;
constexpr uint32_t kBarX = 1;

struct DensePlan {
  int C, KS, NC, KR, PC;   // cluster size, K-slice, output columns per CTA, K*r, pushed columns per row
  int rounds, KSR;         // the K-slice is gathered in `rounds` rounds of KSR columns through one buffer
  int router;              // the learned router's 64 hidden columns ride along with the shrink
  uint32_t off_a, off_w1;  // phase 1: the stacked A rows (and W1's rows) of a round, after its x tile
  uint32_t off_g, off_b;   // phase 2: G hi/lo tiles, two B pass buffers
  uint32_t off_s;          // epilogue staging (also the receive slots, used earlier)
  uint32_t region, smem;
  uint32_t off_rt;         // router parameters and per-row scratch, after the control block
  uint32_t g_blk;          // bytes of one 64-column block of a G tile (128 rows x 128 B)
  uint32_t b_pass;         // bytes of one B pass buffer
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Per-CTA scratch (fp32): the router's W2 [64 x K], b1 [64] and b2 [8] (router variant only),
// and the owner rows' adapter coefficients [RPC][K].
inline size_t router_scratch_bytes(int K, int RPC) {
  return sizeof(float) * ((size_t)kRouterHidden * K + kRouterHidden + 8 + (size_t)RPC * K);
}

// Shared memory: phase 1 holds one round's x tile [KSR/64 blocks][64 rows][128 B] (plus room
// for the M = 128 MMA to read 64 rows past its last block), its rows of the stacked A
// operand and, with the router, of W1.  Phase 2 (after the shrink) reuses it for the G tiles
// and the B pass buffers.  The staging lines of the epilogue come after both and share their
// space with the receive slots of the cluster reduction: remote CTAs push their partials
// while this CTA's MMAs may still read phase 1, and the epilogue starts only after every
// partial has been consumed.  Two rounds halve phase 1, which is what lets the router's 64
// extra columns (and d_in = 4096) keep two CTAs per SM.
bool dense_plan(int32_t d_in, int32_t d_out, int32_t K, int32_t r, int C, int rounds, size_t budget, bool router,
                DensePlan* s) {
  if (d_in % (C * kKBlock * rounds) || d_out % (C * kKBlock)) return false;
  s->C = C;
  s->KS = d_in / C;
  s->rounds = rounds;
  s->KSR = s->KS / rounds;
  s->NC = d_out / C;
  s->KR = K * r;
  s->PC = s->KR + (router ? kRouterHidden : 0);
  s->router = router ? 1 : 0;
  if (s->KSR > 512) return false;
  const size_t x_bytes = (size_t)(s->KSR / kKBlock) * kTileRows * 128;
  const size_t a_bytes = (size_t)s->KSR * s->KR * 2;
  const size_t w1_bytes = router ? (size_t)s->KSR * kRouterHidden * 2 : 0;
  const size_t over = (size_t)(kMmaM - kTileRows) * 128;
  const size_t phase1 = x_bytes + (a_bytes + w1_bytes > over ? a_bytes + w1_bytes : over);
  const int kblocks = (s->KR + 63) / 64;  // 64-column blocks of a G tile
  s->g_blk = (uint32_t)(kMmaM * 128);
  const size_t g_bytes = 2 * (size_t)kblocks * s->g_blk;
  s->b_pass = (uint32_t)((kPassW / 64) * s->KR * 128);
  const size_t phase2 = align_up(g_bytes, 1024) + 2 * (size_t)s->b_pass;
  const size_t stage = (size_t)kTileRows * (kPiece * 4 + 16);
  const size_t recv = (size_t)kTileRows * s->PC * 4;
  s->off_a = (uint32_t)x_bytes;
  s->off_w1 = (uint32_t)(x_bytes + a_bytes);
  s->off_g = 0;
  s->off_b = (uint32_t)align_up(g_bytes, 1024);
  s->off_s = (uint32_t)align_up(phase1 > phase2 ? phase1 : phase2, 1024);
  s->region = (uint32_t)align_up(s->off_s + (stage > recv ? stage : recv), 1024);
  s->off_rt = s->region + (uint32_t)kCtrlBytes;
  s->smem = (uint32_t)(s->off_rt + align_up(router_scratch_bytes(K, kTileRows / C), 16) + 1024);
  return s->smem <= budget;
}

// Two CTAs per SM first, else one per SM.  Among the plans of a tier (one round first), the
// widest cluster whose CTAs all fit one wave (tiles x C <= CTAs resident at once): a second,
// partial wave repeats every CTA's serial front (gather, cluster reduction) behind the first
// wave's epilogue.  Measured on GB300 for the top-2 dense apply at 4096 tokens, 2048 -> 6144,
// K = 4, r = 16: clusters of 4 in one wave 49.1 us, clusters of 8 in 1.7 waves 53.2 us.  When
// no cluster fits one wave, the widest that fits the tier.
bool dense_choose(int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r, bool router, DensePlan* s) {
  // K*r = 256 would need 128 KB of G tiles alone (hi and lo, M = 128 rows): it never fits.
  // The stacked shrink operand is made of 64-column blocks: K*r is 64 or 128.
  if (!(r == 16 || r == 32 || r == 64) || (K * r != 64 && K * r != 128)) return false;
  int only_c = 0, only_rounds = 0;
#ifdef MOLORA_TUNING_ENV
  if (const char* e = getenv("MOLORA_DENSE_CLUSTER")) only_c = atoi(e);
  if (const char* e = getenv("MOLORA_DENSE_ROUNDS")) only_rounds = atoi(e);
#endif
  const int64_t tiles = (N + kTileRows - 1) / kTileRows;
  for (size_t budget : {kTwoPerSm, kMaxSmem}) {
    const int64_t resident = (budget == kTwoPerSm ? 2 : 1) * (int64_t)num_sms();
    bool found = false;
    DensePlan widest{};
    for (int C : {8, 4, 2, 1})
      for (int rounds : {1, 2, 4}) {
        if ((only_c && C != only_c) || (only_rounds && rounds != only_rounds)) continue;
        if (!dense_plan(d_in, d_out, K, r, C, rounds, budget, router, s)) continue;
        if (tiles * C <= resident) return true;
        if (!found) widest = *s, found = true;
        break;  // this cluster size's first fitting plan
      }
    if (found) {
      *s = widest;
      return true;
    }
  }
  return false;
}

// The learned router's parameters and outputs, for the fused variant (router + apply).
struct RouterIo {
  const __nv_bfloat16* W2;  // [64 x K]
  const float* b1;          // [64] or null
  const float* b2;          // [K] or null
  float* logits;            // [N x K] or null
  int32_t* ids;             // [N x k]
  float* w;                 // [N x k]
};

struct __align__(8) DCtrl {
  uint64_t bar_a;        // TMA of W1's slice (router variant)
  uint64_t bar_x;        // shrink MMAs done
  uint64_t bar_round;    // shrink MMAs of a round done: its buffer may be refilled (one phase per round)
  uint64_t bar_bp[2];    // B pass buffer loaded (one phase per use)
  uint64_t bar_full[2];  // expand pass done, per TMEM buffer
  uint64_t bar_empty[2]; // epilogue drained a TMEM buffer
  uint64_t bar_recv;     // this CTA's rows of partial H have arrived from every CTA
  uint64_t bar_g;        // all 64 rows of G (hi and lo) have arrived
  uint32_t tmem_base;
  int32_t abort;
  int32_t tok[kMmaM];    // token of each tile row, -1 past the batch
};
static_assert(sizeof(DCtrl) <= kCtrlBytes, "control block");

__device__ __forceinline__ SmemLayout layout_for_row_bytes(uint32_t row_bytes) {
  return row_bytes == 32 ? kSwizzle32B : (row_bytes == 64 ? kSwizzle64B : kSwizzle128B);
}

}  // namespace

// kRouter = false: ids and w are given.  kRouter = true: the kernel also runs the learned
// router on the same x tile (its W1 product is 64 more columns of the shrink) and writes
// logits, ids and w before using them.
template <bool kRouter>
__global__ void __launch_bounds__(kThreads, 1)
    lora_dense_kernel(const __nv_bfloat16* __restrict__ x, int64_t N, int32_t d_in, int32_t d_out, int32_t K,
                      int32_t r, int32_t k, const int32_t* __restrict__ ids, const float* __restrict__ w,
                      float scale, void* __restrict__ y, int32_t y_bf16, const DensePlan P, int32_t* err_word,
                      const RouterIo rio, const __nv_bfloat16* __restrict__ A,
                      const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_w1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DCtrl* ctrl = reinterpret_cast<DCtrl*>(sm + P.region);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = P.C, KS = P.KS, NC = P.NC, KR = P.KR, PC = P.PC, R = P.rounds, KSR = P.KSR;
  const int crank = (int)cluster_ctarank();
  const int64_t t0 = (int64_t)(blockIdx.x / C) * kTileRows;
  const int nvalid = (int)(N - t0 < kTileRows ? N - t0 : kTileRows);
  uint8_t* const yb = static_cast<uint8_t*>(y);
  const uint32_t ysz = y_bf16 ? 2u : 4u;

  uint8_t* xs = sm;
  uint8_t* as = sm + P.off_a;
  uint8_t* w1s = sm + P.off_w1;
  uint8_t* g_hi = sm + P.off_g;
  const int gblocks = (KR + 63) / 64;
  uint8_t* g_lo = g_hi + (size_t)gblocks * P.g_blk;
  const uint32_t g_row_bytes = KR >= 64 ? 128u : (uint32_t)KR * 2u;
  uint8_t* bs = sm + P.off_b;
  uint8_t* stage = sm + P.off_s;
  float* recv = reinterpret_cast<float*>(sm + P.off_s);  // [C sources][64/C rows][PC], before the epilogue
  const uint32_t stage_stride = (uint32_t)kPiece * 4u + 16u;
  const int RPC = kTileRows / C;
  // router scratch: W2 and the biases as fp32, per-row adapter coefficients
  float* w2s = reinterpret_cast<float*>(sm + P.off_rt);
  float* b1s = w2s + kRouterHidden * K;
  float* b2s = b1s + kRouterHidden;
  float* coef_s = b2s + 8;  // [RPC][K]

  if (warp == 4) {
    tmem_alloc(&ctrl->tmem_base, kTmemCols);
    tmem_relinquish();
    if (lane == 0) {
      mbar_init(&ctrl->bar_a, 1);
      mbar_init(&ctrl->bar_x, 1);
      mbar_init(&ctrl->bar_round, 1);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&ctrl->bar_bp[i], 1);
        mbar_init(&ctrl->bar_full[i], 1);
        mbar_init(&ctrl->bar_empty[i], kEpilogueThreads);
      }
      mbar_init(&ctrl->bar_recv, 1);
      mbar_init(&ctrl->bar_g, 1);
      mbar_fence_init();
      mbar_arrive_expect_tx(&ctrl->bar_recv, (uint32_t)kTileRows * PC * 4u);
      mbar_arrive_expect_tx(&ctrl->bar_g, (uint32_t)kTileRows * KR * 4u);
      ctrl->abort = 0;
      tma_prefetch_desc(&map_b);
      if (kRouter) tma_prefetch_desc(&map_w1);
    }
  }
  pdl_wait();
  pdl_launch_dependents();
  if (warp < 4) ctrl->tok[tid] = tid < nvalid ? (int32_t)(t0 + tid) : -1;
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  __syncwarp();
  cluster_arrive();  // barriers of every CTA initialised and armed

  // ---- shrink, in R rounds of KSR columns through one buffer
  auto load_w1 = [&](int rd) {  // W1 rows of round rd: 64 x 64 boxes landing MN-major (128-byte
                                // swizzle), one more 64-column block right after the stacked A blocks
    mbar_arrive_expect_tx(&ctrl->bar_a, (uint32_t)KSR * kRouterHidden * 2);
    for (int kb = 0; kb < KSR / kKBlock; ++kb)
      tma_load_2d(smem_u32(w1s + (size_t)kb * kKBlock * 128), &map_w1, 0, crank * KS + rd * KSR + kb * kKBlock,
                  &ctrl->bar_a);
  };
  if (kRouter && warp == 4 && lane == 0) load_w1(0);
  bool shrink_ok = true;
  for (int rd = 0; rd < R; ++rd) {
    if (warp < 4) {
      if (rd > 0 && !mbar_wait(&ctrl->bar_round, (uint32_t)(rd - 1) & 1u)) {  // the buffer is free again
        ctrl->abort = 1;
        report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
      }
      const int sub = lane >> 3, chunk = lane & 7;
      for (int kb = 0; kb < KSR / kKBlock; ++kb) {
        const uint32_t blk = smem_u32(xs + (size_t)kb * kTileRows * 128);
        const int col = crank * KS + rd * KSR + kb * kKBlock + chunk * 8;
#pragma unroll 4
        for (int it = 0; it < kTileRows / 16; ++it) {
          const int row = it * 16 + warp * 4 + sub;
          const int32_t tok = ctrl->tok[row];
          const __nv_bfloat16* src = tok >= 0 ? x + (int64_t)tok * d_in + col : x;
          cp_async_16(blk + sw128_offset(row, chunk), src, tok >= 0 ? 16u : 0u);
        }
      }
      // every adapter's rows of this round, stacked as one MN-major [KSR x K*r] operand:
      // 64-column blocks of KSR rows x 128 B with the 128-byte swizzle (column a*r + j is A_a[., j])
      const int cpr = r / 8;  // 16-byte chunks per adapter row
      const int per_a = KSR * cpr;
      for (int q = tid; q < K * per_a; q += kEpilogueThreads) {
        const int a = q / per_a, rem = q - a * per_a, i = rem / cpr, c = rem - i * cpr;
        const int n = a * r + c * 8;
        cp_async_16(smem_u32(as + (size_t)(n / 64) * KSR * 128 + sw128_offset(i, (n % 64) / 8)),
                    A + ((int64_t)a * d_in + crank * KS + rd * KSR + i) * r + c * 8, 16u);
      }
      cp_async_commit();
      if (rd == 0 && !kRouter) {
        // the owner rows' coefficients sum_j [ids[t,j] == a] w[t,j], while the gather is in flight
        for (int q = tid; q < RPC * K; q += kEpilogueThreads) {
          const int rl = q / K, a = q - rl * K;
          const int64_t t = t0 + crank * RPC + rl;
          float c = 0.f;
          if (t < N) {
            for (int j = 0; j < k; ++j) {
              const int32_t id = ids[t * k + j];
              if (id == a) c += w ? w[t * k + j] : 1.f;
              if ((id < 0 || id >= K) && a == 0) report(err_word, MOLORA_DEV_BAD_ADAPTER_ID);
            }
          }
          coef_s[q] = c;
        }
      }
      if (rd == 0 && kRouter) {  // the router's second layer, while the gather is in flight
        for (int i = tid; i < kRouterHidden * K; i += kEpilogueThreads) w2s[i] = __bfloat162float(rio.W2[i]);
        if (tid < kRouterHidden) b1s[tid] = rio.b1 ? rio.b1[tid] : 0.f;
        if (tid < K) b2s[tid] = rio.b2 ? rio.b2[tid] : 0.f;
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
    }
    __syncwarp();
    named_barrier(kBarX, kThreads);  // round rd's x, A (and the coefficients or W2) are in shared memory
    if (warp == 4 && lane == 0) {
      if (shrink_ok && kRouter) shrink_ok = mbar_wait(&ctrl->bar_a, (uint32_t)rd & 1u);
      shrink_ok = shrink_ok && !ctrl->abort;
      tc_fence_after();
      if (shrink_ok) {
        // one MMA per 16-row K step over all adapters at once (and the router's W1): the x
        // tile is read once per step, not once per adapter.  TMEM columns [0, K*r) take x A_a
        // for every adapter in order, [K*r, K*r + 64) the router's hidden partials.
        const uint32_t idesc = idesc_bf16_f32(kMmaM, (uint32_t)PC, false, true);
        for (int kb = 0; kb < KSR / kKBlock; ++kb)
          for (int ks = 0; ks < kKBlock / 16; ++ks) {
            // 128 MMA rows from the block's start: the tile's 64 rows, then 64 unused rows
            const uint64_t da = smem_desc(smem_u32(xs + (size_t)kb * kTileRows * 128 + ks * 32), 16, 1024,
                                          kSwizzle128B);
            const uint64_t db = smem_desc(smem_u32(as + (size_t)kb * kKBlock * 128 + ks * 2048),
                                          (uint32_t)KSR * 128u, 1024, kSwizzle128B);
            umma_f16(tmem, da, db, idesc, (rd | kb | ks) != 0);
          }
      }
      if (rd + 1 < R) {
        // this round's MMAs release the buffer; the last round's completion is bar_x
        if (shrink_ok) umma_commit(&ctrl->bar_round);
        else mbar_arrive(&ctrl->bar_round);
        if (kRouter && shrink_ok) {
          shrink_ok = mbar_wait(&ctrl->bar_round, (uint32_t)rd & 1u);
          if (shrink_ok) load_w1(rd + 1);
        }
      } else if (shrink_ok) {
        umma_commit(&ctrl->bar_x);
      } else {
        ctrl->abort = 1;
        report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
        mbar_arrive(&ctrl->bar_x);
      }
    }
  }
  const int npass = (NC + kPassW - 1) / kPassW;
  auto load_b = [&](int p) {  // B rows [0, KR) of columns [c*NC + p*128, +128), into buffer p % 2
    uint8_t* bb = bs + (size_t)(p & 1) * P.b_pass;
    const int width = min(kPassW, NC - p * kPassW);
    mbar_arrive_expect_tx(&ctrl->bar_bp[p & 1], (uint32_t)(width / 64) * KR * 128);
    for (int q = 0; q < width / 64; ++q)
      tma_load_2d(smem_u32(bb + (size_t)q * KR * 128), &map_b, crank * NC + p * kPassW + q * 64, 0,
                  &ctrl->bar_bp[p & 1]);
  };
  if (warp == 4 && lane == 0) {
    // the first two B passes land in phase-1 space once the shrink MMAs have read it
    if (mbar_wait(&ctrl->bar_x, 0)) {
      for (int p = 0; p < npass && p < 2; ++p) load_b(p);
    } else {
      ctrl->abort = 1;
      report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
    }
  }

  // ---- cluster reduction of H, pushed to the row owners
  bool have_h = true;
  if (warp < 4) {
    if (tid < nvalid) prefetch_l2_bulk(yb + ((t0 + tid) * d_out + crank * NC) * ysz, (uint32_t)NC * ysz);
    have_h = mbar_wait(&ctrl->bar_x, 0);
    tc_fence_after();
    if (!have_h) {
      ctrl->abort = 1;
      report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
    }
  }
  __syncwarp();
  cluster_wait();
  if (warp < 2) {  // rows 0..63
    const int row = tid;
    const uint32_t owner = (uint32_t)(row / RPC);
    const uint32_t dst = dsmem_addr(smem_u32(recv + ((size_t)crank * RPC + (row % RPC)) * PC), owner);
    const uint32_t dst_bar = dsmem_addr(smem_u32(&ctrl->bar_recv), owner);
    float v[16];
    for (int c0 = 0; c0 < PC; c0 += 16) {
      if (have_h)
        tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
      else
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        st_async_v4(dst + (c0 + 4 * i) * 4,
                    make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]), __float_as_uint(v[4 * i + 2]),
                               __float_as_uint(v[4 * i + 3])),
                    dst_bar);
    }
  }
  if (warp < 4) {
    tc_fence_before();
    const bool got = mbar_wait(&ctrl->bar_recv, 0);
    if (!got) {
      ctrl->abort = 1;
      report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
    }
    if (kRouter) {
      // the learned router for the owner's rows: hidden units from the C partials,
      // logits, top k and softmax; logits, ids and w go out, the coefficients to scratch
      // (the plan takes K*r of 64 or 128 with r >= 16, so K <= 8: one logit per lane)
      router_rows_jl<1, 1>(recv, C, RPC, PC, KR, false, w2s, b1s, b2s, K, k, t0 + crank * RPC, N, got && have_h,
                        rio.logits, rio.ids, rio.w, coef_s, tid, kEpilogueThreads, true);
      named_barrier(2, kEpilogueThreads);  // coefficients ready
    }
    // owner: rows [crank*RPC, (crank+1)*RPC) of the tile; each item is 8 columns of one row
    const int groups = KR / 8;
    for (int item = tid; item < RPC * groups; item += kEpilogueThreads) {
      const int rl = item / groups, c0 = (item % groups) * 8;
      const int trow = crank * RPC + rl;
      const int a = c0 / r;
      const float coef = coef_s[rl * K + a] * scale;
      float h[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int cc = 0; cc < C; ++cc) {
        const float4* src = reinterpret_cast<const float4*>(recv + ((size_t)cc * RPC + rl) * PC + c0);
        const float4 p0 = src[0], p1 = src[1];
        h[0] += p0.x, h[1] += p0.y, h[2] += p0.z, h[3] += p0.w;
        h[4] += p1.x, h[5] += p1.y, h[6] += p1.z, h[7] += p1.w;
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float g0 = coef * h[2 * i], g1 = coef * h[2 * i + 1];
        const __nv_bfloat16 h0 = __float2bfloat16_rn(g0), h1 = __float2bfloat16_rn(g1);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(g0 - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(g1 - __bfloat162float(h1));
        hi[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
        lo[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
      }
      // G is K-major: 64-column blocks of 128 rows x 128 B (or one narrower block)
      const uint32_t off = (uint32_t)(c0 / 64) * P.g_blk + swz_offset(trow, (c0 % 64) / 8, g_row_bytes);
      const uint4 vh = make_uint4(hi[0], hi[1], hi[2], hi[3]), vl = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      for (int d = 0; d < C; ++d) {
        const uint32_t bar_d = dsmem_addr(smem_u32(&ctrl->bar_g), (uint32_t)d);
        st_async_v4(dsmem_addr(smem_u32(g_hi + off), (uint32_t)d), vh, bar_d);
        st_async_v4(dsmem_addr(smem_u32(g_lo + off), (uint32_t)d), vl, bar_d);
      }
    }
  }
  __syncwarp();

  // ---- expand and epilogue
  if (warp == 4) {
    if (lane == 0) {
      bool ok = !ctrl->abort && mbar_wait(&ctrl->bar_g, 0);
      fence_proxy_async_smem();
      tc_fence_after();
      const SmemLayout gl = layout_for_row_bytes(g_row_bytes);
      for (int p = 0; p < npass; ++p) {
        const int buf = p & 1;
        const int width = min(kPassW, NC - p * kPassW);
        if (ok) ok = mbar_wait(&ctrl->bar_bp[buf], (uint32_t)(p >> 1) & 1u);
        if (p >= 2 && ok) ok = mbar_wait(&ctrl->bar_empty[buf], (uint32_t)((p >> 1) - 1) & 1u);
        if (!ok) {
          ctrl->abort = 1;
          report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
          mbar_arrive(&ctrl->bar_full[buf]);
          continue;
        }
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(kMmaM, width, false, true);
        const uint32_t d = tmem + (uint32_t)(buf * kPassW);
        const uint8_t* bb = bs + (size_t)buf * P.b_pass;
        for (int ks = 0; ks < KR / 16; ++ks) {
          const uint64_t db = smem_desc(smem_u32(bb + (size_t)ks * 2048), (uint32_t)KR * 128u, 1024, kSwizzle128B);
          const uint32_t goff = (uint32_t)(ks / 4) * P.g_blk + (uint32_t)(ks % 4) * 32u;
          umma_f16(d, smem_desc(smem_u32(g_hi + goff), 16, 8 * g_row_bytes, gl), db, idesc, ks != 0);
          umma_f16(d, smem_desc(smem_u32(g_lo + goff), 16, 8 * g_row_bytes, gl), db, idesc, 1);
        }
        umma_commit(&ctrl->bar_full[buf]);
        if (p + 2 < npass) {
          // this buffer's B tile is free once these MMAs are done
          ok = mbar_wait(&ctrl->bar_full[buf], (uint32_t)(p >> 1) & 1u);
          if (ok) load_b(p + 2);
        }
      }
    }
    __syncwarp();
  } else {
    const int row = tid;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float* srow = reinterpret_cast<float*>(stage + row * stage_stride);
    const int32_t my_tok = row < nvalid ? (int32_t)(t0 + row) : -1;
    for (int p = 0; p < npass; ++p) {
      const int buf = p & 1;
      const int width = min(kPassW, NC - p * kPassW);
      const bool ok = mbar_wait(&ctrl->bar_full[buf], (uint32_t)(p >> 1) & 1u);
      tc_fence_after();
      if (!ok) report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
      for (int q = 0; ok && !ctrl->abort && warp < 2 && q < width; q += kPiece) {
        const int cols = min(kPiece, width - q);
        bulk_wait_read<0>();  // the previous reduction has read the line
        for (int c0 = 0; c0 < cols; c0 += 32) {
          float v[32];
          tmem_ld32(lane_base + (uint32_t)(buf * kPassW + q + c0), v);
          if (my_tok >= 0) {
            if (y_bf16) {
              uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(srow) + c0 * 2);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t u[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * i + 2 * j], v[8 * i + 2 * j + 1]);
                  u[j] = *reinterpret_cast<const uint32_t*>(&b2);
                }
                dst[i] = make_uint4(u[0], u[1], u[2], u[3]);
              }
            } else {
              float4* dst = reinterpret_cast<float4*>(srow + c0);
#pragma unroll
              for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            }
          }
        }
        fence_proxy_async_smem();
        if (my_tok >= 0) {
          void* dst = yb + ((int64_t)my_tok * d_out + crank * NC + p * kPassW + q) * ysz;
          if (y_bf16)
            bulk_reduce_add_bf16(dst, smem_u32(srow), (uint32_t)cols * 2u);
          else
            bulk_reduce_add_f32(static_cast<float*>(dst), smem_u32(srow), (uint32_t)cols * 4u);
          bulk_commit();
        }
      }
      tc_fence_before();
      mbar_arrive(&ctrl->bar_empty[buf]);
    }
    bulk_wait_all();
  }
  __syncthreads();
  cluster_arrive();
  cluster_wait();  // no CTA leaves while another may still write into its shared memory
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 dense_encoder() {
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

bool dense_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows,
               CUtensorMapSwizzle swz) {
  auto enc = dense_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool dense_supported(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r) {
  DensePlan s;
  return dtype == MOLORA_BF16 && dense_choose(N, d_in, d_out, K, r, false, &s) && dense_encoder() != nullptr;
}

bool router_dense_supported(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r) {
  DensePlan s;
  return dtype == MOLORA_BF16 && dense_choose(N, d_in, d_out, K, r, true, &s) && dense_encoder() != nullptr;
}

// Where the dense path beat the scalar and grouped ones on GB300 (top-2, r = 16, warm and L2
// flushed alike): with a plan of two CTAs per SM (one or two gather rounds) from 512 tokens --
// 4096 -> 4096 at K = 4: 18.6 vs 19.4 us at 512 and 23.8 vs 32.9 us at 2048 tokens; 2048 -> 6144
// at K = 4: 18.2 vs 21.3 us at 512 and 49 vs 71 us at 4096.  A one-CTA-per-SM plan (K*r = 128
// at d_in = 4096) leaves too few clusters resident, and small batches pay for the extra
// adapters: the scalar or grouped path won all of those points.
bool dense_preferred(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r) {
  if (dtype != MOLORA_BF16 || N < 512 || !(r == 16 || r == 32 || r == 64) || (K * r != 64 && K * r != 128))
    return false;
  DensePlan s;
  for (int C : {8, 4, 2, 1})
    for (int rounds : {1, 2})
      if (dense_plan(d_in, d_out, K, r, C, rounds, kTwoPerSm, false, &s)) return dense_encoder() != nullptr;
  return false;
}

namespace {

cudaError_t launch_dense(const void* x, int64_t N, int32_t d_in, int32_t d_out, const void* A, const void* B,
                         int32_t K, int32_t r, const int32_t* ids, const float* w, int32_t k, float scale, void* y,
                         bool y_bf16, int32_t* err_word, const void* W1, const RouterIo& rio, cudaStream_t stream) {
  const bool router = W1 != nullptr;
  DensePlan s;
  if (!dense_choose(N, d_in, d_out, K, r, router, &s)) return cudaErrorNotSupported;
  CUtensorMap map_b, map_w1;
  // B seen as [K*r x d_out]: a box is all K*r rows (every adapter) by 64 columns
  if (!dense_map(&map_b, B, (uint64_t)K * r, (uint64_t)d_out, 64, (uint32_t)(K * r), CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  if (router) {
    // W1 [d_in x 64]: boxes of 64 rows x 64 columns (128 B rows, 128-byte swizzle)
    if (!dense_map(&map_w1, W1, (uint64_t)d_in, kRouterHidden, kRouterHidden, kKBlock, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  } else {
    std::memset(&map_w1, 0, sizeof(map_w1));
  }
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(lora_dense_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kMaxSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(lora_dense_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kMaxSmem);
    if (attr_err != cudaSuccess) cudaGetLastError();
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t tiles = (N + kTileRows - 1) / kTileRows;
  return launch_kernel(router ? lora_dense_kernel<true> : lora_dense_kernel<false>, dim3((unsigned)(tiles * s.C)),
                       dim3(kThreads), s.smem, stream, s.C, static_cast<const __nv_bfloat16*>(x), N, d_in, d_out, K,
                       r, k, ids, w, scale, y, (int32_t)(y_bf16 ? 1 : 0), s, err_word, rio,
                       static_cast<const __nv_bfloat16*>(A), map_b, map_w1);
}

}  // namespace

cudaError_t launch_lora_dense(const void* x, int64_t N, int32_t d_in, int32_t d_out, const void* A, const void* B,
                              int32_t K, int32_t r, const int32_t* ids, const float* w, int32_t k, float scale,
                              void* y, bool y_bf16, int32_t* err_word, cudaStream_t stream) {
  const RouterIo none = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  return launch_dense(x, N, d_in, d_out, A, B, K, r, ids, w, k, scale, y, y_bf16, err_word, nullptr, none, stream);
}

cudaError_t launch_router_lora_dense(const void* x, int64_t N, int32_t d_in, int32_t d_out, const void* W1,
                                     const float* b1, const void* W2, const float* b2, const void* A, const void* B,
                                     int32_t K, int32_t r, int32_t k, float scale, float* logits, int32_t* ids,
                                     float* w, void* y, bool y_bf16, int32_t* err_word, cudaStream_t stream) {
  const RouterIo rio = {static_cast<const __nv_bfloat16*>(W2), b1, b2, logits, ids, w};
  return launch_dense(x, N, d_in, d_out, A, B, K, r, nullptr, nullptr, k, scale, y, y_bf16, err_word, W1, rio,
                      stream);
}

}  // namespace molora
