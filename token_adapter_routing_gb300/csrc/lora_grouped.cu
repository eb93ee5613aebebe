// lora_grouped.cu -- the grouped tensor-core LoRA apply of "MoLoRA: Composable
// Specialization via Per-Token Adapter Routing" (Figure 2 right: tokens grouped by their
// selected adapter run as grouped GEMMs; Table 1: grouped GEMM dispatch shared by both
// routing modes; Figure 4: adapters at fixed addresses in a GPU-resident hot set).
//
// One fused kernel per call.  A work tile is TM (64 or 128) consecutive slots of one
// adapter's group (dispatch order), handled by a thread-block cluster of C CTAs:
//   0. before the tile is known, each CTA prefetches an equal share of the start of y into
//      L2 (DRAM is otherwise idle then); once its x rows have landed, each row prefetches
//      its y segment;
//   1. shrink, split over d_in: CTA c gathers its TM token rows x[tok, c*KS:(c+1)*KS)
//      with 16-byte cp.async (the gather is fused as an index list: no permuted copy of
//      x), TMA-loads A_a's matching K-slice, and accumulates h_c = x A_a (fp32) in TMEM
//      with tcgen05.mma (M = 128; with TM = 64 the other 64 rows are unused);
//   2. the C partial h_c are summed through distributed shared memory in a fixed order
//      (deterministic), scaled by scale * w(slot), and split into two bf16 terms
//      g = g_hi + g_lo (relative error 2^-17) to feed the next MMA;
//   3. expand, split over d_out: CTA c computes D = g B_a[:, c*NC:(c+1)*NC) into TMEM in
//      double-buffered passes of PW columns, B_a's columns TMA-loaded;
//   4. epilogue: D goes TMEM -> registers -> shared memory, then each row segment is added
//      into y[tok, cols] by one TMA bulk reduction in L2 (this un-permutes: scatter by
//      token).  With k = 1 every y element receives one addition; with k > 1 a token's k
//      slots live in different tiles and their additions may land in any order.
// The same kernel runs one masked per-sequence pass when given a fixed adapter (tiles are
// then consecutive tokens and the slot weight is the 0/1 mask), takes the adapters from a
// table of addresses instead of the slabs (indirect layout), and updates a bf16 y.
//
// Shapes small enough for two CTAs per SM (shared memory <= 113 KB, 256 TMEM columns) use
// 128-column passes; larger ones run one CTA per SM with 512 TMEM columns.  Either way the
// TMEM of all resident CTAs fits in the SM's 512 columns, so an allocation never waits on
// a CTA that is itself waiting at a cluster barrier.
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

constexpr int kTileM = 128;   // slots per tile = TMEM lanes = MMA M
constexpr int kKBlock = 64;   // K elements per 128-byte swizzle row (bf16)
constexpr int kEpilogueThreads = 128;
constexpr int kThreads = kEpilogueThreads + 32;  // + one producer/MMA warp
constexpr size_t kSmemPerSm = 228 * 1024;
constexpr size_t kSmemReservedPerCta = 1024;
constexpr size_t kMaxSmem = 227 * 1024;
constexpr size_t kCtrlBytes = 2048;
constexpr uint32_t kBarX = 1;  // named barrier: x round staged (warps 0-4)

struct GroupedPlan {
  int TM;            // valid rows per tile (64 or 128; the MMA always has M = 128)
  int C;             // cluster size: split of d_in and of d_out
  int KS;            // d_in / C: K-slice per CTA
  int NC;            // d_out / C: output columns per CTA
  int XR;            // x columns gathered per round
  int PW;            // expand pass width (TMEM columns per buffer)
  int piece;         // columns per bulk reduction
  uint32_t tmem_cols;
  uint32_t off_a;    // phase 1: A slice after the x round buffer
  uint32_t off_g;    // phase 2: g_hi (g_lo follows at +128*r*2 bytes)
  uint32_t off_b;    // phase 2: B column chunk
  uint32_t off_s;    // phase 2: epilogue staging
  uint32_t off_recv; // receive slots for partial h, [C sources][128/C rows][r] fp32
  uint32_t region;   // bytes before the control block (1024-aligned)
  int prefetch_y;    // send this CTA's y row segments to L2 once its x gather has landed
  uint64_t early_y;  // bytes at the start of y prefetched as contiguous shares before the tile is known
  uint32_t smem;     // dynamic shared memory requested
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool plan_layout(int32_t r, size_t g_tile, size_t budget, bool two_per_sm, GroupedPlan* s);

bool plan_one(int32_t d_in, int32_t d_out, int32_t r, int C, int TM, bool two_per_sm, GroupedPlan* s) {
  if (d_in % (C * kKBlock) || d_out % (C * 64)) return false;
  s->TM = TM;
  s->C = C;
  s->KS = d_in / C;
  s->NC = d_out / C;
  s->PW = two_per_sm ? 128 : 256;
  s->tmem_cols = two_per_sm ? 256 : 512;
  const size_t budget = two_per_sm ? kSmemPerSm / 2 - kSmemReservedPerCta : kMaxSmem;
  // g tiles are K-major with rows of r bf16 and the swizzle that matches that row width
  const size_t g_tile = (size_t)kTileM * r * 2;
  for (int piece : {128, 64}) {
#ifdef MOLORA_TUNING_ENV
    if (const char* e = getenv("MOLORA_PIECE"))
      if (piece != atoi(e)) continue;
#endif
    s->piece = piece;
    if (plan_layout(r, g_tile, budget, two_per_sm, s)) return true;
  }
  return false;
}

bool plan_layout(int32_t r, size_t g_tile, size_t budget, bool two_per_sm, GroupedPlan* s) {
  // phase 2 (after this CTA's shrink): g tiles, B chunk, epilogue staging.  g arrives from
  // the row owners only after every CTA of the cluster finished its shrink, so it may reuse
  // phase-1 space.  The receive slots for partial h get their own region: other CTAs may
  // push into them while this CTA's tensor core still reads its x tile.
  const size_t stage = (size_t)kTileM * (s->piece * 4 + 16);
  const size_t off_b = align_up(2 * g_tile, 1024);
  const size_t off_s = align_up(off_b + (size_t)s->NC * r * 2, 1024);
  const size_t phase2 = off_s + stage;
  const size_t recv = align_up((size_t)kTileM * r * 4, 1024);
  s->off_g = 0;
  s->off_b = (uint32_t)off_b;
  s->off_s = (uint32_t)off_s;
  int max_xr = 512;  // one round when the whole K-slice fits: fewer barrier round trips
#ifdef MOLORA_TUNING_ENV
  if (const char* e = getenv("MOLORA_XR")) max_xr = atoi(e);
#endif
  for (int XR = s->KS > max_xr ? max_xr : s->KS; XR >= kKBlock; XR -= kKBlock) {
    if (s->KS % XR) continue;
    const int nbuf = s->KS / XR > 1 ? 2 : 1;  // rounds alternate between two x buffers
    // x buffers hold TM rows; the M = 128 MMA over a 64-row buffer also reads the next 64 rows'
    // worth of shared memory (finite, unused), so at least 8 KB of this region follows the ring
    const size_t ring = (size_t)nbuf * XR * s->TM * 2;
    const size_t a_bytes = (size_t)s->KS * r * 2;
    const size_t over = s->TM < kTileM ? (size_t)(kTileM - s->TM) * 128 : 0;
    const size_t phase1 = ring + (a_bytes > over ? a_bytes : over);
    const size_t shared_region = align_up(phase1 > phase2 ? phase1 : phase2, 1024);
    size_t smem = shared_region + recv + 1024 /* base alignment slack */ + kCtrlBytes;
    if (!two_per_sm && smem < kSmemPerSm / 2) smem = kSmemPerSm / 2;  // keep it at one CTA per SM
    if (smem <= budget) {
      s->XR = XR;
      s->off_a = (uint32_t)ring;
      s->off_recv = (uint32_t)shared_region;
      s->region = (uint32_t)(shared_region + recv);
      s->smem = (uint32_t)smem;
      return true;
    }
  }
  return false;
}

// Picks cluster size, tile rows and CTAs per SM from what the host knows at launch: the slot
// count S and the number of groups K (so the mean group size S/K; the group sizes themselves
// are only on the device, and a launch captured in a CUDA graph must not depend on them).  A
// launch has ceil(S/TM) + K clusters (every group's last tile may be partial); the clusters of
// empty tiles leave at once, so the tiles that run are about ceil(S/TM) + K/2.  Measured on
// GB300 (decode sweep, d = 4096, r = 16, 256..2048 tokens, K = 8..64, uniform and Zipf(1.1);
// the 4-modality workload with uniform, 80/10/5/5 and 95/2/2/1 shares):
//   - 64-row tiles at two CTAs per SM win while their running tiles fit one wave (K = 8 at
//     2048 tokens: 22.7 vs 31.8 us for 128-row tiles); once they do not, 128-row tiles win if
//     the groups average at least 32 slots (K = 16 at 2048 tokens: 32.6 vs 36.8 us);
//   - with 64-row tiles, clusters of 4 beat clusters of 8 when all the clusters of 8 would
//     fill more than about 1.5 waves (K = 64 at 256..1024 tokens: 37.4 vs 42.3 us, 40.3 vs 43.9,
//     46.3 vs 47.0); clusters of 2 and 1 lose everywhere at this width.
//   - the skewed shares cost nothing: tiles follow the groups (20.6-20.9 us for all three).
// What the host cannot see costs at most this much: a Zipf draw over K = 32 at 2048 tokens
// prefers 64-row tiles (40.8 vs 46.7 us), a uniform draw over K = 64 at 2048 tokens clusters of
// 4 (52.6 vs 60.0 us).  Shapes that fit neither fall back through the list below.
bool choose(int32_t d_in, int32_t d_out, int32_t r, int64_t S, int32_t K, GroupedPlan* s) {
  int only_c = 0, only_one = 0, only_tm = 0;
#ifdef MOLORA_TUNING_ENV
  if (const char* e = getenv("MOLORA_CLUSTER")) only_c = atoi(e);
  if (const char* e = getenv("MOLORA_ONE_PER_SM")) only_one = atoi(e);
  if (const char* e = getenv("MOLORA_TILE_ROWS")) only_tm = atoi(e);
#endif
  struct Cand { int C, TM; bool two; };
  const int64_t sms = num_sms();
  const int64_t tiles64 = (S + 63) / 64;
  const int64_t running64 = tiles64 + (K + 1) / 2;  // 64-row tiles that run (empty ones leave)
  int pref_tm = (running64 * 8 > 2 * sms && 2 * tiles64 >= K) ? 128 : 64;
  GroupedPlan probe;
  if (!plan_one(d_in, d_out, r, 8, 64, true, &probe) && plan_one(d_in, d_out, r, 8, 64, false, &probe)) {
    // One CTA per SM (rank 64 at d = 4096: the B slice, staging and receive slots take an SM's
    // shared memory).  Then about sms / 9 clusters of 8 are resident at once (two per GPC of
    // 18-20 SMs), and the time steps with the waves of launched clusters: take the tile rows
    // with fewer waves, 64 rows on a tie.  Measured, rank 64, K = 4..32, 512..4096 tokens, 64
    // vs 128 rows forced: this choice loses 31 us summed over 36 points, the two-per-SM rule
    // above 103 us (e.g. 4 adapters, 1536 tokens: 25.8 us with 128 rows, 36.7 with 64).
    const int64_t wave = sms / 9 > 0 ? sms / 9 : 1;
    const int64_t w64 = (tiles64 + K + wave - 1) / wave;
    const int64_t w128 = ((S + 127) / 128 + K + wave - 1) / wave;
    pref_tm = w128 < w64 ? 128 : 64;
  }
  // (clusters of 4 measured with 64-row tiles only; large groups keep clusters of 8)
  const int pref_c = (pref_tm == 64 && (tiles64 + K) * 8 > 3 * sms) ? 4 : 8;
  const Cand preferred[] = {{pref_c, pref_tm, true}, {pref_c, pref_tm, false}};
  static const Cand order[] = {{8, 128, true}, {8, 128, false}, {4, 128, true}, {4, 128, false},
                               {2, 128, true}, {2, 128, false}, {1, 128, true}, {1, 128, false},
                               {8, 64, true}, {4, 64, true}, {4, 64, false}, {8, 64, false},
                               {2, 64, true}, {2, 64, false}, {1, 64, true}, {1, 64, false}};
  auto allowed = [&](const Cand& c) {
    return !((only_c && c.C != only_c) || (only_one && c.two) || (only_tm && c.TM != only_tm));
  };
  for (const Cand& c : preferred)
    if (allowed(c) && plan_one(d_in, d_out, r, c.C, c.TM, c.two, s)) return true;
  for (const Cand& c : order)
    if (allowed(c) && plan_one(d_in, d_out, r, c.C, c.TM, c.two, s)) return true;
  return false;
}

struct TileInfo {
  int32_t adapter;  // -1: idle cluster
  int32_t row0;     // first row of the tile inside the adapter's group (or first token)
  int32_t nvalid;   // valid rows in the tile
  int32_t group_off;
};

struct __align__(8) Ctrl {
  uint64_t bar_a;         // TMA of the A slice
  uint64_t bar_b;         // TMA of the B chunk
  uint64_t bar_x[2];      // shrink MMAs reading x buffer b done (one phase per use of the buffer)
  uint64_t bar_full[2];   // expand pass done, per TMEM buffer
  uint64_t bar_empty[2];  // epilogue drained a TMEM buffer
  uint64_t bar_recv;      // partial-h rows this CTA owns have arrived from every CTA
  uint64_t bar_g;         // all TM rows of g (hi and lo) have arrived from their owners
  uint64_t bar_perm;      // the dispatch permutation, copied whole into the x buffers
  uint32_t tmem_base;
  int32_t abort;
  TileInfo tile;
  int32_t tok[kTileM];    // token of each tile row, -1 for padding (drives the gather)
  int32_t live[kTileM];   // row passed validation and gets a reduction
  float wgt[kTileM];      // weight of each tile row (0 for padding or invalid)
  int32_t offs[kMaxAdapters + 1];  // the dispatch offsets, loaded once by K+1 threads at a time
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

__device__ __forceinline__ SmemLayout sw_for_rank(int r) {
  return r == 16 ? kSwizzle32B : (r == 32 ? kSwizzle64B : kSwizzle128B);
}

}  // namespace

// At most 168 registers: two CTAs (10 warps) must fit the 16K registers of an SM partition.
// kYBf16: y is bf16 (a separate instantiation, so the fp32 epilogue carries no bf16 branch).
template <bool kYBf16>
__global__ void __maxnreg__(168)
    lora_grouped_kernel(const __nv_bfloat16* __restrict__ x, int64_t N, int32_t d_in, int32_t d_out, int32_t K,
                        int32_t r, int32_t k, const int32_t* __restrict__ ids, const float* __restrict__ w,
                        const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm, float scale,
                        void* __restrict__ y, int32_t mask_adapter, const GroupedPlan P,
                        int32_t* err_word, const __grid_constant__ CUtensorMap map_a,
                        const __grid_constant__ CUtensorMap map_b, int32_t indirect,
                        const __grid_constant__ AdapterTable table) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(sm + P.region);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = P.C, KS = P.KS, NC = P.NC, TM = P.TM;
  uint8_t* const yb = static_cast<uint8_t*>(y);
  constexpr uint32_t ysz = kYBf16 ? 2u : 4u;  // bytes per y element: fp32, or bf16
  const int crank = (int)cluster_ctarank();
  const int cluster_id = blockIdx.x / C;
  const int64_t S = N * (int64_t)k;

  // ---- prologue that reads nothing the previous kernel writes: overlaps it under PDL
  if (warp == 4) {
    tmem_alloc(&ctrl->tmem_base, P.tmem_cols);
    tmem_relinquish();
    if (lane == 0) {
      // indirect layout: the 32 lanes of this warp load A and B with cp.async, one arrival each
      mbar_init(&ctrl->bar_a, indirect ? 32 : 1);
      mbar_init(&ctrl->bar_b, indirect ? 32 : 1);
      mbar_init(&ctrl->bar_x[0], 1);
      mbar_init(&ctrl->bar_x[1], 1);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&ctrl->bar_full[i], 1);
        mbar_init(&ctrl->bar_empty[i], kEpilogueThreads);
      }
      mbar_init(&ctrl->bar_recv, 1);
      mbar_init(&ctrl->bar_g, 1);
      mbar_init(&ctrl->bar_perm, 1);
      mbar_fence_init();
      // both receive the tile's TM rows x r values: fp32 partials, and g as two bf16 halves
      mbar_arrive_expect_tx(&ctrl->bar_recv, (uint32_t)P.TM * r * 4u);
      mbar_arrive_expect_tx(&ctrl->bar_g, (uint32_t)P.TM * r * 4u);
      if (!indirect) {
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
      }
    }
  }
  if (P.early_y > 0 && warp == 0) {
    // The first P.early_y bytes of y, an equal contiguous share per CTA, in 32 KB pieces.
    // Nothing here depends on the previous kernel (a prefetch only moves lines into L2), and
    // DRAM is otherwise idle until the tile's rows are known and the x gather starts.
    const uint64_t total = P.early_y;
    const uint64_t share = ((total + gridDim.x - 1) / gridDim.x + 15) & ~uint64_t(15);
    const uint64_t begin = (uint64_t)blockIdx.x * share;
    const uint64_t end = begin + share < total ? begin + share : total;
    for (uint64_t off = begin + (uint64_t)lane * 32768u; off < end; off += 32u * 32768u) {
      const uint64_t len = end - off < 32768u ? end - off : 32768u;
      prefetch_l2_bulk(reinterpret_cast<const uint8_t*>(y) + off, (uint32_t)(len & ~uint64_t(15)));
    }
  }
  pdl_wait();
  pdl_launch_dependents();
  // The whole permutation (S slots) is copied into the x buffers, which stay idle until the
  // gather, in parallel with the offsets: the tile's tokens then come from shared memory
  // instead of a second dependent global load after the tile is decoded.
  const int rounds = KS / P.XR;
  const int nbuf = rounds > 1 ? 2 : 1;
  const size_t blk_bytes = (size_t)TM * 128;          // one 64-column K-block of a buffer
  const size_t buf_bytes = (size_t)(P.XR / kKBlock) * blk_bytes;
  const bool perm_smem = mask_adapter < 0 && S > 0 && (S & 3) == 0 && S * 4 <= (int64_t)(nbuf * buf_bytes) &&
                         (reinterpret_cast<uintptr_t>(perm) & 15) == 0;
  if (perm_smem && warp == 4 && lane == 0) {
    mbar_arrive_expect_tx(&ctrl->bar_perm, (uint32_t)(S * 4));
    bulk_load_g2s(smem_u32(sm), perm, (uint32_t)(S * 4), &ctrl->bar_perm);
  }

  // ---- which tile this cluster owns (identical in every CTA of the cluster)
  if (mask_adapter < 0)
    for (int i = tid; i <= K; i += kThreads) ctrl->offs[i] = offsets[i];
  __syncthreads();
  if (tid == 0) {
    TileInfo ti{-1, 0, 0, 0};
    if (mask_adapter >= 0) {
      const int64_t t0 = (int64_t)cluster_id * TM;
      if (t0 < N) ti = TileInfo{mask_adapter, (int32_t)t0, (int32_t)(N - t0 < TM ? N - t0 : TM), 0};
    } else {
      int32_t cum = 0;
      int32_t prev = ctrl->offs[0];
      bool bad = prev != 0;
      for (int a = 0; a < K && ti.adapter < 0 && !bad; ++a) {
        const int32_t nxt = ctrl->offs[a + 1];
        if (nxt < prev || nxt > S) {
          bad = true;
          break;
        }
        const int32_t n_a = nxt - prev;
        const int32_t tiles = (n_a + TM - 1) / TM;
        if (cluster_id < cum + tiles) {
          const int32_t row0 = (cluster_id - cum) * TM;
          ti = TileInfo{a, row0, min(TM, n_a - row0), prev};
        }
        cum += tiles;
        prev = nxt;
      }
      if (bad) {
        if (crank == 0 && cluster_id == 0) report(err_word, MOLORA_DEV_BAD_PERMUTATION);
        ti.adapter = -1;
      }
    }
    ctrl->tile = ti;
    ctrl->abort = 0;
  }
  __syncthreads();
  const TileInfo tile = ctrl->tile;
  if (tile.adapter < 0) {  // the whole cluster idles: every CTA computed the same tile
    // the permutation copy must land before the CTA leaves
    if (perm_smem && warp == 4 && lane == 0) mbar_wait(&ctrl->bar_perm, 0);
    if (warp == 4) {
      tc_fence_after();
      tmem_dealloc(ctrl->tmem_base, P.tmem_cols);
    }
    return;
  }
  const int a = tile.adapter;

  uint8_t* xs = sm;              // phase 1: two x round buffers, XR/64 blocks of [TM rows x 128 B], 128B swizzle
  uint8_t* as = sm + P.off_a;    // phase 1: A slice [KS x r], MN-major, swizzled by TMA
  uint8_t* g_hi = sm + P.off_g;  // phase 2: g as two bf16 K-major tiles, rows of r elements
  uint8_t* g_lo = g_hi + (size_t)kTileM * r * 2;
  const uint32_t g_row_bytes = (uint32_t)r * 2u;
  uint8_t* bs = sm + P.off_b;    // phase 2: B chunk, NC/64 boxes of [r rows x 128 B]
  uint8_t* stage = sm + P.off_s;
  const uint32_t stage_stride = (uint32_t)P.piece * 4u + 16u;

  int32_t slot = -1;
  if (warp < 4) {
    const int row = tid;
    int32_t tok = -1;
    if (row < tile.nvalid) {
      if (mask_adapter >= 0) {
        tok = tile.row0 + row;
      } else if (perm_smem) {
        if (!mbar_wait(&ctrl->bar_perm, 0)) report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
        slot = reinterpret_cast<const volatile int32_t*>(sm)[tile.group_off + tile.row0 + row];
        if (slot >= 0 && slot < S) tok = slot / k;
      } else {
        slot = perm[tile.group_off + tile.row0 + row];
        if (slot >= 0 && slot < S) tok = slot / k;
      }
    }
    ctrl->tok[row] = tok;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  __syncwarp();
  cluster_arrive();  // barriers of every CTA initialised and armed (waited on before the first remote store)

  // ---- shrink: rounds of XR columns, each gathered, then consumed by XR/16 MMAs.  Rounds
  // alternate between two x buffers: round rd+1 is in flight while round rd is multiplied.
  const uint32_t idesc_shrink = idesc_bf16_f32(kTileM, r, false, true);
  if (warp == 4) {
    if (indirect) {
      // the same bytes the TMA box would write: rows of r elements, swizzled to match r
      const __nv_bfloat16* Aa = static_cast<const __nv_bfloat16*>(table.a[a]) + (int64_t)crank * KS * r;
      const int cpr = r / 8;  // 16-byte chunks per row
      for (int i = lane; i < KS * cpr; i += 32) {
        const int row = i / cpr, chunk = i % cpr;
        cp_async_16(smem_u32(as) + (uint32_t)((row / kKBlock) * kKBlock * r * 2) +
                        swz_offset(row % kKBlock, chunk, (uint32_t)r * 2u),
                    Aa + (int64_t)row * r + chunk * 8, 16u);
      }
      cp_async_mbar_arrive(&ctrl->bar_a);
    } else if (lane == 0) {
      mbar_arrive_expect_tx(&ctrl->bar_a, (uint32_t)KS * r * 2);
      for (int kb = 0; kb < KS / kKBlock; ++kb)
        tma_load_2d(smem_u32(as + (size_t)kb * kKBlock * r * 2), &map_a, 0, a * d_in + crank * KS + kb * kKBlock,
                    &ctrl->bar_a);
    }
  }
  // lanes 8q..8q+7 copy the eight 16-byte chunks of one 128-byte row segment
  // x is read once: its lines go first, so that the prefetched y lines stay for the reductions
  // (measured: 19.30 -> 18.76 us on the 4-modality apply; the same hint on the y reductions
  // changed nothing)
  const uint64_t x_policy = l2_policy_evict_first();
  auto gather = [&](int rd) {
    uint8_t* xb = xs + (rd % nbuf) * buf_bytes;
    const int sub = lane >> 3, chunk = lane & 7;
    for (int kb = 0; kb < P.XR / kKBlock; ++kb) {
      const uint32_t blk = smem_u32(xb + (size_t)kb * blk_bytes);
      const int col = crank * KS + rd * P.XR + kb * kKBlock + chunk * 8;
#pragma unroll 4
      for (int it = 0; it < TM / 16; ++it) {
        const int row = it * 16 + warp * 4 + sub;
        const int32_t tok = ctrl->tok[row];
        const __nv_bfloat16* src = tok >= 0 ? x + (int64_t)tok * d_in + col : x;
        cp_async_16_hint(blk + sw128_offset(row, chunk), src, tok >= 0 ? 16u : 0u, x_policy);
      }
    }
    cp_async_commit();
  };
  // checks this row's slot against the tile's adapter and records its weight; its loads go
  // out once the x rounds are in flight, so their latency hides behind the gather
  auto validate = [&]() {
    const int row = tid;
    int32_t live = 0;
    float wt = 0.f;
    const int32_t tok = ctrl->tok[row];
    if (tok >= 0) {
      if (mask_adapter >= 0) {
        live = 1;
        wt = ids[tok] == mask_adapter ? 1.f : 0.f;
      } else if (ids[slot] == a) {
        live = 1;
        wt = w ? w[slot] : 1.f;
      } else if (crank == 0) {
        report(err_word, MOLORA_DEV_BAD_PERMUTATION);
      }
    } else if (row < tile.nvalid && crank == 0) {
      report(err_word, MOLORA_DEV_BAD_PERMUTATION);
    }
    ctrl->live[row] = live;
    ctrl->wgt[row] = wt;
  };
  if (warp < 4) {
    gather(0);
    if (rounds == 1) validate();
  }
  for (int rd = 0; rd < rounds; ++rd) {
    if (warp < 4) {
      if (rd + 1 < rounds) {
        const int nb = (rd + 1) % nbuf;
        // buffer nb was last read by the MMAs of round rd-1 (its ((rd-1)/2)-th use)
        if (rd >= 1 && !mbar_wait(&ctrl->bar_x[nb], ((rd - 1) >> 1) & 1)) {
          ctrl->abort = 1;
          report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
        }
        gather(rd + 1);
        if (rd == 0) validate();
        cp_async_wait_group<1>();  // round rd has landed; round rd+1 stays in flight
      } else {
        cp_async_wait_all();
      }
      fence_proxy_async_smem();
    }
    __syncwarp();
    named_barrier(kBarX, kThreads);  // round rd is in shared memory
    if (warp == 4 && lane == 0) {
      bool ok = !ctrl->abort;
      if (ok && rd == 0) {
        ok = mbar_wait(&ctrl->bar_a, 0);
        fence_proxy_async_smem();  // A written by cp.async (indirect layout) is read by the MMA
      }
      tc_fence_after();
      uint64_t* done = &ctrl->bar_x[rd % nbuf];
      if (ok) {
        const uint32_t atom = 8u * r * 2u;
        const SmemLayout swz = sw_for_rank(r);
        const uint8_t* xb = xs + (rd % nbuf) * buf_bytes;
        for (int kb = 0; kb < P.XR / kKBlock; ++kb)
          for (int ks = 0; ks < kKBlock / 16; ++ks) {
            const int krow = rd * P.XR + kb * kKBlock + ks * 16;
            // 128 MMA rows from here: the tile's TM rows, then (TM = 64) 64 unused rows
            const uint64_t da = smem_desc(smem_u32(xb + (size_t)kb * blk_bytes + ks * 32), 16, 1024, kSwizzle128B);
            const uint64_t db = smem_desc(smem_u32(as + (size_t)krow * r * 2), atom, atom, swz);
            umma_f16(tmem, da, db, idesc_shrink, (rd | kb | ks) != 0);
          }
        umma_commit(done);
      } else {
        ctrl->abort = 1;
        report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
        mbar_arrive(done);
      }
    }
  }
  // the last round's commit covers every shrink MMA issued before it
  uint64_t* const last_bar = &ctrl->bar_x[(rounds - 1) % nbuf];
  const uint32_t last_parity = (uint32_t)((rounds - 1) / nbuf) & 1u;
  if (warp == 4 && (indirect || lane == 0)) {
    // B chunk lands in the phase-1 region once the last shrink MMAs have read it
    if (mbar_wait(last_bar, last_parity)) {
      if (indirect) {
        // boxes of r rows x 64 columns, 128-byte rows swizzled, as the TMA would write them
        const __nv_bfloat16* Ba = static_cast<const __nv_bfloat16*>(table.b[a]) + (int64_t)crank * NC;
        for (int i = lane; i < r * (NC / 8); i += 32) {
          const int row = i / (NC / 8), c8 = i % (NC / 8);  // c8: 16-byte chunk along the columns
          cp_async_16(smem_u32(bs) + (uint32_t)((c8 / 8) * r * 128) + sw128_offset(row, c8 % 8),
                      Ba + (int64_t)row * d_out + c8 * 8, 16u);
        }
        cp_async_mbar_arrive(&ctrl->bar_b);
      } else {
        mbar_arrive_expect_tx(&ctrl->bar_b, (uint32_t)NC * r * 2);
        for (int q = 0; q < NC / 64; ++q)
          tma_load_2d(smem_u32(bs + (size_t)q * r * 128), &map_b, crank * NC + q * 64, a * r, &ctrl->bar_b);
      }
    } else {
      ctrl->abort = 1;
      report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
      mbar_arrive(&ctrl->bar_b);
    }
  }
  // ---- cluster reduction of h, pushed rather than pulled: CTA c owns tile rows
  // [c*RPC, (c+1)*RPC).  Every CTA sends each row's partial h to the row's owner
  // (st.async into the owner's receive slots, counted by its bar_recv); the owner sums the
  // C partials in rank order (deterministic), forms g = scale * w * h, splits it into bf16
  // hi + lo, and sends both rows to every CTA's g tiles (counted by their bar_g).
  const int RPC = TM / C;  // only the tile's TM rows travel; MMA rows past them stay local
  float* recv = reinterpret_cast<float*>(sm + P.off_recv);  // [C sources][RPC rows][r]
  bool have_h = true;
  if (warp < 4) {
    // x has landed and only the last shrink MMAs are running: start pulling this row's y
    // segment into L2, so the reductions of the expand find it there.  Earlier, the prefetch
    // competed with the x gather and slowed it more than it helped.
    if (P.prefetch_y && ctrl->tok[tid] >= 0)
      prefetch_l2_bulk(yb + ((int64_t)ctrl->tok[tid] * d_out + crank * NC) * ysz, (uint32_t)NC * ysz);
    have_h = mbar_wait(last_bar, last_parity);
    tc_fence_after();
    if (!have_h) {
      ctrl->abort = 1;
      report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
    }
  }
  __syncwarp();
  cluster_wait();  // every CTA's barriers are armed
  if (warp < 4) {
    const int row = tid;
    if (warp * 32 < TM) {  // whole warps: TM is 64 or 128
      const uint32_t owner = (uint32_t)(row / RPC);
      const uint32_t dst = dsmem_addr(smem_u32(recv + ((size_t)crank * RPC + (row % RPC)) * r), owner);
      const uint32_t dst_bar = dsmem_addr(smem_u32(&ctrl->bar_recv), owner);
      float v[16];
      for (int c0 = 0; c0 < r; c0 += 16) {
        if (have_h)
          tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
        else
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          st_async_v4(dst + (c0 + 4 * i) * 4,
                      make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                                 __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3])),
                      dst_bar);
      }
    }
    tc_fence_before();
    // owner: reduce its rows once every source has delivered them
    const bool got = mbar_wait(&ctrl->bar_recv, 0);
    if (!got) {
      ctrl->abort = 1;
      report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
    }
    const int groups = r / 8;
    for (int item = tid; item < RPC * groups; item += kEpilogueThreads) {
      const int rl = item / groups, c0 = (item % groups) * 8;
      const int trow = crank * RPC + rl;
      float h[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int cc = 0; cc < C; ++cc) {
        const float4* src = reinterpret_cast<const float4*>(recv + ((size_t)cc * RPC + rl) * r + c0);
        const float4 p0 = src[0], p1 = src[1];
        h[0] += p0.x, h[1] += p0.y, h[2] += p0.z, h[3] += p0.w;
        h[4] += p1.x, h[5] += p1.y, h[6] += p1.z, h[7] += p1.w;
      }
      const float coef = scale * ctrl->wgt[trow];
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
      const uint32_t off = swz_offset(trow, c0 / 8, g_row_bytes);
      const uint4 vh = make_uint4(hi[0], hi[1], hi[2], hi[3]), vl = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      for (int d = 0; d < C; ++d) {
        const uint32_t bar_d = dsmem_addr(smem_u32(&ctrl->bar_g), (uint32_t)d);
        st_async_v4(dsmem_addr(smem_u32(g_hi + off), (uint32_t)d), vh, bar_d);
        st_async_v4(dsmem_addr(smem_u32(g_lo + off), (uint32_t)d), vl, bar_d);
      }
    }
  }
  __syncwarp();

  const int npass = (NC + P.PW - 1) / P.PW;
  if (warp == 4) {
    if (lane == 0) {
      bool ok = !ctrl->abort && mbar_wait(&ctrl->bar_b, 0) && mbar_wait(&ctrl->bar_g, 0);
      fence_proxy_async_smem();
      tc_fence_after();
      for (int p = 0; p < npass; ++p) {
        const int buf = p & 1;
        const int width = min(P.PW, NC - p * P.PW);
        if (p >= 2 && ok) ok = mbar_wait(&ctrl->bar_empty[buf], ((p >> 1) - 1) & 1);
        if (!ok) {
          ctrl->abort = 1;
          report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
          mbar_arrive(&ctrl->bar_full[buf]);
          continue;
        }
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(kTileM, width, false, true);
        const uint32_t d = tmem + buf * P.PW;
        for (int ks = 0; ks < r / 16; ++ks) {
          const uint64_t db = smem_desc(smem_u32(bs + (size_t)(p * (P.PW / 64)) * r * 128 + ks * 2048), r * 128,
                                        1024, kSwizzle128B);
          const SmemLayout gl = sw_for_rank(r);
          umma_f16(d, smem_desc(smem_u32(g_hi + ks * 32), 16, 8 * g_row_bytes, gl), db, idesc, ks != 0);
          umma_f16(d, smem_desc(smem_u32(g_lo + ks * 32), 16, 8 * g_row_bytes, gl), db, idesc, 1);
        }
        umma_commit(&ctrl->bar_full[buf]);
      }
    }
    __syncwarp();
  } else {
    // Each thread drains its own TMEM lane (tile row) into its staging row, then hands the
    // row segment to the TMA unit as one bulk fp32 add into y.
    const int row = tid;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float* srow = reinterpret_cast<float*>(stage + row * stage_stride);
    const int32_t my_tok = ctrl->live[row] ? ctrl->tok[row] : -1;
    for (int p = 0; p < npass; ++p) {
      const int buf = p & 1;
      const int width = min(P.PW, NC - p * P.PW);
      const bool ok = mbar_wait(&ctrl->bar_full[buf], (p >> 1) & 1);
      tc_fence_after();
      if (!ok) report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
      // warps whose rows all lie past the tile (TM = 64) have nothing to drain
      for (int q = 0; ok && !ctrl->abort && warp * 32 < TM && q < width; q += P.piece) {
        const int cols = min(P.piece, width - q);
        bulk_wait_read<0>();  // the previous reduction has read the stage
        for (int c0 = 0; c0 < cols; c0 += 32) {
          float v[32];
          tmem_ld32(lane_base + buf * P.PW + q + c0, v);
          if (my_tok >= 0) {
            if (kYBf16) {
              // round each contribution to bf16 (nearest even); the bulk add rounds the sum
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
        // one bulk reduction per row segment, performed by the TMA unit in L2
        fence_proxy_async_smem();
        if (my_tok >= 0) {
          void* dst = yb + ((int64_t)my_tok * d_out + crank * NC + p * P.PW + q) * ysz;
          if (kYBf16)
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
    tmem_dealloc(tmem, P.tmem_cols);
  }
}

// ---------------------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

// 2-D bf16 tensor map over a row-major [rows x cols] array.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows,
              CUtensorMapSwizzle swz) {
  auto enc = encoder();
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

bool grouped_supported(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r, int32_t k) {
  if (dtype != MOLORA_BF16 || !(r == 16 || r == 32 || r == 64)) return false;
  GroupedPlan s;
  return choose(d_in, d_out, r, N * (int64_t)k, K, &s) && encoder() != nullptr;
}

cudaError_t launch_lora_grouped(const void* x, int64_t N, int32_t d_in, int32_t d_out, const void* A, const void* B,
                                int32_t K, int32_t r, const int32_t* ids, const float* w, int32_t k,
                                const int32_t* counts, const int32_t* offsets, const int32_t* perm, float scale,
                                void* y, bool y_bf16, int32_t mask_adapter, int32_t* err_word,
                                cudaStream_t stream, const AdapterTable* table) {
  (void)counts;
  GroupedPlan s;
  if (!choose(d_in, d_out, r, mask_adapter >= 0 ? N : N * (int64_t)k, mask_adapter >= 0 ? 1 : K, &s))
    return cudaErrorNotSupported;
  s.prefetch_y = 1;
  // DRAM idles for about 2 us while the tile is decoded; prefetching 45% of y (at most
  // 24 MiB) fills that window and measured best on GB300 (4-modality workload, back-to-back
  // steps, x gathered evict-first: 20, 30, 40, 50, 60, 80 and 100% tried, 40-50% best).  The
  // rest of y follows per row, late.
  const uint64_t y_bytes = (uint64_t)N * d_out * (y_bf16 ? 2u : 4u);
  const uint64_t early = y_bytes * 9u / 20u;
  s.early_y = (early < (24ull << 20) ? early : (24ull << 20)) & ~uint64_t(15);
#ifdef MOLORA_TUNING_ENV
  if (const char* e = getenv("MOLORA_PREFETCH_Y")) s.prefetch_y = atoi(e);
  if (const char* e = getenv("MOLORA_EARLY_Y")) {
    const int pct = atoi(e) < 0 ? 0 : (atoi(e) > 100 ? 100 : atoi(e));
    s.early_y = (y_bytes * (uint64_t)pct / 100u) & ~uint64_t(15);
  }
#endif
  CUtensorMap map_a, map_b;
  AdapterTable tab;
  memset(&tab, 0, sizeof(tab));
  if (table) {
    // indirect layout: the kernel reads the adapters through the table; the maps stay unused
    memset(&map_a, 0, sizeof(map_a));
    memset(&map_b, 0, sizeof(map_b));
    tab = *table;
  } else {
    const CUtensorMapSwizzle swa =
        r == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : (r == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
    if (!make_map(&map_a, A, (uint64_t)K * d_in, (uint64_t)r, (uint32_t)r, kKBlock, swa)) return cudaErrorInvalidValue;
    if (!make_map(&map_b, B, (uint64_t)K * r, (uint64_t)d_out, 64, (uint32_t)r, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(lora_grouped_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kMaxSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(lora_grouped_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kMaxSmem);
    if (attr_err != cudaSuccess) cudaGetLastError();
  });
  if (attr_err != cudaSuccess) return attr_err;

  const int64_t tiles = mask_adapter >= 0 ? (N + s.TM - 1) / s.TM : (N * k + s.TM - 1) / s.TM + K;
  return launch_kernel(y_bf16 ? lora_grouped_kernel<true> : lora_grouped_kernel<false>, dim3((unsigned)(tiles * s.C)),
                       dim3(kThreads), s.smem, stream, s.C, static_cast<const __nv_bfloat16*>(x), N, d_in, d_out, K, r,
                       k, ids, w, offsets, perm, scale, y, mask_adapter, s, err_word, map_a, map_b,
                       (int32_t)(table ? 1 : 0), tab);
}

}  // namespace molora
