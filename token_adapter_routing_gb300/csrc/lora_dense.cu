// lora_dense.cu -- the top-k LoRA apply of "MoLoRA: Composable Specialization via
// Per-Token Adapter Routing" computed token-major over the whole hot set (Figure 2: a
// token's output is the weighted sum over its top-k adapters; Table 10's shapes):
//
//   y[t,:] += scale * sum_a c[t,a] (x[t,:] A_a) B_a,   c[t,a] = sum_j [ids[t,j] == a] w[t,j]
//
// which is the pages' sum written over all K adapters, with weight zero for the ones a
// token did not select.  When K*r is small (the hot set's ranks stacked: at most 128
// columns) this evaluates every adapter for every token on the tensor cores instead of
// grouping slots by adapter, and in exchange reads each token's x row once and adds into
// each y row once, whatever k is -- the grouped path reads x and reduces into y once per
// slot, k times per token.  No dispatch is needed.
//
// A tile is 64 consecutive tokens, handled by a cluster of C CTAs:
//   1. shrink, split over d_in: CTA c gathers x[t0:t0+64, c*KS:(c+1)*KS) with 16-byte
//      cp.async, TMA-loads the K-slices of all K adapters' A, and accumulates
//      H = x [A_0 | ... | A_{K-1}] (K*r columns, fp32) in TMEM, one tcgen05.mma per adapter
//      and 16-element K step (M = 128: rows past 64 are unused);
//   2. the C partial H are summed through distributed shared memory in rank order
//      (deterministic), each adapter's r columns are scaled by scale * c[t,a], and the
//      result G is split into bf16 hi + lo and sent to every CTA of the cluster;
//   3. expand, split over d_out: D = G [B_0; ...; B_{K-1}] -- the B slab seen as
//      [K*r x d_out] is exactly the stacked operand -- in double-buffered passes of 128
//      columns whose B tiles stream in by TMA, two buffers deep;
//   4. epilogue: D goes TMEM -> registers -> shared memory -> one bulk fp32 (or bf16) add
//      per row segment into y, performed by the TMA unit in L2.  Every y element receives
//      one addition, so results are reproducible for any k.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

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
  int C, KS, NC, KR;       // cluster size, K-slice, output columns per CTA, K*r
  uint32_t off_a;          // phase 1: all adapters' A slices after the x tile
  uint32_t off_g, off_b;   // phase 2: G hi/lo tiles, two B pass buffers
  uint32_t off_s;          // epilogue staging (also the receive slots, used earlier)
  uint32_t region, smem;
  uint32_t g_blk;          // bytes of one 64-column block of a G tile (128 rows x 128 B)
  uint32_t b_pass;         // bytes of one B pass buffer
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Shared memory: phase 1 holds the x tile [KS/64 blocks][64 rows][128 B] (plus room for the
// M = 128 MMA to read 64 rows past its last block) and the adapters' A slices.  Phase 2
// (after the shrink) reuses it for the G tiles and the B pass buffers.  The staging lines
// of the epilogue come after both; the receive slots of the cluster reduction share them,
// because remote CTAs may push their partials while this CTA's MMAs still read phase 1,
// and the epilogue starts only after every partial has been consumed.
bool dense_plan(int32_t d_in, int32_t d_out, int32_t K, int32_t r, int C, size_t budget, DensePlan* s) {
  if (d_in % (C * kKBlock) || d_out % (C * kKBlock)) return false;
  s->C = C;
  s->KS = d_in / C;
  s->NC = d_out / C;
  s->KR = K * r;
  if (s->KS > 512) return false;  // one gather round
  const size_t x_bytes = (size_t)(s->KS / kKBlock) * kTileRows * 128;
  const size_t a_bytes = (size_t)K * s->KS * r * 2;
  const size_t over = (size_t)(kMmaM - kTileRows) * 128;
  const size_t phase1 = x_bytes + (a_bytes > over ? a_bytes : over);
  const int kblocks = (s->KR + 63) / 64;  // 64-column blocks of a G tile (KR >= 64), else one narrow tile
  s->g_blk = (uint32_t)(kMmaM * (s->KR >= 64 ? 128 : s->KR * 2));
  const size_t g_bytes = 2 * (size_t)kblocks * s->g_blk;
  s->b_pass = (uint32_t)((kPassW / 64) * s->KR * 128);
  const size_t phase2 = align_up(g_bytes, 1024) + 2 * (size_t)s->b_pass;
  const size_t stage = (size_t)kTileRows * (kPiece * 4 + 16);
  const size_t recv = (size_t)kTileRows * s->KR * 4;
  s->off_a = (uint32_t)x_bytes;
  s->off_g = 0;
  s->off_b = (uint32_t)align_up(g_bytes, 1024);
  s->off_s = (uint32_t)align_up(phase1 > phase2 ? phase1 : phase2, 1024);
  s->region = (uint32_t)align_up(s->off_s + (stage > recv ? stage : recv), 1024);
  s->smem = s->region + (uint32_t)kCtrlBytes + 1024;
  return s->smem <= budget;
}

bool dense_choose(int32_t d_in, int32_t d_out, int32_t K, int32_t r, DensePlan* s) {
  // K*r = 256 would need 128 KB of G tiles alone (hi and lo, M = 128 rows): it never fits
  if (!(r == 16 || r == 32 || r == 64) || K * r > 128 || (K * r) % 16) return false;
  for (size_t budget : {kTwoPerSm, kMaxSmem})
    for (int C : {8, 4, 2, 1})
      if (dense_plan(d_in, d_out, K, r, C, budget, s)) return true;
  return false;
}

struct __align__(8) DCtrl {
  uint64_t bar_a;        // TMA of all adapters' A slices
  uint64_t bar_x;        // shrink MMAs done
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

__global__ void __launch_bounds__(kThreads, 1)
    lora_dense_kernel(const __nv_bfloat16* __restrict__ x, int64_t N, int32_t d_in, int32_t d_out, int32_t K,
                      int32_t r, int32_t k, const int32_t* __restrict__ ids, const float* __restrict__ w,
                      float scale, void* __restrict__ y, int32_t y_bf16, const DensePlan P, int32_t* err_word,
                      const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DCtrl* ctrl = reinterpret_cast<DCtrl*>(sm + P.region);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = P.C, KS = P.KS, NC = P.NC, KR = P.KR;
  const int crank = (int)cluster_ctarank();
  const int64_t t0 = (int64_t)(blockIdx.x / C) * kTileRows;
  const int nvalid = (int)(N - t0 < kTileRows ? N - t0 : kTileRows);
  uint8_t* const yb = static_cast<uint8_t*>(y);
  const uint32_t ysz = y_bf16 ? 2u : 4u;

  uint8_t* xs = sm;
  uint8_t* as = sm + P.off_a;
  uint8_t* g_hi = sm + P.off_g;
  const int gblocks = (KR + 63) / 64;
  uint8_t* g_lo = g_hi + (size_t)gblocks * P.g_blk;
  const uint32_t g_row_bytes = KR >= 64 ? 128u : (uint32_t)KR * 2u;
  uint8_t* bs = sm + P.off_b;
  uint8_t* stage = sm + P.off_s;
  float* recv = reinterpret_cast<float*>(sm + P.off_s);  // [C sources][64/C rows][KR], before the epilogue
  const uint32_t stage_stride = (uint32_t)kPiece * 4u + 16u;
  const int RPC = kTileRows / C;

  if (warp == 4) {
    tmem_alloc(&ctrl->tmem_base, kTmemCols);
    tmem_relinquish();
    if (lane == 0) {
      mbar_init(&ctrl->bar_a, 1);
      mbar_init(&ctrl->bar_x, 1);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&ctrl->bar_bp[i], 1);
        mbar_init(&ctrl->bar_full[i], 1);
        mbar_init(&ctrl->bar_empty[i], kEpilogueThreads);
      }
      mbar_init(&ctrl->bar_recv, 1);
      mbar_init(&ctrl->bar_g, 1);
      mbar_fence_init();
      mbar_arrive_expect_tx(&ctrl->bar_recv, (uint32_t)kTileRows * KR * 4u);
      mbar_arrive_expect_tx(&ctrl->bar_g, (uint32_t)kTileRows * KR * 4u);
      ctrl->abort = 0;
      tma_prefetch_desc(&map_a);
      tma_prefetch_desc(&map_b);
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

  // ---- shrink
  if (warp == 4 && lane == 0) {
    mbar_arrive_expect_tx(&ctrl->bar_a, (uint32_t)K * KS * r * 2);
    for (int a = 0; a < K; ++a)
      for (int kb = 0; kb < KS / kKBlock; ++kb)
        tma_load_2d(smem_u32(as + ((size_t)a * KS + (size_t)kb * kKBlock) * r * 2), &map_a, 0,
                    a * d_in + crank * KS + kb * kKBlock, &ctrl->bar_a);
  }
  if (warp < 4) {
    const int sub = lane >> 3, chunk = lane & 7;
    for (int kb = 0; kb < KS / kKBlock; ++kb) {
      const uint32_t blk = smem_u32(xs + (size_t)kb * kTileRows * 128);
      const int col = crank * KS + kb * kKBlock + chunk * 8;
#pragma unroll 4
      for (int it = 0; it < kTileRows / 16; ++it) {
        const int row = it * 16 + warp * 4 + sub;
        const int32_t tok = ctrl->tok[row];
        const __nv_bfloat16* src = tok >= 0 ? x + (int64_t)tok * d_in + col : x;
        cp_async_16(blk + sw128_offset(row, chunk), src, tok >= 0 ? 16u : 0u);
      }
    }
    cp_async_commit();
    cp_async_wait_all();
    fence_proxy_async_smem();
  }
  __syncwarp();
  named_barrier(kBarX, kThreads);  // the x tile is in shared memory
  if (warp == 4 && lane == 0) {
    bool ok = mbar_wait(&ctrl->bar_a, 0);
    tc_fence_after();
    if (ok) {
      const uint32_t atom = 8u * r * 2u;
      const SmemLayout swz = layout_for_row_bytes((uint32_t)r * 2u);
      const uint32_t idesc = idesc_bf16_f32(kMmaM, r, false, true);
      for (int kb = 0; kb < KS / kKBlock; ++kb)
        for (int ks = 0; ks < kKBlock / 16; ++ks) {
          // 128 MMA rows from the block's start: the tile's 64 rows, then 64 unused rows
          const uint64_t da = smem_desc(smem_u32(xs + (size_t)kb * kTileRows * 128 + ks * 32), 16, 1024,
                                        kSwizzle128B);
          const int krow = kb * kKBlock + ks * 16;
          for (int a = 0; a < K; ++a) {
            const uint64_t db = smem_desc(smem_u32(as + ((size_t)a * KS + krow) * r * 2), atom, atom, swz);
            umma_f16(tmem + (uint32_t)(a * r), da, db, idesc, (kb | ks) != 0);
          }
        }
      umma_commit(&ctrl->bar_x);
    } else {
      ctrl->abort = 1;
      report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
      mbar_arrive(&ctrl->bar_x);
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
    const uint32_t dst = dsmem_addr(smem_u32(recv + ((size_t)crank * RPC + (row % RPC)) * KR), owner);
    const uint32_t dst_bar = dsmem_addr(smem_u32(&ctrl->bar_recv), owner);
    float v[16];
    for (int c0 = 0; c0 < KR; c0 += 16) {
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
    // owner: rows [crank*RPC, (crank+1)*RPC) of the tile; each item is 8 columns of one row
    const int groups = KR / 8;
    for (int item = tid; item < RPC * groups; item += kEpilogueThreads) {
      const int rl = item / groups, c0 = (item % groups) * 8;
      const int trow = crank * RPC + rl;
      const int a = c0 / r;
      float coef = 0.f;
      const int64_t t = t0 + trow;
      if (t < N) {
        for (int j = 0; j < k; ++j) {
          const int32_t id = ids[t * k + j];
          if (id == a) coef += w ? w[t * k + j] : 1.f;
          if ((id < 0 || id >= K) && a == 0 && crank == 0) report(err_word, MOLORA_DEV_BAD_ADAPTER_ID);
        }
      }
      coef *= scale;
      float h[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int cc = 0; cc < C; ++cc) {
        const float4* src = reinterpret_cast<const float4*>(recv + ((size_t)cc * RPC + rl) * KR + c0);
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
  (void)N;
  DensePlan s;
  return dtype == MOLORA_BF16 && dense_choose(d_in, d_out, K, r, &s) && dense_encoder() != nullptr;
}

// Where the dense path beat the grouped one on GB300 (top-2, r = 16, L2 flushed): with a plan
// of two CTAs per SM and at least a few thousand tokens (2048 -> 6144 at N = 4096: 64 vs 82 us).
// One CTA per SM (d_in = 4096 at K*r = 64) leaves too few clusters resident, and small batches
// pay for the extra adapters: the grouped path won all of those points.
bool dense_preferred(molora_dtype dtype, int64_t N, int32_t d_in, int32_t d_out, int32_t K, int32_t r) {
  if (dtype != MOLORA_BF16 || N < 2048 || !(r == 16 || r == 32 || r == 64) || K * r > 128) return false;
  DensePlan s;
  for (int C : {8, 4, 2, 1})
    if (dense_plan(d_in, d_out, K, r, C, kTwoPerSm, &s)) return dense_encoder() != nullptr;
  return false;
}

cudaError_t launch_lora_dense(const void* x, int64_t N, int32_t d_in, int32_t d_out, const void* A, const void* B,
                              int32_t K, int32_t r, const int32_t* ids, const float* w, int32_t k, float scale,
                              void* y, bool y_bf16, int32_t* err_word, cudaStream_t stream) {
  DensePlan s;
  if (!dense_choose(d_in, d_out, K, r, &s)) return cudaErrorNotSupported;
  CUtensorMap map_a, map_b;
  const CUtensorMapSwizzle swa =
      r == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : (r == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
  if (!dense_map(&map_a, A, (uint64_t)K * d_in, (uint64_t)r, (uint32_t)r, kKBlock, swa)) return cudaErrorInvalidValue;
  // B seen as [K*r x d_out]: a box is all K*r rows (every adapter) by 64 columns
  if (!dense_map(&map_b, B, (uint64_t)K * r, (uint64_t)d_out, 64, (uint32_t)(K * r), CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(lora_dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
    if (attr_err != cudaSuccess) cudaGetLastError();
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t tiles = (N + kTileRows - 1) / kTileRows;
  return launch_kernel(lora_dense_kernel, dim3((unsigned)(tiles * s.C)), dim3(kThreads), s.smem, stream, s.C,
                       static_cast<const __nv_bfloat16*>(x), N, d_in, d_out, K, r, k, ids, w, scale, y,
                       (int32_t)(y_bf16 ? 1 : 0), s, err_word, map_a, map_b);
}

}  // namespace molora
