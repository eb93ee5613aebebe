// lora_grouped.cu -- the grouped tensor-core LoRA apply of "MoLoRA: Composable
// Specialization via Per-Token Adapter Routing" (Figure 2 right: tokens grouped by their
// selected adapter run as grouped GEMMs; Table 1: grouped GEMM dispatch shared by both
// routing modes; Figure 4: adapters at fixed addresses in a GPU-resident hot set).
//
// One fused kernel per call.  A work tile is up to 128 consecutive slots of one adapter's
// group (dispatch order), handled by a thread-block cluster of C CTAs:
//   1. shrink, split over d_in: CTA c gathers its 128 token rows x[tok, c*KS:(c+1)*KS)
//      with 16-byte cp.async (the gather fused as an index list: no permuted copy of x),
//      TMA-loads A_a's matching K-slice, and accumulates h_c = x A_a (128 x r, fp32) in
//      TMEM with tcgen05.mma;
//   2. the C partial h_c are summed through distributed shared memory in a fixed order
//      (deterministic), scaled by scale * w(slot), and split into two bf16 terms
//      g = g_hi + g_lo (relative error 2^-17) to feed the next MMA;
//   3. expand, split over d_out: CTA c computes D = g B_a[:, c*NC:(c+1)*NC) into TMEM in
//      passes of up to 256 columns (double-buffered), B_a's columns TMA-loaded;
//   4. epilogue: D goes TMEM -> registers -> shared memory, and each row is added into
//      y[tok, cols] by one cp.reduce.async.bulk .add.f32: the TMA unit performs the fp32
//      read-modify-write in L2, which also un-permutes (scatter by token) and, for top-k
//      with k > 1, combines the k slots of a token.
// The same kernel runs one masked per-sequence pass when given a fixed adapter: tiles are
// then 128 consecutive tokens and the slot weight is the 0/1 mask.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace molora {

namespace {

constexpr int kTileM = 128;          // slots per tile = TMEM lanes = MMA M
constexpr int kKBlock = 64;          // K elements per 128-byte swizzle row (bf16)
constexpr int kPassN = 256;          // columns per expand pass (one MMA N, one TMEM buffer)
constexpr int kPieceN = 128;         // columns per epilogue bulk reduction
constexpr int kEpilogueThreads = 128;
constexpr int kThreads = kEpilogueThreads + 32;  // + one producer/MMA warp
constexpr uint32_t kTmemCols = 512;
constexpr size_t kMinSmem = 116 * 1024;  // at most one CTA per SM, so a 512-column TMEM allocation never waits
constexpr size_t kMaxSmem = 227 * 1024;

struct GroupedShape {
  int C;          // cluster size (split of d_in and of d_out)
  int KS;         // d_in / C
  int NC;         // d_out / C
  size_t off_a;   // phase 1: A slice after the x tile
  size_t off_g;   // phase 2: g_hi (g_lo follows at +16 KB)
  size_t off_b;   // phase 2: B column chunk
  size_t off_s;   // phase 2: epilogue staging
  size_t region;  // bytes of the reused region
  size_t smem;    // dynamic shared memory requested
};

__host__ __device__ constexpr uint32_t p_stride(int r) { return (uint32_t)r * 4u + 16u; }
constexpr uint32_t kStageStride = kPieceN * 4 + 16;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool plan(int32_t d_in, int32_t d_out, int32_t r, int C, GroupedShape* s) {
  if (d_in % (C * kKBlock) || d_out % (C * 64)) return false;
  s->C = C;
  s->KS = d_in / C;
  s->NC = d_out / C;
  const size_t phase1 = (size_t)s->KS * (kTileM * 2 + 2 * r);
  s->off_a = (size_t)s->KS * kTileM * 2;
  s->off_g = align_up((size_t)kTileM * p_stride(r), 1024);
  s->off_b = s->off_g + 2 * 16384;
  s->off_s = align_up(s->off_b + (size_t)s->NC * r * 2, 1024);
  const size_t phase2 = s->off_s + (size_t)kTileM * kStageStride;
  s->region = phase1 > phase2 ? phase1 : phase2;
  s->smem = align_up(s->region, 1024) + 1024 /* base alignment slack */ + 2048 /* control block */;
  if (s->smem < kMinSmem) s->smem = kMinSmem;
  return s->smem <= kMaxSmem;
}

bool choose(int32_t d_in, int32_t d_out, int32_t r, GroupedShape* s) {
  for (int C : {8, 4, 2, 1})
    if (plan(d_in, d_out, r, C, s)) return true;
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
  uint64_t bar_shrink;    // shrink MMAs done
  uint64_t bar_full[2];   // expand pass done, per TMEM buffer
  uint64_t bar_empty[2];  // epilogue drained a TMEM buffer
  uint32_t tmem_base;
  int32_t abort;
  TileInfo tile;
  int32_t tok[kTileM];  // token of each tile row (-1: padding or skipped)
  float wgt[kTileM];    // weight of each tile row (0 for padding)
};

__device__ __forceinline__ uint64_t sw_for_rank(int r) {
  return r == 16 ? kSwizzle32B : (r == 32 ? kSwizzle64B : kSwizzle128B);
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    lora_grouped_kernel(const __nv_bfloat16* __restrict__ x, int64_t N, int32_t d_in, int32_t d_out, int32_t K,
                        int32_t r, int32_t k, const int32_t* __restrict__ ids, const float* __restrict__ w,
                        const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm, float scale,
                        float* __restrict__ y, int32_t mask_adapter, int32_t C, int32_t KS, int32_t NC,
                        uint32_t off_a, uint32_t off_g, uint32_t off_b, uint32_t off_s, uint32_t region,
                        int32_t* err_word, const __grid_constant__ CUtensorMap map_a,
                        const __grid_constant__ CUtensorMap map_b) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(sm + region);  // region is 1024-aligned by the host
  int32_t* s_tok = ctrl->tok;
  float* s_w = ctrl->wgt;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int crank = (int)cluster_ctarank();
  const int cluster_id = blockIdx.x / C;
  const int64_t S = N * (int64_t)k;

  // ---- which tile this cluster owns (identical in every CTA of the cluster)
  if (tid == 0) {
    TileInfo ti{-1, 0, 0, 0};
    if (mask_adapter >= 0) {
      const int64_t t0 = (int64_t)cluster_id * kTileM;
      if (t0 < N) ti = TileInfo{mask_adapter, (int32_t)t0, (int32_t)(N - t0 < kTileM ? N - t0 : kTileM), 0};
    } else {
      int32_t cum = 0;
      int32_t prev = offsets[0];
      bool bad = prev != 0;
      for (int a = 0; a < K && ti.adapter < 0; ++a) {
        const int32_t nxt = offsets[a + 1];
        if (nxt < prev || nxt > S) {
          bad = true;
          break;
        }
        const int32_t n_a = nxt - prev;
        const int32_t tiles = (n_a + kTileM - 1) / kTileM;
        if (cluster_id < cum + tiles) {
          const int32_t row0 = (cluster_id - cum) * kTileM;
          ti = TileInfo{a, row0, min(kTileM, n_a - row0), prev};
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
  if (tile.adapter < 0) return;  // whole cluster idles (every CTA computed the same tile)
  const int a = tile.adapter;

  uint8_t* xs = sm;             // phase 1: x tile, KS/64 blocks of [128 rows x 128 B]
  uint8_t* as = sm + off_a;     // phase 1: A slice [KS x r], MN-major, swizzled by TMA
  uint8_t* ps = sm;             // phase 2: partial h, [128][r] fp32 (row stride r*4+16)
  uint8_t* g_hi = sm + off_g;   // phase 2: g as two bf16 K-major tiles
  uint8_t* g_lo = g_hi + 16384;
  uint8_t* bs = sm + off_b;     // phase 2: B chunk, NC/64 boxes of [r rows x 128 B]
  float* stage = reinterpret_cast<float*>(sm + off_s);

  if (warp == 4) {
    tmem_alloc(&ctrl->tmem_base, kTmemCols);
    tmem_relinquish();
    if (lane == 0) {
      mbar_init(&ctrl->bar_a, 1);
      mbar_init(&ctrl->bar_b, 1);
      mbar_init(&ctrl->bar_shrink, 1);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&ctrl->bar_full[i], 1);
        mbar_init(&ctrl->bar_empty[i], kEpilogueThreads);
      }
      mbar_fence_init();
      tma_prefetch_desc(&map_a);
      tma_prefetch_desc(&map_b);
    }
  } else {
    // per-row metadata: token and weight (weight 0 for padding rows)
    const int row = tid;
    int32_t tok = -1;
    float wt = 0.f;
    if (row < tile.nvalid) {
      if (mask_adapter >= 0) {
        tok = tile.row0 + row;
        wt = ids[tok] == mask_adapter ? 1.f : 0.f;
      } else {
        const int32_t slot = perm[tile.group_off + tile.row0 + row];
        if (slot >= 0 && slot < S && ids[slot] == a) {
          tok = slot / k;
          wt = w ? w[slot] : 1.f;
        } else if (crank == 0) {
          report(err_word, MOLORA_DEV_BAD_PERMUTATION);
        }
      }
    }
    s_tok[row] = tok;
    s_w[row] = wt;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;

  if (warp == 4) {
    if (lane == 0) {
      // A slice rows a*d_in + crank*KS + [0, KS), in boxes of 64 rows
      mbar_arrive_expect_tx(&ctrl->bar_a, (uint32_t)KS * r * 2);
      for (int kb = 0; kb < KS / kKBlock; ++kb)
        tma_load_2d(smem_u32(as + (size_t)kb * kKBlock * r * 2), &map_a, 0, a * d_in + crank * KS + kb * kKBlock,
                    &ctrl->bar_a);
    }
  } else {
    // gather: lanes 8q..8q+7 copy the eight 16-byte chunks of one 128-byte row segment
    const int sub = lane >> 3, chunk = lane & 7;
    const int nkb = KS / kKBlock;
    for (int kb = 0; kb < nkb; ++kb) {
      const uint32_t blk = smem_u32(xs + (size_t)kb * kTileM * 128);
#pragma unroll 4
      for (int it = 0; it < kTileM / 16; ++it) {
        const int row = it * 16 + warp * 4 + sub;
        const int32_t tok = s_tok[row];
        const __nv_bfloat16* src =
            tok >= 0 ? x + (int64_t)tok * d_in + crank * KS + kb * kKBlock + chunk * 8 : x;
        cp_async_16(blk + sw128_offset(row, chunk), src, tok >= 0 ? 16u : 0u);
      }
    }
    cp_async_commit();
    cp_async_wait_all();
    fence_proxy_async_smem();
  }
  __syncthreads();  // x tile in shared memory

  const uint32_t idesc_shrink = idesc_bf16_f32(kTileM, r, false, true);
  if (warp == 4 && lane == 0) {
    bool ok = mbar_wait(&ctrl->bar_a, 0);
    tc_fence_after();
    if (ok) {
      const uint32_t atom = 8u * r * 2u;
      const SmemLayout swz = (SmemLayout)sw_for_rank(r);
      for (int kb = 0; kb < KS / kKBlock; ++kb)
        for (int ks = 0; ks < kKBlock / 16; ++ks) {
          const uint64_t da = smem_desc(smem_u32(xs + (size_t)kb * kTileM * 128 + ks * 32), 16, 1024, kSwizzle128B);
          const uint64_t db = smem_desc(smem_u32(as + (size_t)(kb * kKBlock + ks * 16) * r * 2), atom, atom, swz);
          umma_f16(tmem, da, db, idesc_shrink, (kb | ks) != 0);
        }
      umma_commit(&ctrl->bar_shrink);
    } else {
      ctrl->abort = 1;
      report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
      mbar_arrive(&ctrl->bar_shrink);
    }
    // B chunk lands in the (now dead) phase-1 region once the shrink has read it
    ok = mbar_wait(&ctrl->bar_shrink, 0);
    if (ok) {
      mbar_arrive_expect_tx(&ctrl->bar_b, (uint32_t)NC * r * 2);
      for (int q = 0; q < NC / 64; ++q)
        tma_load_2d(smem_u32(bs + (size_t)q * r * 128), &map_b, crank * NC + q * 64, a * r, &ctrl->bar_b);
    } else {
      ctrl->abort = 1;
      report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
      mbar_arrive(&ctrl->bar_b);
    }
  }
  if (warp < 4) {
    // partial h of this CTA: TMEM -> registers -> shared memory (for the cluster reduction)
    const bool ok = mbar_wait(&ctrl->bar_shrink, 0);
    tc_fence_after();
    const int row = tid;
    if (ok) {
      float v[16];
      for (int c0 = 0; c0 < r; c0 += 16) {
        tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
        float4* dst = reinterpret_cast<float4*>(ps + row * p_stride(r) + c0 * 4);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    } else {
      ctrl->abort = 1;
      report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
    }
    tc_fence_before();
  }
  __syncwarp();
  cluster_sync();  // every CTA's partial h is in its shared memory

  if (warp < 4) {
    const int row = tid;
    const float coef = scale * s_w[row];
    const uint32_t mine = smem_u32(ps + row * p_stride(r));
    for (int c0 = 0; c0 < r; c0 += 8) {
      float h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = 0.f;
      for (int cc = 0; cc < C; ++cc) {
        const uint32_t src = dsmem_addr(mine, (uint32_t)cc) + c0 * 4;
        const float4 p0 = dsmem_ld_f4(src), p1 = dsmem_ld_f4(src + 16);
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
      const uint32_t off = sw128_offset(row, c0 / 8);
      *reinterpret_cast<uint4*>(g_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(g_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    fence_proxy_async_smem();
  }
  __syncwarp();
  cluster_arrive();  // done reading the other CTAs' partials (waited on before exit)
  __syncthreads();   // g ready for the tensor core

  const int npass = (NC + kPassN - 1) / kPassN;
  if (warp == 4) {
    if (lane == 0) {
      bool ok = !ctrl->abort && mbar_wait(&ctrl->bar_b, 0);
      tc_fence_after();
      for (int p = 0; p < npass; ++p) {
        const int buf = p & 1;
        const int width = min(kPassN, NC - p * kPassN);
        if (p >= 2 && ok) ok = mbar_wait(&ctrl->bar_empty[buf], ((p >> 1) - 1) & 1);
        if (!ok) {
          ctrl->abort = 1;
          report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
          mbar_arrive(&ctrl->bar_full[buf]);
          continue;
        }
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(kTileM, width, false, true);
        const uint32_t d = tmem + buf * kPassN;
        for (int ks = 0; ks < r / 16; ++ks) {
          const uint64_t db = smem_desc(smem_u32(bs + (size_t)(p * (kPassN / 64)) * r * 128 + ks * 2048), r * 128,
                                        1024, kSwizzle128B);
          umma_f16(d, smem_desc(smem_u32(g_hi + ks * 32), 16, 1024, kSwizzle128B), db, idesc, ks != 0);
          umma_f16(d, smem_desc(smem_u32(g_lo + ks * 32), 16, 1024, kSwizzle128B), db, idesc, 1);
        }
        umma_commit(&ctrl->bar_full[buf]);
      }
    }
    __syncwarp();
  } else {
    const int row = tid;
    const int32_t tok = s_tok[row];
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    float* srow = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(stage) + row * kStageStride);
    for (int p = 0; p < npass; ++p) {
      const int buf = p & 1;
      const int width = min(kPassN, NC - p * kPassN);
      const bool ok = mbar_wait(&ctrl->bar_full[buf], (p >> 1) & 1);
      tc_fence_after();
      if (!ok) report(err_word, MOLORA_DEV_WAIT_TIMEOUT);
      for (int q = 0; ok && !ctrl->abort && q < width; q += kPieceN) {
        const int cols = min(kPieceN, width - q);
        bulk_wait_read<0>();  // this row's previous reduction has finished reading the stage
        float v[16];
        for (int c0 = 0; c0 < cols; c0 += 16) {
          tmem_ld16(lane_base + buf * kPassN + q + c0, v);
          float4* dst = reinterpret_cast<float4*>(srow + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        fence_proxy_async_smem();
        if (tok >= 0) {
          bulk_reduce_add_f32(y + (int64_t)tok * d_out + crank * NC + p * kPassN + q, smem_u32(srow), cols * 4);
          bulk_commit();
        }
      }
      tc_fence_before();
      mbar_arrive(&ctrl->bar_empty[buf]);
    }
    bulk_wait_all();
  }
  __syncthreads();
  cluster_wait();  // no CTA leaves while another may still read its partials
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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
  (void)N, (void)K, (void)k;
  if (dtype != MOLORA_BF16 || !(r == 16 || r == 32 || r == 64)) return false;
  GroupedShape s;
  return choose(d_in, d_out, r, &s) && encoder() != nullptr;
}

cudaError_t launch_lora_grouped(const void* x, int64_t N, int32_t d_in, int32_t d_out, const void* A, const void* B,
                                int32_t K, int32_t r, const int32_t* ids, const float* w, int32_t k,
                                const int32_t* counts, const int32_t* offsets, const int32_t* perm, float scale,
                                float* y, int32_t mask_adapter, int32_t* err_word, cudaStream_t stream) {
  (void)counts;
  GroupedShape s;
  if (!choose(d_in, d_out, r, &s)) return cudaErrorNotSupported;
  CUtensorMap map_a, map_b;
  const CUtensorMapSwizzle swa =
      r == 16 ? CU_TENSOR_MAP_SWIZZLE_32B : (r == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
  if (!make_map(&map_a, A, (uint64_t)K * d_in, (uint64_t)r, (uint32_t)r, kKBlock, swa)) return cudaErrorInvalidValue;
  if (!make_map(&map_b, B, (uint64_t)K * r, (uint64_t)d_out, 64, (uint32_t)r, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(lora_grouped_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
    if (attr_err != cudaSuccess) cudaGetLastError();
  });
  if (attr_err != cudaSuccess) return attr_err;
  static_assert(sizeof(Ctrl) <= 2048, "control block");

  const int64_t tiles = mask_adapter >= 0 ? (N + kTileM - 1) / kTileM : (N * k + kTileM - 1) / kTileM + K;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * s.C));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = s.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)s.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, lora_grouped_kernel, static_cast<const __nv_bfloat16*>(x), N, d_in, d_out, K, r,
                            k, ids, w, offsets, perm, scale, y, mask_adapter, (int32_t)s.C, (int32_t)s.KS,
                            (int32_t)s.NC, (uint32_t)s.off_a, (uint32_t)s.off_g, (uint32_t)s.off_b,
                            (uint32_t)s.off_s, (uint32_t)align_up(s.region, 1024), err_word, map_a, map_b);
  const cudaError_t last = cudaGetLastError();  // clears the runtime's error state either way
  return e != cudaSuccess ? e : last;
}

}  // namespace molora
