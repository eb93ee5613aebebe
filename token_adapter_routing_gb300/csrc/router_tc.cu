// router_tc.cu -- the learned router TopK(g(x)) of "MoLoRA: Composable Specialization via
// Per-Token Adapter Routing" (Table 1: routing cost O(64d + 64K); Figure 2: top-k adapters
// combined by a weighted sum; Table 10: softmax(Wx + b) gating) on tcgen05 tensor cores.
//
// The d_in x 64 projection is the only dense contraction (64 flops per byte of x), so it
// runs as a tcgen05 GEMM: a cluster of C CTAs owns 128 consecutive tokens and splits d_in;
// each CTA streams its K-slice of x (K-major, 128-byte swizzle) and the matching W1 rows
// (MN-major) through a ring of TMA stages, and accumulates 128 x 64 fp32 partials in TMEM.
// CTA c owns tokens [c*128/C, (c+1)*128/C) of the tile: every CTA stages its partials in
// shared memory and sends each owner its rows with one bulk copy (counted by the owner's
// mbarrier), and the owner sums the C partials in rank order (deterministic).  Eight lanes per
// token then form the hidden units, the logits, the top k (strictly greater wins, so equal
// logits keep the lower index) and the softmax over the k, all in registers (router_rows in
// common.cuh, shared with the fused router + apply kernel: the same arithmetic, so both give
// identical results whenever they split d_in the same way).
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace molora {

namespace {

constexpr int kTileM = 128;
constexpr int kKBlock = 64;
constexpr int kEpi = 128;                 // warps 0-3: reduction and second stage, one row each
constexpr int kThreads = kEpi + 64;       // + TMA producer warp (4) + MMA warp (5)
constexpr uint32_t kTmemCols = 64;
constexpr size_t kMaxSmem = 227 * 1024;
constexpr size_t kTwoPerSm = 113 * 1024;
constexpr int kMaxStages = 4;
constexpr uint32_t kStageBytes = (uint32_t)(kTileM + kRouterHidden) * kKBlock * 2;  // x block + W1 block

struct RouterShape {
  int C, KS, S;  // cluster size (split of d_in), K-slice per CTA, stages in the ring
  size_t off_recv, off_w2, region, smem;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr size_t kStagingBytes = (size_t)kTileM * kRouterHidden * 4;  // the tile's partials, fp32

bool plan(int32_t d_in, int32_t K, int C, size_t budget, RouterShape* s) {
  if (d_in % (C * kKBlock) || kTileM % C) return false;
  s->C = C;
  s->KS = d_in / C;
  const int nkb = s->KS / kKBlock;
  for (int S = kMaxStages < nkb ? kMaxStages : nkb; S >= 1; --S) {
    s->S = S;
    // the outgoing partials are staged in the ring (x and W1 are consumed by then); the
    // receive slots are not: other CTAs may copy in while this CTA's tensor core still reads
    const size_t ring = (size_t)S * kStageBytes;
    s->off_recv = align_up(ring > kStagingBytes ? ring : kStagingBytes, 1024);
    s->off_w2 = s->off_recv + kStagingBytes;
    // W2 as fp32 [64 x K], b1 [64], b2 [K]
    s->region = align_up(s->off_w2 + sizeof(float) * ((size_t)kRouterHidden * K + kRouterHidden + K), 1024);
    s->smem = s->region + 1024 + 256;
    if (s->smem <= budget) return true;
  }
  return false;
}

// Two CTAs per SM where they fit (the deepest ring that does), else one.  The cluster is the
// widest whose CTAs (tiles x C) are all resident at once: every CTA pays the same serial tail
// (exchange, second stage, cluster exit), so a second, partial wave costs a whole CTA time (at
// 8192 tokens, d_in = 4096: clusters of 4 in one wave beat clusters of 8 in 1.7 waves).  When
// even C = 1 takes more than one wave, C = 1 (no exchange at all).
bool choose(int64_t N, int32_t d_in, int32_t K, RouterShape* s) {
  const int64_t tiles = (N + kTileM - 1) / kTileM;
  for (size_t budget : {kTwoPerSm, kMaxSmem}) {
    const int64_t slots = (budget == kTwoPerSm ? 2 : 1) * (int64_t)num_sms();
    bool found = false;
    RouterShape narrowest{};
    for (int C : {8, 4, 2, 1}) {
      if (!plan(d_in, K, C, budget, s)) continue;
      if (tiles * C <= slots) return true;
      narrowest = *s;
      found = true;
    }
    if (found) {
      *s = narrowest;
      return true;
    }
  }
  return false;
}

struct __align__(8) RCtrl {
  uint64_t full[kMaxStages];   // x and W1 blocks of a stage landed
  uint64_t empty[kMaxStages];  // the MMAs reading a stage are done
  uint64_t bar_mma;            // all MMAs done
  uint64_t bar_recv;           // every CTA's partials of this CTA's rows arrived
  uint32_t tmem_base;
  int32_t abort;
};

}  // namespace

// A warp-specialized CTA: warp 4 streams the CTA's K-slice of x (128 rows) and W1 through a ring
// of S stages of 64-column K-blocks by TMA; warp 5 issues tcgen05.mma (M = 128, N = 64) into TMEM
// and releases each stage when its MMAs complete; warps 0-3 meanwhile stage W2 and the biases,
// then move the 128 x 64 partials from TMEM to shared memory (row-major, 16-byte chunks swizzled
// by row) and send each owner its RPC = 128 / C rows with one bulk copy (counted by the owner's
// mbarrier), and as owner run the second stage for their rows (router_rows).
__global__ void __launch_bounds__(kThreads, 2)
    router_tc_kernel(int64_t N, int32_t d_in, const __nv_bfloat16* __restrict__ W2, const float* __restrict__ b1,
                     const float* __restrict__ b2, int32_t K, int32_t k, float* __restrict__ logits,
                     int32_t* __restrict__ ids, float* __restrict__ w, const RouterShape P,
                     const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  RCtrl* ctrl = reinterpret_cast<RCtrl*>(sm + P.region);
  uint8_t* stg = sm;                                        // [128 rows][64] fp32 partials, after the MMAs
  float* recv = reinterpret_cast<float*>(sm + P.off_recv);  // [C sources][RPC rows][64]
  float* w2s = reinterpret_cast<float*>(sm + P.off_w2);
  float* b1s = w2s + kRouterHidden * K;
  float* b2s = b1s + kRouterHidden;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = P.C, KS = P.KS, S = P.S;
  const int crank = (int)cluster_ctarank();
  const int64_t t0 = (int64_t)(blockIdx.x / C) * kTileM;
  const int nkb = KS / kKBlock;
  const int RPC = kTileM / C;
  volatile int32_t* abort = &ctrl->abort;

  if (warp == 5) {
    tmem_alloc(&ctrl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&ctrl->full[i], 1);
      mbar_init(&ctrl->empty[i], 1);
    }
    mbar_init(&ctrl->bar_mma, 1);
    mbar_init(&ctrl->bar_recv, 1);
    ctrl->abort = 0;
    mbar_fence_init();
    mbar_arrive_expect_tx(&ctrl->bar_recv, (uint32_t)kStagingBytes);
    tma_prefetch_desc(&map_x);
    tma_prefetch_desc(&map_w1);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  cluster_arrive();  // every CTA's receive barrier is initialised and armed
  pdl_wait();        // the inputs may come from the previous kernel; the setup above overlapped it
  pdl_launch_dependents();

  if (warp == 4) {
    if (lane == 0) {
      int issued = 0;
      for (int kb = 0; kb < nkb; ++kb, ++issued) {
        const int s = kb % S, use = kb / S;
        if (use > 0 && !mbar_wait_or_abort(&ctrl->empty[s], (uint32_t)(use - 1) & 1u, abort)) break;
        uint8_t* st = sm + (size_t)s * kStageBytes;
        const int32_t col = crank * KS + kb * kKBlock;
        mbar_arrive_expect_tx(&ctrl->full[s], kStageBytes);
        tma_load_2d(smem_u32(st), &map_x, col, (int32_t)t0, &ctrl->full[s]);
        tma_load_2d(smem_u32(st + kTileM * kKBlock * 2), &map_w1, 0, col, &ctrl->full[s]);
      }
      // nothing may land in shared memory after the CTA has left
      for (int s = 0; s < S && s < issued; ++s) mbar_wait(&ctrl->full[s], (uint32_t)((issued - 1 - s) / S) & 1u);
    }
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTileM, kRouterHidden, false, true);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % S;
        if (!mbar_wait_or_abort(&ctrl->full[s], (uint32_t)(kb / S) & 1u, abort)) break;
        tc_fence_after();
        const uint8_t* st = sm + (size_t)s * kStageBytes;
        for (int ks = 0; ks < kKBlock / 16; ++ks) {
          const uint64_t da = smem_desc(smem_u32(st + ks * 32), 16, 1024, kSwizzle128B);
          const uint64_t db = smem_desc(smem_u32(st + kTileM * kKBlock * 2 + ks * 2048), 1024, 1024, kSwizzle128B);
          umma_f16(tmem, da, db, idesc, (kb | ks) != 0);
        }
        umma_commit(&ctrl->empty[s]);
      }
      umma_commit(&ctrl->bar_mma);  // arrives once every MMA issued above has completed
    }
    __syncwarp();
  } else {
    // W2 and the biases while the loads stream (only these four warps read them)
    for (int i = tid; i < kRouterHidden * K; i += kEpi) w2s[i] = __bfloat162float(W2[i]);
    if (tid < kRouterHidden) b1s[tid] = b1 ? b1[tid] : 0.f;
    for (int i = tid; i < K; i += kEpi) b2s[i] = b2 ? b2[i] : 0.f;
    const bool have = __all_sync(0xffffffffu, mbar_wait_or_abort(&ctrl->bar_mma, 0, abort) && !*abort);
    tc_fence_after();
    // row `tid` of the tile: its 64 partial hidden sums, TMEM -> staging (chunk c at c ^ (row & 7))
    const int row = tid;
    uint32_t v[64];
    if (have) {
      tmem_ld32_start(tmem + ((uint32_t)(warp * 32) << 16), *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld32_start(tmem + ((uint32_t)(warp * 32) << 16) + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld_bind(*reinterpret_cast<uint32_t(*)[32]>(v + 32));
    } else {
#pragma unroll
      for (int i = 0; i < 64; ++i) v[i] = 0u;
    }
    uint4* srow = reinterpret_cast<uint4*>(stg + (size_t)row * kRouterHidden * 4);
#pragma unroll
    for (int c = 0; c < 16; ++c) srow[c ^ (row & 7)] = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    fence_proxy_async_smem();  // the staged rows, visible to the bulk copies
    named_barrier(1, kEpi);
    cluster_wait();  // every owner's receive barrier is armed
    if (tid < C) {
      // owner `tid` gets rows [tid * RPC, (tid + 1) * RPC) into its slot for this CTA
      const uint32_t bytes = (uint32_t)RPC * kRouterHidden * 4;
      bulk_copy_to_cluster(dsmem_addr(smem_u32(recv) + (uint32_t)crank * bytes, (uint32_t)tid),
                           smem_u32(stg) + (uint32_t)tid * bytes, bytes, dsmem_addr(smem_u32(&ctrl->bar_recv), (uint32_t)tid));
    }
    named_barrier(2, kEpi);  // W2 and the biases staged by every epilogue thread
    const bool got = __all_sync(0xffffffffu, mbar_wait(&ctrl->bar_recv, 0));
    // owner: ReLU, logits, top k and softmax for this CTA's rows
    router_rows(recv, C, RPC, kRouterHidden, 0, true, w2s, b1s, b2s, K, k, t0 + crank * RPC, N, got && have, logits,
                ids, w, nullptr, tid, kEpi);
  }
  if (warp >= 4) cluster_wait();
  __syncthreads();
  cluster_arrive();
  cluster_wait();  // no CTA leaves while another may still copy into its shared memory, or from it
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

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

bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows) {
  auto enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool router_tc_supported(molora_dtype dtype, int64_t N, int32_t d_in, int32_t K, int32_t k) {
  (void)k;
  RouterShape s;
  return dtype == MOLORA_BF16 && choose(N, d_in, K, &s) && encoder() != nullptr;
}

cudaError_t launch_router_tc(const void* x, int64_t N, int32_t d_in, const void* W1, const float* b1, const void* W2,
                             const float* b2, int32_t K, int32_t k, float* logits, int32_t* ids, float* w,
                             cudaStream_t stream) {
  RouterShape s;
  if (!choose(N, d_in, K, &s)) return cudaErrorNotSupported;
  CUtensorMap map_x, map_w1;
  if (!make_map(&map_x, x, (uint64_t)N, (uint64_t)d_in, kKBlock, kTileM)) return cudaErrorInvalidValue;
  if (!make_map(&map_w1, W1, (uint64_t)d_in, kRouterHidden, kRouterHidden, kKBlock)) return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
    if (attr_err != cudaSuccess) cudaGetLastError();
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int64_t tiles = (N + kTileM - 1) / kTileM;
  return launch_kernel(router_tc_kernel, dim3((unsigned)(tiles * s.C)), dim3(kThreads), s.smem, stream, s.C, N, d_in,
                       static_cast<const __nv_bfloat16*>(W2), b1, b2, K, k, logits, ids, w, s, map_x, map_w1);
}

}  // namespace molora
