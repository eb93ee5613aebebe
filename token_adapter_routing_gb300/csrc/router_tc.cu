// router_tc.cu -- the learned router TopK(g(x)) of "MoLoRA: Composable Specialization via
// Per-Token Adapter Routing" (Table 1: routing cost O(64d + 64K); Figure 2: top-k adapters
// combined by a weighted sum; Table 10: softmax(Wx + b) gating) on tcgen05 tensor cores.
//
// The d_in x 64 projection is the only dense contraction (64 flops per byte of x), so it
// runs as a tcgen05 GEMM: a cluster of C CTAs owns 128 consecutive tokens and splits d_in;
// each CTA TMA-loads its x tile (K-major, 128-byte swizzle) and the matching W1 rows
// (MN-major), and accumulates 128 x 64 fp32 partials in TMEM.  CTA c owns tokens
// [c*128/C, (c+1)*128/C) of the tile: every CTA pushes those rows' partials to their owner
// with st.async (counted by the owner's mbarrier), and the owner sums the C partials in rank
// order (deterministic).  The owner's 128 threads then split each token's 64 hidden units
// into 8 groups: ReLU, partial logits over the group's 8 units, and a fixed-order sum of the
// 8 group partials (combined by warp shuffles); one thread per token selects the top k
// (strictly greater wins, so equal logits keep the lower index) and renormalises the softmax
// over the k (router_rows in common.cuh, shared with the fused router + apply kernel).
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace molora {

namespace {

constexpr int kTileM = 128;
constexpr int kKBlock = 64;
constexpr int kThreads = 160;
constexpr uint32_t kTmemCols = 64;
constexpr size_t kMaxSmem = 227 * 1024;
constexpr size_t kTwoPerSm = 113 * 1024;

struct RouterShape {
  int C, KS, XR;  // XR: x columns loaded per round (the x and W1 buffers are reused per round)
  size_t off_w1, off_recv, off_w2, region, smem;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool plan(int32_t d_in, int32_t K, int C, size_t budget, RouterShape* s) {
  if (d_in % (C * kKBlock) || kTileM % C) return false;
  s->C = C;
  s->KS = d_in / C;
  for (int XR = s->KS > 512 ? 512 : s->KS; XR >= kKBlock; XR -= kKBlock) {
    if (s->KS % XR) continue;
    s->XR = XR;
    s->off_w1 = (size_t)XR * kTileM * 2;
    const size_t phase1 = s->off_w1 + (size_t)XR * kRouterHidden * 2;
    // the logits of the owner's rows reuse the phase-1 space (x and W1 are consumed by then)
    const size_t plog = (size_t)(kTileM / C) * K * 4;
    // receive slots: other CTAs may push while this CTA's tensor core still reads x
    s->off_recv = align_up(phase1 > plog ? phase1 : plog, 1024);
    s->off_w2 = s->off_recv + (size_t)kTileM * kRouterHidden * 4;
    // W2 as fp32 [64 x K], b1 [64], b2 [K]
    s->region = align_up(s->off_w2 + sizeof(float) * ((size_t)kRouterHidden * K + kRouterHidden + K), 1024);
    s->smem = s->region + 1024 + 256;
    if (s->smem <= budget) return true;
  }
  return false;
}

// Clusters of 8 first; the widest x round that still fits two CTAs per SM (so a cluster's
// rounds overlap another CTA's), else one CTA per SM.
bool choose(int32_t d_in, int32_t K, RouterShape* s) {
  for (size_t budget : {kTwoPerSm, kMaxSmem})
    for (int C : {8, 4, 2, 1})
      if (plan(d_in, K, C, budget, s)) return true;
  return false;
}

struct __align__(8) RCtrl {
  uint64_t bar_load;   // TMA of one round (one phase per round)
  uint64_t bar_round;  // MMAs of one round done (one phase per round; waited only by the producer)
  uint64_t bar_mma;    // all MMAs done (one phase)
  uint64_t bar_recv;
  uint32_t tmem_base;
  int32_t abort;
};

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(int64_t N, int32_t d_in, const __nv_bfloat16* __restrict__ W2, const float* __restrict__ b1,
                     const float* __restrict__ b2, int32_t K, int32_t k, float* __restrict__ logits,
                     int32_t* __restrict__ ids, float* __restrict__ w, int32_t C, int32_t KS, int32_t XR,
                     uint32_t off_w1,
                     uint32_t off_recv, uint32_t off_w2, uint32_t region, const __grid_constant__ CUtensorMap map_x,
                     const __grid_constant__ CUtensorMap map_w1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  RCtrl* ctrl = reinterpret_cast<RCtrl*>(sm + region);
  uint8_t* xs = sm;
  uint8_t* w1s = sm + off_w1;
  float* plog = reinterpret_cast<float*>(sm);  // [RPC rows][K] logits, after the MMA
  float* recv = reinterpret_cast<float*>(sm + off_recv);  // [C sources][RPC rows][64]
  float* w2s = reinterpret_cast<float*>(sm + off_w2);
  float* b1s = w2s + kRouterHidden * K;
  float* b2s = b1s + kRouterHidden;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int crank = (int)cluster_ctarank();
  const int64_t tile = blockIdx.x / C;
  const int64_t t0 = tile * kTileM;
  const int nkb = XR / kKBlock;  // K-blocks per round
  const int rounds = KS / XR;
  const int RPC = kTileM / C;

  if (warp == 4) {
    tmem_alloc(&ctrl->tmem_base, kTmemCols);
    tmem_relinquish();
    if (lane == 0) {
      mbar_init(&ctrl->bar_load, 1);
      mbar_init(&ctrl->bar_round, 1);
      mbar_init(&ctrl->bar_mma, 1);
      mbar_init(&ctrl->bar_recv, 1);
      ctrl->abort = 0;
      mbar_fence_init();
      mbar_arrive_expect_tx(&ctrl->bar_recv, (uint32_t)kTileM * kRouterHidden * 4u);
      tma_prefetch_desc(&map_x);
      tma_prefetch_desc(&map_w1);
    }
  }
  pdl_wait();  // the inputs may come from the previous kernel; the prologue above overlapped it
  pdl_launch_dependents();
  if (warp < 4) {
    for (int i = tid; i < kRouterHidden * K; i += kTileM) w2s[i] = __bfloat162float(W2[i]);
    if (tid < kRouterHidden) b1s[tid] = b1 ? b1[tid] : 0.f;
    if (tid < K) b2s[tid] = b2 ? b2[tid] : 0.f;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  __syncwarp();
  cluster_arrive();  // every CTA's receive barrier is initialised and armed

  if (warp == 4 && lane == 0) {
    bool ok = true;
    const uint32_t idesc = idesc_bf16_f32(kTileM, kRouterHidden, false, true);
    for (int rd = 0; rd < rounds && ok; ++rd) {
      if (rd > 0) ok = mbar_wait(&ctrl->bar_round, (rd - 1) & 1);  // the buffers are free again
      if (!ok) break;
      mbar_arrive_expect_tx(&ctrl->bar_load, (uint32_t)XR * (kTileM + kRouterHidden) * 2);
      for (int kb = 0; kb < nkb; ++kb) {
        const int32_t col = crank * KS + rd * XR + kb * kKBlock;
        tma_load_2d(smem_u32(xs + (size_t)kb * kTileM * 128), &map_x, col, (int32_t)t0, &ctrl->bar_load);
        tma_load_2d(smem_u32(w1s + (size_t)kb * kKBlock * 128), &map_w1, 0, col, &ctrl->bar_load);
      }
      ok = mbar_wait(&ctrl->bar_load, rd & 1);
      tc_fence_after();
      if (!ok) break;
      for (int kb = 0; kb < nkb; ++kb)
        for (int ks = 0; ks < kKBlock / 16; ++ks) {
          const uint64_t da = smem_desc(smem_u32(xs + (size_t)kb * kTileM * 128 + ks * 32), 16, 1024, kSwizzle128B);
          const uint64_t db =
              smem_desc(smem_u32(w1s + (size_t)kb * kKBlock * 128 + ks * 2048), 1024, 1024, kSwizzle128B);
          umma_f16(tmem, da, db, idesc, (rd | kb | ks) != 0);
        }
      umma_commit(&ctrl->bar_round);
    }
    if (ok) {
      umma_commit(&ctrl->bar_mma);  // covers every MMA issued above
    } else {
      ctrl->abort = 1;
      mbar_arrive(&ctrl->bar_mma);
    }
  }
  bool have = true;
  if (warp < 4) {
    have = mbar_wait(&ctrl->bar_mma, 0) && !ctrl->abort;
    tc_fence_after();
  }
  __syncwarp();
  cluster_wait();
  if (warp < 4) {
    // push this row's 64 partial hidden sums to the row's owner
    const int row = tid;
    const uint32_t owner = (uint32_t)(row / RPC);
    const uint32_t dst = dsmem_addr(smem_u32(recv + ((size_t)crank * RPC + (row % RPC)) * kRouterHidden), owner);
    const uint32_t dst_bar = dsmem_addr(smem_u32(&ctrl->bar_recv), owner);
    float v[16];
    for (int c0 = 0; c0 < kRouterHidden; c0 += 16) {
      if (have)
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
    tc_fence_before();
    const bool got = mbar_wait(&ctrl->bar_recv, 0);
    // owner: ReLU, logits, top k and softmax for this CTA's rows (plog holds the logit rows)
    router_rows(recv, C, RPC, kRouterHidden, 0, w2s, b1s, b2s, K, k, t0 + crank * RPC, N, got && have, logits, ids,
                w, plog, nullptr, tid, kTileM);
  }
  __syncwarp();
  __syncthreads();
  cluster_arrive();
  cluster_wait();  // no CTA leaves while another may still write into its shared memory
  if (warp == 4) {
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
  (void)N, (void)k;
  RouterShape s;
  return dtype == MOLORA_BF16 && choose(d_in, K, &s) && encoder() != nullptr;
}

cudaError_t launch_router_tc(const void* x, int64_t N, int32_t d_in, const void* W1, const float* b1, const void* W2,
                             const float* b2, int32_t K, int32_t k, float* logits, int32_t* ids, float* w,
                             cudaStream_t stream) {
  RouterShape s;
  if (!choose(d_in, K, &s)) return cudaErrorNotSupported;
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
                       static_cast<const __nv_bfloat16*>(W2), b1, b2, K, k, logits, ids, w, (int32_t)s.C,
                       (int32_t)s.KS, (int32_t)s.XR, (uint32_t)s.off_w1, (uint32_t)s.off_recv, (uint32_t)s.off_w2,
                       (uint32_t)s.region, map_x, map_w1);
}

}  // namespace molora
