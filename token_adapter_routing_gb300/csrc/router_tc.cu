// router_tc.cu -- the learned router TopK(g(x)) of "MoLoRA: Composable Specialization via
// Per-Token Adapter Routing" (Table 1: routing cost O(64d + 64K); Figure 2: top-k adapters
// combined by a weighted sum; Table 10: softmax(Wx + b) gating) on tcgen05 tensor cores.
//
// The d_in x 64 projection is the only dense contraction (64 flops per byte of x), so it
// runs as a tcgen05 GEMM: a cluster of C CTAs owns 128 consecutive tokens and splits d_in;
// each CTA TMA-loads its x tile (K-major, 128-byte swizzle) and the matching W1 rows
// (MN-major), accumulates 128 x 64 fp32 partials in TMEM, and the partials are summed
// through distributed shared memory in a fixed order.  Each CTA then finishes 128/C of the
// tokens on CUDA cores: ReLU, the 64 x K second layer, top-k selection (strictly greater
// wins, so equal logits keep the lower index) and the softmax renormalised over the k.
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
constexpr uint32_t kPStride = kRouterHidden * 4 + 16;
constexpr size_t kMaxSmem = 227 * 1024;

struct RouterShape {
  int C, KS;
  size_t off_w1, off_w2, region, smem;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool plan(int32_t d_in, int32_t K, int C, RouterShape* s) {
  if (d_in % (C * kKBlock) || kTileM % C) return false;
  s->C = C;
  s->KS = d_in / C;
  s->off_w1 = (size_t)s->KS * kTileM * 2;
  const size_t phase1 = s->off_w1 + (size_t)s->KS * kRouterHidden * 2;
  const size_t phase2 = (size_t)kTileM * kPStride;
  s->off_w2 = align_up(phase1 > phase2 ? phase1 : phase2, 1024);
  // W2 as fp32 [64 x K], b1 [64], b2 [K], per-row logits [128/C x K]
  s->region = s->off_w2 + sizeof(float) * ((size_t)kRouterHidden * K + kRouterHidden + K + (kTileM / C) * K);
  s->region = align_up(s->region, 1024);
  s->smem = s->region + 1024 + 256;
  return s->smem <= kMaxSmem;
}

bool choose(int32_t d_in, int32_t K, RouterShape* s) {
  for (int C : {8, 4, 2, 1})
    if (plan(d_in, K, C, s)) return true;
  return false;
}

struct __align__(8) RCtrl {
  uint64_t bar_load;
  uint64_t bar_mma;
  uint32_t tmem_base;
  int32_t abort;
};

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(int64_t N, int32_t d_in, const __nv_bfloat16* __restrict__ W2, const float* __restrict__ b1,
                     const float* __restrict__ b2, int32_t K, int32_t k, float* __restrict__ logits,
                     int32_t* __restrict__ ids, float* __restrict__ w, int32_t C, int32_t KS, uint32_t off_w1,
                     uint32_t off_w2, uint32_t region, const __grid_constant__ CUtensorMap map_x,
                     const __grid_constant__ CUtensorMap map_w1) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  RCtrl* ctrl = reinterpret_cast<RCtrl*>(sm + region);
  uint8_t* xs = sm;
  uint8_t* w1s = sm + off_w1;
  uint8_t* ps = sm;  // partial hidden, after the MMA has consumed x
  float* w2s = reinterpret_cast<float*>(sm + off_w2);
  float* b1s = w2s + kRouterHidden * K;
  float* b2s = b1s + kRouterHidden;
  float* lgs = b2s + K;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int crank = (int)cluster_ctarank();
  const int64_t tile = blockIdx.x / C;
  const int64_t t0 = tile * kTileM;
  const int nkb = KS / kKBlock;

  if (warp == 4) {
    tmem_alloc(&ctrl->tmem_base, kTmemCols);
    tmem_relinquish();
    if (lane == 0) {
      mbar_init(&ctrl->bar_load, 1);
      mbar_init(&ctrl->bar_mma, 1);
      ctrl->abort = 0;
      mbar_fence_init();
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

  if (warp == 4 && lane == 0) {
    mbar_arrive_expect_tx(&ctrl->bar_load, (uint32_t)KS * (kTileM + kRouterHidden) * 2);
    for (int kb = 0; kb < nkb; ++kb) {
      const int32_t col = crank * KS + kb * kKBlock;
      tma_load_2d(smem_u32(xs + (size_t)kb * kTileM * 128), &map_x, col, (int32_t)t0, &ctrl->bar_load);
      tma_load_2d(smem_u32(w1s + (size_t)kb * kKBlock * 128), &map_w1, 0, col, &ctrl->bar_load);
    }
    const bool ok = mbar_wait(&ctrl->bar_load, 0);
    tc_fence_after();
    if (ok) {
      const uint32_t idesc = idesc_bf16_f32(kTileM, kRouterHidden, false, true);
      for (int kb = 0; kb < nkb; ++kb)
        for (int ks = 0; ks < kKBlock / 16; ++ks) {
          const uint64_t da = smem_desc(smem_u32(xs + (size_t)kb * kTileM * 128 + ks * 32), 16, 1024, kSwizzle128B);
          const uint64_t db =
              smem_desc(smem_u32(w1s + (size_t)kb * kKBlock * 128 + ks * 2048), 1024, 1024, kSwizzle128B);
          umma_f16(tmem, da, db, idesc, (kb | ks) != 0);
        }
      umma_commit(&ctrl->bar_mma);
    } else {
      ctrl->abort = 1;
      mbar_arrive(&ctrl->bar_mma);
    }
  }
  bool timed_out = false;
  if (warp < 4) {
    const bool ok = mbar_wait(&ctrl->bar_mma, 0);
    tc_fence_after();
    if (ok && !ctrl->abort) {
      float v[16];
      float* prow = reinterpret_cast<float*>(ps + tid * kPStride);
      for (int c0 = 0; c0 < kRouterHidden; c0 += 16) {
        tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<float4*>(prow + c0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      }
    } else {
      timed_out = true;
    }
    tc_fence_before();
  }
  __syncwarp();
  cluster_sync();

  const int rows_per = kTileM / C;
  if (tid < rows_per) {
    const int row = crank * rows_per + tid;
    const int64_t t = t0 + row;
    if (t < N && !timed_out) {
      float h[kRouterHidden];
#pragma unroll
      for (int j = 0; j < kRouterHidden; ++j) h[j] = 0.f;
      const uint32_t mine = smem_u32(ps + row * kPStride);
      for (int cc = 0; cc < C; ++cc) {
        const uint32_t src = dsmem_addr(mine, (uint32_t)cc);
#pragma unroll
        for (int j = 0; j < kRouterHidden; j += 4) {
          const float4 p = dsmem_ld_f4(src + j * 4);
          h[j] += p.x, h[j + 1] += p.y, h[j + 2] += p.z, h[j + 3] += p.w;
        }
      }
#pragma unroll
      for (int j = 0; j < kRouterHidden; ++j) h[j] = fmaxf(h[j] + b1s[j], 0.f);
      float* lg = lgs + tid * K;
      for (int a = 0; a < K; ++a) {
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < kRouterHidden; ++j) s = fmaf(h[j], w2s[j * K + a], s);
        s += b2s[a];
        lg[a] = s;
        if (logits) logits[t * K + a] = s;
      }
      uint64_t used = 0;
      float m = 0.f, denom = 0.f;
      float e[kMaxAdapters];
      int sel[kMaxAdapters];
      for (int js = 0; js < k; ++js) {
        int best = -1;
        for (int a = 0; a < K; ++a)
          if (!((used >> a) & 1ull) && (best < 0 || lg[a] > lg[best])) best = a;
        used |= 1ull << best;
        if (js == 0) m = lg[best];
        sel[js] = best;
        e[js] = expf(lg[best] - m);
        denom += e[js];
      }
      const float inv = 1.f / denom;
      for (int js = 0; js < k; ++js) {
        ids[t * k + js] = sel[js];
        w[t * k + js] = e[js] * inv;
      }
    }
  }
  __syncwarp();
  cluster_arrive();
  cluster_wait();
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
                       (int32_t)s.KS, (uint32_t)s.off_w1, (uint32_t)s.off_w2, (uint32_t)s.region, map_x, map_w1);
}

}  // namespace molora
