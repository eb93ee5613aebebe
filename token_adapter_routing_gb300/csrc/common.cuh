// common.cuh -- shared device helpers for the sm_103a kernels: inline PTX for mbarriers,
// cp.async, bulk async copies / reductions, TMA, thread-block clusters and tcgen05 (5th-gen
// tensor cores with TMEM accumulators).  Every on-chip wait here is bounded in time.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "molora.h"

namespace molora {

constexpr int kMaxAdapters = MOLORA_MAX_ADAPTERS;
constexpr int kRouterHidden = MOLORA_ROUTER_HIDDEN;
// Bounded waits give up after this many nanoseconds (then report MOLORA_DEV_WAIT_TIMEOUT).
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;

__device__ __forceinline__ void report(int32_t* err_word, int32_t bits) {
  if (err_word) atomicOr(err_word, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ programmatic dependent launch
// Every kernel here is launched with programmatic stream serialization: it may start while the
// previous kernel in the stream is still running, does only work that reads none of that
// kernel's outputs, then waits for it (griddepcontrol.wait: the previous grid has completed and
// its memory is visible) and lets the next kernel begin its own prologue.  Without a
// programmatic predecessor both instructions are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity to complete; false if `limit_ns` ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// As mbar_wait, but also gives up as soon as *abort is set by another thread of the CTA, and
// sets *abort itself when the time limit runs out, so that one failed wait ends every other
// role's waits promptly instead of each running out its own limit.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity, volatile int32_t* abort,
                                                   uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      return false;
    }
  }
}

// ------------------------------------------------------------------ cp.async (16 B, L2 only)
// src_bytes < 16 zero-fills the rest of the 16 destination bytes (0 = pure zero fill).
__device__ __forceinline__ void cp_async_16(uint32_t sdst, const void* gsrc, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sdst), "l"(gsrc), "r"(src_bytes)
               : "memory");
}
// An L2 policy that makes the lines it touches the first to be evicted: for data read exactly
// once (x), so that it does not push out lines that are still to be used (y prefetched ahead).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// cp_async_16 under an L2 cache policy (l2_policy_evict_first).
__device__ __forceinline__ void cp_async_16_hint(uint32_t sdst, const void* gsrc, uint32_t src_bytes, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(sdst), "l"(gsrc),
               "r"(src_bytes), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// One arrival on `bar` once every cp.async this thread issued so far has landed (the
// barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Wait until at most N committed cp.async groups of this thread are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ proxies / bulk async
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// y[gdst .. gdst+bytes) += smem[ssrc .. ssrc+bytes) as fp32, performed in L2 by the TMA unit.
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst),
               "r"(ssrc), "r"(bytes)
               : "memory");
}
// The same for bf16 elements: each destination element becomes the bf16 sum of itself and
// the staged bf16 value.
__device__ __forceinline__ void bulk_reduce_add_bf16(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.noftz.bf16 [%0], [%1], %2;" ::"l"(gdst),
               "r"(ssrc), "r"(bytes)
               : "memory");
}
// *gdst += v, four consecutive fp32, as one L2 reduction (no value returned).
__device__ __forceinline__ void red_add_v4(float* gdst, float4 v) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(gdst), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N committed bulk groups of this thread still READ shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// bulk_wait_read<n> for a run-time n in 0..7 (larger values wait as for 7).
__device__ __forceinline__ void bulk_wait_read_upto(int n) {
  switch (n) {
    case 0: bulk_wait_read<0>(); break;
    case 1: bulk_wait_read<1>(); break;
    case 2: bulk_wait_read<2>(); break;
    case 3: bulk_wait_read<3>(); break;
    case 4: bulk_wait_read<4>(); break;
    case 5: bulk_wait_read<5>(); break;
    case 6: bulk_wait_read<6>(); break;
    default: bulk_wait_read<7>(); break;
  }
}

// ------------------------------------------------------------------ TMA (tensor maps)
__device__ __forceinline__ void tma_load_2d(uint32_t sdst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(sdst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}
// As tma_load_2d, but the box lands at the same shared-memory offset in every CTA of
// `cta_mask` (this cluster's ranks), each counting the bytes on its own mbarrier at bar's offset.
__device__ __forceinline__ void tma_load_2d_multicast(uint32_t sdst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                                      uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster "
      "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(sdst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "h"(cta_mask)
      : "memory");
}
// smem box -> global through a tensor map, each element ADDED to the destination (the
// element type of the map: fp32 add for a FLOAT32 map); rows and columns outside the tensor
// are skipped.  Completes as a bulk group of the issuing thread.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t ssrc, int32_t c0, int32_t c1) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(ssrc)
               : "memory");
}
// Asks L2 to fetch one box of a tensor map (no shared memory involved, no completion).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t c0, int32_t c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ clusters / DSMEM
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}
// Address of the same shared-memory variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local_saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_saddr), "r"(rank));
  return r;
}
// One fp32 store into CTA-cluster shared memory (address from dsmem_addr).
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float4 dsmem_ld_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}
// 16 bytes into CTA-cluster shared memory (address from dsmem_addr); completes `bytes` of
// the transaction count of the mbarrier at `remote_bar` (a cluster address too).
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint4 v, uint32_t remote_bar) {
  asm volatile("st.async.weak.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
               : "memory");
}
// `bytes` (a multiple of 16) from global memory (16-byte aligned) into this CTA's shared memory
// (16-byte aligned), counted on the mbarrier `bar` of this CTA.
__device__ __forceinline__ void bulk_load_g2s(uint32_t sdst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(sdst),
               "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// `bytes` (a multiple of 16) from this CTA's shared memory to CTA-cluster shared memory (a
// dsmem_addr address, 16-byte aligned), counted on the mbarrier at `remote_bar` (a cluster address).
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t remote_bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "r"(src), "r"(bytes), "r"(remote_bar)
               : "memory");
}
// Named barrier over `count` threads (a multiple of 32) of this CTA; threads of one warp
// may arrive separately (non-.aligned form).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Asks L2 to fetch [gptr, gptr + bytes) ahead of use (bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* gptr, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gptr), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ tcgen05 / TMEM
// Allocation is warp-collective; the TMEM base address is written to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bf16/fp16 inputs, fp32 accumulate; issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on *bar when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// As umma_commit, arriving on the mbarrier at bar's offset in every CTA of `cta_mask`.
__device__ __forceinline__ void umma_commit_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(cta_mask)
               : "memory");
}

// Loads 16 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per thread) and
// waits for the load, so the registers are valid on return.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Loads 32 consecutive fp32 columns of this warp's 32 TMEM lanes and waits for the load.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// tcgen05.ld of 32 consecutive fp32 columns of this warp's 32 TMEM lanes WITHOUT waiting: the
// registers are not valid until tmem_ld_wait() has run on them.  Several loads may be in flight.
__device__ __forceinline__ void tmem_ld32_start(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// Waits for every tcgen05.ld this thread issued; the registers of `r` are read-write operands, so
// no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
// Binds a second register block to the same completed wait (a wait covers every load issued
// before it): marks `r` as produced here without waiting again.
__device__ __forceinline__ void tmem_ld_bind(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma (sm_100 family layout):
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-47  descriptor version (1)
//   bits 49-51  base offset (0: every swizzled tile here starts on its swizzle-span boundary)
//   bits 61-63  layout: 0 none, 2 128B swizzle, 4 64B swizzle, 6 32B swizzle
enum SmemLayout : uint32_t { kSwizzleNone = 0, kSwizzle128B = 2, kSwizzle64B = 4, kSwizzle32B = 6 };

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              SmemLayout layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)layout << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format (1 = bf16),
//   bit 15 A major (0 = K-major), bit 16 B major (1 = MN-major), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Byte offset of the 16-byte chunk `chunk` (0..7) of row `row` inside a K-major tile whose
// rows are 128 bytes and which uses the 128-byte swizzle (8-row, 1024-byte atoms).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a K-major tile whose rows are
// `row_bytes` long (32, 64 or 128) and which uses the swizzle of that width (8-row atoms):
// the chunk index is XOR-ed with the row bits that sit at address bits 7.. of the atom.
__device__ __forceinline__ uint32_t swz_offset(uint32_t row, uint32_t chunk, uint32_t row_bytes) {
  const uint32_t f = row_bytes == 32 ? (row >> 2) & 1u : (row_bytes == 64 ? (row >> 1) & 3u : row & 7u);
  return row * row_bytes + ((chunk ^ f) << 4);
}

// The learned router's second stage (Table 1's O(64K) part; Table 10's softmax gating; Figure
// 2's top-k) for `rows` consecutive tokens starting at t_first, eight lanes per token (nthreads a
// multiple of 32).  recv holds C partial hidden vectors per token, source-major: source cc, row
// rl at recv + (cc * rows + rl) * stride + col0, 64 floats; with `swz` its 16-byte chunks are
// stored at chunk ^ (rl & 7) (the layout a conflict-free staging store leaves).
//   hidden  h = ReLU(sum over sources in rank order + b1); lane g of a token sums units 8g..8g+7
//           and hands them to the token's other lanes by shuffles;
//   logits  lane g owns logits a = g + 8j (j < JL = ceil(K / 8)); each is eight group partials
//           (an fmaf chain over the group's 8 units, from 0) added in group order, then b2;
//   top k   k rounds of an 8-lane butterfly on (logit, index): larger logit wins, equal logits
//           keep the lower index (the result of a sequential strictly-greater scan);
//   softmax over the k, shifted by the largest: e_j = exp(l_j - l_0), denominator summed in
//           selection order, w_j = e_j * (1 / denominator).
// The arithmetic, and so every bit of the results, does not depend on the lane mapping.
// Stores logits (if non-null and `store`), ids and w for tokens t < N when `ok`; writes the
// token's coefficients coef[rl * K + a] (0 for unselected adapters) when coef is non-null.
// JL is a template parameter so that no lane issues work for logits it does not own.
template <int JL, int RPT>
__device__ __forceinline__ void router_rows_jl(const float* recv, int C, int rows, int stride, int col0, bool swz,
                                               const float* w2s, const float* b1s, const float* b2s, int K, int k,
                                               int64_t t_first, int64_t N, bool ok, float* logits, int32_t* ids,
                                               float* w, float* coef, int tid, int nthreads, bool store) {
  const int lane = tid & 31, g = lane & 7, gbase = lane & ~7;
  // each thread carries RPT tokens at once (items tid, tid + nthreads, ...): independent chains
  for (int base = 0; base < rows * 8; base += nthreads * RPT) {  // warp-uniform trip count
    int rl[RPT];
    bool valid[RPT];
    float hg[RPT][8];
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
      const int item = base + q * nthreads + tid;
      rl[q] = item >> 3;
      valid[q] = item < rows * 8;
#pragma unroll
      for (int i = 0; i < 8; ++i) hg[q][i] = 0.f;
      if (valid[q]) {
        const int c0 = swz ? (2 * g) ^ (rl[q] & 7) : 2 * g, c1 = swz ? (2 * g + 1) ^ (rl[q] & 7) : 2 * g + 1;
        for (int cc = 0; cc < C; ++cc) {
          const float4* src = reinterpret_cast<const float4*>(recv + ((size_t)cc * rows + rl[q]) * stride + col0);
          const float4 p0 = src[c0], p1 = src[c1];
          hg[q][0] += p0.x, hg[q][1] += p0.y, hg[q][2] += p0.z, hg[q][3] += p0.w;
          hg[q][4] += p1.x, hg[q][5] += p1.y, hg[q][6] += p1.z, hg[q][7] += p1.w;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) hg[q][i] = fmaxf(hg[q][i] + b1s[g * 8 + i], 0.f);
      }
    }
    // logits g + 8j: group gg's units come from lane gg of the token (8 shuffles), then each
    // logit's chain over them is added to its running sum (group order)
    bool own[RPT][JL];
    float lv[RPT][JL];
#pragma unroll
    for (int q = 0; q < RPT; ++q)
#pragma unroll
      for (int j = 0; j < JL; ++j) own[q][j] = valid[q] && g + 8 * j < K, lv[q][j] = 0.f;
#pragma unroll(JL <= 2 ? 4 : 1)
    for (int gg = 0; gg < 8; ++gg) {
#pragma unroll
      for (int q = 0; q < RPT; ++q) {
        float hc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) hc[i] = __shfl_sync(0xffffffffu, hg[q][i], gbase | gg);
#pragma unroll
        for (int j = 0; j < JL; ++j) {
          if (own[q][j]) {
            const float* wc = w2s + (gg * 8) * K + g + 8 * j;
            float sg = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) sg = fmaf(hc[i], wc[i * K], sg);
            lv[q][j] = gg == 0 ? sg : lv[q][j] + sg;
          }
        }
      }
    }
    int64_t t[RPT];
    bool out[RPT];
#pragma unroll
    for (int q = 0; q < RPT; ++q) {
#pragma unroll
      for (int j = 0; j < JL; ++j)
        if (own[q][j]) lv[q][j] += b2s[g + 8 * j];
      t[q] = t_first + rl[q];
      out[q] = valid[q] && t[q] < N && ok;
      if (coef)
#pragma unroll
        for (int j = 0; j < JL; ++j)
          if (own[q][j]) coef[rl[q] * K + g + 8 * j] = 0.f;
      if (out[q] && logits && store)
#pragma unroll
        for (int j = 0; j < JL; ++j)
          if (own[q][j]) logits[t[q] * K + g + 8 * j] = lv[q][j];
    }
    __syncwarp();  // the zeroed coefficients before the selected ones
    // One selection round for token q: its best unselected logit, known to all 8 lanes.
    uint32_t used[RPT];  // bit j: logit g + 8j already selected
    auto select = [&](int q, float& bv, int& bi) {
      bv = 0.f, bi = -1;
#pragma unroll
      for (int j = 0; j < JL; ++j)
        if (own[q][j] && !((used[q] >> j) & 1u) && (bi < 0 || lv[q][j] > bv)) bv = lv[q][j], bi = g + 8 * j;
#pragma unroll
      for (int off = 1; off < 8; off <<= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (oi >= 0 && (bi < 0 || ov > bv || (ov == bv && oi < bi))) bv = ov, bi = oi;
      }
      if (bi >= 0 && (bi & 7) == g) used[q] |= 1u << (bi >> 3);
    };
    float m[RPT], denom[RPT];
#pragma unroll
    for (int q = 0; q < RPT; ++q) m[q] = 0.f, denom[q] = 0.f, used[q] = 0;
    if (k <= 8) {  // lane g keeps slot g: one selection pass
      float my_e[RPT];
      int my_i[RPT];
#pragma unroll
      for (int q = 0; q < RPT; ++q) my_e[q] = 0.f, my_i[q] = 0;
      for (int js = 0; js < k; ++js) {
#pragma unroll
        for (int q = 0; q < RPT; ++q) {
          float bv;
          int bi;
          select(q, bv, bi);
          if (js == 0) m[q] = bv;
          const float e = expf(bv - m[q]);
          denom[q] += e;
          if (js == g) my_e[q] = e, my_i[q] = bi;
        }
      }
#pragma unroll
      for (int q = 0; q < RPT; ++q) {
        if (out[q] && g < k) {
          const float wj = my_e[q] * (1.f / denom[q]);
          if (store) {
            ids[t[q] * k + g] = my_i[q];
            w[t[q] * k + g] = wj;
          }
          if (coef) coef[rl[q] * K + my_i[q]] = wj;
        }
      }
    } else {  // the selection runs twice (denominator, then weights)
      for (int pass = 0; pass < 2; ++pass) {
        float inv[RPT];
#pragma unroll
        for (int q = 0; q < RPT; ++q) inv[q] = pass ? 1.f / denom[q] : 0.f, used[q] = 0;
        for (int js = 0; js < k; ++js) {
#pragma unroll
          for (int q = 0; q < RPT; ++q) {
            float bv;
            int bi;
            select(q, bv, bi);
            if (js == 0) m[q] = bv;
            const float e = expf(bv - m[q]);
            if (pass == 0) {
              denom[q] += e;
            } else if (out[q] && g == (js & 7)) {
              const float wj = e * inv[q];
              if (store) {
                ids[t[q] * k + js] = bi;
                w[t[q] * k + js] = wj;
              }
              if (coef) coef[rl[q] * K + bi] = wj;
            }
          }
        }
      }
    }
  }
}

// Chooses the instantiation: logits per lane from K, and two tokens per thread when the rows
// need more than one pass of the threads and K <= 8 (the registers allow it there).
__device__ __forceinline__ void router_rows(const float* recv, int C, int rows, int stride, int col0, bool swz,
                                            const float* w2s, const float* b1s, const float* b2s, int K, int k,
                                            int64_t t_first, int64_t N, bool ok, float* logits, int32_t* ids,
                                            float* w, float* coef, int tid, int nthreads, bool store = true) {
  if (K <= 8 && rows * 8 > nthreads)
    router_rows_jl<1, 2>(recv, C, rows, stride, col0, swz, w2s, b1s, b2s, K, k, t_first, N, ok, logits, ids, w,
                         coef, tid, nthreads, store);
  else if (K <= 8)
    router_rows_jl<1, 1>(recv, C, rows, stride, col0, swz, w2s, b1s, b2s, K, k, t_first, N, ok, logits, ids, w,
                         coef, tid, nthreads, store);
  else if (K <= 16)
    router_rows_jl<2, 1>(recv, C, rows, stride, col0, swz, w2s, b1s, b2s, K, k, t_first, N, ok, logits, ids, w,
                         coef, tid, nthreads, store);
  else if (K <= 32)
    router_rows_jl<4, 1>(recv, C, rows, stride, col0, swz, w2s, b1s, b2s, K, k, t_first, N, ok, logits, ids, w,
                         coef, tid, nthreads, store);
  else
    router_rows_jl<8, 1>(recv, C, rows, stride, col0, swz, w2s, b1s, b2s, K, k, t_first, N, ok, logits, ids, w,
                         coef, tid, nthreads, store);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

}  // namespace molora
