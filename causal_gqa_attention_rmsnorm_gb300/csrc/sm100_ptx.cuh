// Thin inline-PTX wrappers for sm_100-family features used by the bf16 path:
// mbarriers, TMA tensor loads, tcgen05 MMA / TMEM, and a globaltimer-bounded
// mbarrier wait.  Written from the PTX ISA's descriptions of these
// instructions; every wait gives up after kWaitLimitNs and reports it.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "../../include/tb.h"

namespace tb {
namespace ptx {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make initialised barriers visible to the async (TMA / tensor) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase of parity `parity` has completed.  Gives up when
// another thread of the CTA has raised *abort, or after kWaitLimitNs, in which
// case it raises *abort and sets TB_DEVERR_TIMEOUT in the device error word.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        *abort = 1;
        atomicOr(err, TB_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Poll the counter at p (global memory, written by other CTAs) until it
// reaches target, for at most limit_ns; false when it did not.  No error is
// raised: the caller has another way to its result.
__device__ __forceinline__ bool poll_count(const int* p, int target, uint64_t limit_ns) {
  auto load = [p]() {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
  };
  if (load() >= target) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
    __nanosleep(128);
    if (load() >= target) return true;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// mbar_wait for roles where the whole warp proceeds together (warp-collective
// tcgen05.ld/st and votes follow): every lane waits, and the warp continues only
// if all lanes saw the phase complete, so a time-out never splits the warp.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort, int* err) {
  const bool ok = mbar_wait(bar, parity, abort, err);
  return __all_sync(0xffffffffu, ok);
}

// Pull [p, p + bytes) into L2 (p 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

// Part i of n of the 16-byte units of [p, p + bytes), pulled into L2 in pieces
// of at most 64 KB.
__device__ __forceinline__ void prefetch_l2_part(const void* p, unsigned long long bytes, int i, int n) {
  const unsigned long long units = bytes >> 4, per = (units + (unsigned long long)n - 1) / (unsigned long long)n;
  unsigned long long u = per * (unsigned long long)i;
  const unsigned long long end = u + per < units ? u + per : units;
  for (; u < end; u += 4096) {
    const unsigned long long len = end - u < 4096 ? end - u : 4096;
    prefetch_l2_bulk(static_cast<const uint8_t*>(p) + (u << 4), (uint32_t)(len << 4));
  }
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled TMA load of the box at (x, y) = (inner, outer) into smem; the
// transaction bytes complete on `bar`.
__device__ __forceinline__ void tma_load_2d(const CUtensorMap* m, void* dst, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// 3-D tiled TMA load of the box at (x, y, z).
__device__ __forceinline__ void tma_load_3d(const CUtensorMap* m, void* dst, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Untiled bulk copy of `bytes` bytes (a multiple of 16; both addresses 16-byte
// aligned) from global memory into smem; the bytes complete on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(static_cast<uint64_t>(__cvta_generic_to_global(src))), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 policy for data read once per call (streamed weights, the KV cache):
// evicted first, so that what the next kernel reads back (partial sums,
// activations) stays in L2.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// tma_load_2d / tma_load_3d / bulk_load with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(const CUtensorMap* m, void* dst, uint64_t* bar, int x, int y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_hint(const CUtensorMap* m, void* dst, uint64_t* bar, int x, int y, int z,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(static_cast<uint64_t>(__cvta_generic_to_global(src))), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 2^x on the special-function unit (flush-to-zero; -inf gives 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction (three-input form of max.f32).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// ---- tcgen05 -------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] · B[smem desc]ᵀ, kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Batched issue of the MMAs of one tile, for an issuing thread that must spend
// as few instructions per MMA as possible: descriptors are passed as their low
// and high 32-bit words, each MMA's operand offset is an immediate added to the
// low word (the address field never carries into the high word below 256 KB of
// shared memory), and one predicate serves every MMA after the first.
//
// S += Q·Kᵀ over dh = 16·NK: both operands K-major with the 128-byte swizzle,
// 64-element column blocks 16 KB apart (128 rows of 128 bytes).
#define TB_MMA_SS_STEP(OFF, PRED)                                              \
  "add.u32 la, %1, " #OFF ";\n\t"                                             \
  "add.u32 lb, %3, " #OFF ";\n\t"                                             \
  "mov.b64 da, {la, %2};\n\t"                                                 \
  "mov.b64 db, {lb, %4};\n\t"                                                 \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, " #PRED ";\n\t"
template <int NK>
__device__ __forceinline__ void mma_tile_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
  static_assert(NK == 4 || NK == 8, "dh 64 or 128");
  const uint32_t alo = (uint32_t)adesc, ahi = (uint32_t)(adesc >> 32);
  const uint32_t blo = (uint32_t)bdesc, bhi = (uint32_t)(bdesc >> 32);
  if constexpr (NK == 4) {
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b32 la, lb;\n\t.reg .b64 da, db;\n\t"
        "setp.ne.b32 pf, 0, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
        TB_MMA_SS_STEP(0, pf) TB_MMA_SS_STEP(2, pt) TB_MMA_SS_STEP(4, pt) TB_MMA_SS_STEP(6, pt) "}" ::"r"(d_tmem),
        "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b32 la, lb;\n\t.reg .b64 da, db;\n\t"
        "setp.ne.b32 pf, 0, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
        TB_MMA_SS_STEP(0, pf) TB_MMA_SS_STEP(2, pt) TB_MMA_SS_STEP(4, pt) TB_MMA_SS_STEP(6, pt)
        TB_MMA_SS_STEP(1024, pt) TB_MMA_SS_STEP(1026, pt) TB_MMA_SS_STEP(1028, pt) TB_MMA_SS_STEP(1030, pt) "}" ::"r"(d_tmem),
        "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc)
        : "memory");
  }
}
#undef TB_MMA_SS_STEP

// O (+)= P·V over 128 keys: P (bf16 pairs) in tensor memory at a_tmem, 8
// columns per 16 keys; V MN-major with 16-key slices 2 KB apart.  `acc` = 0
// overwrites O with the first slice's product.
#define TB_MMA_TS_STEP(K, PRED)                                                \
  "add.u32 ta, %1, " #K "*8;\n\t"                                             \
  "add.u32 lb, %2, " #K "*128;\n\t"                                           \
  "mov.b64 db, {lb, %3};\n\t"                                                 \
  "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], db, %4, " #PRED ";\n\t"
__device__ __forceinline__ void mma_tile_ts128(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t acc) {
  const uint32_t blo = (uint32_t)bdesc, bhi = (uint32_t)(bdesc >> 32);
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b32 ta, lb;\n\t.reg .b64 db;\n\t"
      "setp.ne.b32 pf, %5, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
      TB_MMA_TS_STEP(0, pf) TB_MMA_TS_STEP(1, pt) TB_MMA_TS_STEP(2, pt) TB_MMA_TS_STEP(3, pt)
      TB_MMA_TS_STEP(4, pt) TB_MMA_TS_STEP(5, pt) TB_MMA_TS_STEP(6, pt) TB_MMA_TS_STEP(7, pt) "}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc)
      : "memory");
}
#undef TB_MMA_TS_STEP

// Arrive on `bar` once every tcgen05 op this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 lanes × 16 consecutive 32-bit columns: thread i gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// 32 lanes × 8 consecutive 32-bit columns: thread i gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
// 32 lanes × 8 consecutive 32-bit columns from registers into TMEM.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
      "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a tile whose rows are 128 bytes with the
// 128-byte swizzle, 8-row core groups 1024 bytes apart (K-major operand).
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                  // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024u >> 4) << 32;       // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;                  // descriptor version for sm_100
  d |= (uint64_t)2 << 61;                  // 128-byte swizzle
  return d;
}

// Descriptor of an MN-major operand tile stored as 128-byte rows along MN,
// swizzled, with K rows 128 bytes apart: 8-row K groups are `sbo` bytes apart
// and 64-element MN blocks `lbo` bytes apart.
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A and B, fp32 D.
// a_mn / b_mn select MN-major operands (transposed in the descriptor).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn = false, bool b_mn = false) {
  return (1u << 4)                          // D format: f32
         | (1u << 7)                        // A format: bf16
         | (1u << 10)                       // B format: bf16
         | ((a_mn ? 1u : 0u) << 15)         // A major-ness
         | ((b_mn ? 1u : 0u) << 16)         // B major-ness
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// ---- CTA pairs (cta_group::2) --------------------------------------------
//
// Two CTAs of a cluster share each tensor-core operation: an M = 256 MMA
// issued by the even CTA (the leader) takes A rows 0..127 from the leader's
// shared memory or tensor memory and rows 128..255 from its peer's, B columns
// 0..N/2-1 from the leader and N/2..N-1 from the peer, and writes D rows
// 0..127 into the leader's tensor memory and 128..255 into the peer's, all at
// the same addresses in both CTAs.  Tensor memory is allocated by one warp in
// each CTA of the pair together.

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Shared::cluster address of the object at shared::cta address `a` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
// Loads from the shared memory of a CTA of the cluster, at a shared::cluster
// address (mapa_shared).
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
// Every thread of every CTA of the cluster: release this CTA's prior writes,
// wait for the others.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier of either CTA, given its shared::cluster address.
// What the arrival publishes is tensor-memory data, ordered by the tcgen05
// fences around the barrier, so the default (CTA-scope) release suffices.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// mbar_wait for barriers that threads of the peer CTA arrive on (acquire at
// cluster scope); same time limit and abort protocol.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort, int* err) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait_cluster(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(a, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        *abort = 1;
        atomicOr(err, TB_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait_cluster_warp(uint64_t* bar, uint32_t parity, volatile int* abort, int* err) {
  const bool ok = mbar_wait_cluster(bar, parity, abort, err);
  return __all_sync(0xffffffffu, ok);
}
// 3-D tiled TMA load into this CTA's shared memory whose bytes complete on the
// mbarrier at shared::cluster address `bar_cluster`, which may be the peer's.
__device__ __forceinline__ void tma_load_3d_pair(const CUtensorMap* m, void* dst, uint32_t bar_cluster, int x, int y,
                                                 int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// 2-D variant of tma_load_3d_pair.
__device__ __forceinline__ void tma_load_2d_pair(const CUtensorMap* m, void* dst, uint32_t bar_cluster, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
// One pair MMA (M = 256 across the two CTAs), both operands in shared memory.
__device__ __forceinline__ void mma2_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Arrive once on the mbarrier at the same shared::cta address in both CTAs of
// the pair when every pair MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}

// Pair S += Q·Kᵀ over dh = 128: A (Q, 128 rows per CTA) K-major, 64-column
// blocks 16 KB apart; B (K, 64 key rows per CTA) K-major, blocks 8 KB apart.
#define TB_MMA2_SS_STEP(OA, OB, PRED)                                          \
  "add.u32 la, %1, " #OA ";\n\t"                                             \
  "add.u32 lb, %3, " #OB ";\n\t"                                             \
  "mov.b64 da, {la, %2};\n\t"                                                 \
  "mov.b64 db, {lb, %4};\n\t"                                                 \
  "tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %5, " #PRED ";\n\t"
__device__ __forceinline__ void mma2_tile_ss128(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc) {
  const uint32_t alo = (uint32_t)adesc, ahi = (uint32_t)(adesc >> 32);
  const uint32_t blo = (uint32_t)bdesc, bhi = (uint32_t)(bdesc >> 32);
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b32 la, lb;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.b32 pf, 0, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
      TB_MMA2_SS_STEP(0, 0, pf) TB_MMA2_SS_STEP(2, 2, pt) TB_MMA2_SS_STEP(4, 4, pt) TB_MMA2_SS_STEP(6, 6, pt)
      TB_MMA2_SS_STEP(1024, 512, pt) TB_MMA2_SS_STEP(1026, 514, pt) TB_MMA2_SS_STEP(1028, 516, pt)
      TB_MMA2_SS_STEP(1030, 518, pt) "}" ::"r"(d_tmem),
      "r"(alo), "r"(ahi), "r"(blo), "r"(bhi), "r"(idesc)
      : "memory");
}
#undef TB_MMA2_SS_STEP

// Pair O (+)= P·V over 128 keys: P (bf16 pairs) in tensor memory, 8 columns
// per 16 keys; V (64 value columns per CTA) MN-major, 16-key slices 2 KB apart.
#define TB_MMA2_TS_STEP(K, PRED)                                               \
  "add.u32 ta, %1, " #K "*8;\n\t"                                             \
  "add.u32 lb, %2, " #K "*128;\n\t"                                           \
  "mov.b64 db, {lb, %3};\n\t"                                                 \
  "tcgen05.mma.cta_group::2.kind::f16 [%0], [ta], db, %4, " #PRED ";\n\t"
__device__ __forceinline__ void mma2_tile_ts128(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                uint32_t acc) {
  const uint32_t blo = (uint32_t)bdesc, bhi = (uint32_t)(bdesc >> 32);
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b32 ta, lb;\n\t.reg .b64 db;\n\t"
      "setp.ne.b32 pf, %5, 0;\n\tsetp.eq.b32 pt, 0, 0;\n\t"
      TB_MMA2_TS_STEP(0, pf) TB_MMA2_TS_STEP(1, pt) TB_MMA2_TS_STEP(2, pt) TB_MMA2_TS_STEP(3, pt)
      TB_MMA2_TS_STEP(4, pt) TB_MMA2_TS_STEP(5, pt) TB_MMA2_TS_STEP(6, pt) TB_MMA2_TS_STEP(7, pt) "}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc)
      : "memory");
}
#undef TB_MMA2_TS_STEP

}  // namespace ptx
}  // namespace tb
