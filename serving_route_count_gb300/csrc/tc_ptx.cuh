// tc_ptx.cuh - inline-PTX wrappers for the Blackwell (sm_103a) data path: mbarriers, TMA
// (cp.async.bulk.tensor), bulk copies, tcgen05 TMEM allocation / copies / MMA / loads.
// Every wait is bounded: after kTimeoutNs of wall time it records kErrTimeout in the call's
// error word and returns false, so a lost arrival can never hang the GPU.
#pragma once

#include <cuda.h>

#include "moe_common.cuh"

namespace moe {
namespace tc {

#define TC_DEV __device__ __forceinline__

constexpr unsigned long long kTimeoutNs = 1000000000ull;  // 1 s

TC_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

TC_DEV uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

TC_DEV void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count));
}
TC_DEV void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
TC_DEV void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
TC_DEV void mbar_arrive_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)),
               "r"(bytes)
               : "memory");
}
// Raises the transaction count the current phase of b waits for, without arriving.
TC_DEV void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)),
               "r"(bytes)
               : "memory");
}
TC_DEV bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for phase `parity` of barrier b to complete; false (and the timeout bit set in *err)
// when it did not within limit_ns (kTimeoutNs unless a test shortens it).
TC_DEV bool mbar_wait(uint64_t* b, uint32_t parity, int32_t* err,
                      unsigned long long limit_ns = kTimeoutNs) {
  if (mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(b, parity)) return true;
    if (globaltimer() - t0 > limit_ns) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}

// mbar_wait taken by every lane of a warp, with one verdict for the warp: true only when the wait
// succeeded in every lane.  The lanes' bounded waits can end differently (one lane times out as
// the phase completes for another), and the warp-collective work that follows (tcgen05.ld / st,
// shuffles, __syncwarp) has to run in all lanes or in none.
TC_DEV bool mbar_wait_warp(uint64_t* b, uint32_t parity, int32_t* err) {
  return __all_sync(0xffffffffu, mbar_wait(b, parity, err));
}

// After a wait gave up: waits (each wait bounded) for the stages this thread filled last - the
// loads of fill numbers max(0, issued - S) .. issued - 1, stage j % S, phase j / S - so that no
// copy still targets the CTA's shared memory when it exits.  A phase that cannot complete (its
// other arrivals never came) ends at the time limit.
template <int S>
TC_DEV void drain_stage_loads(uint64_t* full, int issued, int32_t* err) {
  for (int j = issued > S ? issued - S : 0; j < issued; ++j)
    mbar_wait(&full[j % S], (uint32_t)(j / S) & 1u, err);
}

// 4-byte asynchronous global -> shared copy (both addresses 4-byte aligned).
TC_DEV void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
TC_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
TC_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's committed cp.async groups are still in flight.
template <int N>
TC_DEV void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

TC_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA tile loads into shared memory, completion counted in bytes on barrier `bar`.
TC_DEV void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
TC_DEV void tma_load_3d(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// L2 policy for data read once per call (streamed weights): evicted first, so that what is
// reused (activation tiles, the combine buffer) stays in L2.
TC_DEV uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// tma_load_3d with an L2 cache policy.
TC_DEV void tma_load_3d_hint(void* dst, const CUtensorMap* tm, int x, int y, int z, uint64_t* bar,
                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Contiguous global -> shared copy (16-byte aligned addresses, size a multiple of 16).
TC_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// bulk_load with an L2 cache policy.
TC_DEV void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
TC_DEV void prefetch_tmap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
}

// Shared-memory matrix descriptor of the 5th-generation tensor core:
// start address, leading / stride byte offsets (16-byte units), version 1, layout type
// (0 = no swizzle, 2 = 128-byte swizzle).
TC_DEV uint64_t smem_desc(const void* p, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  const uint64_t a = (smem_u32(p) >> 4) & 0x3FFF;
  return a | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) | ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) |
         (1ull << 46) | ((uint64_t)layout << 61);
}
// K-major operand tile written by TMA with 128-byte swizzle: rows of 128 bytes, 8-row atoms.
TC_DEV uint64_t desc_sw128(const void* p) { return smem_desc(p, 16, 1024, 2); }
// Scale-factor chunk: 32 rows of 16 bytes, contiguous.
TC_DEV uint64_t desc_sf(const void* p) { return smem_desc(p, 0, 128, 0); }

TC_DEV void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
TC_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
TC_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Tensor memory is allocated, and the allocation permit given up, before anything else a CTA
// does (warp 0; the other warps go on).  While a CTA of a kernel that uses tensor memory still
// holds its permit, no further CTA of that kernel starts on the same SM (measured: the SM's
// second CTA starts only once the first has relinquished, or exited if it never does, with
// shared memory and tensor memory to spare), so a global read or a dependency wait placed
// before the allocation holds back the SM's other CTAs by its whole latency.
TC_DEV void tmem_alloc_first(uint32_t* dst, uint32_t ncols) {
  if ((threadIdx.x >> 5) == 0) {
    tmem_alloc(dst, ncols);
    tmem_relinquish();
  }
}
// Early exit of a CTA that allocated at entry: every thread of the CTA takes the branch.
TC_DEV void tmem_exit_early(const uint32_t* s_tmem, uint32_t ncols);

TC_DEV void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
TC_DEV void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
TC_DEV void tmem_exit_early(const uint32_t* s_tmem, uint32_t ncols) {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if ((threadIdx.x >> 5) == 0) tmem_dealloc(*s_tmem, ncols);
}
// 32 rows x 16 bytes of scale factors -> TMEM, replicated to the four 32-lane quadrants.
TC_DEV void tc_cp_sf(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
}
// D[tmem] (+)= A[smem] x B[smem]^T with UE8M0 block scales from TMEM (MXFP8/6/4 kind).
TC_DEV void mma_mxf8f6f4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                         uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem] x B[smem]^T with E2M1 A and B and UE4M3 block scales per 16 along K
// from TMEM (NVFP4 x NVFP4, K = 64 per instruction: four scales per row).
TC_DEV void mma_mxf4nvf4_4x(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                            uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem] x B[smem]^T, bf16 / fp16 operands, fp32 accumulation.
TC_DEV void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] x B[smem]^T, f16 / bf16 operands, fp32 accumulation; A is M rows over
// the 128 lanes, two 16-bit elements along K per 32-bit column (the even one in the low half).
TC_DEV void mma_f16_ta(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns from registers; the warp writes its own quadrant.
TC_DEV void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
// Waits until this thread's tcgen05.st stores have completed.
TC_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Arrive on `bar` once all tcgen05 operations issued so far by this thread have completed.
TC_DEV void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns; the warp reads its own lane quadrant.
TC_DEV void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Instruction descriptor of kind::mxf8f6f4 with UE8M0 scales, K-major A and B, M = 128:
// a / b formats (E4M3 = 0, E2M1 = 5), N, and the scale-factor byte selectors of A and B.
__host__ __device__ constexpr uint32_t idesc_mxf8f6f4(uint32_t afmt, uint32_t bfmt, uint32_t n,
                                                      uint32_t sf_id) {
  return (sf_id << 4) | (afmt << 7) | (bfmt << 10) | ((n >> 3) << 17) | (1u << 23) |
         ((128u >> 4) << 24) | (sf_id << 29);
}
// Instruction descriptor of kind::f16 with bf16 A/B, fp32 D, K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}
// Instruction descriptor of kind::mxf4nvf4 with 4X scale vectors: A and B E2M1 (format 1 of
// this kind), UE4M3 scales (scale-format bit 23 clear), scale ids 0, fp32 D, K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_mxf4nvf4(uint32_t n) {
  return (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}
constexpr uint32_t kFmtE4M3 = 0;
constexpr uint32_t kFmtE2M1 = 5;

}  // namespace tc
}  // namespace moe
