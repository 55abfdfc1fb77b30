// Inline-PTX wrappers for the sm_103a tensor-memory path: mbarriers with bounded waits,
// TMA tensor loads, tcgen05 allocation / MMA / commit / tensor-memory loads and stores.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace ql {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: gives up after `limit` unsuccessful polls, or as soon as *abort is set.
// Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit, volatile int* abort) {
  for (uint32_t n = 0;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if (n >= limit || (abort && *abort)) return false;
  }
}

// ------------------------------------------------------------------ L2 cache policies
// evict_first: data read once (a weight stream) leaves L2 before anything else; evict_last:
// data fetched ahead of its use stays until then
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* m, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// shared memory -> global, one 2D box (rows / columns past the tensor's edge are not written);
// the caller fences its generic writes to the box first (fence.proxy.async) and waits with
// bulk_wait_all before the CTA exits
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, uint32_t smem_src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(x), "r"(y), "r"(smem_src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_and_wait_all() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* m, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_result)),
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

// D[tmem] (+)= A[smem] x B[smem]^T with per-32-K UE8M0 scale vectors read from tensor memory
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// D[tmem] (+)= A[smem] x B[smem]^T, f16 operands, fp32 accumulation
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One 64-K stage of f16 MMAs (four K = 16 steps: descriptors advance by 2 units = 32 bytes)
// issued in the same instruction stream as a non-blocking test of the next stage's two
// barriers: a completed-phase test costs ~150 cycles of latency in the issuing thread, which
// the MMA issue (~110 cycles each) hides.  Returns bit 0 / bit 1 = barrier 0 / 1 complete.
__device__ __forceinline__ uint32_t mma4_f16_test2(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                   uint32_t accumulate, uint32_t bar0, uint32_t bar1,
                                                   uint32_t parity) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p0, p1, pa;\n\t.reg .u32 r0, r1;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p0, [%6], %8;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p1, [%7], %8;\n\t"
      "setp.ne.b32 pa, %5, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], %2, %3, %4, pa;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], %9, %10, %4, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], %11, %12, %4, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], %13, %14, %4, 1;\n\t"
      "selp.u32 r0, 1, 0, p0;\n\t"
      "selp.u32 r1, 2, 0, p1;\n\t"
      "or.b32 %0, r0, r1;\n\t}"
      : "=r"(r)
      : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(bar0), "r"(bar1), "r"(parity),
        "l"(a_desc + 2), "l"(b_desc + 2), "l"(a_desc + 4), "l"(b_desc + 4), "l"(a_desc + 6), "l"(b_desc + 6)
      : "memory");
  return r;
}

// One stage of block-scaled MMAs (four K = 32 steps, scale byte j of each vector chosen by
// idesc j) issued in the same instruction stream as a non-blocking test of the next stage's two
// barriers, as mma4_f16_test2.  Returns bit 0 / bit 1 = barrier 0 / 1 complete.
__device__ __forceinline__ uint32_t mma4_mxf8f6f4_test2(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                        const uint32_t (&idesc)[4], uint32_t sfa_tmem,
                                                        uint32_t sfb_tmem, uint32_t accumulate, uint32_t bar0,
                                                        uint32_t bar1, uint32_t parity) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p0, p1, pa;\n\t.reg .u32 r0, r1;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p0, [%5], %7;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p1, [%6], %7;\n\t"
      "setp.ne.b32 pa, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], %2, %3, %8, [%12], [%13], pa;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], %14, %15, %9, [%12], [%13], 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], %16, %17, %10, [%12], [%13], 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%1], %18, %19, %11, [%12], [%13], 1;\n\t"
      "selp.u32 r0, 1, 0, p0;\n\t"
      "selp.u32 r1, 2, 0, p1;\n\t"
      "or.b32 %0, r0, r1;\n\t}"
      : "=r"(r)
      : "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(accumulate), "r"(bar0), "r"(bar1), "r"(parity), "r"(idesc[0]),
        "r"(idesc[1]), "r"(idesc[2]), "r"(idesc[3]), "r"(sfa_tmem), "r"(sfb_tmem), "l"(a_desc + 2), "l"(b_desc + 2),
        "l"(a_desc + 4), "l"(b_desc + 4), "l"(a_desc + 6), "l"(b_desc + 6)
      : "memory");
  return r;
}

// arrive on `bar` once every tcgen05 operation issued so far by this thread has completed
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_st_x4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v0), "r"(v1),
               "r"(v2), "r"(v3)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%"
      "20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_x8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile written by TMA with 128-byte
// swizzling: rows of 128 bytes, 8-row swizzle atoms 1024 bytes apart (stride byte offset),
// descriptor version 1, layout type 2 (128B swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);        // start address
  d |= (uint64_t)1 << 16;                          // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;                // stride byte offset
  d |= (uint64_t)1 << 46;                          // version
  d |= (uint64_t)2 << 61;                          // 128B swizzle
  return d;
}

// Instruction descriptor of kind::mxf8f6f4 with UE8M0 scales: A and B K-major,
// M = 128, N = n, formats (E4M3 = 0, E2M1 = 5), scale-vector byte ids.
__host__ __device__ constexpr uint32_t idesc_mxf8f6f4(uint32_t a_fmt, uint32_t b_fmt, uint32_t n, uint32_t a_sf_id,
                                                      uint32_t b_sf_id) {
  return (b_sf_id << 4) | (a_fmt << 7) | (b_fmt << 10) | ((n >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24) |
         (a_sf_id << 29);
}

// Instruction descriptor of kind::f16 with f16 A and B (both K-major) and an fp32 accumulator:
// accumulator format 1 (bits 4-5), A / B format 0 = f16, N = n (bits 17-22, n / 8), M = 128.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t n) {
  return (1u << 4) | ((n >> 3) << 17) | ((128u >> 4) << 24);
}

}  // namespace tc
}  // namespace ql
