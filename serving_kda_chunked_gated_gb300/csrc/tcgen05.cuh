// Blackwell (sm_100a family, here sm_103a) tensor-core building blocks in
// inline PTX: tcgen05 TMEM allocation, MMA issue/commit, TMEM loads and
// stores, shared-memory matrix descriptors, mbarriers with bounded waits, and
// the warp-level mma.sync used for 16x16 sub-blocks.
//
// Shared-memory operand layout used everywhere ("SW128 K-major"): an R x K
// operand (R rows = M or N, K = reduction dim) is stored as slabs of R rows x
// 128 bytes (32 four-byte or 64 two-byte elements of K per slab); row r of a slab sits at
// (r/8)*1024 + (r%8)*128 and its 16-byte chunk c is stored at chunk c ^ (r%8)
// (the 128-byte swizzle), so slabs must be 1024-byte aligned.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#define TC_DEV __device__ __forceinline__

namespace tc {

TC_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// byte offset of element (r, k) inside an SW128 K-major operand with R rows
TC_DEV uint32_t sw128_offset(int r, int k, int R) {
    const int slab = k >> 5, kk = k & 31;
    return (uint32_t)(slab * R * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                      ((((kk >> 2) ^ (r & 7)) << 4)) + ((kk & 3) << 2));
}

// byte offset of 2-byte element (r, k) inside an SW128 K-major operand with R rows
// (slabs of 64 elements)
TC_DEV uint32_t sw128_offset_h(int r, int k, int R) {
    const int slab = k >> 6, kk = k & 63;
    return (uint32_t)(slab * R * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                      ((((kk >> 3) ^ (r & 7)) << 4)) + ((kk & 7) << 1));
}

// Shared-memory matrix descriptor for an SW128 K-major operand; `addr` is the
// shared address of element (0, k0) (k0 a multiple of 8 for 4-byte types).
TC_DEV uint64_t sw128_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)(1u) << 16;                        // leading byte offset (unused for SW128 K-major)
    d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;    // stride byte offset: 8-row groups
    d |= (uint64_t)1 << 46;                           // descriptor version
    d |= (uint64_t)2 << 61;                           // 128-byte swizzle
    return d;
}

// descriptor for k-step `ks` of an SW128 K-major operand: 32 bytes per step, i.e.
// 8 tf32 elements (kind::tf32) or 16 fp16 elements (kind::f16)
TC_DEV uint64_t sw128_desc_k(uint32_t base, int R, int ks) {
    const int k0 = ks * 8;
    return sw128_desc(base + (uint32_t)((k0 >> 5) * R * 128 + (k0 & 31) * 4));
}

// Instruction descriptor, kind::tf32, FP32 accumulate, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool neg_a = false) {
    return (1u << 4)                 // D = F32
         | (2u << 7) | (2u << 10)    // A, B = TF32
         | ((neg_a ? 1u : 0u) << 13)
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::f16 with fp16 A and B, FP32 accumulate, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4)                 // D = F32 (A, B = F16: format 0)
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

// FP32 -> FP16 (round to nearest even): one value, and a pair packed as (lo, hi)
TC_DEV uint16_t f32_to_f16(float x) {
    uint16_t h;
    asm("cvt.rn.f16.f32 %0, %1;" : "=h"(h) : "f"(x));
    return h;
}
TC_DEV uint32_t pack_f16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// ---------------------------------------------------------------------------
// TMEM allocation (one warp executes these)
// ---------------------------------------------------------------------------
TC_DEV void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(smem_dst)), "r"(ncols) : "memory");
}
TC_DEV void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
TC_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

TC_DEV void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
TC_DEV void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy shared-memory writes -> visible to the tensor core (async proxy)
TC_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---------------------------------------------------------------------------
// MMA issue (a single thread issues)
// ---------------------------------------------------------------------------
TC_DEV void mma_tf32_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc) : "memory");
}
TC_DEV void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc) : "memory");
}
TC_DEV void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc) : "memory");
}
// arrive on an mbarrier once all previously issued MMAs of this thread complete
TC_DEV void mma_commit(uint64_t* mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(mbar)) : "memory");
}

// ---------------------------------------------------------------------------
// TMEM <-> registers, 32x32b shape: thread i of warp w <-> lane 32*(w%4)+i,
// register j <-> column col+j.  `taddr` must carry the warp's lane base.
// ---------------------------------------------------------------------------
TC_DEV void tmem_ld16(uint32_t taddr, float* r) {
    uint32_t* u = reinterpret_cast<uint32_t*>(r);
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
                   "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]),
                   "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
                 : "r"(taddr));
}
TC_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

TC_DEV void tmem_st16(uint32_t taddr, const float* r) {
    const uint32_t* u = reinterpret_cast<const uint32_t*>(r);
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 :: "r"(taddr), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]),
                    "r"(u[6]), "r"(u[7]), "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]),
                    "r"(u[13]), "r"(u[14]), "r"(u[15])
                 : "memory");
}
TC_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// mbarrier with a bounded wait
// ---------------------------------------------------------------------------
TC_DEV void mbar_init(uint64_t* mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(mbar)), "r"(count) : "memory");
}
TC_DEV void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

TC_DEV bool mbar_try_wait(uint64_t* mbar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_u32(mbar)), "r"(parity) : "memory");
    return ok != 0;
}
// Wait for phase `parity` to complete; gives up after `limit` polls and
// returns false (the caller records the timeout and stops issuing work).
TC_DEV bool mbar_wait_bounded(uint64_t* mbar, uint32_t parity, uint32_t limit = (1u << 26)) {
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(mbar, parity)) return true;
    return false;
}

// Default bound of a wait, in polls (seconds at most); kernels take the bound
// of their waits on local copies and tensor-core work as a launch parameter.
constexpr uint32_t WAIT_POLLS = 1u << 22;

// The give-up path of a kernel whose bounded wait ran out: the thread that
// issues asynchronous copies and tensor-core work stops issuing, and before
// the CTA releases its shared memory and TMEM it waits here for the last phase
// it issued on each mbarrier (n_issued phases so far; phases complete in order
// and the kernels keep at most one outstanding per mbarrier, so the last
// phase's parity identifies it).  Returns false if that wait ran out too.
TC_DEV bool drain_phase(uint64_t* mbar, uint32_t n_issued) {
    return n_issued == 0 || mbar_wait_bounded(mbar, (n_issued - 1) & 1u, WAIT_POLLS);
}

// Error word bits set by a kernel whose bounded wait ran out
constexpr int ERR_WAIT = 1;    // a wait gave up: the call's outputs are invalid
constexpr int ERR_DRAIN = 2;   // and the wait for work already issued gave up as well

// expect `bytes` more transaction bytes on the mbarrier and arrive once
TC_DEV void mbar_arrive_expect_tx(uint64_t* mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(mbar)), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------------------
// TMA: 2-D tiled bulk copy global -> shared, completion counted on an mbarrier.
// `map` is the address of a CUtensorMap kernel parameter (__grid_constant__);
// (x, y) = (innermost, outer) element coordinates of the box origin.
// ---------------------------------------------------------------------------
TC_DEV void tma_load_2d(void* dst, const void* map, int x, int y, uint64_t* mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(mbar))
        : "memory");
}
// untiled bulk copy global -> shared: dst, src 16-byte aligned, bytes a multiple of 16
TC_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* mbar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(mbar))
        : "memory");
}
// TMA: 2-D tiled bulk copy shared -> global, completion tracked by this thread's bulk
// groups (commit with bulk_commit; bulk_wait_read -- or bulk_wait_read_but1, which
// leaves the newest group pending -- before a source is rewritten, bulk_wait_all
// before the CTA exits)
TC_DEV void tma_store_2d(const void* map, int x, int y, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
}
TC_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
TC_DEV void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
TC_DEV void bulk_wait_read_but1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
TC_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
TC_DEV void tma_prefetch_desc(const void* map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// FP32 -> TF32 (round to nearest, ties away), result kept in a 32-bit float
// ---------------------------------------------------------------------------
// (integer form: add half a tf32 ulp to the magnitude and clear the 13 low
// mantissa bits -- two full-rate integer operations; finite inputs)
TC_DEV float to_tf32(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

// ---------------------------------------------------------------------------
// Warp-level MMA, m16n8k8, tf32 inputs, fp32 accumulate.
//   A (16x8, row): a0=(g,t) a1=(g+8,t) a2=(g,t+4) a3=(g+8,t+4)
//   B (8x8, col):  b0=(k=t,n=g) b1=(k=t+4,n=g)
//   C (16x8):      c0=(g,2t) c1=(g,2t+1) c2=(g+8,2t) c3=(g+8,2t+1)
// with g = lane/4, t = lane%4.
// ---------------------------------------------------------------------------
TC_DEV void mma_m16n8k8_tf32(float* c, const float* a, const float* b) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(__float_as_uint(a[0])), "r"(__float_as_uint(a[1])), "r"(__float_as_uint(a[2])),
          "r"(__float_as_uint(a[3])), "r"(__float_as_uint(b[0])), "r"(__float_as_uint(b[1])));
}

}  // namespace tc
