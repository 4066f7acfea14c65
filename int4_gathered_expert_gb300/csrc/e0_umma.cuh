// Blackwell (sm_103a) building blocks written as inline PTX: mbarriers with
// time-bounded waits, TMA tile loads, and the 5th-generation tensor-core path
// (TMEM allocation, tcgen05.mma kind::f16 with operands in shared memory and
// the fp32 accumulator in tensor memory, commit to an mbarrier, tcgen05.ld).
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "e0_common.cuh"

namespace e0 {

E0_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

E0_DEV uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier

E0_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
E0_DEV void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
E0_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
E0_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
E0_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase with the given parity to complete.  Gives up (returns
// false) after `limit_ns` of wall time or as soon as *abort becomes non-zero.
// try_wait with a suspend-time hint: the thread sleeps in hardware until the
// phase completes or about `hint_ns` pass, instead of spinning on issue slots
// the working warps of the SM need
E0_DEV bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
E0_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, const volatile uint32_t* abort, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ------------------------------------------------------------------ TMA

E0_DEV void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
E0_DEV void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
E0_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ------------------------------------------------------------------ tcgen05

// one full warp executes these two
E0_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
E0_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
E0_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
E0_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, fp16 inputs, fp32 accumulate; issued by one thread.
E0_DEV void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, fp16 inputs, fp32 accumulate; A is M rows in
// M lanes of tensor memory, K-major, two fp16 of consecutive k per 32-bit column
// (one MMA of K = 16 reads 8 columns).  Issued by one thread.
E0_DEV void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(
            d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive (once) on `bar` when every tcgen05.mma issued so far by this thread has completed
E0_DEV void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread t of the warp gets TMEM
// lane (32*(warp%4) + t), columns col..col+15.
E0_DEV void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
E0_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 bits, 32 consecutive columns: thread t of the warp writes
// TMEM lane (32*(warp%4) + t), columns col..col+31.
E0_DEV void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
                 : "memory");
}
E0_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes (64 fp16) stored in 8-row groups of 1024 bytes (the layout a TMA
// load with CU_TENSOR_MAP_SWIZZLE_128B writes).  Fields: start address >> 4
// (bits 0-13), leading-dimension offset (16-29, unused for this layout: 1),
// stride between 8-row groups >> 4 (32-45), descriptor version 1 (46-47),
// layout type 2 = 128B swizzle (61-63).
E0_DEV uint64_t sdesc_k_sw128(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits 4-5
// = 1), A and B fp16 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Position of 16-byte chunk c of row r inside a 128B-swizzled K-major tile.
E0_DEV uint32_t sw128_offset(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

E0_DEV uint32_t lop_and_or(uint32_t a, uint32_t mask, uint32_t magic) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(magic));
    return d;
}

// Dequantise one 64-element group of a row (8 code words in kernel nibble
// order + its (scale, bias)) to fp16 w = scale*q + bias and store it as row r
// of a 128B-swizzled tile.  Each word gives 8 consecutive fp16 = one chunk:
// the codes become exact fp16 integers via the exponent trick (OR into the
// mantissa of 1024 or 64, then subtract), then one fp16 FMA applies scale and
// bias (a single rounding).
E0_DEV void dequant64_to_tile(const uint4 c0, const uint4 c1, uint32_t sb_bits, uint8_t* tile, int r) {
    const __half2 sb = *reinterpret_cast<const __half2*>(&sb_bits);
    const __half2 s2 = __low2half2(sb), b2 = __high2half2(sb);
    const uint32_t m1024 = 0x64006400u, m64 = 0x54005400u;
    const __half2 h1024 = *reinterpret_cast<const __half2*>(&m1024);
    const __half2 h64 = *reinterpret_cast<const __half2*>(&m64);
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    uint8_t* rowp = tile + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t x = w[k], y = x >> 8;
        uint32_t p0 = lop_and_or(x, 0x000F000Fu, m1024);
        uint32_t p1 = lop_and_or(x, 0x00F000F0u, m64);
        uint32_t p2 = lop_and_or(y, 0x000F000Fu, m1024);
        uint32_t p3 = lop_and_or(y, 0x00F000F0u, m64);
        __half2 q0 = __hsub2(*reinterpret_cast<__half2*>(&p0), h1024);
        __half2 q1 = __hsub2(*reinterpret_cast<__half2*>(&p1), h64);
        __half2 q2 = __hsub2(*reinterpret_cast<__half2*>(&p2), h1024);
        __half2 q3 = __hsub2(*reinterpret_cast<__half2*>(&p3), h64);
        __half2 o0 = __hfma2(q0, s2, b2), o1 = __hfma2(q1, s2, b2), o2 = __hfma2(q2, s2, b2), o3 = __hfma2(q3, s2, b2);
        uint4 out;
        out.x = *reinterpret_cast<uint32_t*>(&o0);
        out.y = *reinterpret_cast<uint32_t*>(&o1);
        out.z = *reinterpret_cast<uint32_t*>(&o2);
        out.w = *reinterpret_cast<uint32_t*>(&o3);
        *reinterpret_cast<uint4*>(rowp + ((k ^ (r & 7)) << 4)) = out;
    }
}

// The same dequantisation into registers: o[c] holds k = 2c, 2c + 1 (the
// column order of a K-major A row in tensor memory).
E0_DEV void dequant64_to_regs(const uint4 c0, const uint4 c1, uint32_t sb_bits, uint32_t (&o)[32]) {
    const __half2 sb = *reinterpret_cast<const __half2*>(&sb_bits);
    const __half2 s2 = __low2half2(sb), b2 = __high2half2(sb);
    const uint32_t m1024 = 0x64006400u, m64 = 0x54005400u;
    const __half2 h1024 = *reinterpret_cast<const __half2*>(&m1024);
    const __half2 h64 = *reinterpret_cast<const __half2*>(&m64);
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t x = w[k], y = x >> 8;
        uint32_t p0 = lop_and_or(x, 0x000F000Fu, m1024);
        uint32_t p1 = lop_and_or(x, 0x00F000F0u, m64);
        uint32_t p2 = lop_and_or(y, 0x000F000Fu, m1024);
        uint32_t p3 = lop_and_or(y, 0x00F000F0u, m64);
        __half2 q0 = __hsub2(*reinterpret_cast<__half2*>(&p0), h1024);
        __half2 q1 = __hsub2(*reinterpret_cast<__half2*>(&p1), h64);
        __half2 q2 = __hsub2(*reinterpret_cast<__half2*>(&p2), h1024);
        __half2 q3 = __hsub2(*reinterpret_cast<__half2*>(&p3), h64);
        __half2 o0 = __hfma2(q0, s2, b2), o1 = __hfma2(q1, s2, b2), o2 = __hfma2(q2, s2, b2), o3 = __hfma2(q3, s2, b2);
        o[4 * k + 0] = *reinterpret_cast<uint32_t*>(&o0);
        o[4 * k + 1] = *reinterpret_cast<uint32_t*>(&o1);
        o[4 * k + 2] = *reinterpret_cast<uint32_t*>(&o2);
        o[4 * k + 3] = *reinterpret_cast<uint32_t*>(&o3);
    }
}

E0_DEV void zero_row_of_tile(uint8_t* tile, int r) {
    uint8_t* rowp = tile + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
    for (int k = 0; k < 8; ++k) *reinterpret_cast<uint4*>(rowp + (k << 4)) = make_uint4(0, 0, 0, 0);
}

}  // namespace e0
