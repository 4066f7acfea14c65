// Device helpers shared by the decode and prefill kernels (sm_103a).
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/e0moe.h"

#define E0_DEV __device__ __forceinline__

namespace e0 {

constexpr int GROUP = 64;

// ---------------------------------------------------------------- status

E0_DEV void set_status(uint32_t* st, uint32_t bits) {
    if (st) atomicOr(st, bits);
}

// ---------------------------------------------------------------- warp reductions

E0_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
E0_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
E0_DEV int warp_sum_int(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// Sum over consecutive segments of G lanes (any G <= 32); the result is valid
// in the first lane of each segment (lane % G == 0).
E0_DEV float seg_sum(float v, int G, int lane) {
    const int pos = lane % G;
    for (int o = 1; o < G; o <<= 1) {
        const float t = __shfl_down_sync(0xffffffffu, v, o);
        if (pos + o < G) v += t;
    }
    return v;
}

// ---------------------------------------------------------------- loads

// L2 policy for data read once (streamed weights): first out when L2 needs
// room, so that the streamed bytes do not push out what is read again.
E0_DEV uint64_t l2_evict_first() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
E0_DEV uint4 ldg_stream(const void* p) {  // weights: read once, kept neither in L1 nor long in L2
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(l2_evict_first()));
    return v;
}
E0_DEV uint32_t ldg_u32(const void* p) {
    uint32_t v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(l2_evict_first()));
    return v;
}

// ---------------------------------------------------------------- fixed-point activations
//
// The int4 GEMV multiplies 4-bit codes by activations held as 16-bit fixed
// point per group of 64: x16_j = rint(x_j * 32767 / M_g), M_g = max|x| over
// the group, so x_j ~= c_g * x16_j with c_g = M_g / 32767 (relative error
// <= 1.5e-5 of the group maximum).  x16 is split into a signed high byte and
// an unsigned low byte (x16 = 256*hi + lo) so that two dp4a instructions give
// the exact integer sum of q_j * x16_j.
//
// In the kernel layout a 32-bit code word k holds elements 8k..8k+7 with
// nibble j (bits 4j..4j+3) = element 8k + P[j], P = {0,2,4,6,1,3,5,7}.  So
// (w & 0x0F0F0F0F) holds elements (0,4,1,5) in bytes 0..3 and
// ((w >> 4) & 0x0F0F0F0F) holds elements (2,6,3,7) (offsets within the word).
// A group's planes are 8 uint4, one per code word: {hi bytes of set A, hi
// bytes of set B, lo bytes of set A, lo bytes of set B} with A = (0,4,1,5) and
// B = (2,6,3,7) in that byte order.

struct XGroup {
    float c;    // M_g / 32767
    float sx;   // sum of x16 over the group (exact integer, as float)
};

E0_DEV int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
E0_DEV uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Loads of data that other blocks of a running persistent kernel may have
// written: served from L2 (L1 is not coherent across SMs).  Shared-memory
// pointers are read directly.
E0_DEV float ld_shared_or_l2(const float* p) { return __isGlobal(p) ? __ldcg(p) : *p; }
E0_DEV float2 ld2_shared_or_l2(const float* p) {
    return __isGlobal(p) ? __ldcg(reinterpret_cast<const float2*>(p)) : *reinterpret_cast<const float2*>(p);
}
E0_DEV int ldi_shared_or_l2(const int32_t* p) { return __isGlobal(p) ? __ldcg(p) : *p; }

// One warp quantises one 64-value group (lane holds elements 2*lane and
// 2*lane + 1) into planes + XGroup.  Plane word k of the group is stored at
// planes[k * pstride].
E0_DEV void quantize_group_v(const float2 v, uint4* planes, XGroup* xg, int lane, uint32_t* st, int pstride = 1) {
    float mx = warp_max(fmaxf(fabsf(v.x), fabsf(v.y)));
    if (!(mx < 3.0e38f)) {  // NaN or inf in the activations
        if (lane == 0) set_status(st, E0_ST_NONFINITE);
        mx = 0.f;
    }
    const float inv = mx > 0.f ? 32767.f / mx : 0.f;
    int qa = __float2int_rn(v.x * inv);
    int qb = __float2int_rn(v.y * inv);
    qa = max(-32767, min(32767, qa));
    qb = max(-32767, min(32767, qb));
    int s = warp_sum_int(qa + qb);
    // this lane holds elements 2m, 2m+1 of its word (m = lane & 3): they sit in
    // set A (m even) or B (m odd), at bytes (m >> 1) and 2 + (m >> 1)
    const int m = lane & 3, p = 8 * (m >> 1);
    const uint32_t hi = (((uint32_t)(qa >> 8) & 0xFFu) << p) | (((uint32_t)(qb >> 8) & 0xFFu) << (p + 16));
    const uint32_t lo = (((uint32_t)qa & 0xFFu) << p) | (((uint32_t)qb & 0xFFu) << (p + 16));
    uint32_t hiA = (m & 1) ? 0u : hi, hiB = (m & 1) ? hi : 0u;
    uint32_t loA = (m & 1) ? 0u : lo, loB = (m & 1) ? lo : 0u;
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        hiA |= __shfl_xor_sync(0xffffffffu, hiA, o);
        hiB |= __shfl_xor_sync(0xffffffffu, hiB, o);
        loA |= __shfl_xor_sync(0xffffffffu, loA, o);
        loB |= __shfl_xor_sync(0xffffffffu, loB, o);
    }
    if ((lane & 3) == 0) planes[(lane >> 2) * pstride] = make_uint4(hiA, hiB, loA, loB);
    if (lane == 0) {
        xg->c = mx / 32767.f;
        xg->sx = (float)s;
    }
}

// One warp quantises group g of x (64 fp32 values) into planes + XGroup.
E0_DEV void quantize_group_warp(const float* x, uint4* planes, XGroup* xg, int lane, uint32_t* st, int pstride = 1) {
    quantize_group_v(ld2_shared_or_l2(x + 2 * lane), planes, xg, lane, st, pstride);
}

// Partial dot product of one 64-element group of an int4 row (two uint4 code
// chunks = 8 words, kernel nibble order) with the matching activation planes;
// sb = (scale, bias).  Plane word k is read at pl[k * pstride].
E0_DEV float q4_group_dot(const uint4 c0, const uint4 c1, const uint4* pl, XGroup xg, uint32_t sb_bits, int pstride = 1) {
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    int hi = 0;
    uint32_t lo = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint4 p = pl[k * pstride];
        const uint32_t a = w[k] & 0x0F0F0F0Fu;
        const uint32_t b = (w[k] >> 4) & 0x0F0F0F0Fu;
        hi = dp4a_us(a, p.x, hi);
        hi = dp4a_us(b, p.y, hi);
        lo = dp4a_uu(a, p.z, lo);
        lo = dp4a_uu(b, p.w, lo);
    }
    const int sqx = hi * 256 + (int)lo;
    __half2 sb = *reinterpret_cast<const __half2*>(&sb_bits);
    const float s = __low2float(sb), b = __high2float(sb);
    return xg.c * fmaf(s, (float)sqx, b * xg.sx);
}

// ---------------------------------------------------------------- 32-element half-groups

// One warp quantises 32 values (one per lane; lanes beyond n hold 0) into
// the planes of a half-group (4 uint4, kernel nibble order) and its XGroup.
E0_DEV void quantize_half_warp(float v, uint4* planes, XGroup* xg, int lane) {
    const float mx = warp_max(fabsf(v));
    const float inv = (mx > 0.f && mx < 3.0e38f) ? 32767.f / mx : 0.f;
    int q = __float2int_rn(v * inv);
    q = max(-32767, min(32767, q));
    const int s = warp_sum_int(q);
    const int e = lane & 7;  // element within its 8-element word
    const int set = (e >> 1) & 1, byte = ((e & 1) << 1) | (e >> 2);
    const uint32_t hi = ((uint32_t)(q >> 8) & 0xFFu) << (8 * byte);
    const uint32_t lo = ((uint32_t)q & 0xFFu) << (8 * byte);
    uint32_t hiA = set ? 0u : hi, hiB = set ? hi : 0u, loA = set ? 0u : lo, loB = set ? lo : 0u;
#pragma unroll
    for (int o = 1; o <= 4; o <<= 1) {
        hiA |= __shfl_xor_sync(0xffffffffu, hiA, o);
        hiB |= __shfl_xor_sync(0xffffffffu, hiB, o);
        loA |= __shfl_xor_sync(0xffffffffu, loA, o);
        loB |= __shfl_xor_sync(0xffffffffu, loB, o);
    }
    if (e == 0) planes[lane >> 3] = make_uint4(hiA, hiB, loA, loB);
    if (lane == 0) {
        xg->c = (inv > 0.f) ? mx / 32767.f : 0.f;
        xg->sx = (float)s;
    }
}

// Dot product of one half-group of an int4 row (16 code bytes) with its planes.
E0_DEV float q4_half_dot(const uint4 c, const uint4* pl, XGroup xg, uint32_t sb_bits) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    int hi = 0;
    uint32_t lo = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint4 p = pl[k];
        const uint32_t a = w[k] & 0x0F0F0F0Fu;
        const uint32_t b = (w[k] >> 4) & 0x0F0F0F0Fu;
        hi = dp4a_us(a, p.x, hi);
        hi = dp4a_us(b, p.y, hi);
        lo = dp4a_uu(a, p.z, lo);
        lo = dp4a_uu(b, p.w, lo);
    }
    const int sqx = hi * 256 + (int)lo;
    __half2 sb = *reinterpret_cast<const __half2*>(&sb_bits);
    return xg.c * fmaf(__low2float(sb), (float)sqx, __high2float(sb) * xg.sx);
}

// fp16 weights x fp32 activations, 8 halves per uint4.
E0_DEV float h8_dot(const uint4 wv, const float* x) {
    const __half2* h = reinterpret_cast<const __half2*>(&wv);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __half22float2(h[i]);
        acc = fmaf(f.x, x[2 * i], acc);
        acc = fmaf(f.y, x[2 * i + 1], acc);
    }
    return acc;
}

// fp16 weights x fp32 activations: 8 halves of wv times a (first 4) and b (last 4).
E0_DEV float h8_dot44(const uint4 wv, const float4 a, const float4 b) {
    const __half2* hw = reinterpret_cast<const __half2*>(&wv);
    const float2 w0 = __half22float2(hw[0]), w1 = __half22float2(hw[1]);
    const float2 w2 = __half22float2(hw[2]), w3 = __half22float2(hw[3]);
    float acc = w0.x * a.x;
    acc = fmaf(w0.y, a.y, acc);
    acc = fmaf(w1.x, a.z, acc);
    acc = fmaf(w1.y, a.w, acc);
    acc = fmaf(w2.x, b.x, acc);
    acc = fmaf(w2.y, b.y, acc);
    acc = fmaf(w3.x, b.z, acc);
    return fmaf(w3.y, b.w, acc);
}

E0_DEV float silu_f(float x) { return x / (1.f + expf(-x)); }
E0_DEV float gelu_erf_f(float x) { return 0.5f * x * (1.f + erff(x * 0.70710678118654752f)); }
E0_DEV float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

// ---------------------------------------------------------------- kernel layout offsets

// Canonical code word (nibble i = element i) -> kernel nibble order.
__host__ __device__ inline uint32_t interleave_word(uint32_t c) {
    const int P[8] = {0, 2, 4, 6, 1, 3, 5, 7};
    uint32_t k = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) k |= ((c >> (4 * P[j])) & 0xFu) << (4 * j);
    return k;
}
E0_DEV uint4 interleave16(uint4 v) {
    return make_uint4(interleave_word(v.x), interleave_word(v.y), interleave_word(v.z), interleave_word(v.w));
}

// Rows of a down block: the down projection is stored in blocks of DROWS
// output rows, each block holding every input of its rows.
constexpr int DROWS = 16;

// Offsets inside one expert slot (the kernel layout documented in e0moe.h).
struct SlotLayout {
    int H, I;
    __host__ __device__ size_t down_codes() const { return (size_t)I * H; }
    __host__ __device__ size_t gu_sb() const { return (size_t)I * H + (size_t)H * I / 2; }
    __host__ __device__ size_t down_sb() const { return gu_sb() + (size_t)I * (H / GROUP) * 2 * 4; }
    __host__ __device__ size_t bytes() const { return down_sb() + (size_t)H * (I / GROUP) * 4; }
    // down codes: the 16 bytes of output row j, half-group c (inputs 32c..32c+31),
    // in row blocks: block j / DROWS holds [half-group][row in block][16 bytes]
    __host__ __device__ size_t down_code_off(int j, int c) const {
        return down_codes() + (((size_t)(j / DROWS) * (I / 32) + c) * DROWS + j % DROWS) * 16;
    }
    // down (scale, bias) word of output row j, 64-group g: [block][group][row in block]
    __host__ __device__ size_t down_sb_off(int j, int g) const {
        return down_sb() + (((size_t)(j / DROWS) * (I / GROUP) + g) * DROWS + j % DROWS) * 4;
    }
    // one row block's down codes / words are contiguous
    __host__ __device__ size_t down_block_code_bytes() const { return (size_t)(I / 32) * DROWS * 16; }
    __host__ __device__ size_t down_block_sb_bytes() const { return (size_t)(I / GROUP) * DROWS * 4; }
};

}  // namespace e0
