// Shared pieces of the tensor-core append kernels (head_dim <= 128, and the
// head_dim 256 kernel that takes one half of the output channels per CTA):
// tile geometry, the measured accumulation bound of kind::f16, bf16 splitting,
// tensor-memory reads of y, the reciprocal-path code decision and the
// description of where a vector's input row lives.
#pragma once

#include "oscar_append_common.cuh"
#include "oscar_tcgen05.cuh"

namespace oscar {
namespace tcq {

constexpr int kTcRows = 128;               // vectors per tile (the MMA's M; one tensor-memory lane each)

constexpr int kMetaInts = 4;               // per vector: slot, head | kind << 16, source offset (int64)
constexpr float kMagic = 12582912.0f;      // 1.5·2^23: x + kMagic rounds x to an integer in the low bits
// Bound on |y - fl(x·R)| per channel, in units of 2^-24·‖y‖₂.  Measured on
// GB300 (kind::f16, fp32 accumulator): within one MMA the terms are aligned to
// the largest one at a resolution of 2^-25 of its binade and truncated, and the
// sum is truncated to fp32 (1 - 2^-26 gives 1, 2^30 + 1 - 2^30 gives 0).  Over
// rows of Gaussian, outlier-channel, wide-exponent and column-aligned inputs the
// largest error of this kernel's order (lo, mid, hi parts) was 7.3·2^-24·‖x‖₂
// (2.1 on outlier-channel rows); the bound takes twice the largest, and ‖x‖₂ =
// ‖y‖₂ for an orthogonal R (1% margin).
constexpr float kTcErr = 16.0f;
constexpr float kTcBound = 1.01f * (kTcErr + 1.0f) / 16777216.0f;

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    return (uint32_t)f32_to_bf16_bits(lo) | ((uint32_t)f32_to_bf16_bits(hi) << 16);
}

// part p (0: hi, 1: mid, 2: lo) of the three-way bf16 split of x
__device__ __forceinline__ float bf16_part(float x, int p) {
    const float h = bf16_bits_to_f32(f32_to_bf16_bits(x));
    if (p == 0) return h;
    const float r1 = x - h;
    const float m = bf16_bits_to_f32(f32_to_bf16_bits(r1));
    if (p == 1) return m;
    return r1 - m;
}

// 32 channels of y for this thread's vector.
__device__ __forceinline__ void load_y(uint32_t taddr, float (&y)[32]) {
    tc5::ld32(taddr, y);
    tc5::wait_ld();
}

__device__ __forceinline__ float min3f(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// min and max of 32 values folded into (mn, mx): four independent chains of
// three-input min / max, then a short combine.
__device__ __forceinline__ void minmax32(const float (&y)[32], float& mn, float& mx) {
    float a[4], b[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float* v = y + 8 * k;
        a[k] = fminf(min3f(min3f(v[0], v[1], v[2]), v[3], v[4]), min3f(v[5], v[6], v[7]));
        b[k] = fmaxf(max3f(max3f(v[0], v[1], v[2]), v[3], v[4]), max3f(v[5], v[6], v[7]));
    }
    mn = min3f(mn, min3f(a[0], a[1], a[2]), a[3]);
    mx = max3f(mx, max3f(b[0], b[1], b[2]), b[3]);
}

__device__ __forceinline__ void pack_codes32(const float2 (&c)[16], uint32_t& w0, uint32_t& w1);

// Codes of 32 channels as two words of 16 (channel i at bits 2i) by the
// reciprocal path on channel pairs (paired fp32 operations); bit 31 of `tie` is
// cleared when some |q - rint(q)|² reaches -nb2 (q within the group's band of a
// half-integer).  s = 0 (a flat group) takes r3 = 0 and gives codes 0.
__device__ __forceinline__ void codes32(const float (&y)[32], float zc, float r3, float nb2, uint32_t& w0, uint32_t& w1,
                                        uint32_t& tie) {
    float2 c[16];                         // codes of channels (2j, 2j+1) as floats
    {
        const float2 nz = make_float2(-zc, -zc), three = make_float2(3.0f, 3.0f);
        const float2 mg = make_float2(kMagic, kMagic), nmg = make_float2(-kMagic, -kMagic);
        const float2 m1 = make_float2(-1.0f, -1.0f);
        const float2 nb = make_float2(nb2, nb2);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float2 a = __fadd2_rn(make_float2(y[2 * j], y[2 * j + 1]), nz);                 // y - z
            const float2 t = make_float2(__saturatef(__fmul_rn(a.x, r3)), __saturatef(__fmul_rn(a.y, r3)));
            const float2 q = __fmul2_rn(t, three);                                               // in [0, 3]
            c[j] = __fadd2_rn(__fadd2_rn(q, mg), nmg);                                          // rint(q)
            const float2 d = __ffma2_rn(c[j], m1, q);                                           // q - rint(q)
            const float2 e = __ffma2_rn(d, d, nb);                                              // >= 0: near a tie
            tie &= __float_as_uint(e.x) & __float_as_uint(e.y);
        }
    }
    pack_codes32(c, w0, w1);
}

// Packs 32 codes held as floats (channels 2j, 2j+1 in c[j]) into two words of
// 16 (channel i at bits 2i): Σ c_i 4^i over 8 channels per value, as a
// depth-3 tree of exact integer FMAs.
__device__ __forceinline__ void pack_codes32(const float2 (&c)[16], uint32_t& w0, uint32_t& w1) {
    const float2 k16 = make_float2(16.0f, 16.0f), k256 = make_float2(256.0f, 256.0f);
    float2 A[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) A[k] = __ffma2_rn(c[2 * k + 1], k16, c[2 * k]);      // c_4k + 16 c_4k+2 | odd
    uint32_t u[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float2 B = __ffma2_rn(A[2 * m + 1], k256, A[2 * m]);
        const float v = __fmaf_rn(B.y, 4.0f, B.x);                                    // channels 8m .. 8m+7
        u[m] = __float_as_uint(__fadd_rn(v, kMagic));                                 // low 16 bits = v
    }
    w0 = __byte_perm(u[0], u[1], 0x5410);
    w1 = __byte_perm(u[2], u[3], 0x5410);
}

// Where a vector's bf16 row lives: kind 1 the recent ring, kind 2 the new
// input (converted to bf16 as it is read); anything else reads as zeros.
struct ExactSrc {
    const uint16_t* recent;
    const void* src_new;
    int kv_dtype;
    int kind;
    int64_t off;
};

// One fp32 column of this thread's tensor-memory lane (warp-collective: the
// column must be the same in every lane).
__device__ __forceinline__ float load_col(uint32_t taddr) {
    uint32_t v;
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v) : "r"(taddr));
    tc5::wait_ld();
    return __uint_as_float(v);
}

}  // namespace tcq
}  // namespace oscar
