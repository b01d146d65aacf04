// Shared declarations of the append kernels (quantise-on-append).
#pragma once

#include <cuda_fp8.h>

#include "oscar_internal.h"
#include "oscar_device.cuh"

namespace oscar {

constexpr int kMaxAppendBatch = 4096;
constexpr int kTileVec = 64;        // head vectors per tile (one matrix: K or V)
constexpr int kColBlock = 64;       // columns of R per GEMM pass
constexpr int kAppendThreads = 256;

struct AppendParams {
    const void* k;
    const void* v;
    int kv_dtype;
    const int32_t* cu_new;
    const int32_t* start_pos;
    const int32_t* req_idx;
    const int32_t* page_table;
    int64_t pt_stride;
    int batch;
    uint8_t* records;
    uint16_t* sink;
    uint16_t* recent;
    const float* rot_k;
    const float* rot_v;
    int64_t num_slots;
    int max_reqs;
    int Hkv, S, W, G, rec_bytes;
    int64_t slot_bytes;         // pool stride of one slot (all KV heads)
    int fp8;                    // (s, z) stored as E4M3 pairs (else fp16 pairs)
    float clip;
    int64_t total_new;
    int* status;
};

__device__ __forceinline__ int hist_hi(int L, int S, int W) { return max(S, L - W); }

// Exclusive prefix over requests of the number of positions entering the
// history; prefix[batch] is the total.  All threads of the block participate.
__device__ __forceinline__ void build_prefix(const AppendParams& P, int* prefix, int* scratch) {
    const int tid = threadIdx.x;
    const int per = (P.batch + blockDim.x - 1) / blockDim.x;
    const int b0 = min(P.batch, tid * per), b1 = min(P.batch, b0 + per);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
        const int L0 = P.start_pos[b];
        const int n = P.cu_new[b + 1] - P.cu_new[b];
        int cnt = 0;
        if (L0 < 0 || n < 0) {
            set_status(P.status, OSCAR_DEV_BAD_LEN);
        } else {
            cnt = hist_hi(L0 + n, P.S, P.W) - hist_hi(L0, P.S, P.W);
        }
        prefix[b] = cnt;  // temporarily the count
        local += cnt;
    }
    int total;
    int run = block_exclusive_scan(local, scratch, &total);
    for (int b = b0; b < b1; ++b) {
        const int c = prefix[b];
        prefix[b] = run;
        run += c;
    }
    if (tid == 0) prefix[P.batch] = total;
    __syncthreads();
}

// Largest b with prefix[b] <= u (prefix non-decreasing, prefix[0] = 0).
__device__ __forceinline__ int find_request(const int* prefix, int batch, int u) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ---- exact code decisions -------------------------------------------------
//
// The codes and (s, z) of a vector are a function of y = x·R rounded to fp32.
// The kernels form y with fp32 accumulation, so their y may differ from that
// value by a bounded amount e.  Every decision below is a monotone function of
// the y values it reads (fp32 operations and fp16 rounding are monotone), so a
// decision taken at both ends of [y - e, y + e] that comes out the same is the
// decision of the exact y.  Where the two ends disagree, the y values that
// decide it are formed again with a compensated dot product (Ogita, Rump and
// Oishi's Dot2: error-free products and sums carried in a second fp32 word),
// which is faithful to the exact product, and the decision is taken on them.

// Storage rounding of a scale or zero: fp16 (nearest even), or float8 E4M3
// (nearest even, finite values beyond ±448 saturated).  Returns the stored bit
// pattern (16 or 8 bits); both roundings are monotone in x.
__device__ __forceinline__ uint32_t sz_bits(float x, bool fp8) {
    return fp8 ? (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3)
               : (uint32_t)__half_as_ushort(__float2half_rn(x));
}

// Value of a stored scale or zero (exact in fp32 for both formats).
__device__ __forceinline__ float sz_value(uint32_t bits, bool fp8) {
    if (fp8) {
        const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)bits, __NV_E4M3);
        return __half2float(__half(h));
    }
    return __half2float(__ushort_as_half((unsigned short)bits));
}

// A group's stored (scale, zero) from its extremes, in the order the quantiser
// defines: lo = r·min, hi = r·max, s = rnd((hi - lo)/3), z = rnd(lo), with rnd
// the fp16 or E4M3 rounding; returns the bit patterns and their values.
struct SZ {
    uint32_t sb, zb;
    float s, z;
};
__device__ __forceinline__ SZ sz_decide(float mn, float mx, float r, bool fp8) {
    const float lo = __fmul_rn(r, mn);
    const float hi = __fmul_rn(r, mx);
    SZ o;
    o.sb = sz_bits(__fdiv_rn(__fsub_rn(hi, lo), 3.0f), fp8);
    o.zb = sz_bits(lo, fp8);
    o.s = sz_value(o.sb, fp8);
    o.z = sz_value(o.zb, fp8);
    return o;
}

// Writes the pair of group gi at byte `off` of a record: fp16 pairs (4 bytes,
// 4-byte aligned) or E4M3 pairs (2 bytes, 2-byte aligned), scale first.
__device__ __forceinline__ void store_sz(uint8_t* rec, int off, int gi, const SZ& v, bool fp8) {
    if (fp8) *reinterpret_cast<uint16_t*>(rec + off + 2 * gi) = (uint16_t)(v.sb | (v.zb << 8));
    else *reinterpret_cast<uint32_t*>(rec + off + 4 * gi) = v.sb | (v.zb << 16);
}

// True when extremes anywhere in [mn - e, mn + e] × [mx - e, mx + e] could give
// another (s, z).  Every step of sz_decide is monotone, so the oracle's values
// at any point of that box lie in intervals bounded with directed rounding:
// lo in [rd(r·(mn - e)), ru(r·(mn + e))], and (hi - lo)/3 in
// [rd((rd(r·(mx - e)) - ru(r·(mn + e)))·⅓↓), ru((ru(r·(mx + e)) - rd(r·(mn - e)))·⅓↑)];
// the decision is certain when both ends of each interval round to the same
// stored value (fp16 or E4M3).
__device__ __forceinline__ bool sz_uncertain(float mn, float mx, float r, float e, bool fp8) {
    constexpr float kThirdDn = 0.333333313465118408203125f;   // the fp32 neighbours of 1/3
    constexpr float kThirdUp = 0.3333333432674407958984375f;
    const float lo_a = __fmul_rd(r, __fsub_rd(mn, e)), lo_b = __fmul_ru(r, __fadd_ru(mn, e));
    const float hi_a = __fmul_rd(r, __fsub_rd(mx, e)), hi_b = __fmul_ru(r, __fadd_ru(mx, e));
    const float s_a = __fmul_rd(__fsub_rd(hi_a, lo_b), kThirdDn);
    const float s_b = __fmul_ru(__fsub_ru(hi_b, lo_a), kThirdUp);
    return sz_bits(lo_a, fp8) != sz_bits(lo_b, fp8) || sz_bits(fmaxf(s_a, 0.0f), fp8) != sz_bits(s_b, fp8);
}

// Half-width in units of the quotient u = (y - z)/s of the band around a
// rounding boundary (0.5, 1.5, 2.5) inside which y ± e may decide another code:
// e/s plus the roundings of y - z and of the division (2^-21 relative for |u|
// up to 3), with margin.  r3 is the fp32 reciprocal of 3s (within half an ulp),
// so 3e·r3 is e/s to 2^-22.
__device__ __forceinline__ float code_band(float e, float r3) {
    return __fmaf_ru(__fmul_ru(3.0f * e, r3), 1.0f + 1.0f / 1048576.0f, 1.0f / 524288.0f);
}

// True when the correctly rounded quotient u lies within `band` of a rounding
// boundary that changes the clamped code.
__device__ __forceinline__ bool code_near_boundary(float u, float band) {
    const float d = fminf(fminf(fabsf(u - 0.5f), fabsf(u - 1.5f)), fabsf(u - 2.5f));
    return d <= band;
}

// Σ_k x_k·R[k][j] over k < D, faithfully rounded (compensated), by the whole
// warp: lane l takes k = l, l + 32, ...; every lane returns the result.  xk(k)
// returns the bf16-exact input element k; R is row-major with row stride ldr.
template <int D, class XF>
__device__ __noinline__ float dot2_warp(XF xk, const float* R, int ldr, int j, int lane) {
    float s = 0.0f, c = 0.0f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
        const int k = lane + 32 * i;
        const float a = xk(k), b = R[(int64_t)k * ldr + j];
        const float p = __fmul_rn(a, b);
        const float pe = __fmaf_rn(a, b, -p);                       // a·b = p + pe exactly
        const float t = __fadd_rn(s, p);
        const float bp = __fsub_rn(t, s);
        const float er = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(p, bp));   // s + p = t + er
        s = t;
        c = __fadd_rn(c, __fadd_rn(er, pe));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float so = __shfl_xor_sync(0xffffffffu, s, off);
        const float co = __shfl_xor_sync(0xffffffffu, c, off);
        const float t = __fadd_rn(s, so);
        const float bp = __fsub_rn(t, s);
        const float er = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(so, bp));
        s = t;
        c = __fadd_rn(__fadd_rn(c, co), er);
    }
    return __fadd_rn(s, c);
}

// Bound on |y_j - fl(x·R_j)| for every channel j of a vector whose y was formed
// by a sequential fp32 FMA chain over k < D (D roundings), given Σ x_k²:
// γ_D·Σ_k |x_k||R_kj| <= γ_D·‖x‖₂·‖R_j‖₂ (R orthogonal: ‖R_j‖₂ = 1 up to
// rounding), plus half an ulp of the rounded result (<= 2^-24·‖x‖₂), with a
// 1% margin for R's rounding and the evaluation of the norm.
template <int D>
__device__ __forceinline__ float fma_chain_bound(float x_sq) {
    constexpr float k = 1.01f * (float)(D + 2) / 16777216.0f;
    return k * sqrtf(x_sq);
}

// Tensor-core rotation + quantisation of large appends (head_dim 64 or 128);
// returns OSCAR_OK after launching, or a negative status.
template <int D>
int launch_quantize_tc(const AppendParams& P, int64_t max_vec, cudaStream_t stream);

// Tensor-core rotation + quantisation of large appends at head_dim 256 (groups
// of 32, 64 or 128 channels); returns OSCAR_OK after launching, or a negative status.
int launch_quantize_tc256(const AppendParams& P, int64_t max_vec, cudaStream_t stream);

}  // namespace oscar
