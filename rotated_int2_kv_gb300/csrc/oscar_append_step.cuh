// Per-vector pieces of the append path shared by the append kernels and the
// fused decode-step kernel: the exact quantise-and-store of one rotated head
// vector, the decode-step row resolution, and the one-block-per-vector
// rotation (thread c forms output channel c).
#pragma once

#include "oscar_append_common.cuh"

namespace oscar {

// Quantises one rotated head vector held by a warp (lane: channels lane·CPL ..
// lane·CPL + CPL - 1) and writes its codes and (s, z) pairs into the record.
// y came from a sequential fp32 FMA chain and lies within e of x·R rounded to
// fp32; every (s, z) or code decision that y ± e could change is taken again on
// y values formed by the compensated dot product of xk (the vector's bf16
// elements) with the columns of R (row-major, row stride D).
template <int D, class XF>
__device__ __forceinline__ void quantize_store(const AppendParams& P, float (&y)[D / 32], int slot, int h, int mat,
                                               int lane, float e, XF xk, const float* R) {
    constexpr int CPL = D / 32;
    const int lpg = P.G / CPL;       // lanes per group (4..32)
    const float r = P.clip;
    const int rec_off_codes = mat ? D / 4 : 0;
    const int ng = D / P.G;
    const bool fp8 = P.fp8 != 0;
    const int rec_off_sz = D / 2 + (mat ? (fp8 ? 2 : 4) * ng : 0);
    auto group_extremes = [&](float& mn, float& mx) {
        mn = y[0];
        mx = y[0];
#pragma unroll
        for (int j = 1; j < CPL; ++j) { mn = fminf(mn, y[j]); mx = fmaxf(mx, y[j]); }
        for (int off = 1; off < lpg; off <<= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        }
    };
    float mn, mx;
    group_extremes(mn, mx);
    uint32_t exact = 0;              // channels j of this lane whose y is already the compensated one
    const bool unc = sz_uncertain(mn, mx, r, e, fp8);
    if (__any_sync(0xffffffffu, unc)) {
        // the extremes of an uncertain group lie among its channels within 2e of
        // the computed ones: form those exactly and take the extremes again
        const float tlo = __fadd_ru(mn, __fmul_ru(2.0f, e)), thi = __fsub_rd(mx, __fmul_ru(2.0f, e));
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            uint32_t m = __ballot_sync(0xffffffffu, unc && (y[j] <= tlo || y[j] >= thi));
            while (m) {
                const int L = __ffs(m) - 1;
                m &= m - 1;
                const float ye = dot2_warp<D>(xk, R, D, L * CPL + j, lane);
                if (lane == L) {
                    y[j] = ye;
                    exact |= 1u << j;
                }
            }
        }
        group_extremes(mn, mx);
    }
    const SZ sz = sz_decide(mn, mx, r, fp8);
    const float s = sz.s, z = sz.z;
    const float band = s != 0.0f ? code_band(e, __frcp_rn(3.0f * s)) : 0.0f;
    uint32_t bits = 0;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        float u = s != 0.0f ? __fdiv_rn(__fsub_rn(y[j], z), s) : 0.0f;
        uint32_t m = __ballot_sync(0xffffffffu, s != 0.0f && !((exact >> j) & 1u) && code_near_boundary(u, band));
        while (m) {
            const int L = __ffs(m) - 1;
            m &= m - 1;
            const float ye = dot2_warp<D>(xk, R, D, L * CPL + j, lane);
            if (lane == L) u = __fdiv_rn(__fsub_rn(ye, z), s);
        }
        const uint32_t c = s != 0.0f ? (uint32_t)fminf(fmaxf(rintf(u), 0.0f), 3.0f) : 0u;
        bits |= c << (2 * j);
    }
    uint8_t* rec = P.records + (int64_t)slot * P.slot_bytes + (int64_t)h * P.rec_bytes;
    if (CPL >= 4) {
#pragma unroll
        for (int bj = 0; bj < CPL / 4; ++bj)
            rec[rec_off_codes + lane * (CPL / 4) + bj] = (uint8_t)(bits >> (8 * bj));
    } else {  // CPL == 2: two lanes share a byte
        const uint32_t other = __shfl_xor_sync(0xffffffffu, bits, 1);
        if ((lane & 1) == 0) rec[rec_off_codes + lane / 2] = (uint8_t)(bits | (other << 4));
    }
    if ((lane % lpg) == 0) store_sz(rec, rec_off_sz, lane / lpg, sz, fp8);
}

// Σ x² of a vector, summed over the warp (lane: channels lane·CPL ..).
template <int CPL>
__device__ __forceinline__ float warp_sum_sq(const float (&x)[CPL]) {
    float q = 0.0f;
#pragma unroll
    for (int j = 0; j < CPL; ++j) q = fmaf(x[j], x[j], q);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) q += __shfl_xor_sync(0xffffffffu, q, off);
    return q;
}

// 32 consecutive rows of one column of a 256-wide fp32 matrix (row stride 1024
// bytes), all loads issued back to back in one statement.
__device__ __forceinline__ void ld32_col256(const float* p, float (&r)[32]) {
    asm volatile(
        "ld.global.nc.f32 %0, [%32+0];\n\t"
        "ld.global.nc.f32 %1, [%32+1024];\n\t"
        "ld.global.nc.f32 %2, [%32+2048];\n\t"
        "ld.global.nc.f32 %3, [%32+3072];\n\t"
        "ld.global.nc.f32 %4, [%32+4096];\n\t"
        "ld.global.nc.f32 %5, [%32+5120];\n\t"
        "ld.global.nc.f32 %6, [%32+6144];\n\t"
        "ld.global.nc.f32 %7, [%32+7168];\n\t"
        "ld.global.nc.f32 %8, [%32+8192];\n\t"
        "ld.global.nc.f32 %9, [%32+9216];\n\t"
        "ld.global.nc.f32 %10, [%32+10240];\n\t"
        "ld.global.nc.f32 %11, [%32+11264];\n\t"
        "ld.global.nc.f32 %12, [%32+12288];\n\t"
        "ld.global.nc.f32 %13, [%32+13312];\n\t"
        "ld.global.nc.f32 %14, [%32+14336];\n\t"
        "ld.global.nc.f32 %15, [%32+15360];\n\t"
        "ld.global.nc.f32 %16, [%32+16384];\n\t"
        "ld.global.nc.f32 %17, [%32+17408];\n\t"
        "ld.global.nc.f32 %18, [%32+18432];\n\t"
        "ld.global.nc.f32 %19, [%32+19456];\n\t"
        "ld.global.nc.f32 %20, [%32+20480];\n\t"
        "ld.global.nc.f32 %21, [%32+21504];\n\t"
        "ld.global.nc.f32 %22, [%32+22528];\n\t"
        "ld.global.nc.f32 %23, [%32+23552];\n\t"
        "ld.global.nc.f32 %24, [%32+24576];\n\t"
        "ld.global.nc.f32 %25, [%32+25600];\n\t"
        "ld.global.nc.f32 %26, [%32+26624];\n\t"
        "ld.global.nc.f32 %27, [%32+27648];\n\t"
        "ld.global.nc.f32 %28, [%32+28672];\n\t"
        "ld.global.nc.f32 %29, [%32+29696];\n\t"
        "ld.global.nc.f32 %30, [%32+30720];\n\t"
        "ld.global.nc.f32 %31, [%32+31744];\n\t"
        : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7]), "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]), "=f"(r[13]), "=f"(r[14]), "=f"(r[15]), "=f"(r[16]), "=f"(r[17]), "=f"(r[18]), "=f"(r[19]), "=f"(r[20]), "=f"(r[21]), "=f"(r[22]), "=f"(r[23]), "=f"(r[24]), "=f"(r[25]), "=f"(r[26]), "=f"(r[27]), "=f"(r[28]), "=f"(r[29]), "=f"(r[30]), "=f"(r[31])
        : "l"(p));
}

// ---------------------------------------------------------------------------
// Decode-step appends in one launch.  When a call appends at most W tokens in
// total, every request's new tokens all land in a BF16 window (sink below S,
// else the ring), and the tokens leaving the window are exactly the positions
// q = p - W >= S of the new positions p: position q's ring row p % W is the one
// that new position p overwrites.  So one warp per (new token, KV head) reads
// the leaving row, writes the new row over it, and quantises the leaving row
// into its history record (each lane reads and then writes the same elements,
// which orders the two), in place of the quantise kernel followed by the
// window copy.
// ---------------------------------------------------------------------------

// Resolves new row t (K or V of head h) of a decode-step append: request b,
// position p, window row rq; false (with status bits) when the row is invalid.
__device__ __forceinline__ bool resolve_new_row(const AppendParams& P, int64_t t, int& b, int& p, int& rq, int& bits) {
    b = find_request(P.cu_new, P.batch, (int)t);
    const int L0 = P.start_pos[b];
    const int c0 = P.cu_new[b], n = P.cu_new[b + 1] - c0;
    p = L0 + (int)(t - c0);
    rq = P.req_idx ? P.req_idx[b] : b;
    bits = 0;
    if (L0 < 0 || t - c0 >= n) bits |= OSCAR_DEV_BAD_LEN;
    if (rq < 0 || rq >= P.max_reqs) bits |= OSCAR_DEV_BAD_REQ;
    return bits == 0;
}

// Row of position p (K or V of head h) in the sink or the recent ring of window row rq.
__device__ __forceinline__ int64_t window_row(const AppendParams& P, int rq, int p, int h, int mat, int D) {
    return p < P.S ? ((((int64_t)rq * P.S + p) * P.Hkv + h) * 2 + mat) * D
                   : ((((int64_t)rq * P.W + p % P.W) * P.Hkv + h) * 2 + mat) * D;
}

// Slot of the history record of position q of request b, or -1 (with status bits).
__device__ __forceinline__ int history_slot(const AppendParams& P, int b, int q, int& bits) {
    if (q >= P.pt_stride) {
        bits |= OSCAR_DEV_BAD_LEN;
        return -1;
    }
    const int sl = P.page_table[(int64_t)b * P.pt_stride + q];
    if (sl < 0 || sl >= P.num_slots) {
        bits |= OSCAR_DEV_BAD_SLOT;
        return -1;
    }
    return sl;
}

// One decode-step vector (new token t, KV head h, K or V) by a block of at
// least 64 threads, thread i taking elements i, i + blockDim, ...: reads the
// row leaving the recent window (position p - W, if it enters the history),
// writes the new row over it, and quantises the leaving row into its record.  y[c] = Σ_k x_k·R[k][c]
// with k sequential (the order of the other CUDA-core kernels: bit-identical
// y); rows of R are read as coalesced lines, 32 in flight.  sx, sy: D floats
// of shared memory each.  Every thread of the block calls it (block barriers).
// The vector after its resolution: input row t is position p of request b
// (window row rq); ok false skips it, with `bits` reported.
template <int D>
__device__ __forceinline__ void append_vec_resolved(const AppendParams& P, int64_t t, int h, int mat, int b, int p,
                                                    int rq, bool ok, int bits, float* sx, float* sy) {
    constexpr int CPL = D / 32;
    const float* R = mat ? P.rot_v : P.rot_k;
    const void* src_new = mat ? P.v : P.k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nth = blockDim.x;                      // threads take elements tid, tid + nth, ...
    const int q = p - P.W;
    const bool spill = ok && q >= P.S;
    const int slot = spill ? history_slot(P, b, q, bits) : -1;
    // every element this thread owns is read before any is written: the new row
    // goes over the leaving one
    float xs[(D + 63) / 64];
#pragma unroll
    for (int u = 0; u < (D + 63) / 64; ++u) {
        const int c = tid + nth * u;
        xs[u] = spill && c < D && u * nth < D ? bf16_bits_to_f32(P.recent[window_row(P, rq, q, h, mat, D) + c]) : 0.f;
    }
    if (ok) {
        for (int c = tid; c < D; c += nth) {
            const float xn = load_elem(src_new, (t * P.Hkv + h) * D + c, P.kv_dtype);
            (p < P.S ? P.sink : P.recent)[window_row(P, rq, p, h, mat, D) + c] = f32_to_bf16_bits(xn);
        }
    }
    if (bits && tid == 0) set_status(P.status, bits);
    if (slot < 0) return;                            // the same decision in every thread
#pragma unroll
    for (int u = 0; u < (D + 63) / 64; ++u) {
        const int c = tid + nth * u;
        if (c < D && u * nth < D) sx[c] = xs[u];
    }
    __syncthreads();
    for (int c = tid; c < D; c += nth) {
        float y = 0.f;
        const float* rc = R + c;
        for (int k0 = 0; k0 < D; k0 += 32) {         // 32 rows of R in flight, then their FMAs in order
            float r[32];
            if constexpr (D == 256) {
                ld32_col256(rc + (int64_t)k0 * D, r);
            } else {
#pragma unroll
                for (int u = 0; u < 32; ++u) r[u] = __ldg(rc + (int64_t)(k0 + u) * D);
            }
#pragma unroll
            for (int u = 0; u < 32; ++u) y = fmaf(sx[k0 + u], r[u], y);
        }
        sy[c] = y;
    }
    __syncthreads();
    if (warp == 0) {
        float yv[CPL], xv[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            yv[j] = sy[lane * CPL + j];
            xv[j] = sx[lane * CPL + j];
        }
        const float eb = fma_chain_bound<D>(warp_sum_sq<CPL>(xv));
        quantize_store<D>(P, yv, slot, h, mat, lane, eb, [&](int k) { return sx[k]; }, R);
    }
    __syncthreads();                                 // sx and sy may be reused
}

template <int D>
__device__ __forceinline__ void append_vec_item(const AppendParams& P, int64_t t, int h, int mat, float* sx,
                                                float* sy) {
    int b, p, rq, bits;
    const bool ok = resolve_new_row(P, t, b, p, rq, bits);
    append_vec_resolved<D>(P, t, h, mat, b, p, rq, ok, bits, sx, sy);
}

}  // namespace oscar
