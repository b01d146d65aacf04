// Tensor-core rotation and quantisation of large appends at head_dim 256
// (prefill chunks of wide-head layers, e.g. the [Escha log] 27B layer with
// CHUNK 8192).
//
// [OSCAR news] "OSCARの違い" / "サービングシステム：混合精度キャッシュレイアウト":
// every head vector entering the INT2 history is rotated, y = x·R, then
// clipped and quantised per group.
//
// At d = 256 the three bf16 parts of R that the head_dim <= 128 kernel keeps in
// shared memory (384 KB) do not fit, so each CTA takes one half of the output
// channels (blockIdx.z; a group of at most 128 channels never straddles two
// halves) and R's half in two bf16 parts, hi = bf16(R) and lo = bf16(R - hi),
// 128 KB as the B operand (N = 128 channels × K = 256, K-major, 128-byte
// swizzle).  One warpgroup per CTA: a tile of 128 vectors (the A operand, 64
// KB) is multiplied into one 128-column fp32 accumulator in tensor memory (lo
// parts first), and while thread i quantises vector i from its tensor-memory
// lane, the next tile's rows are already loading (one tensor-map TMA load per
// 64 channels when they are a contiguous block of the bf16 input, else 16-byte
// cp.async per chunk).
//
// Exact decisions as in the head_dim <= 128 kernel: y differs from x·R rounded
// to fp32 by at most e = (kAcc256 + ρ)·‖x‖₂, the sum of the accumulation bound of
// kind::f16 (twice the one measured over 8 k-steps, for 16 k-steps, plus 1 ulp
// of the result) and the two-part residual: with r = R - hi - lo,
// |Σ_k x_k r[k][c]| <= ‖x‖₂·‖r[:, c]‖₂ (Cauchy-Schwarz), and ρ, the largest
// column norm of r over the CTA's channels, is formed from R itself when the
// parts are built (rounded up).  Elementwise |r| reaches 2^-17·|R|, so ρ
// depends on R; for a dense orthogonal R of order 256 it is about 50·2^-24.
// Any (s, z) or code decision that y ± e could change is taken again on y
// formed by a compensated dot product of the input row with R's fp32 column.
//
// For the (s, z) decisions those products run on chip and in parallel: R's
// half is also kept in tensor memory in fp32, each group of 8 lanes holding
// the eight 32-k parts of eight channels (see rt_exact_dots), a vector with an
// uncertain group copies its bf16 row from the x tile into shared memory
// before the next tile overwrites it, and each candidate (vector, channel) is
// queued to the lane group that holds the channel, whose lanes form 32-term
// parts of the product and add them.  A request that finds its channel's queue
// or the row stash full takes the warp-serial path over global memory instead.
#include <algorithm>
#include <cstring>

#include <cuda.h>

#include "oscar_append_tc_common.cuh"

namespace oscar {

bool tc_encode_rows(CUtensorMap* m, const void* base, int64_t rows, int d);

namespace {

using namespace tcq;

constexpr int kD = 256;                           // input channels: K of the MMA
constexpr int kN = 128;                           // output channels per CTA: one half of y
constexpr int kKS = kD / 16;                      // k-steps of 16
constexpr int kThreads = 128;                     // one warpgroup: thread i owns tile row i
constexpr uint32_t kCols = 512;                   // tensor-memory columns: accumulator 0 .. 127, R's half 256 .. 511
constexpr uint32_t kRtCol = 256;                  // first column of R's half in tensor memory (fp32)
constexpr int kQ = 12;                            // exact-y requests one channel takes per batch
constexpr int kXS = kD + 8;                       // stride of a stashed bf16 row (528 B: rows on different banks)
constexpr int kABytes = kTcRows * kD * 2;         // one x tile (64 KB)
constexpr int kBPart = kN * kD * 2;               // one part of R's half (64 KB)
constexpr int kCPR = kD / 8;                      // 16-byte chunks per input row (32)
constexpr size_t kSmem = 1024 + 2 * (size_t)kBPart + kABytes + (size_t)2 * kTcRows * kMetaInts * 4 + 128;
// accumulation part of the bound on |y - fl(x·R)| / ‖x‖₂: 2·kTcErr + 1 ulp of the
// result, in units of 2^-24 (the residual part ρ is added per CTA; 1% margin on both)
constexpr float kAcc256 = (2.0f * kTcErr + 1.0f) / 16777216.0f;

__device__ __forceinline__ void cta_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ bool cta_bar_or(bool v) {
    int r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, 1, 128, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((int)v) : "memory");
    return r != 0;
}

// fl(x·R[:, ch]) (compensated, faithful to the exact product) for the vector of
// lane L, by the whole warp: lane l takes k = 8l .. 8l + 7, x from the vector's
// row in global memory, R's fp32 column ch from global memory.
__device__ __forceinline__ float tc256_dot2(const float* R, const ExactSrc& src, int L, int ch, int lane) {
    constexpr int KPL = kD / 32;
    const int kd = __shfl_sync(0xffffffffu, src.kind, L);
    const uint32_t olo = __shfl_sync(0xffffffffu, (uint32_t)(uint64_t)src.off, L);
    const uint32_t ohi = __shfl_sync(0xffffffffu, (uint32_t)((uint64_t)src.off >> 32), L);
    const int64_t o = (int64_t)(((uint64_t)ohi << 32) | olo) + lane * KPL;
    const int k0 = lane * KPL;
    float x[KPL], r[KPL];
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
        x[i] = kd == 1 ? bf16_bits_to_f32(src.recent[o + i])
             : kd == 2 ? bf16_bits_to_f32(f32_to_bf16_bits(load_elem(src.src_new, o + i, src.kv_dtype)))
                       : 0.0f;
        r[i] = __ldg(R + (int64_t)(k0 + i) * kD + ch);
    }
    float s = 0.0f, c = 0.0f;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
        const float pr = __fmul_rn(x[i], r[i]);
        const float pe = __fmaf_rn(x[i], r[i], -pr);                 // x·r = pr + pe exactly
        const float t = __fadd_rn(s, pr);
        const float bp = __fsub_rn(t, s);
        const float er = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(pr, bp));
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

// Exact extremes of one group for the lanes whose (s, z) y ± e could change
// (warp-collective, out of line): the candidates are the channels within 2e of
// the computed extremes (y reloaded from the group's tensor-memory columns
// tgrp); ch0 is the group's first channel of y (global index).
template <int G>
__device__ __noinline__ float2 tc256_exact_extremes(uint32_t tgrp, const float* R, ExactSrc src, bool unc, float mn,
                                                    float mx, float e2, int ch0, int lane) {
    const float tlo = __fadd_ru(mn, e2), thi = __fsub_rd(mx, e2);
    float mne = INFINITY, mxe = -INFINITY;
#pragma unroll 1
    for (int c = 0; c < G / 32; ++c) {
        float y[32];
        load_y(tgrp + 32 * c, y);
        uint32_t cm = 0;
#pragma unroll
        for (int q = 0; q < 32; ++q) cm |= (unc && (y[q] <= tlo || y[q] >= thi)) ? (1u << q) : 0u;
        uint32_t bal;
        while ((bal = __ballot_sync(0xffffffffu, cm != 0u)) != 0u) {
            const int L = __ffs(bal) - 1;
            const int q = __shfl_sync(0xffffffffu, __ffs(cm) - 1, L);
            const float ye = tc256_dot2(R, src, L, ch0 + 32 * c + q, lane);
            if (lane == L) {
                cm &= cm - 1u;
                mne = fminf(mne, ye);
                mxe = fmaxf(mxe, ye);
            }
        }
    }
    return make_float2(mne, mxe);
}

// Shared-memory queues of one batch of on-chip exact products.
struct RtQueues {
    int* cnt;                 // [kN] requests queued to each channel
    int* vec;                 // [kN][kQ] stash row of each request
    float* y;                 // [kN][kQ] its exact y
    const uint16_t* xs;       // stashed bf16 rows [xcap][kXS]
};

__device__ __forceinline__ void dot2_step(float& s, float& c, float x, float r) {
    const float p = __fmul_rn(x, r);
    const float pe = __fmaf_rn(x, r, -p);                            // x·r = p + pe exactly
    const float t = __fadd_rn(s, p);
    const float bp = __fsub_rn(t, s);
    const float er = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(p, bp));   // s + p = t + er
    s = t;
    c = __fadd_rn(c, __fadd_rn(er, pe));
}

// R's half in tensor memory: the kLPC lanes of a lane group (lanes kLPC·i ..
// kLPC·i + kLPC - 1 of warp w) hold the kLPC parts (kKP consecutive k each) of
// the same kLPC channels; lane L holds, for m = 0 .. kLPC - 1, part L mod kLPC of
// channel 32w + L/kLPC + (32/kLPC)·m of the half, R[kKP·(L mod kLPC) + kk][..]
// at column kRtCol + kKP·m + kk (kk < kKP).  One exact product is split over
// the lanes of a group.
constexpr int kLPC = 8;                           // lanes per channel
constexpr int kKP = kD / kLPC;                    // k per lane (32)
static_assert(kKP == 32 && 32 % kLPC == 0, "one 32-column tensor-memory load per channel");

// fl(x·R[:, ch]) for every stashed row queued to the channels of this thread's
// lane group (cnt, vec: the queues; yq: the results, [kN][kQ]): each lane forms
// the compensated dot product over its kKP k in order, and the group sums its
// (sum, error) pairs with log2(kLPC) compensated shuffle steps.  Warp-collective
// (tensor-memory loads, shuffles): every thread of the warp calls it.
__device__ __noinline__ void rt_exact_dots(uint32_t trt, const uint16_t* xs, const int* cnt, const int* vec,
                                           float* yq, int warp, int lane) {
    const int part = lane % kLPC, ci = lane / kLPC;
#pragma unroll 1
    for (int m = 0; m < kLPC; ++m) {
        const int ch = 32 * warp + ci + (32 / kLPC) * m;   // channel of the half
        const int n = min(cnt[ch], kQ);
        const int nmax = __reduce_max_sync(0xffffffffu, n);
        if (nmax == 0) continue;                    // warp-uniform
        float rr[32];
        tc5::ld32(trt + kKP * m, rr);
        tc5::wait_ld();
#pragma unroll 1
        for (int r = 0; r < nmax; ++r) {
            float s = 0.0f, c = 0.0f;
            if (r < n) {
                const uint4* p = reinterpret_cast<const uint4*>(xs + (int64_t)vec[ch * kQ + r] * kXS + kKP * part);
#pragma unroll
                for (int w = 0; w < kKP / 8; ++w) {
                    const uint4 u = p[w];
                    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        dot2_step(s, c, __uint_as_float(wd[i] << 16), rr[8 * w + 2 * i]);
                        dot2_step(s, c, __uint_as_float(wd[i] & 0xFFFF0000u), rr[8 * w + 2 * i + 1]);
                    }
                }
            }
#pragma unroll
            for (int off = 1; off < kLPC; off <<= 1) {  // the group's partial sums
                const float so = __shfl_xor_sync(0xffffffffu, s, off);
                const float co = __shfl_xor_sync(0xffffffffu, c, off);
                const float t = __fadd_rn(s, so);
                const float bp = __fsub_rn(t, s);
                const float er = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(so, bp));
                s = t;
                c = __fadd_rn(__fadd_rn(c, co), er);
            }
            if (part == 0 && r < n) yq[ch * kQ + r] = __fadd_rn(s, c);
        }
    }
}

// Exact extremes of one group for the threads whose (s, z) y ± e could change,
// one batch for the whole CTA: every such thread queues its channels within 2e
// of the computed extremes (tensor-memory columns tgrp; lch0 / gch0: the
// group's first channel within the half / in y) with its stashed row xslot,
// the lane groups holding the channels form them, and the thread takes the min /
// max of its exact values.  A thread without a stashed row, or whose request
// does not fit a queue, takes the warp-serial path.  All threads call it (CTA
// barriers).
template <int G>
__device__ __noinline__ float2 rt_exact_extremes(RtQueues Q, uint32_t tgrp, uint32_t trt, bool unc, int xslot,
                                                 float mn, float mx, float e2, int lch0, int gch0, const float* R,
                                                 ExactSrc xsrc, int tid, int lane) {
    const float tlo = __fadd_ru(mn, e2), thi = __fsub_rd(mx, e2);
    bool over = unc && xslot < 0;
    uint64_t mine = 0;                             // (channel | slot << 7) of each request, 12 bits apiece
    static_assert(kQ <= 16 && kN <= 128, "a request fits 12 bits");
    int nm = 0;
#pragma unroll 1
    for (int c = 0; c < G / 32; ++c) {
        float y[32];
        load_y(tgrp + 32 * c, y);
        uint32_t cm = 0;
#pragma unroll
        for (int q = 0; q < 32; ++q) cm |= (unc && (y[q] <= tlo || y[q] >= thi)) ? (1u << q) : 0u;
        while (cm && !over) {
            const int ch = lch0 + 32 * c + __ffs(cm) - 1;
            cm &= cm - 1u;
            if (nm == 5) {                         // no room in `mine`: reserve nothing
                over = true;
                break;
            }
            const int sl = atomicAdd(Q.cnt + ch, 1);
            if (sl < kQ) {                         // every reserved slot below kQ is written
                Q.vec[ch * kQ + sl] = xslot;
                mine |= (uint64_t)(ch | (sl << 7)) << (12 * nm);
                ++nm;
            } else {
                over = true;
            }
        }
    }
    cta_bar();                                     // every request queued
    rt_exact_dots(trt, Q.xs, Q.cnt, Q.vec, Q.y, tid >> 5, lane);
    cta_bar();                                     // every exact y formed; every count read
    Q.cnt[tid] = 0;                                // the next batch queues after a later barrier
    float mne = INFINITY, mxe = -INFINITY;
    if (unc && !over)
        for (int i = 0; i < nm; ++i) {
            const uint32_t en = (uint32_t)(mine >> (12 * i)) & 4095u;
            const float v = Q.y[(en & 127u) * kQ + (en >> 7)];
            mne = fminf(mne, v);
            mxe = fmaxf(mxe, v);
        }
    if (__any_sync(0xffffffffu, over)) {
        const float2 ex = tc256_exact_extremes<G>(tgrp, R, xsrc, over, mn, mx, e2, gch0, lane);
        if (over) {
            mne = ex.x;
            mxe = ex.y;
        }
    }
    return make_float2(mne, mxe);
}

// Re-decides the codes of one 32-channel chunk whose reciprocal-path quotient
// lies near a half-integer (warp-collective, out of line); ch0: the chunk's
// first channel of y (global index).
__device__ __noinline__ uint2 tc256_exact_codes(uint32_t tchunk, const float* R, ExactSrc src, float zc, float sc,
                                                float r3, float nb2, float be, uint2 w, int ch0, int lane) {
    float y[32];
    load_y(tchunk, y);
    uint32_t cm = 0;
#pragma unroll
    for (int q = 0; q < 32; ++q) {
        const float t = __saturatef(__fmul_rn(__fsub_rn(y[q], zc), r3));
        const float qq = __fmul_rn(t, 3.0f);
        const float dd = qq - rintf(qq);
        cm |= (__fmaf_rn(dd, dd, nb2) >= 0.0f ? 1u : 0u) << q;
    }
    uint32_t bal;
    while ((bal = __ballot_sync(0xffffffffu, cm != 0u)) != 0u) {
        const int L = __ffs(bal) - 1;
        const int q = __shfl_sync(0xffffffffu, __ffs(cm) - 1, L);
        const float yq = load_col(tchunk + q);
        float u = sc != 0.0f ? __fdiv_rn(__fsub_rn(yq, zc), sc) : 0.0f;
        if (__shfl_sync(0xffffffffu, (int)(sc != 0.0f && code_near_boundary(u, be)), L)) {
            const float ye = tc256_dot2(R, src, L, ch0 + q, lane);
            u = __fdiv_rn(__fsub_rn(ye, zc), sc);
        }
        if (lane == L) {
            cm &= cm - 1u;
            const uint32_t c = sc != 0.0f ? (uint32_t)fminf(fmaxf(rintf(u), 0.0f), 3.0f) : 0u;
            if (q < 16) w.x = (w.x & ~(3u << (2 * q))) | (c << (2 * q));
            else w.y = (w.y & ~(3u << (2 * q - 32))) | (c << (2 * q - 32));
        }
    }
    return w;
}

}  // namespace

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
quantize_tc256_kernel(AppendParams P, const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      int use_tma, int xcap) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    static_assert(kN % G == 0, "a group lies within one half of the channels");
    constexpr int ngh = kN / G;                     // groups in this CTA's half
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sB = smem;                                               // [2 parts][128 rows n][256 k] swizzled
    unsigned char* A = smem + 2 * kBPart;                                   // [128 rows][256 k] swizzled
    int* meta = reinterpret_cast<int*>(A + kABytes);                        // [2 buffers][128][4]
    uint64_t* bar = reinterpret_cast<uint64_t*>(meta + 2 * kTcRows * kMetaInts);   // MMAs done
    uint64_t* full = bar + 1;                                               // TMA rows landed
    uint32_t* tslot = reinterpret_cast<uint32_t*>(full + 1);
    int* prefix = reinterpret_cast<int*>(tslot + 2);                       // batch + 1
    int* scratch = prefix + P.batch + 1;                                    // kThreads
    int* nx = scratch + kThreads;                                           // rows stashed in this tile
    RtQueues Q;
    Q.cnt = nx + 4;                                                         // kN
    Q.vec = Q.cnt + kN;                                                     // kN × kQ
    Q.y = reinterpret_cast<float*>(Q.vec + kN * kQ);                        // kN × kQ
    uint16_t* xs = reinterpret_cast<uint16_t*>((reinterpret_cast<uintptr_t>(Q.y + kN * kQ) + 15) & ~uintptr_t(15));
    Q.xs = xs;                                                              // xcap × kXS

    const int mat = blockIdx.y, half = blockIdx.z;
    const float* R = mat ? P.rot_v : P.rot_k;
    const void* src_new = mat ? P.v : P.k;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gt = tid;                             // tile row = tensor-memory lane

    build_prefix(P, prefix, scratch);
    const int64_t total_vec = (int64_t)prefix[P.batch] * P.Hkv;
    const int64_t ntiles = (total_vec + kTcRows - 1) / kTcRows;
    if ((int64_t)blockIdx.x >= ntiles) return;    // uniform over the CTA, before any allocation

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(full, 1);
        fence_mbar_init();
        *nx = 0;
    }
    Q.cnt[tid] = 0;                                 // kThreads == kN
    if (warp == 0) {
        tc5::alloc(tslot, kCols);
        tc5::relinquish();
    }
    tc5::fence_before();
    __syncthreads();
    tc5::fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tacc = tmem + ((uint32_t)(32 * warp) << 16);   // this warp's lanes, column 0
    const uint32_t trt = tacc + kRtCol;             // this lane's share of R's half (lane-group layout)
    // B: the two parts of R[:, 128·half .. +127] as 128 rows n × 256 k.  Item (n, j)
    // reads R[8j .. 8j+7][128·half + n] and stores its 16-byte chunk of both parts.
    // Thread tid builds every chunk of channel n = tid (kThreads == kN) and sums
    // the squares of r = R - hi - lo over its column, rounding up.
    static_assert(kThreads == kN, "one channel of B per thread");
    constexpr int NB = kN * kCPR;
    static_assert(NB % (2 * kThreads) == 0, "every item of the loop below is in range");
    float rsq = 0.0f;
#pragma unroll 1
    for (int i0 = tid; i0 < NB; i0 += 2 * kThreads) {
        float v[2][8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = i0 + u * kThreads;
            const int n = i % kN, j = i / kN;
#pragma unroll
            for (int q = 0; q < 8; ++q) v[u][q] = R[(int64_t)(8 * j + q) * kD + kN * half + n];
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = i0 + u * kThreads;
            const int n = i % kN, j = i / kN;
#pragma unroll
            for (int p = 0; p < 2; ++p) {             // part 0: bf16(R), part 1: bf16(R - part 0)
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) w[q] = pack_bf16(bf16_part(v[u][2 * q], p), bf16_part(v[u][2 * q + 1], p));
                *reinterpret_cast<uint4*>(sB + p * kBPart + tc5::sw128_offset(kN, n, j)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {             // r = bf16_part(v, 2) exactly (R - hi and R - hi - lo are exact in fp32)
                const float r = bf16_part(v[u][q], 2);
                rsq = __fmaf_ru(r, r, rsq);
            }
        }
    }
    {   // R's half into tensor memory, lane-group layout (see rt_exact_dots): this
        // lane's part of its kLPC channels, 32 rows of R in flight
        const int part = lane % kLPC, ci = lane / kLPC;
#pragma unroll 1
        for (int m = 0; m < kLPC; ++m) {
            const float* src = R + (int64_t)(kKP * part) * kD + kN * half + 32 * warp + ci + (32 / kLPC) * m;
            float v[kKP];
#pragma unroll
            for (int i = 0; i < kKP; ++i) v[i] = __ldg(src + (int64_t)i * kD);
#pragma unroll
            for (int j = 0; j < kKP / 8; ++j) {
                uint32_t col[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) col[i] = __float_as_uint(v[8 * j + i]);
                tc5::st8(trt + kKP * m + 8 * j, col);   // the same columns in every lane
            }
        }
        tc5::wait_st();
    }
    {   // ρ: the largest column norm of r over this CTA's channels (scratch is free after build_prefix)
        float m = __fsqrt_ru(rsq);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) reinterpret_cast<float*>(scratch)[warp] = m;
    }
    tc5::fence_proxy_async();
    tc5::fence_before();
    __syncthreads();
    tc5::fence_after();
    float rho = 0.0f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) rho = fmaxf(rho, reinterpret_cast<const float*>(scratch)[w]);
    const float kBound = __fmul_ru(1.01f, __fadd_ru(kAcc256, rho));   // e = kBound·‖x‖₂

    const bool vec_in = (reinterpret_cast<uintptr_t>(src_new) & 15) == 0;
    const float rclip = P.clip;
    const bool fp8 = P.fp8 != 0;
    constexpr int ng = kD / G;                      // groups of the whole vector
    const int rec_off_codes = (mat ? kD / 4 : 0) + (kN / 4) * half;
    const int rec_off_sz = kD / 2 + (mat ? (fp8 ? 2 : 4) * ng : 0);
    const int gi0 = ngh * half;                     // first group of this half
    const CUtensorMap* tmap = mat ? &tm_v : &tm_k;

    // Vector gt of a tile is resolved in two stages one loop iteration apart (as
    // in the head_dim <= 128 kernel): locate() starts the page-table load,
    // publish() checks the slot and writes the entry.
    struct Loc {
        int b, p, h, sl;
        bool valid;
    };
    auto locate = [&](int64_t tile) {
        Loc L{0, 0, 0, -1, false};
        const int64_t ev = tile * kTcRows + gt;
        if (tile < ntiles && ev < total_vec) {
            const int u = (int)(ev / P.Hkv);
            L.h = (int)(ev % P.Hkv);
            L.b = find_request(prefix, P.batch, u);
            L.p = hist_hi(P.start_pos[L.b], P.S, P.W) + (u - prefix[L.b]);
            L.valid = true;
            if (L.p < P.pt_stride) L.sl = P.page_table[(int64_t)L.b * P.pt_stride + L.p];
        }
        return L;
    };
    auto publish = [&](const Loc& L, int buf) {
        int slot = -1, kind = 0;
        int64_t off = 0;
        if (L.valid) {
            const int b = L.b, p = L.p, h = L.h;
            const int L0 = P.start_pos[b];
            if (p >= P.pt_stride) set_status(P.status, OSCAR_DEV_BAD_LEN);
            else if (L.sl < 0 || L.sl >= P.num_slots) set_status(P.status, OSCAR_DEV_BAD_SLOT);
            else slot = L.sl;
            const int rq = P.req_idx ? P.req_idx[b] : b;
            if (p < L0 && (rq < 0 || rq >= P.max_reqs)) {
                set_status(P.status, OSCAR_DEV_BAD_REQ);
                slot = -1;
            }
            if (p >= L0 && (int64_t)P.cu_new[b] + (p - L0) >= P.total_new) {
                set_status(P.status, OSCAR_DEV_BAD_LEN);
                slot = -1;
            }
            if (slot >= 0) {
                if (p < L0) {
                    kind = 1;
                    off = ((((int64_t)rq * P.W + p % P.W) * P.Hkv + h) * 2 + mat) * kD;
                } else {
                    kind = 2;
                    off = ((int64_t)(P.cu_new[b] + (p - L0)) * P.Hkv + h) * kD;
                }
            }
        }
        int* m = meta + (buf * kTcRows + gt) * kMetaInts;
        m[0] = slot;
        m[1] = L.h | (kind << 16);
        *reinterpret_cast<int64_t*>(m + 2) = off;
    };
    // rows 32·warp .. +31 of a tile into the x tile, one row per warp instruction
    auto gather = [&](int buf) {
#pragma unroll 4
        for (int rr = 0; rr < 32; ++rr) {
            const int row = 32 * warp + rr, j = lane;
            unsigned char* dst = A + tc5::sw128_offset(kTcRows, row, j);
            const int4 m = *reinterpret_cast<const int4*>(meta + (buf * kTcRows + row) * kMetaInts);
            const int kind = m.y >> 16;
            const int64_t off = (int64_t)(((uint64_t)(uint32_t)m.w << 32) | (uint32_t)m.z) + 8 * j;
            if (kind == 1) {
                cp_async16(dst, P.recent + off);
            } else if (kind == 2 && vec_in && P.kv_dtype == OSCAR_DTYPE_BF16) {
                cp_async16(dst, reinterpret_cast<const uint16_t*>(src_new) + off);
            } else if (kind == 2 && vec_in) {
                const float4 f0 = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src_new) + off);
                const float4 f1 = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src_new) + off + 4);
                *reinterpret_cast<uint4*>(dst) =
                    make_uint4(pack_bf16(f0.x, f0.y), pack_bf16(f0.z, f0.w), pack_bf16(f1.x, f1.y), pack_bf16(f1.z, f1.w));
            } else if (kind == 2) {
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    w[q] = pack_bf16(load_elem(src_new, off + 2 * q, P.kv_dtype), load_elem(src_new, off + 2 * q + 1, P.kv_dtype));
                *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            } else {
                *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        cp_async_commit();
    };
    // a tile whose valid rows are the consecutive rows of the bf16 input from
    // row 0's offset on comes by TMA; called after the barrier that follows publish(buf)
    auto contiguous = [&](int buf) -> bool {
        const int4 m0 = *reinterpret_cast<const int4*>(meta + buf * kTcRows * kMetaInts);
        const int4 m = *reinterpret_cast<const int4*>(meta + (buf * kTcRows + gt) * kMetaInts);
        const int64_t off0 = (int64_t)(((uint64_t)(uint32_t)m0.w << 32) | (uint32_t)m0.z);
        const int64_t off = (int64_t)(((uint64_t)(uint32_t)m.w << 32) | (uint32_t)m.z);
        const bool row_ok = m.x < 0 || ((m.y >> 16) == 2 && off == off0 + (int64_t)gt * kD);
        const bool head_ok = m0.x >= 0 && (m0.y >> 16) == 2;
        return !cta_bar_or(!(row_ok && head_ok));
    };
    auto issue_tma = [&](int buf) {
        if (gt == 0) {
            const int4 m0 = *reinterpret_cast<const int4*>(meta + buf * kTcRows * kMetaInts);
            const int64_t off0 = (int64_t)(((uint64_t)(uint32_t)m0.w << 32) | (uint32_t)m0.z);
            mbar_arrive_expect_tx(full, (uint32_t)kABytes);
#pragma unroll
            for (int xb = 0; xb < kD / 64; ++xb)
                tc5::tma_load_2d(A + xb * kTcRows * 128, tmap, 64 * xb, (int)(off0 / kD), full);
        }
    };

    long long budget = 2000000000LL;            // cycles per wait (~1 s); 0 after a timeout
    bool aborted = false;
    uint32_t it = 0;
    const int64_t step = gridDim.x;
    int64_t tile = blockIdx.x;
    uint32_t tma_n = 0;                         // TMA tiles so far (parity of `full`)
    bool cur_tma = false;
    int drain_full = -1, drain_mma = -1;
    publish(locate(tile), 0);
    cta_bar();
    cur_tma = use_tma && contiguous(0);
    if (cur_tma) issue_tma(0);
    else gather(0);
    Loc pend = locate(tile + step);
    for (; tile < ntiles; tile += step, ++it) {
        const int buf = it & 1;
        bool to = false;
        if (cur_tma) {
            // every thread observes the TMA completion: all of them read the x tile (‖x‖² below)
            if (!mbar_wait_bounded(full, tma_n & 1, P.status, budget)) {
                to = true;
                if (gt == 0) drain_full = (int)(tma_n & 1);
            }
            ++tma_n;
        } else {
            cp_async_wait<0>();
            tc5::fence_proxy_async();
        }
        tc5::fence_before();
        if (cta_bar_or(to)) {                   // rows in place; the last epilogue's tensor-memory loads done
            aborted = true;
            break;
        }
        if (gt == 0) {
            tc5::fence_after();
            constexpr uint32_t idesc = tc5::idesc_bf16_f32(kTcRows, kN);
            const uint64_t ad0 = tc5::sw128_desc(smem_addr(A)), bd0 = tc5::sw128_desc(smem_addr(sB));
#pragma unroll
            for (int p = 1; p >= 0; --p)          // lo parts first, hi parts last
#pragma unroll
                for (int kk = 0; kk < kKS; ++kk) {
                    // start addresses in 16-byte units stay below 2^14 (shared memory < 256 KB)
                    const uint32_t ao = (uint32_t)((kk >> 2) * kTcRows * 128 + (kk & 3) * 32);
                    const uint32_t bo = (uint32_t)(p * kBPart + (kk >> 2) * kN * 128 + (kk & 3) * 32);
                    tc5::mma_bf16(tmem, ad0 + (ao >> 4), bd0 + (bo >> 4), idesc, !(p == 1 && kk == 0));
                }
            tc5::commit(bar);
            *nx = 0;                              // the last tile's stashed rows are done with (barrier above)
        }
        const int64_t nxt = tile + step;
        publish(pend, buf ^ 1);
        pend = locate(nxt + step);
        // ‖x‖² of this thread's row from the x tile (read alongside the tensor core)
        float xsq;
        {
            float2 q2 = make_float2(0.0f, 0.0f);
#pragma unroll 8
            for (int j = 0; j < kCPR; ++j) {
                const uint4 u = *reinterpret_cast<const uint4*>(A + tc5::sw128_offset(kTcRows, gt, j));
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 v = make_float2(__uint_as_float(w4[q] << 16), __uint_as_float(w4[q] & 0xFFFF0000u));
                    q2 = __ffma2_rn(v, v, q2);
                }
            }
            xsq = q2.x + q2.y;
        }
        to = false;
        if (gt == 0 && !mbar_wait_bounded(bar, it & 1, P.status, budget)) {
            to = true;
            drain_mma = (int)(it & 1);
        }
        if (cta_bar_or(to)) {                   // MMAs done (A free); next tile's vectors resolved
            aborted = true;
            break;
        }
        tc5::fence_after();
        constexpr int NC = G / 32;
        const float e = kBound * sqrtf(xsq);
        const float e2 = __fmul_ru(2.0f, e);
        // extremes of this thread's groups, and its x row stashed when one of
        // their (s, z) could change (before the next tile's rows overwrite it)
        float gmn[ngh], gmx[ngh];
        uint32_t umask = 0;
#pragma unroll
        for (int gl = 0; gl < ngh; ++gl) {
            float mn = INFINITY, mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                float y[32];
                load_y(tacc + gl * G + 32 * c, y);
                minmax32(y, mn, mx);
            }
            gmn[gl] = mn;
            gmx[gl] = mx;
            umask |= sz_uncertain(mn, mx, rclip, e, fp8) ? (1u << gl) : 0u;
        }
        int xslot = -1;
        if (umask) {
            const int sl = atomicAdd(nx, 1);
            if (sl < xcap) {
                xslot = sl;
                uint4* dst = reinterpret_cast<uint4*>(xs + (int64_t)sl * kXS);
#pragma unroll 8
                for (int j = 0; j < kCPR; ++j) dst[j] = *reinterpret_cast<const uint4*>(A + tc5::sw128_offset(kTcRows, gt, j));
            }
        }
        cta_bar();                                // rows stashed: the x tile may be overwritten
        cur_tma = false;
        if (nxt < ntiles) {
            cur_tma = use_tma && contiguous(buf ^ 1);
            if (cur_tma) issue_tma(buf ^ 1);
            else gather(buf ^ 1);
        }

        // ---- quantise this half of vector gt ----
        const int* m = meta + (buf * kTcRows + gt) * kMetaInts;
        const int slot = m[0];
        const ExactSrc xsrc{P.recent, src_new, P.kv_dtype, m[1] >> 16, *reinterpret_cast<const int64_t*>(m + 2)};
        uint8_t* rec = P.records + (int64_t)(slot < 0 ? 0 : slot) * P.slot_bytes + (int64_t)(m[1] & 0xFFFF) * P.rec_bytes;
#pragma unroll 1
        for (int gl = 0; gl < ngh; ++gl) {
            const int gch = kN * half + gl * G;   // first channel of the group in y
            uint32_t words[G / 16];
            float mn = gmn[0], mx = gmx[0];
#pragma unroll
            for (int i = 1; i < ngh; ++i)
                if (gl == i) {
                    mn = gmn[i];
                    mx = gmx[i];
                }
            const bool unc = (umask >> gl) & 1u;
            if (cta_bar_or(unc)) {                // some (s, z) of the tile could change: one batch for the CTA
                const float2 ex = rt_exact_extremes<G>(Q, tacc + gl * G, trt, unc, xslot, mn, mx, e2, gl * G, gch,
                                                       R, xsrc, gt, lane);
                if (unc) {
                    mn = ex.x;
                    mx = ex.y;
                }
            }
            const SZ sz = sz_decide(mn, mx, rclip, fp8);
            const float sc = sz.s, zc = sz.z;
            const float r3 = sc != 0.0f ? __frcp_rn(3.0f * sc) : 0.0f;
            const float be = code_band(e, r3);
            const float hb = 0.5f - (be + 1.0f / 2097152.0f);
            const float nb2 = hb > 0.0f ? -hb * hb : 0.0f;
            uint32_t tie = 0xFFFFFFFFu;
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                float y[32];
                load_y(tacc + gl * G + 32 * c, y);
                codes32(y, zc, r3, nb2, words[2 * c], words[2 * c + 1], tie);
            }
            if (__any_sync(0xffffffffu, !(tie >> 31))) {
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const uint2 w = tc256_exact_codes(tacc + gl * G + 32 * c, R, xsrc, zc, sc, r3, nb2, be,
                                                      make_uint2(words[2 * c], words[2 * c + 1]), gch + 32 * c, lane);
                    words[2 * c] = w.x;
                    words[2 * c + 1] = w.y;
                }
            }
            if (slot >= 0) {
                store_sz(rec, rec_off_sz, gi0 + gl, sz, fp8);
                uint8_t* dst = rec + rec_off_codes + gl * (G / 4);
                // records start on 8-byte boundaries (E4M3 pairs) or 16-byte ones (fp16)
#pragma unroll
                for (int q = 0; q < G / 32; ++q)
                    *reinterpret_cast<uint2*>(dst + 8 * q) = make_uint2(words[2 * q], words[2 * q + 1]);
            }
        }
    }
    if (aborted && gt == 0) {                     // copies or MMAs may still run: bounded drain
        long long drain = 2000000000LL;
        if (drain_full >= 0) mbar_wait_bounded(full, (uint32_t)drain_full, P.status, drain);
        if (drain_mma >= 0) mbar_wait_bounded(bar, (uint32_t)drain_mma, P.status, drain);
    }
    cp_async_wait<0>();
    tc5::fence_before();
    __syncthreads();
    if (warp == 0) {
        tc5::fence_after();
        tc5::dealloc(tmem, kCols);
    }
}

template <int G>
static int launch_tc256(const AppendParams& P, int64_t max_vec, cudaStream_t stream) {
    // prefix, scratch, the stash counter, the queues, 16 bytes of alignment, then
    // as many stashed rows (up to 64) as the block's shared memory still holds
    const size_t fixed = kSmem + (size_t)(P.batch + 1 + kThreads + 4 + kN + 2 * kN * kQ) * 4 + 16;
    const int lim = max_dynamic_smem();
    if (lim <= 0) return OSCAR_ERR_CUDA;
    const int xcap = (int)std::min<int64_t>(64, std::max<int64_t>(0, ((int64_t)lim - (int64_t)fixed) / (kXS * 2)));
    const size_t smem = fixed + (size_t)xcap * kXS * 2;
    auto kern = quantize_tc256_kernel<G>;
    if (const int rc_ = ensure_dynamic_smem((const void*)kern, smem, "cudaFuncSetAttribute(quantize_tc256_kernel)"))
        return rc_;
    const int64_t tiles = (max_vec + kTcRows - 1) / kTcRows;
    // grid (x, K|V, channel half): one CTA per SM in all
    const int64_t grid_x = std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)sm_count() / 4));
    CUtensorMap tk, tv;
    memset(&tk, 0, sizeof tk);
    memset(&tv, 0, sizeof tv);
    const int64_t rows = P.total_new * P.Hkv;
    const int use_tma = P.kv_dtype == OSCAR_DTYPE_BF16 && rows > 0 && rows < 0x7FFFFFFF &&
                        (reinterpret_cast<uintptr_t>(P.k) & 15) == 0 && (reinterpret_cast<uintptr_t>(P.v) & 15) == 0 &&
                        tc_encode_rows(&tk, P.k, rows, kD) && tc_encode_rows(&tv, P.v, rows, kD);
    launch_dependent(kern, dim3((unsigned)grid_x, 2, 2), dim3(kThreads), smem, stream, P, tk, tv, use_tma, xcap);
    return check_cuda("quantize_tc256_kernel launch");
}

int launch_quantize_tc256(const AppendParams& P, int64_t max_vec, cudaStream_t stream) {
    if (P.G == 32) return launch_tc256<32>(P, max_vec, stream);
    if (P.G == 64) return launch_tc256<64>(P, max_vec, stream);
    if (P.G == 128) return launch_tc256<128>(P, max_vec, stream);
    return OSCAR_ERR_ARG;
}

}  // namespace oscar
