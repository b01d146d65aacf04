// Tensor-core split-K history kernel for decode attention over the INT2 region.
//
// [OSCAR news] "サービングシステム：混合精度キャッシュレイアウト": the history
// tokens between the 64 BF16 sink tokens and the 256 BF16 recent tokens are
// INT2 after the OSCAR rotation; this kernel attends over them in the rotated
// domain (q·R_K against k̂, Σ p·v̂ mapped back by R_Vᵀ in the combine kernel).
// [Escha log] part 2, fix 4: query head h reads KV head h / (Hq/Hkv); here a
// warp owns one KV head and all of its query heads, so the mapping holds by
// construction for any group count (including 6).
//
// Structure (persistent CTAs, one per SM; CTA i owns flattened history chunks
// [i·N/n, (i+1)·N/n)):
//  * every warp owns one KV head (two warps per head: token-interleaved
//    16-token tiles for d <= 128, channel halves for d = 256) and runs its own
//    gather pipeline: page-table entries are fetched 2·kNPF tiles ahead and the
//    head's records (rec bytes per token, a slot-major pool) kNPF tiles ahead,
//    both with cp.async into a private shared-memory ring; waits are
//    cp.async.wait_group, so warps never block on one another's loads;
//  * each tile runs mma.sync.m16n8k16 f16 → f32.  A code c enters the MMA as
//    the exact fp16 value 1 + α·c, α = 1/4 for odd and 1/16 for even channels
//    (one funnel shift exposes two adjacent code positions at bits 8-9 and
//    6-7, and one LOP3 each turns them into fp16); the channel weights 1/α
//    sit in the other operand or in the epilogue, and the per-group scale s
//    and zero z are applied in fp32 afterwards:
//        logit = Σ_g [s_g·(Σ (q̃/α)(1 + α c) − Σ q̃/α) + z_g·Σ q̃]
//        o_rot[ch] = (Σ_t w_t (1 + α_ch c_t) − Σ_t w_t)/α_ch + Σ_t p_t z_t,   w = p·s
//    q̃/α and p·s are split into fp16 hi + lo parts that occupy the n8 columns
//    (head, part), so the products carry ~22 bits;
//  * online softmax in log2 units, partials (m, l, o) per (CTA, request).
#include <algorithm>
#include <cmath>

#include "oscar_internal.h"
#include "oscar_device.cuh"
#include "oscar_decode_common.cuh"

namespace oscar {

namespace mma_detail {

constexpr int kNPF = 8;     // 16-token tiles in flight per warp
constexpr int kTile = 16;

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// From x (the word rotated so that code position m sits at bits 8-9 and
// m-1 at bits 6-7 of each half): half2 of 1 + c/4 for position m, and of
// 1 + c/16 for position m-1.  Both values are exact in fp16.
// (x & mask) | one as a single LOP3 (look-up table 0xEA = (a & b) | c).
__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t mask, uint32_t one) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "r"(mask), "r"(one));
    return d;
}
__device__ __forceinline__ uint32_t code_q4(uint32_t x) { return and_or(x, 0x03000300u, 0x3C003C00u); }
__device__ __forceinline__ uint32_t code_q16(uint32_t x) { return and_or(x, 0x00C000C0u, 0x3C003C00u); }
__device__ __forceinline__ uint32_t rotr(uint32_t w, uint32_t n) { return __funnelshift_r(w, w, n); }

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Packs (x0, x1) as fp16 hi parts, or as the lo parts x - fp16(x) when lo is set.
__device__ __forceinline__ uint32_t pack_part(float x0, float x1, bool lo) {
    __half2 h = __floats2half2_rn(x0, x1);
    if (lo) {
        const float2 f = __half22float2(h);
        h = __floats2half2_rn(x0 - f.x, x1 - f.y);
    }
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 h2f(uint32_t v) {
    return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

}  // namespace mma_detail

// Shared row stride of one token's record: rounded up to an odd multiple of
// 16 B, so that 8 consecutive rows start in 8 different 4-bank groups.
__host__ __device__ constexpr int row_bytes(int rec) {
    return ((rec + 15) / 16) % 2 == 1 ? (rec + 15) / 16 * 16 : (rec + 15) / 16 * 16 + 16;
}

// Walks the segments (one per request) of a CTA's chunk run [f, f1) and, in
// each, the 16-token tiles first, first + step, ... that belong to one warp.
struct TileIter {
    int64_t f, f1, fe;
    int b, t_seg, t_end, t0, step16;
    bool valid;

    __device__ void seg(const DecodeParams& P) {
        valid = f < f1;
        if (!valid) return;
        int lo = 0, hi = P.batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (P.cprefix[mid] <= f) lo = mid; else hi = mid - 1;
        }
        b = lo;
        fe = min(f1, (int64_t)P.cprefix[b + 1]);
        const int L = P.len[b];
        const int h_end = max(P.S, L - P.W);
        t_seg = P.S + (int)(f - P.cprefix[b]) * P.chunk;
        t_end = min(h_end, P.S + (int)(fe - P.cprefix[b]) * P.chunk);
    }
    // segment iteration (consumers)
    __device__ void init_seg(const DecodeParams& P, int64_t f0_, int64_t f1_) {
        f = f0_;
        f1 = f1_;
        seg(P);
    }
    __device__ void next_seg(const DecodeParams& P) {
        f = fe;
        seg(P);
    }
    // tile iteration (producers): skips segments with no tile for this warp
    __device__ void skip_empty(const DecodeParams& P, int first) {
        while (valid && t_seg + first * mma_detail::kTile >= t_end) next_seg(P);
        if (valid) t0 = t_seg + first * mma_detail::kTile;
    }
    __device__ void init_tiles(const DecodeParams& P, int64_t f0_, int64_t f1_, int first, int step) {
        step16 = step * mma_detail::kTile;
        init_seg(P, f0_, f1_);
        skip_empty(P, first);
    }
    __device__ void next_tile(const DecodeParams& P, int first) {
        t0 += step16;
        if (t0 >= t_end) {
            next_seg(P);
            skip_empty(P, first);
        }
    }
};

// D: head_dim; G: group size; NT: n8 tiles of (head, hi/lo) columns; WPH:
// warps per head along channels (2 for d = 256); TI: token-interleaved warps
// per (head, channel slice).
template <int D, int G, int NT, int WPH, int TI>
struct MmaCfg {
    static constexpr int kSliceCh = D / WPH;        // channels per warp
    static constexpr int kKS = kSliceCh / 16;       // k-steps (words of 16 codes) per warp
    static constexpr int kGW = kSliceCh / G > 0 ? kSliceCh / G : 1;  // groups per warp slice
    static constexpr int kMT = kSliceCh / 16;       // P·V m-tiles per warp
    static constexpr int kMTG = G / 16;             // m-tiles per group
    static_assert(G <= kSliceCh, "a warp's channel slice must hold whole groups");
    static_assert(G >= 32, "group size below 32 has no fast path");
    static_assert(WPH * TI <= 2, "at most two warps share a KV head");
};

// Shared-memory layout: per warp [kNPF][16][row] records, [2·kNPF][16] slot
// ids, [kNPF] tile masks (warp_bytes apiece), then per head the logit
// exchange / merge area at x_off.
template <int D, int G, int NT, int WPH, int TI>
__global__ void __launch_bounds__(32 * (D == 256 ? 4 : 8) * WPH * TI, 1)
history_mma_kernel(DecodeParams P, int x_off) {
    using namespace mma_detail;
    using C = MmaCfg<D, G, NT, WPH, TI>;
    constexpr int KS = C::kKS, GW = C::kGW, MT = C::kMT, MTG = C::kMTG;
    constexpr int kXFloats = 2 * 32 * 2 * NT * 2 + 32 * NT * MT * 2 + 64;  // logits x2 buffers + merge
    constexpr int REC = (D / 2 + 8 * (D / G) + 15) / 16 * 16;   // record bytes (== P.rec_bytes)
    constexpr int row = row_bytes(REC);         // shared row stride of one token's record
    constexpr int warp_bytes = (kNPF * kTile * row + 2 * kNPF * kTile * 4 + kNPF * 4 + 127) / 128 * 128;
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int Hkv = P.Hkv;
    const int h = warp / (WPH * TI);            // KV head
    const int sub = warp % (WPH * TI);
    const int wsl = (WPH == 2) ? sub : 0;       // channel slice
    const int ti = (TI == 2) ? sub : 0;         // token interleave index
    const int r = lane >> 2, j = lane & 3;
    const int g = P.g;
    unsigned char* ring = smem + warp * warp_bytes;                             // [kNPF][16][row]
    int32_t* pts = reinterpret_cast<int32_t*>(ring + kNPF * kTile * row);      // [2 kNPF][16]
    uint32_t* tmask = reinterpret_cast<uint32_t*>(pts + 2 * kNPF * kTile);     // [kNPF]
    float* xb = reinterpret_cast<float*>(smem + x_off) + h * kXFloats;
    const int bar_id = 1 + h;

    const int64_t N = P.cprefix[P.batch];
    const int64_t f0 = (int64_t)blockIdx.x * N / gridDim.x;
    const int64_t f1 = (int64_t)(blockIdx.x + 1) * N / gridDim.x;
    if (f0 >= f1) return;
    const int first = ti;
    constexpr int CPR = REC / 16;               // 16-byte chunks per record
    constexpr int CPH = (CPR + 1) / 2;          // chunks per half-warp lane
    const uint8_t* recbase = P.records + (int64_t)h * REC;
    // zero the ring once: rows of invalid tokens then always hold finite values
    for (int i = lane; i < warp_bytes / 16; i += 32)
        *reinterpret_cast<uint4*>(ring + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();

    // ---- gather pipeline of this warp ----
    TileIter itp, itr;
    itp.init_tiles(P, f0, f1, first, TI);
    itr = itp;
    uint32_t kp = 0, kr = 0;
    auto issue_pt = [&]() {                     // slot ids of tile kp -> pts[kp % 2kNPF]
        if (itp.valid) {
            const int p = itp.t0 + lane;
            if (lane < kTile && p < itp.t_end)
                cp_async4(pts + (kp % (2 * kNPF)) * kTile + lane, P.page_table + (int64_t)itp.b * P.pt_stride + p);
            itp.next_tile(P, first);
        }
        ++kp;
    };
    auto issue_rec = [&]() {                    // records of tile kr -> ring[kr % kNPF]; commits a group
        if (itr.valid) {
            const int ntok = min(kTile, itr.t_end - itr.t0);
            const int32_t* ps = pts + (kr % (2 * kNPF)) * kTile;
            unsigned char* dst = ring + (kr % kNPF) * kTile * row;
            // lanes t and t+16 copy token t: chunks [0, CPH) and [CPH, CPR)
            const int t = lane & 15, c0 = (lane >> 4) * CPH;
            bool ok = false;
            int sl = 0;
            if (t < ntok) {
                sl = ps[t];
                ok = sl >= 0 && sl < P.num_slots;
                if (!ok && lane < 16) set_status(P.status, OSCAR_DEV_BAD_SLOT);
            }
            if (ok) {
                const uint8_t* src = recbase + (int64_t)sl * (Hkv * REC);
#pragma unroll
                for (int c = 0; c < CPH; ++c)
                    if (c0 + c < CPR) cp_async16(dst + t * row + (c0 + c) * 16, src + (c0 + c) * 16);
            }
            const uint32_t vm = __ballot_sync(0xffffffffu, ok) & 0xFFFFu;
            if (lane == 0) tmask[kr % kNPF] = vm;
            itr.next_tile(P, first);
        }
        cp_async_commit();
        ++kr;
    };
    for (int i = 0; i < kNPF; ++i) issue_pt();  // slot ids of the first kNPF tiles
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();
    for (int i = 0; i < kNPF; ++i) {            // their records, and the next kNPF slot-id tiles
        issue_pt();
        issue_rec();
    }

    // funnel shift for the K extraction: code position 2j+1 to bits 8-9 (2j to 6-7)
    const uint32_t rotK = (uint32_t)(4 * j - 6) & 31u;
    int xpar = 0;   // logit-exchange buffer parity; continuous across segments
    uint32_t k = 0; // tiles consumed

    TileIter sg;
    sg.init_seg(P, f0, f1);
    while (sg.valid) {
        const int b = sg.b;
        // ---- per-segment query state ----
        uint32_t bq[NT][KS][2];
        {
            const uint2* qf = P.qfrag + (((int64_t)b * Hkv + h) * P.n_frag_tiles) * (D / 16) * 32;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const uint2 v = qf[((int64_t)nt * (D / 16) + wsl * KS + kk) * 32 + lane];
                    bq[nt][kk][0] = v.x;
                    bq[nt][kk][1] = v.y;
                }
        }
        float2 qs[NT][GW];          // (Σ q̃, Σ q̃/α) per group, head 4nt + j
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hh = 4 * nt + j;
#pragma unroll
            for (int gi = 0; gi < GW; ++gi)
                qs[nt][gi] = hh < g ? P.qsum[((int64_t)b * P.Hq + h * g + hh) * P.ng + wsl * GW + gi]
                                    : make_float2(0.f, 0.f);
        }
        float m_run[NT], l_run[NT];
        float acc[NT][MT][4];
        float Wsum[NT][GW], Zsum[NT][GW];   // for head 4nt + r/2 (B-fragment layout)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m_run[nt] = -1e30f;     // finite: 2^(m_run - m) never sees -inf - -inf
            l_run[nt] = 0.f;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[nt][mt][e] = 0.f;
#pragma unroll
            for (int gi = 0; gi < GW; ++gi) { Wsum[nt][gi] = 0.f; Zsum[nt][gi] = 0.f; }
        }

        for (int t0 = sg.t_seg + first * kTile; t0 < sg.t_end; t0 += TI * kTile, ++k) {
            cp_async_wait<kNPF - 1>();          // records of tile k have landed
            __syncwarp();
            const uint32_t vmask = tmask[k % kNPF];
            const unsigned char* tb = ring + (k % kNPF) * kTile * row;
            {
                const bool v_r = (vmask >> r) & 1u;
                const bool v_r8 = (vmask >> (r + 8)) & 1u;
            // ---------------- QK ----------------
            float sc[GW][NT][4];
#pragma unroll
            for (int gi = 0; gi < GW; ++gi)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[gi][nt][e] = 0.f;
            const uint32_t* krow0 = reinterpret_cast<const uint32_t*>(tb + r * row) + wsl * KS;
            const uint32_t* krow1 = reinterpret_cast<const uint32_t*>(tb + (r + 8) * row) + wsl * KS;
#pragma unroll
            for (int k4 = 0; k4 < KS; k4 += 4) {
                const uint4 w0 = *reinterpret_cast<const uint4*>(krow0 + k4);
                const uint4 w1 = *reinterpret_cast<const uint4*>(krow1 + k4);
                const uint32_t a0s[4] = {w0.x, w0.y, w0.z, w0.w};
                const uint32_t a1s[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int kk = k4 + q;
                    const int gi = (kk * 16) / G;
                    const uint32_t y0 = rotr(a0s[q], rotK), y1 = rotr(a1s[q], rotK);
                    const uint32_t x0 = code_q16(y0), x1 = code_q16(y1);   // channels 2j, 2j+8
                    const uint32_t x2 = code_q4(y0), x3 = code_q4(y1);     // channels 2j+1, 2j+9
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16816(sc[gi][nt], x0, x1, x2, x3, bq[nt][kk][0], bq[nt][kk][1]);
                }
            }
            // logits (log2 units) for rows r, r+8 and head 4nt + j
            float lg[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) { lg[nt][0] = 0.f; lg[nt][1] = 0.f; }
#pragma unroll
            for (int gi = 0; gi < GW; ++gi) {
                const int gg = wsl * GW + gi;
                const float2 sz0 = h2f(*reinterpret_cast<const uint32_t*>(tb + r * row + D / 2 + 4 * gg));
                const float2 sz1 = h2f(*reinterpret_cast<const uint32_t*>(tb + (r + 8) * row + D / 2 + 4 * gg));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float2 Q = qs[nt][gi];       // (Σ q̃, Σ q̃/α)
                    lg[nt][0] += sz0.x * (sc[gi][nt][0] + sc[gi][nt][1] - Q.y) + sz0.y * Q.x;
                    lg[nt][1] += sz1.x * (sc[gi][nt][2] + sc[gi][nt][3] - Q.y) + sz1.y * Q.x;
                }
            }
            if (WPH == 2) {   // add the other channel slice's partial logits
                float* my = xb + xpar * (2 * 32 * 2 * NT) + wsl * (32 * 2 * NT);
                float* ot = xb + xpar * (2 * 32 * 2 * NT) + (1 - wsl) * (32 * 2 * NT);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    my[(nt * 2 + 0) * 32 + lane] = lg[nt][0];
                    my[(nt * 2 + 1) * 32 + lane] = lg[nt][1];
                }
                named_bar(bar_id, 64);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    lg[nt][0] += ot[(nt * 2 + 0) * 32 + lane];
                    lg[nt][1] += ot[(nt * 2 + 1) * 32 + lane];
                }
                xpar ^= 1;
            }
            // ---------------- online softmax ----------------
            float pr[NT][2];
            bool grew = false;
            float alpha[NT];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const bool hv = (4 * nt + j) < g;
                const float x0 = (v_r && hv) ? lg[nt][0] : -INFINITY;
                const float x1 = (v_r8 && hv) ? lg[nt][1] : -INFINITY;
                float tm = fmaxf(x0, x1);
                tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
                tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
                tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
                const float mn = fmaxf(m_run[nt], tm);
                grew |= mn > m_run[nt];
                alpha[nt] = fast_exp2(m_run[nt] - mn);           // m_run starts at a finite -1e30
                m_run[nt] = mn;
                pr[nt][0] = fast_exp2(x0 - mn);                  // masked tokens: 2^-inf = 0
                pr[nt][1] = fast_exp2(x1 - mn);
                l_run[nt] = l_run[nt] * alpha[nt] + pr[nt][0] + pr[nt][1];
            }
            if (__any_sync(0xffffffffu, grew)) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float ab = __shfl_sync(0xffffffffu, alpha[nt], r >> 1);  // head 4nt + r/2
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[nt][mt][e] *= alpha[nt];
#pragma unroll
                    for (int gi = 0; gi < GW; ++gi) { Wsum[nt][gi] *= ab; Zsum[nt][gi] *= ab; }
                }
            }
            // ---------------- P·V ----------------
            // p of tokens 2j, 2j+1, 2j+8, 2j+9 for head 4nt + r/2
            const int srcA = 8 * j + (r >> 1), srcB = srcA + 4;
            float pb[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                pb[nt][0] = __shfl_sync(0xffffffffu, pr[nt][0], srcA);
                pb[nt][1] = __shfl_sync(0xffffffffu, pr[nt][0], srcB);
                pb[nt][2] = __shfl_sync(0xffffffffu, pr[nt][1], srcA);
                pb[nt][3] = __shfl_sync(0xffffffffu, pr[nt][1], srcB);
            }
            const int tk[4] = {2 * j, 2 * j + 1, 2 * j + 8, 2 * j + 9};
            const bool lo_part = r & 1;
#pragma unroll
            for (int gi = 0; gi < GW; ++gi) {
                const int gg = wsl * GW + gi;
                float sv[4], zv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    // rows of invalid tokens hold finite stale data and get p = 0
                    const float2 sz = h2f(*reinterpret_cast<const uint32_t*>(
                        tb + tk[e] * row + D / 2 + 4 * (D / G) + 4 * gg));
                    sv[e] = sz.x;
                    zv[e] = sz.y;
                }
                uint32_t bv[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        w[e] = pb[nt][e] * sv[e];
                        Wsum[nt][gi] += w[e];
                        Zsum[nt][gi] = fmaf(pb[nt][e], zv[e], Zsum[nt][gi]);
                    }
                    bv[nt][0] = pack_part(w[0], w[1], lo_part);
                    bv[nt][1] = pack_part(w[2], w[3], lo_part);
                }
                // this thread's V code slice of group gg: G/32 bytes per token
                const int vb = D / 4 + gg * (G / 4) + r * (G / 32);   // byte offset in the record
                if constexpr (G == 32) {
                    const uint32_t* w0p = reinterpret_cast<const uint32_t*>(tb + tk[0] * row + (vb & ~3));
                    const uint32_t* w1p = reinterpret_cast<const uint32_t*>(tb + tk[1] * row + (vb & ~3));
                    const uint32_t* w2p = reinterpret_cast<const uint32_t*>(tb + tk[2] * row + (vb & ~3));
                    const uint32_t* w3p = reinterpret_cast<const uint32_t*>(tb + tk[3] * row + (vb & ~3));
                    const uint32_t bsel = (uint32_t)(vb & 3);
                    const uint32_t sel = bsel | ((4u + bsel) << 8) | (bsel << 4) | ((4u + bsel) << 12);
                    const uint32_t u01 = prmt(*w0p, *w1p, sel);
                    const uint32_t u23 = prmt(*w2p, *w3p, sel);
#pragma unroll
                    for (int mu = 0; mu < 2; ++mu) {
                        const int mt = gi * MTG + mu;
                        const uint32_t rb = (uint32_t)(4 * mu - 6) & 31u;   // position 2mu+1 -> bits 8-9
                        const uint32_t y01 = rotr(u01, rb), y23 = rotr(u23, rb);
                        const uint32_t a0 = code_q16(y01), a1 = code_q4(y01);
                        const uint32_t a2 = code_q16(y23), a3 = code_q4(y23);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma16816(acc[nt][mt], a0, a1, a2, a3, bv[nt][0], bv[nt][1]);
                    }
                } else {
#pragma unroll
                    for (int hw = 0; hw < G / 64; ++hw) {
                        const int off = vb + 2 * hw;
                        const uint32_t wsel = (off & 2) ? 0x7632u : 0x5410u;
                        const int wo = off & ~3;
                        const uint32_t u01 = prmt(*reinterpret_cast<const uint32_t*>(tb + tk[0] * row + wo),
                                                  *reinterpret_cast<const uint32_t*>(tb + tk[1] * row + wo), wsel);
                        const uint32_t u23 = prmt(*reinterpret_cast<const uint32_t*>(tb + tk[2] * row + wo),
                                                  *reinterpret_cast<const uint32_t*>(tb + tk[3] * row + wo), wsel);
#pragma unroll
                        for (int mu = 0; mu < 4; ++mu) {
                            const int mt = gi * MTG + hw * 4 + mu;
                            const uint32_t rb = (uint32_t)(4 * mu - 6) & 31u;   // position 2mu+1 -> bits 8-9
                            const uint32_t y01 = rotr(u01, rb), y23 = rotr(u23, rb);
                            const uint32_t a0 = code_q16(y01), a1 = code_q4(y01);
                            const uint32_t a2 = code_q16(y23), a3 = code_q4(y23);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                mma16816(acc[nt][mt], a0, a1, a2, a3, bv[nt][0], bv[nt][1]);
                        }
                    }
                }
            }
            }
            __syncwarp();                       // ring slot k % kNPF is free again
            issue_pt();
            issue_rec();
        }

        // ---------------- segment end: reduce, merge, write the partial ----------------
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 4);
            l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 8);
            l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 16);
#pragma unroll
            for (int gi = 0; gi < GW; ++gi) {
                Wsum[nt][gi] += __shfl_xor_sync(0xffffffffu, Wsum[nt][gi], 1);
                Wsum[nt][gi] += __shfl_xor_sync(0xffffffffu, Wsum[nt][gi], 2);
                Zsum[nt][gi] += __shfl_xor_sync(0xffffffffu, Zsum[nt][gi], 1);
                Zsum[nt][gi] += __shfl_xor_sync(0xffffffffu, Zsum[nt][gi], 2);
            }
        }
        // out[head 4nt+j][ch] = (acc_hi + acc_lo − W)/α_ch + Z, with α = 1/16 on the
        // rows r (even code positions) and 1/4 on the rows r+8; W, Z of head 4nt+j sit in lane 8j
        float ov[NT][MT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int gi = 0; gi < GW; ++gi) {
                const float Wh = __shfl_sync(0xffffffffu, Wsum[nt][gi], 8 * j);
                const float Zh = __shfl_sync(0xffffffffu, Zsum[nt][gi], 8 * j);
#pragma unroll
                for (int mu = 0; mu < MTG; ++mu) {
                    const int mt = gi * MTG + mu;
                    ov[nt][mt][0] = 16.f * (acc[nt][mt][0] + acc[nt][mt][1] - Wh) + Zh;
                    ov[nt][mt][1] = 4.f * (acc[nt][mt][2] + acc[nt][mt][3] - Wh) + Zh;
                }
            }
        }
        if (TI == 2) {   // merge the two token-interleaved warps of this head
            float* mb = xb + 2 * 32 * 2 * NT;
            if (ti == 1) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        mb[((nt * MT + mt) * 2 + 0) * 32 + lane] = ov[nt][mt][0];
                        mb[((nt * MT + mt) * 2 + 1) * 32 + lane] = ov[nt][mt][1];
                    }
                    if (r == 0) {
                        mb[NT * MT * 64 + nt * 8 + j] = m_run[nt];
                        mb[NT * MT * 64 + nt * 8 + 4 + j] = l_run[nt];
                    }
                }
            }
            named_bar(bar_id, 64);
            if (ti == 0) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float m1 = mb[NT * MT * 64 + nt * 8 + j];
                    const float l1 = mb[NT * MT * 64 + nt * 8 + 4 + j];
                    const float M = fmaxf(m_run[nt], m1);
                    const float a0 = fast_exp2(m_run[nt] - M);
                    const float a1 = fast_exp2(m1 - M);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        ov[nt][mt][0] = ov[nt][mt][0] * a0 + mb[((nt * MT + mt) * 2 + 0) * 32 + lane] * a1;
                        ov[nt][mt][1] = ov[nt][mt][1] * a0 + mb[((nt * MT + mt) * 2 + 1) * 32 + lane] * a1;
                    }
                    l_run[nt] = l_run[nt] * a0 + l1 * a1;
                    m_run[nt] = M;
                }
            }
            named_bar(bar_id, 64);
        }
        if (ti == 0) {
            const int64_t slot = (int64_t)blockIdx.x + b;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hh = 4 * nt + j;
                if (hh >= g) continue;
                const int hq = h * g + hh;
                if (r == 0 && wsl == 0) P.ml[slot * P.Hq + hq] = make_float2(m_run[nt], l_run[nt]);
                float* o = P.po + (slot * P.Hq + hq) * D;
#pragma unroll
                for (int gi = 0; gi < GW; ++gi) {
                    const int gg = wsl * GW + gi;
#pragma unroll
                    for (int mu = 0; mu < MTG; ++mu) {
                        const int mt = gi * MTG + mu;
                        int ch0;
                        if constexpr (G == 32) ch0 = gg * G + 4 * r + 2 * mu;
                        else ch0 = gg * G + r * (G / 8) + 8 * (mu / 4) + 2 * (mu % 4);
                        o[ch0] = ov[nt][mt][0];
                        o[ch0 + 1] = ov[nt][mt][1];
                    }
                }
            }
        }
        sg.next_seg(P);
    }
    cp_async_wait<0>();
}

// Shared-memory plan: (offset of the exchange areas, total bytes).
template <int D, int G, int NT, int WPH, int TI>
static void mma_smem_plan(int Hkv, int* x_off, size_t* total) {
    using namespace mma_detail;
    constexpr int kXFloats = 2 * 32 * 2 * NT * 2 + 32 * NT * MmaCfg<D, G, NT, WPH, TI>::kMT * 2 + 64;
    constexpr int REC = (D / 2 + 8 * (D / G) + 15) / 16 * 16;
    constexpr int row = row_bytes(REC);
    constexpr int warp_bytes = (kNPF * kTile * row + 2 * kNPF * kTile * 4 + kNPF * 4 + 127) / 128 * 128;
    *x_off = Hkv * WPH * TI * warp_bytes;
    *total = (size_t)*x_off + (size_t)Hkv * kXFloats * 4;
}

template <int D, int G, int NT, int WPH, int TI>
static int launch_mma(DecodeParams P, cudaStream_t st) {
    const int threads = 32 * P.Hkv * WPH * TI;
    int x_off;
    size_t smem;
    mma_smem_plan<D, G, NT, WPH, TI>(P.Hkv, &x_off, &smem);
    if (smem > 225 * 1024) return OSCAR_ERR_ARG;
    auto kern = history_mma_kernel<D, G, NT, WPH, TI>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return check_cuda("cudaFuncSetAttribute(history_mma_kernel)");
    const int grid = std::min(P.n_ctas, sm_count());
    P.n_ctas = grid;
    kern<<<grid, threads, smem, st>>>(P, x_off);
    return check_cuda("history_mma_kernel launch");
}

// Chooses the tensor-core kernel for the shape, or reports that none fits
// (the caller then runs the CUDA-core kernel).  P.n_ctas is updated to the
// grid that was launched.
int launch_history_mma(DecodeParams& P, int head_dim, cudaStream_t st, bool* launched) {
    *launched = false;
    if (P.Hkv > (head_dim == 256 ? 4 : 8) || P.g > 8) return OSCAR_OK;
    const int nt = (2 * P.g + 7) / 8;
    int rc = OSCAR_OK;
    auto go = [&](auto plan, auto fn) {
        int xo;
        size_t smem;
        plan(P.Hkv, &xo, &smem);
        if (smem > 225 * 1024) return;           // does not fit: CUDA-core kernel instead
        rc = fn(P, st);
        *launched = true;
    };
#define OSCAR_MMA(D_, G_, NT_, WPH_, TI_) go(mma_smem_plan<D_, G_, NT_, WPH_, TI_>, launch_mma<D_, G_, NT_, WPH_, TI_>)
    if (head_dim == 128) {
        if (P.G == 64) { if (nt == 1) OSCAR_MMA(128, 64, 1, 1, 2); else OSCAR_MMA(128, 64, 2, 1, 1); }
        else if (P.G == 128) { if (nt == 1) OSCAR_MMA(128, 128, 1, 1, 2); else OSCAR_MMA(128, 128, 2, 1, 1); }
        else if (P.G == 32) { if (nt == 1) OSCAR_MMA(128, 32, 1, 1, 2); else OSCAR_MMA(128, 32, 2, 1, 1); }
    } else if (head_dim == 256) {
        if (P.G == 128) { if (nt == 1) OSCAR_MMA(256, 128, 1, 2, 1); else OSCAR_MMA(256, 128, 2, 2, 1); }
        else if (P.G == 64) { if (nt == 1) OSCAR_MMA(256, 64, 1, 2, 1); else OSCAR_MMA(256, 64, 2, 2, 1); }
    }
#undef OSCAR_MMA
    if (*launched) P.n_ctas = std::min(P.n_ctas, sm_count());
    return rc;
}

}  // namespace oscar
