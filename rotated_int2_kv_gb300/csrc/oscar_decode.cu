// Decode attention over the mixed-precision cache: prep (query rotation and
// request metadata), split-K history kernel over the INT2 region, and the
// combine kernel (BF16 windows, log-sum-exp merge of the history partials,
// R_Vᵀ epilogue).
//
// [OSCAR news] "サービングシステム：混合精度キャッシュレイアウト": 64 BF16 sink
// tokens, 256 BF16 recent tokens, INT2 history in between, paged attention.
// "OSCARの違い": keys and values are stored rotated (x·R_K, x·R_V), so the
// history logit is taken with q·R_K and the weighted sum of rotated values is
// mapped back with R_Vᵀ once, after the sum.  [Escha log] part 2, fix 4: query
// head h reads KV head h / (Hq/Hkv).
//
// This file holds the CUDA-core history kernel (history_simt_kernel); the
// tensor-core one lives in oscar_decode_mma.cu.  Both write the same partials.
#include <algorithm>
#include <cmath>

#include "oscar_internal.h"
#include "oscar_device.cuh"
#include "oscar_decode_common.cuh"
#include "oscar_append_step.cuh"

namespace oscar {

constexpr int kMaxDecodeBatch = 4096;

__device__ __forceinline__ int d_hist_hi(int L, int S, int W) { return max(S, L - W); }

// Number of history chunks of a request of L tokens.
__device__ __forceinline__ int n_chunks(int L, const DecodeParams& P) {
    const int h = d_hist_hi(L, P.S, P.W) - P.S;
    return h > 0 ? (h + P.chunk - 1) / P.chunk : 0;
}

__device__ __forceinline__ bool request_valid(const DecodeParams& P, int b, int* L_out, int* rq_out) {
    const int L = P.seq_lens[b];
    const int rq = P.req_idx ? P.req_idx[b] : b;
    *rq_out = rq;
    *L_out = L;
    return L >= 1 && L <= P.max_seq_len && L <= P.pt_stride && rq >= 0 && rq < P.max_reqs;
}

// ---------------------------------------------------------------------------
// prep: per (KV head, request), q̃ = q·R_K·(log2 e/√d) for the KV head's query
// heads (fp32), its fp16 hi/lo split (of q̃/α) packed as mma B fragments, the
// per-group sums; block (0, b) also the effective length / window row of
// request b, and block (0, 0) the chunk prefix.  It runs as the first z-slice
// of the window kernel's grid (128 threads, scheduled ahead of the window
// tiles), so the two need one launch.
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 128;

// Shared floats the prep slice needs: q and q̃ of up to 16 query heads.
__host__ __device__ constexpr int prep_smem_floats(int D, int g) { return 2 * g * D; }

template <int D, int GQ>
__device__ __forceinline__ void prep_slice(const DecodeParams& P, int hk, int b, float* sm) {
    __shared__ int scan[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = P.g;
    float* sq = sm;              // [GQ][D] q (rows >= g zero)
    float* sqt = sm + GQ * D;    // [g][D] q̃
    if (hk == 0 && b == 0) {
        // chunk prefix over all requests (re-derives validity locally)
        const int per = (P.batch + kPrepThreads - 1) / kPrepThreads;
        const int b0 = min(P.batch, tid * per), b1 = min(P.batch, b0 + per);
        int local = 0;
        for (int r = b0; r < b1; ++r) {
            int L, rq;
            if (request_valid(P, r, &L, &rq)) local += n_chunks(L, P);
        }
        int total;
        int run = block_exclusive_scan(local, scan, &total);
        for (int r = b0; r < b1; ++r) {
            P.cprefix[r] = run;
            int L, rq;
            if (request_valid(P, r, &L, &rq)) run += n_chunks(L, P);
        }
        if (tid == 0) P.cprefix[P.batch] = total;
    }
    int L, rq;
    const bool ok = request_valid(P, b, &L, &rq);
    if (hk == 0 && tid == 0) {
        P.len[b] = ok ? L : 0;
        for (int h = 0; h < P.Hkv * kCombGroups; ++h) P.comb_count[(int64_t)b * P.Hkv * kCombGroups + h] = 0;
        P.req[b] = ok ? rq : 0;
        if (!ok) {
            int bits = 0;
            if (!(L >= 1 && L <= P.max_seq_len && L <= P.pt_stride)) bits |= OSCAR_DEV_BAD_LEN;
            if (!(rq >= 0 && rq < P.max_reqs)) bits |= OSCAR_DEV_BAD_REQ;
            set_status(P.status, bits);
        }
    }
    {   // the q rows of the KV head's query heads: every thread's loads in flight together
        constexpr int NQ = GQ * D / kPrepThreads;
        const int64_t qb = ((int64_t)b * P.Hq + hk * g) * D;
        float qv[NQ];
#pragma unroll
        for (int u = 0; u < NQ; ++u) {
            const int i = tid + kPrepThreads * u;
            qv[u] = i < g * D ? load_elem(P.q, qb + i, P.q_dtype) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < NQ; ++u) sq[tid + kPrepThreads * u] = qv[u];   // rows >= g hold zeros
    }
    __syncthreads();
    // thread (column, head subset): 32 rows of R_K in flight from L2 per batch of k
    constexpr int kSplit = D < kPrepThreads ? kPrepThreads / D : 1;   // threads per column
    constexpr int kHPT = GQ / kSplit;                                   // heads per thread
    for (int ci = tid; ci < D * kSplit; ci += kPrepThreads) {
        const int col = ci % D, hs = ci / D;
        float acc[kHPT];
#pragma unroll
        for (int j = 0; j < kHPT; ++j) acc[j] = 0.f;
        for (int k0 = 0; k0 < D; k0 += 32) {
            float r[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) r[u] = __ldg(P.rot_k + (int64_t)(k0 + u) * D + col);
#pragma unroll
            for (int u = 0; u < 32; ++u)
#pragma unroll
                for (int j = 0; j < kHPT; ++j) acc[j] = fmaf(sq[(j * kSplit + hs) * D + k0 + u], r[u], acc[j]);
        }
#pragma unroll
        for (int j = 0; j < kHPT; ++j) {
            const int h = j * kSplit + hs;
            if (h < g) {
                const float v = acc[j] * P.qscale;
                sqt[h * D + col] = v;
                P.qt[((int64_t)b * P.Hq + hk * g + h) * D + col] = v;
            }
        }
    }
    __syncthreads();
    // Per group, from the fp16 hi + lo parts actually fed to the MMA: Q = Σ q̃
    // and Q' = Σ (fed value).  The fed value of channel c is q̃·2^(kQkExp - bit)
    // for groups >= 64 (subnormal codes; Q' unused there) and q̃/α for group
    // size 32, whose codes enter as 1 + α·c with α = 1/16 on even and 1/4 on
    // odd channels (Q' is subtracted from the accumulator).
    for (int i = warp; i < g * P.ng; i += kPrepThreads / 32) {
        const int j = i / P.ng, gi = i % P.ng;
        float sq_ = 0.f, sqa = 0.f;
        for (int c = gi * P.G + lane; c < (gi + 1) * P.G; c += 32) {
            const float inv = P.G >= 64 ? (float)(1u << (kQkExp - sub_bit(c & 7))) : ((c & 1) ? 4.f : 16.f);
            const float x = sqt[j * D + c] * inv;
            const __half hi = __float2half_rn(x);
            const __half lo = __float2half_rn(x - __half2float(hi));
            const float v = __half2float(hi) + __half2float(lo);
            sqa += v;
            sq_ += v / inv;
        }
        for (int off = 16; off; off >>= 1) {
            sq_ += __shfl_xor_sync(0xffffffffu, sq_, off);
            sqa += __shfl_xor_sync(0xffffffffu, sqa, off);
        }
        if (lane == 0) P.qsum[((int64_t)b * P.Hq + hk * g + j) * P.ng + gi] = make_float2(sq_, sqa);
    }
    // B fragments of KV head hk: [n_tiles][D/16][32 lanes] of (b0b1, b2b3);
    // column n of tile nt is (head 4nt + n/2 of the KV group, part n%2).
    const int nfr = P.n_frag_tiles * (D / 16) * 32;
    uint2* qf = P.qfrag + ((int64_t)b * P.Hkv + hk) * nfr;
    for (int i = tid; i < nfr; i += kPrepThreads) {
        const int ln = i & 31;
        const int kk = (i >> 5) % (D / 16);
        const int nt = i / (32 * (D / 16));
        const int n = ln >> 2, j = ln & 3;
        const int hh = 4 * nt + (n >> 1);
        const int part = n & 1;
        if (hh >= g) {                               // padding column: zero
            qf[i] = make_uint2(0u, 0u);
            continue;
        }
        // Group size 32: k-cols (2j, 2j+1) <- channels (16kk+2j, 16kk+2j+8), even:
        // scaled by 16; k-cols (2j+8, 2j+9) <- channels (16kk+2j+1, 16kk+2j+9), odd:
        // scaled by 4.  Groups >= 64: lane j owns word w = 4(kk/4) + j; k-step kk
        // takes slot kk%4 of it: k-cols (2j, 2j+1) <- first position p of both
        // halves (channels 16w + p, 16w + 8 + p), (2j+8, 2j+9) <- second position.
        int chans[4];
        float scl[4];
        if (P.G >= 64) {
            const int w = 4 * (kk / 4) + j, p0 = slot_pos(kk % 4, 0), p1 = slot_pos(kk % 4, 1);
            chans[0] = 16 * w + p0; chans[1] = 16 * w + 8 + p0;
            chans[2] = 16 * w + p1; chans[3] = 16 * w + 8 + p1;
            scl[0] = scl[1] = (float)(1u << (kQkExp - sub_bit(p0)));
            scl[2] = scl[3] = (float)(1u << (kQkExp - sub_bit(p1)));
        } else {
            chans[0] = 16 * kk + 2 * j; chans[1] = 16 * kk + 2 * j + 8;
            chans[2] = 16 * kk + 2 * j + 1; chans[3] = 16 * kk + 2 * j + 9;
            scl[0] = scl[1] = 16.f;
            scl[2] = scl[3] = 4.f;
        }
        uint16_t hv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float x = sqt[hh * D + chans[e]] * scl[e];
            const __half hi = __float2half_rn(x);
            const __half v = part ? __float2half_rn(x - __half2float(hi)) : hi;
            hv[e] = *reinterpret_cast<const uint16_t*>(&v);
        }
        qf[i] = make_uint2((uint32_t)hv[0] | ((uint32_t)hv[1] << 16), (uint32_t)hv[2] | ((uint32_t)hv[3] << 16));
    }
}

// Query-head bucket of the prep slice: the smallest of 4, 8, 16 that holds the
// query group.  The window kernels are instantiated per bucket, so each carries
// one prep variant (one copy of its code in the instruction cache).
__host__ __device__ constexpr int prep_bucket(int g) { return g <= 4 ? 4 : g <= 8 ? 8 : 16; }

// True when CTA i of an n-CTA history grid owns at least one of N chunks.
__device__ __forceinline__ bool cta_has_work(int64_t i, int64_t N, int64_t n) {
    return i * N / n < (i + 1) * N / n;
}

// Maps flattened chunk index f to (request, chunk-in-request) by binary search
// over the exclusive prefix cprefix[0..batch].
__device__ __forceinline__ int chunk_request(const int32_t* cprefix, int batch, int64_t f) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cprefix[mid] <= f) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ---------------------------------------------------------------------------
// CUDA-core history kernel.  Persistent grid; CTA i owns flattened chunks
// [i·N/n, (i+1)·N/n).  One warp per KV head (heads loop when Hkv exceeds the
// warp count).  Per 32-token tile: lane = token for the logits (factored
// dequant: logit = Σ_g s_g·Σ q̃·c + z_g·Σ q̃), warp-wide online softmax, then
// lane = channel slice for P·V (again factored: Σ (p·s)·c + Σ p·z).
// Codes enter the fp32 arithmetic as 1 + c/4 (exact), and the offset is
// removed with the group sums.
// ---------------------------------------------------------------------------
template <int D, int GQ>
__global__ void __launch_bounds__(512) history_simt_kernel(DecodeParams P) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    constexpr int CPL = D / 32;                 // channels per lane in P·V
    extern __shared__ __align__(16) float s_dyn[];
    float* sQ = s_dyn;                          // [Hq][D] q̃ of the current request
    float* sP = sQ + P.Hq * D;                  // [warps][GQ][32] probabilities
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int64_t N = P.cprefix[P.batch];
    const int64_t f0 = (int64_t)blockIdx.x * N / gridDim.x;
    const int64_t f1 = (int64_t)(blockIdx.x + 1) * N / gridDim.x;
    if (f0 >= f1) return;
    const int ng = P.ng;
    int cur_b = -1;
    float* myP = sP + warp * GQ * 32;
    int64_t f = f0;
    while (f < f1) {
        // segment: chunks [f, fe) of one request
        const int b = chunk_request(P.cprefix, P.batch, f);
        const int64_t fe = min(f1, (int64_t)P.cprefix[b + 1]);
        const int c_first = (int)(f - P.cprefix[b]);
        const int L = P.len[b];
        const int h_end = d_hist_hi(L, P.S, P.W);
        if (b != cur_b) {
            __syncthreads();
            for (int i = threadIdx.x; i < P.Hq * D; i += blockDim.x)
                sQ[i] = P.qt[(int64_t)b * P.Hq * D + i];
            __syncthreads();
            cur_b = b;
        }
        const int t_begin = P.S + c_first * P.chunk;
        const int t_end = min(h_end, P.S + (int)(fe - P.cprefix[b]) * P.chunk);
        for (int hk = warp; hk < P.Hkv; hk += nwarps) {
            const float* q = sQ + hk * P.g * D;
            float m[GQ], l[GQ], acc[GQ][CPL], zacc[GQ];
#pragma unroll
            for (int j = 0; j < GQ; ++j) {
                m[j] = -INFINITY;
                l[j] = 0.f;
                zacc[j] = 0.f;
#pragma unroll
                for (int c = 0; c < CPL; ++c) acc[j][c] = 0.f;
            }
            const int my_gi = (lane * CPL) / P.G;   // group of this lane's channels
            for (int t0 = t_begin; t0 < t_end; t0 += 32) {
                const int p = t0 + lane;
                const bool valid = p < t_end;
                int slot = 0;
                if (valid) {
                    slot = P.page_table[(int64_t)b * P.pt_stride + p];
                    if (slot < 0 || slot >= P.num_slots) {
                        set_status(P.status, OSCAR_DEV_BAD_SLOT);
                        slot = -1;
                    }
                }
                const bool use = valid && slot >= 0;
                const uint8_t* rec = P.records + (int64_t)(use ? slot : 0) * P.slot_bytes + (int64_t)hk * P.rec_bytes;
                // ---- logits, lane = token ----
                float logit[GQ];
#pragma unroll
                for (int j = 0; j < GQ; ++j) logit[j] = 0.f;
                if (use) {
                    for (int gi = 0; gi < ng; ++gi) {
                        float dot[GQ];
#pragma unroll
                        for (int j = 0; j < GQ; ++j) dot[j] = 0.f;
                        for (int w = gi * P.G / 16; w < (gi + 1) * P.G / 16; ++w) {
                            const uint32_t word = *reinterpret_cast<const uint32_t*>(rec + 4 * w);
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                float cf[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    cf[e] = __uint_as_float(0x3F800000u | (((word >> (8 * q4 + 2 * e)) & 3u) << 21));
#pragma unroll
                                for (int j = 0; j < GQ; ++j) {
                                    if (j < P.g) {
                                        const float4 qv = *reinterpret_cast<const float4*>(q + j * D + 16 * w + 4 * q4);
                                        dot[j] = fmaf(qv.x, cf[0], fmaf(qv.y, cf[1], fmaf(qv.z, cf[2], fmaf(qv.w, cf[3], dot[j]))));
                                    }
                                }
                            }
                        }
                        const float2 sz = load_sz(rec + D / 2, gi, P.fp8);
                        const float s = sz.x, z = sz.y;
#pragma unroll
                        for (int j = 0; j < GQ; ++j) {
                            if (j < P.g) {
                                const float Q = P.qsum[((int64_t)b * P.Hq + hk * P.g + j) * ng + gi].x;
                                // Σ q̃(1 + c/4) = Q + Σq̃c/4  =>  s·Σq̃c + z·Q = 4s·(dot - Q) + z·Q
                                logit[j] += 4.f * s * (dot[j] - Q) + z * Q;
                            }
                        }
                    }
                }
                // ---- online softmax over the tile ----
                float alpha[GQ];
#pragma unroll
                for (int j = 0; j < GQ; ++j) {
                    float x = use ? logit[j] : -INFINITY;
                    float tm = x;
#pragma unroll
                    for (int off = 16; off; off >>= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, off));
                    const float mn = fmaxf(m[j], tm);
                    alpha[j] = (m[j] == -INFINITY) ? 0.f : exp2f(m[j] - mn);
                    const float pj = use ? exp2f(x - mn) : 0.f;
                    m[j] = mn;
                    float ps = pj;
#pragma unroll
                    for (int off = 16; off; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
                    l[j] = l[j] * alpha[j] + ps;
                    myP[j * 32 + lane] = pj;
                }
#pragma unroll
                for (int j = 0; j < GQ; ++j) {
                    zacc[j] *= alpha[j];
#pragma unroll
                    for (int c = 0; c < CPL; ++c) acc[j][c] *= alpha[j];
                }
                __syncwarp();
                // ---- P·V, lane = channels [lane·CPL, lane·CPL + CPL) ----
                const int ntok = min(32, t_end - t0);
                for (int t = 0; t < ntok; ++t) {
                    const int st = __shfl_sync(0xffffffffu, use ? slot : -1, t);
                    if (st < 0) continue;
                    const uint8_t* rt = P.records + (int64_t)st * P.slot_bytes + (int64_t)hk * P.rec_bytes;
                    uint32_t bits;
                    if (CPL == 8) bits = *reinterpret_cast<const uint16_t*>(rt + D / 4 + lane * 2);
                    else if (CPL == 4) bits = rt[D / 4 + lane];
                    else bits = (rt[D / 4 + lane / 2] >> (4 * (lane & 1))) & 0xFu;
                    const float2 sz = load_sz(rt + D / 2 + (P.fp8 ? 2 : 4) * ng, my_gi, P.fp8);
                    const float s = sz.x, z = sz.y;
                    float cf[CPL];
#pragma unroll
                    for (int c = 0; c < CPL; ++c) cf[c] = (float)((bits >> (2 * c)) & 3u);
#pragma unroll
                    for (int j = 0; j < GQ; ++j) {
                        const float pj = myP[j * 32 + t];
                        const float w = pj * s;
                        zacc[j] = fmaf(pj, z, zacc[j]);
#pragma unroll
                        for (int c = 0; c < CPL; ++c) acc[j][c] = fmaf(w, cf[c], acc[j][c]);
                    }
                }
                __syncwarp();
            }
            // ---- write the segment partial at slot (CTA + request) ----
            const int64_t slot0 = (int64_t)blockIdx.x + b;
#pragma unroll
            for (int j = 0; j < GQ; ++j) {
                if (j >= P.g) break;
                const int hq = hk * P.g + j;
                if (lane == 0) P.ml[slot0 * P.Hq + hq] = make_float2(m[j], l[j]);
                float* o = P.po + (slot0 * P.Hq + hq) * D + lane * CPL;
#pragma unroll
                for (int c = 0; c < CPL; ++c) o[c] = acc[j][c] + zacc[j];
            }
        }
        f = fe;
    }
}

// ---------------------------------------------------------------------------
// window: one block of 128 threads per (KV head, request, 64-token tile of the
// BF16 sink + recent tokens).  K and V rows are staged in shared memory (rows
// padded to an odd number of words), logits in fp32 against the unrotated q,
// and the tile's (m, l, o) partial is written for the combine.
// ---------------------------------------------------------------------------
constexpr int kCombThreads = 128;      // window kernel
constexpr int kMergeThreads = 512;     // combine kernel
constexpr int kWinTile = 64;

// The new token of each request (position L - 1) read from the step's input
// rows (row b: [batch][Hkv][d] K and V, element type dtype) instead of the
// recent ring, for the fused decode step, whose append writes the ring in the
// same launch.
struct NewRowSrc {
    const void* k;
    const void* v;
    int dtype;
    int on;
};

// One 64-token window tile (wt) of KV head hk, request b on the CUDA cores:
// the (m, l, o) partial of every query head of the KV head.  kCombThreads threads.
template <int D>
__device__ __forceinline__ void window_tile_simt(const DecodeParams& P, int hk, int b, int wt, float* s_w,
                                                 NewRowSrc nr) {
    constexpr int kRowW = D / 2 + 1;               // words per staged bf16 row (odd: conflict-free)
    const int g = P.g, S = P.S, W = P.W;
    float* sq = s_w;                               // [g][D] q · qscale
    float* sp = sq + g * D;                        // [g][kWinTile] logits -> probabilities
    float* sml = sp + g * kWinTile;                // [g][2] (m, l)
    uint32_t* sk = reinterpret_cast<uint32_t*>(sml + 2 * g);   // [kWinTile][kRowW] K tile
    uint32_t* sv = sk + kWinTile * kRowW;                      // [kWinTile][kRowW] V tile
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int L, rq;                                     // the prep slice of this grid writes the same to len / req
    if (!request_valid(P, b, &L, &rq)) L = rq = 0;
    const int sink_end = min(S, L);
    const int rec_lo = d_hist_hi(L, S, W);
    const int nplain = L > 0 ? sink_end + max(0, L - rec_lo) : 0;
    const int t0 = wt * kWinTile;
    const int nt = min(kWinTile, nplain - t0);
    const int64_t pbase = ((int64_t)b * P.Hq + hk * g) * P.n_win_tiles + wt;   // + j * n_win_tiles
    if (nt <= 0) {                                 // empty tile: neutral partial
        for (int j = tid; j < g; j += kCombThreads) P.wml[pbase + (int64_t)j * P.n_win_tiles] = make_float2(-1e30f, 0.f);
        return;
    }
    // q of the first 8 heads: its loads are issued with the tile's, in one round
    constexpr int NQ = 8 * D / kCombThreads;
    float qv[NQ];
    const int64_t qb = ((int64_t)b * P.Hq + hk * g) * D;
#pragma unroll
    for (int u = 0; u < NQ; ++u) {
        const int i = tid + kCombThreads * u;
        qv[u] = i < g * D ? load_elem(P.q, qb + i, P.q_dtype) : 0.f;
    }
    {   // stage the tile: every thread issues all of its 16-byte loads before storing
        constexpr int C8 = D / 8;                       // 16-byte chunks per K (or V) row
        constexpr int NU = kWinTile * C8 / kCombThreads;
        uint4 kq[NU], vq[NU];
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            const int i = tid + kCombThreads * u;
            const int t = i / C8, c8 = i % C8;
            const int tt = t0 + t;
            if (t < nt) {
                const int pos = tt < sink_end ? tt : rec_lo + tt - sink_end;   // position in the request
                if (nr.on && pos == L - 1) {           // the step's new token: from the input row
                    const int64_t e0 = ((int64_t)b * P.Hkv + hk) * D + 8 * c8;
                    uint32_t kw[4], vw[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        kw[e] = (uint32_t)f32_to_bf16_bits(load_elem(nr.k, e0 + 2 * e, nr.dtype)) |
                                ((uint32_t)f32_to_bf16_bits(load_elem(nr.k, e0 + 2 * e + 1, nr.dtype)) << 16);
                        vw[e] = (uint32_t)f32_to_bf16_bits(load_elem(nr.v, e0 + 2 * e, nr.dtype)) |
                                ((uint32_t)f32_to_bf16_bits(load_elem(nr.v, e0 + 2 * e + 1, nr.dtype)) << 16);
                    }
                    kq[u] = make_uint4(kw[0], kw[1], kw[2], kw[3]);
                    vq[u] = make_uint4(vw[0], vw[1], vw[2], vw[3]);
                } else {
                    const uint16_t* base = (tt < sink_end)
                        ? P.sink + (((int64_t)rq * S + tt) * P.Hkv + hk) * 2 * D
                        : P.recent + (((int64_t)rq * W + (rec_lo + tt - sink_end) % W) * P.Hkv + hk) * 2 * D;
                    kq[u] = *reinterpret_cast<const uint4*>(base + c8 * 8);
                    vq[u] = *reinterpret_cast<const uint4*>(base + D + c8 * 8);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            const int i = tid + kCombThreads * u;
            const int t = i / C8, c8 = i % C8;
            if (t < nt) {
                uint32_t* kd = sk + t * kRowW + c8 * 4;
                uint32_t* vd = sv + t * kRowW + c8 * 4;
                kd[0] = kq[u].x; kd[1] = kq[u].y; kd[2] = kq[u].z; kd[3] = kq[u].w;
                vd[0] = vq[u].x; vd[1] = vq[u].y; vd[2] = vq[u].z; vd[3] = vq[u].w;
            }
        }
    }
#pragma unroll
    for (int u = 0; u < NQ; ++u) {
        const int i = tid + kCombThreads * u;
        if (i < g * D) sq[i] = qv[u] * P.qscale;
    }
    // heads 8 .. g-1 of larger query groups (up to 16): one more round
    for (int i = 8 * D + tid; i < g * D; i += kCombThreads) sq[i] = load_elem(P.q, qb + i, P.q_dtype) * P.qscale;
    __syncthreads();
    // logits: thread per (token, head pair j, j + hs); two heads share the K row
    // loads and each dot product runs as two independent chains
    {
        const int hs = (g + 1) / 2;
        for (int i = tid; i < nt * hs; i += kCombThreads) {
            const int t = i % nt, j = i / nt;
            const bool two_h = j + hs < g;
            const uint32_t* kr = sk + t * kRowW;
            const float* qa = sq + j * D;
            const float* qb = sq + (two_h ? j + hs : j) * D;
            float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll 8
            for (int w = 0; w < D / 2; ++w) {
                const uint32_t two = kr[w];
                const float k0 = __uint_as_float(two << 16), k1 = __uint_as_float(two & 0xFFFF0000u);
                a0 = fmaf(qa[2 * w], k0, a0);
                a1 = fmaf(qa[2 * w + 1], k1, a1);
                b0 = fmaf(qb[2 * w], k0, b0);
                b1 = fmaf(qb[2 * w + 1], k1, b1);
            }
            sp[j * kWinTile + t] = a0 + a1;
            if (two_h) sp[(j + hs) * kWinTile + t] = b0 + b1;
        }
    }
    __syncthreads();
    for (int j = warp; j < g; j += kCombThreads / 32) {    // softmax of the tile, per head
        float mx = -INFINITY;
        for (int t = lane; t < nt; t += 32) mx = fmaxf(mx, sp[j * kWinTile + t]);
        for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float sum = 0.f;
        for (int t = lane; t < nt; t += 32) {
            const float pv = exp2f(sp[j * kWinTile + t] - mx);
            sp[j * kWinTile + t] = pv;
            sum += pv;
        }
        for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane == 0) {
            sml[2 * j] = mx;
            sml[2 * j + 1] = sum;
            P.wml[pbase + (int64_t)j * P.n_win_tiles] = make_float2(mx, sum);
        }
    }
    __syncthreads();
    {   // P·V: thread per (head pair j, j + hs; channel pair), sharing the V loads
        const int hs = (g + 1) / 2;
        for (int i = tid; i < hs * (D / 2); i += kCombThreads) {
            const int j = i / (D / 2), w = i % (D / 2);
            const bool two_h = j + hs < g;
            float x0 = 0.f, x1 = 0.f, y0 = 0.f, y1 = 0.f;
            const float* pa = sp + j * kWinTile;
            const float* pb = sp + (two_h ? j + hs : j) * kWinTile;
#pragma unroll 4
            for (int t = 0; t < nt; ++t) {
                const uint32_t two = sv[t * kRowW + w];
                const float v0 = __uint_as_float(two << 16), v1 = __uint_as_float(two & 0xFFFF0000u);
                x0 = fmaf(pa[t], v0, x0);
                x1 = fmaf(pa[t], v1, x1);
                y0 = fmaf(pb[t], v0, y0);
                y1 = fmaf(pb[t], v1, y1);
            }
            float* o = P.wo + (pbase + (int64_t)j * P.n_win_tiles) * D;
            o[2 * w] = x0;
            o[2 * w + 1] = x1;
            if (two_h) {
                float* o2 = P.wo + (pbase + (int64_t)(j + hs) * P.n_win_tiles) * D;
                o2[2 * w] = y0;
                o2[2 * w + 1] = y1;
            }
        }
    }
}

template <int D, int GQ>
__global__ void __launch_bounds__(kCombThreads, D >= 256 ? 2 : 6) window_kernel(DecodeParams P) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    extern __shared__ __align__(16) float s_w[];
    const int hk = blockIdx.x, b = blockIdx.y, wt = (int)blockIdx.z - 1;
    if (wt < 0) {                                  // the first z-slice: query preparation
        prep_slice<D, GQ>(P, hk, b, s_w);
        return;
    }
    window_tile_simt<D>(P, hk, b, wt, s_w, NewRowSrc{nullptr, nullptr, 0, 0});
}

// ---------------------------------------------------------------------------
// window on the tensor cores (d <= 128, g <= 8): the same per-tile partials as
// window_kernel, one block of 4 warps per (KV head, request, 64-token tile).
// The block issues every load of its tile at once (16-byte cp.async of the K
// and V rows, rows past the tile's end read as zero; q with them), then:
//  * warp w computes the logits of tokens 16w .. 16w+15 with
//    mma.sync.m16n8k16 bf16 → fp32: q is the A operand (rows 0..7 the bf16
//    parts of the g heads, rows 8..15 their lo parts q - bf16(q), zero for
//    bf16 q), K enters through ldmatrix; products are exact and
//    S = row h + row h + 8, times log2(e)/√d;
//  * the tile's max and sum per head are combined across the warps in shared
//    memory; p = 2^(S - m) goes to shared memory as A fragments (rows 0..7
//    bf16(p), rows 8..15 the lo parts p - bf16(p));
//  * warp w computes P·V for channels [d/4·w, d/4·(w+1)) over all 64 tokens,
//    V entering through ldmatrix.trans; o = row h + row h + 8.
// ---------------------------------------------------------------------------
namespace wmma_detail {

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&d)[4], uint32_t saddr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]) : "r"(saddr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&d)[4], uint32_t saddr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]) : "r"(saddr));
}
// 16-byte cp.async that copies src_bytes (16 or 0) and fills the rest with zeros
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
// bf16 pair (lower element in the low half) and the pair of lo parts x - bf16(x)
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const uint16_t h0 = f32_to_bf16_bits(x0), h1 = f32_to_bf16_bits(x1);
    hi = (uint32_t)h0 | ((uint32_t)h1 << 16);
    lo = (uint32_t)f32_to_bf16_bits(x0 - bf16_bits_to_f32(h0)) |
         ((uint32_t)f32_to_bf16_bits(x1 - bf16_bits_to_f32(h1)) << 16);
}

}  // namespace wmma_detail

template <int D>
struct WinMmaCfg {
    static constexpr int KS = D / 16;          // k-steps of the logits
    static constexpr int RW = D / 2 + 4;       // words per staged row (≡ 4 mod 32: ldmatrix rows in distinct banks)
    static constexpr int CPR = D / 8;          // 16-byte chunks per row
    static constexpr int NTW = D / 32;         // n-tiles of 8 channels per warp in P·V
    // shared words: one K-then-V tile, q fragments [KS][32][4], P fragments [4][32][4], max / sum [4][8] each
    static constexpr int SMEM_WORDS = kWinTile * RW + KS * 128 + 4 * 128 + 2 * 32;
};

// One 64-token window tile (wt) of KV head hk, request b: the (m, l, o) partial
// of every query head of the KV head.  128 threads; s_wm: WinMmaCfg<D>::SMEM_WORDS.
template <int D>
__device__ __forceinline__ void window_tile_mma(const DecodeParams& P, int hk, int b, int wt, uint32_t* s_wm,
                                                NewRowSrc nr) {
    using namespace wmma_detail;
    using C = WinMmaCfg<D>;
    constexpr int KS = C::KS, RW = C::RW, CPR = C::CPR, NTW = C::NTW;
    // one row tile: K rows for the logits, then V rows over them for P·V (half
    // the shared memory of two tiles: more blocks of the grid per SM)
    uint32_t* sk = s_wm;                               // [64][RW] K rows, then V rows
    uint32_t* sv = sk;
    uint32_t* sqa = sk + kWinTile * RW;                // [KS][32 lanes][4] q fragments
    uint32_t* spa = sqa + KS * 128;                    // [4 sub-tiles][32 lanes][4] P fragments
    float* smx = reinterpret_cast<float*>(spa + 4 * 128);   // [4 warps][8 heads] sub-tile max
    float* ssm = smx + 32;                                   // [4 warps][8 heads] sub-tile sum
    const int g = P.g, S = P.S, W = P.W;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = lane >> 2, j = lane & 3;
    int L, rq;                                     // the prep slice of this grid writes the same to len / req
    if (!request_valid(P, b, &L, &rq)) L = rq = 0;
    const int sink_end = min(S, L);
    const int rec_lo = d_hist_hi(L, S, W);
    const int nplain = L > 0 ? sink_end + max(0, L - rec_lo) : 0;
    const int t0 = wt * kWinTile;
    const int nt = min(kWinTile, nplain - t0);
    const int nwt = P.n_win_tiles;
    const int64_t pbase = ((int64_t)b * P.Hq + hk * g) * nwt + wt;   // + head · nwt
    if (nt <= 0) {                                     // empty tile: neutral partial
        if (tid < g) P.wml[pbase + (int64_t)tid * nwt] = make_float2(-1e30f, 0.f);
        return;
    }
    // ---- the tile's rows of matrix mat (K 0, V 1) into the row tile (cp.async) ----
    auto load_rows = [&](int mat) {
#pragma unroll
        for (int u = 0; u < kWinTile * CPR / 128; ++u) {
            const int i = tid + 128 * u;
            const int t = i / CPR, c = i % CPR;
            const bool ok = t < nt;
            const int tt = t0 + (ok ? t : 0);
            const int pos = tt < sink_end ? tt : rec_lo + tt - sink_end;   // position in the request
            uint32_t* dst = sk + t * RW + 4 * c;
            if (nr.on && ok && pos == L - 1) {         // the step's new token: from the input row
                const int64_t e0 = ((int64_t)b * P.Hkv + hk) * D + 8 * c;
                const void* src = mat ? nr.v : nr.k;
                uint32_t w[4];
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    w[v] = (uint32_t)f32_to_bf16_bits(load_elem(src, e0 + 2 * v, nr.dtype)) |
                           ((uint32_t)f32_to_bf16_bits(load_elem(src, e0 + 2 * v + 1, nr.dtype)) << 16);
                *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
                continue;
            }
            const uint16_t* row = (tt < sink_end)
                ? P.sink + (((int64_t)rq * S + tt) * P.Hkv + hk) * 2 * D
                : P.recent + (((int64_t)rq * W + (rec_lo + tt - sink_end) % W) * P.Hkv + hk) * 2 * D;
            cp_async16_zfill(dst, row + mat * D + 8 * c, ok ? 16u : 0u);
        }
        cp_async_commit();
    };
    load_rows(0);                                      // K rows and q in one round
    {   // q A fragments: entry (kk, lane l, reg e): row (l>>2) + 8·(e&1) (bf16 part / lo part),
        // channels 16kk + 8·(e>>1) + 2·(l&3), +1.  Pairs (e = 2h, 2h+1) share their
        // loads, and every thread's loads are issued before the first is used.
        constexpr int NQ = KS * 64 / 128;
        static_assert(KS % 2 == 0, "whole rounds of 128 fragment pairs");
        const int64_t qb = ((int64_t)b * P.Hq + hk * g) * D;
        float q0[NQ], q1[NQ];
#pragma unroll
        for (int u = 0; u < NQ; ++u) {
            const int x = tid + 128 * u;
            const int kk = x / 64, l = (x / 2) % 32, h = x % 2;
            const int hr = l >> 2, ch = 16 * kk + 8 * h + 2 * (l & 3);
            q0[u] = 0.f;
            q1[u] = 0.f;
            if (hr < g) {
                q0[u] = load_elem(P.q, qb + (int64_t)hr * D + ch, P.q_dtype);
                q1[u] = load_elem(P.q, qb + (int64_t)hr * D + ch + 1, P.q_dtype);
            }
        }
#pragma unroll
        for (int u = 0; u < NQ; ++u) {
            const int x = tid + 128 * u;
            const int kk = x / 64, l = (x / 2) % 32, h = x % 2;
            uint32_t hi, lo;
            split_bf16x2(q0[u], q1[u], hi, lo);
            sqa[(kk * 32 + l) * 4 + 2 * h] = hi;
            sqa[(kk * 32 + l) * 4 + 2 * h + 1] = lo;
        }
    }
    cp_async_wait<0>();
    __syncthreads();
    // ---- logits of sub-tile `warp`: n-tiles tokens 0..7 and 8..15 of it ----
    const int ts = 16 * warp;                          // first token of the sub-tile
    float sv4[4];
    {
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        const int mi = lane >> 3;                      // matrix: tokens +8·(mi >> 1), channels +8·(mi & 1)
        const uint32_t rowa = smem_addr(sk + (ts + (mi >> 1) * 8 + (lane & 7)) * RW) + (mi & 1) * 16;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            const uint4 a = *reinterpret_cast<const uint4*>(sqa + (kk * 32 + lane) * 4);
            uint32_t bk[4];
            ldsm_x4(bk, rowa + kk * 32);
            mma_bf16(c0, a.x, a.y, a.z, a.w, bk[0], bk[1]);
            mma_bf16(c1, a.x, a.y, a.z, a.w, bk[2], bk[3]);
        }
        // head r: tokens 2j, 2j+1 (n-tile 0) and 8+2j, 9+2j (n-tile 1) of the sub-tile
        sv4[0] = (c0[0] + c0[2]) * P.qscale;
        sv4[1] = (c0[1] + c0[3]) * P.qscale;
        sv4[2] = (c1[0] + c1[2]) * P.qscale;
        sv4[3] = (c1[1] + c1[3]) * P.qscale;
        const int tk = ts + 2 * j;
        if (tk >= nt) sv4[0] = -INFINITY;
        if (tk + 1 >= nt) sv4[1] = -INFINITY;
        if (tk + 8 >= nt) sv4[2] = -INFINITY;
        if (tk + 9 >= nt) sv4[3] = -INFINITY;
    }
    float mx = fmaxf(fmaxf(sv4[0], sv4[1]), fmaxf(sv4[2], sv4[3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (j == 0) smx[warp * 8 + r] = mx;
    __syncthreads();                                   // every warp's logits read the K rows
    load_rows(1);                                      // V rows over them, in flight through the softmax
    const float m = fmaxf(fmaxf(smx[r], smx[8 + r]), fmaxf(smx[16 + r], smx[24 + r]));   // token 0 is valid: finite
    float pv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) pv[e] = exp2f(sv4[e] - m);   // masked: 2^-inf = 0
    float sum = (pv[0] + pv[1]) + (pv[2] + pv[3]);
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    if (j == 0) ssm[warp * 8 + r] = sum;
    {
        uint32_t pa[4];
        split_bf16x2(pv[0], pv[1], pa[0], pa[1]);      // rows r (bf16 p) and r + 8 (lo parts), tokens 2j, 2j+1
        split_bf16x2(pv[2], pv[3], pa[2], pa[3]);      // tokens 8+2j, 9+2j
        *reinterpret_cast<uint4*>(spa + (warp * 32 + lane) * 4) = make_uint4(pa[0], pa[1], pa[2], pa[3]);
    }
    cp_async_wait<0>();                                // this thread's V rows landed
    __syncthreads();
    // ---- P·V: channels [d/4·warp, d/4·(warp+1)), all sub-tiles with tokens ----
    float o[NTW][4];
#pragma unroll
    for (int n = 0; n < NTW; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    {
        const int mi = lane >> 3;                      // matrix: tokens +8·(mi & 1), channels +8·(mi >> 1)
        const uint32_t rowv = smem_addr(sv + ((mi & 1) * 8 + (lane & 7)) * RW) + (mi >> 1) * 16 + warp * (D / 4) * 2;
        const int nsub = (nt + 15) / 16;
        for (int ks = 0; ks < nsub; ++ks) {
            const uint4 a = *reinterpret_cast<const uint4*>(spa + (ks * 32 + lane) * 4);
#pragma unroll
            for (int q2 = 0; q2 < NTW / 2; ++q2) {
                uint32_t bv[4];
                ldsm_x4_trans(bv, rowv + ks * 16 * RW * 4 + q2 * 32);
                mma_bf16(o[2 * q2], a.x, a.y, a.z, a.w, bv[0], bv[1]);
                mma_bf16(o[2 * q2 + 1], a.x, a.y, a.z, a.w, bv[2], bv[3]);
            }
        }
    }
    // ---- the tile's partial: m, l per head and o = row r + row r + 8 ----
    if (r < g) {
        const int64_t slot = pbase + (int64_t)r * nwt;
        if (warp == 0 && j == 0)
            P.wml[slot] = make_float2(m, (ssm[r] + ssm[8 + r]) + (ssm[16 + r] + ssm[24 + r]));
        float* op = P.wo + slot * D + warp * (D / 4);
#pragma unroll
        for (int n = 0; n < NTW; ++n)
            *reinterpret_cast<float2*>(op + 8 * n + 2 * j) = make_float2(o[n][0] + o[n][2], o[n][1] + o[n][3]);
    }
}

template <int D, int GQ>
__global__ void __launch_bounds__(128) window_mma_kernel(DecodeParams P) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    extern __shared__ __align__(16) uint32_t s_wm[];
    const int hk = blockIdx.x, b = blockIdx.y, wt = (int)blockIdx.z - 1;
    if (wt < 0) {                                  // the first z-slice (scheduled first): query preparation
        prep_slice<D, GQ>(P, hk, b, reinterpret_cast<float*>(s_wm));
        return;
    }
    window_tile_mma<D>(P, hk, b, wt, s_wm, NewRowSrc{nullptr, nullptr, 0, 0});
}

// ---------------------------------------------------------------------------
// Fused decode step (oscar_decode_step), first of its three launches.  A decode
// step appends one token per request and then attends; the append touches
// only the BF16 ring row of the new token (over the token leaving the window)
// and the history record of the leaving token, and the window attention reads
// the new token from the step's input rows instead of the ring.  So the three
// independent parts of a step's front run in one grid of 128-thread blocks:
//  z = 0, 1:         the append of request y's new K (V) row of KV head x
//                    (the leaving row quantised into its record by one
//                    block per vector, thread c forming output channel c);
//  z = 2:            query preparation of (KV head x, request y);
//  z = 3 .. nwt + 2: window tile z - 3 of (KV head x, request y).
// Blocks start in index order, so the longest chains (the appends) start first.
// The history kernel and the combine follow as in oscar_decode_attention.
// ---------------------------------------------------------------------------
// With the tensor-core window tiles (one 24 KB row tile per block) 9 blocks fit
// an SM's shared memory, so their registers are bounded to match (56 per thread).
template <int D, int GQ, bool MMA>
__global__ void __launch_bounds__(128, MMA ? 9 : 1) step_pre_kernel(DecodeParams P, AppendParams A, NewRowSrc nr) {
    {   // R_K and R_V are no kernel's output: their lines head for L2 while the
        // previous grid drains (two lines per block; the first 2d²·4/256 blocks
        // cover both matrices)
        constexpr int64_t nl = (int64_t)D * D * 4 / 128;            // 128-byte lines of one matrix
        const int64_t bid = blockIdx.x + (int64_t)gridDim.x * (blockIdx.y + (int64_t)gridDim.y * blockIdx.z);
        if (threadIdx.x < 2) {
            const int64_t l = (2 * bid + threadIdx.x) % (2 * nl);
            prefetch_l2(reinterpret_cast<const char*>(l < nl ? A.rot_k : A.rot_v) + 128 * (l % nl));
        }
    }
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    extern __shared__ __align__(16) uint32_t s_step[];
    const int hk = blockIdx.x, b = blockIdx.y, z = (int)blockIdx.z;
    if (z < 2) {
        // request b's new token (input row b) is position L - 1; an invalid
        // request is reported by its prep slice and appends nothing
        int L, rq;
        const bool ok = request_valid(P, b, &L, &rq);
        float* sx = reinterpret_cast<float*>(s_step);
        append_vec_resolved<D>(A, b, hk, z, b, L - 1, rq, ok, 0, sx, sx + D);
        return;
    }
    if (z == 2) {
        prep_slice<D, GQ>(P, hk, b, reinterpret_cast<float*>(s_step));
        return;
    }
    if constexpr (MMA) window_tile_mma<D>(P, hk, b, z - 3, s_step, nr);
    else window_tile_simt<D>(P, hk, b, z - 3, reinterpret_cast<float*>(s_step), nr);
}

// ---------------------------------------------------------------------------
// combine: one block of 512 threads per (KV head, request).  Merges the BF16
// window tiles and, separately, the history partials by log-sum-exp, applies
// R_Vᵀ once to the merged rotated-domain sum, and merges the two domains:
//   out = (e^{m_p-M}·Σ_bf16 p v + e^{m_r-M}·(Σ_hist p v̂)·R_Vᵀ) / (e^{m_p-M} l_p + e^{m_r-M} l_r).
// The kernel is latency-bound, so it is organised around few rounds of global
// loads: every thread issues the (m, l) pairs and o values of all partials of
// its (head, channel) items together and merges them with a running maximum;
// R_Vᵀ is applied with one warp per row of R_V (coalesced row loads, all rows
// of the warp in flight) and warp reductions.
// ---------------------------------------------------------------------------
template <int D>
struct CombCfg {
    static constexpr int NV = (kCombHeads * D + kMergeThreads - 1) / kMergeThreads;   // (head, channel) items per thread
    static constexpr int RPW = D / (kMergeThreads / 32);                     // R_V rows per warp
    static constexpr int F4 = (D / 4 + 31) / 32;                             // float4 of a row per lane
};

// Running log-sum-exp merge of one (m, l) partial and its o value into (M, l, a).
__device__ __forceinline__ void lse_merge(float m, float lv, float x, float& M, float& l, float& a) {
    if (m > M) {
        const float sc = M > -INFINITY ? exp2f(M - m) : 0.f;
        l *= sc;
        a *= sc;
        M = m;
    }
    const float w = exp2f(m - M);
    l = fmaf(w, lv, l);
    a = fmaf(w, x, a);
}

// A request with more than kCombSlice history partials (few requests over
// many CTAs: a single request splits over every CTA) is merged in slices:
// blocks z, z + gridDim.z, ... each merge kCombSlice partials of the request
// in place into the slice's first slot, and the block whose arrival completes
// the count (an atomic per request and KV head, zeroed by prep) merges the
// slices and finishes.
constexpr int kCombSlice = 32;

// Per-block facts of one (KV head, request) of the combine.
struct CombReq {
    int hk, b, nwt, psh, nsl;
    int hq0, gh, grp;                           // first query head of the block, heads in it, head group
    int64_t N, i_lo, sl0;
    float* outp;
};

// Whether history partial slot u of the request belongs to a CTA with a chunk run.
__device__ __forceinline__ uint8_t comb_slot_valid(const DecodeParams& P, const CombReq& R, int u) {
    const int64_t ci = R.i_lo + (u >> R.psh);
    if ((ci + 1) * R.N < 0x7FFFFFFF) {              // 32-bit division when the products fit
        const uint32_t n = (uint32_t)P.n_ctas;
        return (uint32_t)(ci * R.N) / n < (uint32_t)((ci + 1) * R.N) / n;
    }
    return cta_has_work(ci, R.N, P.n_ctas);
}

// Row c of R_V against the merged rotated sums of heads j0 .. j0 + g - 1: the
// lane's partial dot products of the (up to) NH heads are summed over the warp by a butterfly
// that halves the values a lane carries at each of the first log2(NH) steps
// (NH - 1 shuffles), then a plain reduction over the remaining lane bits; head
// h = bits 4, 3, ... of the lane then holds its total, and the first lane of
// each head's group writes the output.
template <int D, int NH>
__device__ __forceinline__ void row_heads(const CombReq& R, const float4 (&rv)[CombCfg<D>::F4], const float* srot,
                                          const float* spl, const float* sst, int g, int c, int lane, int j0 = 0) {
    srot += j0 * D;
    spl += j0 * D;
    sst += 4 * j0;
    float* outp = R.outp + j0 * D;
    float v[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
        float y = 0.f;
        if (j < g) {
#pragma unroll
            for (int f = 0; f < CombCfg<D>::F4; ++f) {
                const int k4 = lane + 32 * f;
                if (k4 < D / 4) {
                    const float4 xv = *reinterpret_cast<const float4*>(srot + j * D + 4 * k4);
                    y = fmaf(xv.x, rv[f].x, fmaf(xv.y, rv[f].y, fmaf(xv.z, rv[f].z, fmaf(xv.w, rv[f].w, y))));
                }
            }
        }
        v[j] = y;
    }
    int off = 16;
#pragma unroll
    for (int cnt = NH; cnt > 1; cnt >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int k = 0; k < cnt / 2; ++k) {
            const float send = upper ? v[k] : v[k + cnt / 2];
            const float keep = upper ? v[k + cnt / 2] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
#pragma unroll
    for (int o2 = off; o2 >= 1; o2 >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o2);
    // head of this lane: bit 4 of the lane selects the upper half, bit 3 the upper quarter, ...
    int h = 0;
#pragma unroll
    for (int cnt = NH, bit = 16; cnt > 1; cnt >>= 1, bit >>= 1) h += (lane & bit) ? cnt / 2 : 0;
    const int first = (lane & ~(2 * off - 1)) == lane;     // lowest lane of the head's group
    if (first && h < g)
        outp[h * D + c] = fmaf(sst[4 * h + 0], spl[h * D + c], sst[4 * h + 1] * v[0]) * sst[4 * h + 2];
}

// Final merge of the window partials and of the history partials at slots
// sl0 + stride·u, u < hn (SLICED: slice results written by other blocks, valid
// when l > 0, read past L1; otherwise the raw partials with their validity in
// sval), then R_Vᵀ and the output.
template <int D, bool SLICED>
__device__ __forceinline__ void combine_finish(const DecodeParams& P, const CombReq& R, float* s_c,
                                               const uint8_t* sval, int hn) {
    using C = CombCfg<D>;
    const int g = R.gh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t stride = SLICED ? kCombSlice : 1;
    float* srot = s_c;                             // [g][D] merged rotated sum
    float* spl = srot + g * D;                     // [g][D] merged window sum
    float* sst = spl + g * D;                      // [g][4]: weights of the two domains and 1 / denominator
    // ---- one round of loads per 8 partials: thread items (head j, channel c) ----
#pragma unroll
    for (int v = 0; v < C::NV; ++v) {
        const int i = tid + kMergeThreads * v;
        if (i >= g * D) break;
        const int j = i / D, c = i % D;
        const int hq = R.hq0 + j;
        float Mp = -INFINITY, lp = 0.f, ap = 0.f;
        const int64_t wb = ((int64_t)R.b * P.Hq + hq) * R.nwt;
        for (int t0 = 0; t0 < R.nwt; t0 += 8) {
            float2 ml[8];
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const bool in = t0 + u < R.nwt;
                ml[u] = in ? P.wml[wb + t0 + u] : make_float2(-INFINITY, 0.f);
                x[u] = in ? P.wo[(wb + t0 + u) * D + c] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (ml[u].y > 0.f) lse_merge(ml[u].x, ml[u].y, x[u], Mp, lp, ap);
        }
        float Mr = -INFINITY, lr = 0.f, ar = 0.f;
        constexpr int UB = 8;                      // partials per round of loads (register budget)
        for (int u0 = 0; u0 < hn; u0 += UB) {
            float2 ml[UB];
            float x[UB];
#pragma unroll
            for (int u = 0; u < UB; ++u) {
                const bool in = u0 + u < hn;
                const int64_t sl = R.sl0 + stride * (u0 + u);
                if (SLICED) {
                    ml[u] = in ? __ldcg(P.ml + sl * P.Hq + hq) : make_float2(-INFINITY, 0.f);
                    x[u] = in ? __ldcg(P.po + (sl * P.Hq + hq) * D + c) : 0.f;
                } else {
                    ml[u] = in ? P.ml[sl * P.Hq + hq] : make_float2(-INFINITY, 0.f);
                    x[u] = in ? P.po[(sl * P.Hq + hq) * D + c] : 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < UB; ++u)
                if (u0 + u < hn && (SLICED || sval[u0 + u]) && ml[u].y > 0.f) lse_merge(ml[u].x, ml[u].y, x[u], Mr, lr, ar);
        }
        srot[i] = ar;
        spl[i] = ap;
        if (c == 0) {                              // every item of head j merged the same (m, l) sequence
            const float Mx = fmaxf(Mp, Mr);
            const float wp = lp > 0.f ? exp2f(Mp - Mx) : 0.f;
            const float wr = lr > 0.f ? exp2f(Mr - Mx) : 0.f;
            sst[4 * j + 0] = wp;
            sst[4 * j + 1] = wr;
            sst[4 * j + 2] = 1.0f / (wp * lp + wr * lr);
        }
    }
    __syncthreads();
    // ---- (Σ_hist p v̂)·R_Vᵀ: y[j][c] = Σ_k x[j][k]·R_V[c][k], one warp per row c ----
    constexpr int RB = C::F4 > 1 ? 2 : 4;          // rows whose loads are in flight together
#pragma unroll 1
    for (int r0 = 0; r0 < C::RPW; r0 += RB) {
        float4 rv[RB][C::F4];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const int c = warp + (kMergeThreads / 32) * (r0 + r);
            const float4* row = reinterpret_cast<const float4*>(P.rot_v + (int64_t)c * D);
#pragma unroll
            for (int f = 0; f < C::F4; ++f) {
                const int k4 = lane + 32 * f;
                rv[r][f] = (r0 + r < C::RPW && k4 < D / 4) ? row[k4] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            if (r0 + r >= C::RPW) break;
            const int c = warp + (kMergeThreads / 32) * (r0 + r);
            for (int j0 = 0; j0 < g; j0 += 4)   // four heads at a time
                row_heads<D, 4>(R, rv[r], srot, spl, sst, min(4, g - j0), c, lane, j0);
        }
    }
}

// The sliced merge of a request with more than kCombSlice history partials
// (kept out of line: the common path's registers stay as they are).
// The sliced request's finish, out of line like the slice merge itself.
template <int D>
__device__ __noinline__ void combine_finish_sliced(const DecodeParams& P, const CombReq& R, float* s_c,
                                                   const uint8_t* sval, int nslice) {
    combine_finish<D, true>(P, R, s_c, sval, nslice);
}

template <int D>
__device__ __noinline__ void combine_sliced(const DecodeParams& P, const CombReq& R, float* s_c, int nslice) {
    using C = CombCfg<D>;
    __shared__ int s_last;
    __shared__ float s_w[kCombHeads][kCombSlice];  // per (head, slot of the slice): weight e^{m - M_head}
    __shared__ float s_ml[kCombHeads][2];          // per head: M and Σ weight·l over the slice
    const int g = R.gh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t* sval = reinterpret_cast<uint8_t*>(s_c + (2 * g * D + 4 * g));
    for (int sc = blockIdx.z; sc < nslice; sc += gridDim.z) {
        const int u_lo = sc * kCombSlice, u_n = min(kCombSlice, R.nsl - u_lo);
        const int64_t sl0 = R.sl0 + u_lo;
        // first (m, l) of the slice through one warp per head (lane = slot) into
        // weights e^{m - M} in shared memory; then every o value of the thread's
        // item in one round of loads
        if (warp < g) {
            const int hq = R.hq0 + warp;
            float m = -INFINITY, l = 0.f;
            if (lane < u_n && comb_slot_valid(P, R, u_lo + lane)) {
                const float2 ml = P.ml[(sl0 + lane) * P.Hq + hq];
                if (ml.y > 0.f) { m = ml.x; l = ml.y; }
            }
            float M = m;
#pragma unroll
            for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            const float w = l > 0.f ? exp2f(m - M) : 0.f;
            float lw = w * l;
#pragma unroll
            for (int o = 16; o; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
            s_w[warp][lane] = w;
            if (lane == 0) { s_ml[warp][0] = M; s_ml[warp][1] = lw; }
        }
        __syncthreads();
#pragma unroll 1
        for (int v = 0; v < C::NV; ++v) {
            const int i = tid + kMergeThreads * v;
            const int j = min(i / D, g - 1), c = i % D;
            const int hq = R.hq0 + j;
            const float* px = P.po + (sl0 * P.Hq + hq) * D + c;
            const int64_t step = (int64_t)P.Hq * D;  // one slot further
            const int un = i < g * D ? u_n : 0;
            // slots of CTAs without a chunk run were never written: weight 0, not loaded
            float x[kCombSlice];
#pragma unroll
            for (int u = 0; u < kCombSlice; ++u) x[u] = (u < un && s_w[j][u] != 0.f) ? px[u * step] : 0.f;
            float a = 0.f;
#pragma unroll
            for (int u = 0; u < kCombSlice; ++u) a = fmaf(s_w[j][u], x[u], a);
            if (i < g * D) s_c[i] = a;             // the finish's scratch is free until the last slice
        }
        __syncthreads();                           // every read of the slice's first slot is done
        const int64_t slw = sl0;                   // the slice's result replaces its first slot
#pragma unroll
        for (int v = 0; v < C::NV; ++v) {
            const int i = tid + kMergeThreads * v;
            if (i >= g * D) continue;
            const int j = i / D, c = i % D;
            const int hq = R.hq0 + j;
            P.po[(slw * P.Hq + hq) * D + c] = s_c[i];
            if (c == 0) P.ml[slw * P.Hq + hq] = s_ml[j][1] > 0.f ? make_float2(s_ml[j][0], s_ml[j][1])
                                                                  : make_float2(-INFINITY, 0.f);
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = atomicAdd(P.comb_count + ((int64_t)R.b * P.Hkv + R.hk) * kCombGroups + R.grp, 1) == nslice - 1;
        __syncthreads();
        if (s_last) {                              // every slice is merged: finish the request
            __threadfence();
            combine_finish_sliced<D>(P, R, s_c, sval, nslice);
            return;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kMergeThreads, D == 128 ? 2 : 1) combine_kernel(DecodeParams P) {
    {   // R_V is no kernel's output: its lines head for L2 while the history grid drains
        constexpr int nl = D * D * 4 / 128;
        const int bid = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        if (threadIdx.x < 8) prefetch_l2(reinterpret_cast<const char*>(P.rot_v) + 128 * ((8 * bid + threadIdx.x) % nl));
    }
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    extern __shared__ __align__(16) float s_c[];
    const int g = P.g;
    const int tid = threadIdx.x;
    CombReq R;
    const int ngrp = (g + kCombHeads - 1) / kCombHeads;
    R.hk = blockIdx.x / ngrp;
    const int grp = blockIdx.x % ngrp;
    R.b = blockIdx.y;
    R.gh = min(kCombHeads, g - grp * kCombHeads);
    R.hq0 = R.hk * g + grp * kCombHeads;
    R.grp = grp;
    const int L = P.len[R.b];
    R.outp = P.out + ((int64_t)R.b * P.Hq + R.hq0) * D;
    if (L <= 0) {
        if (blockIdx.z == 0)
            for (int i = tid; i < R.gh * D; i += kMergeThreads) R.outp[i] = 0.f;
        return;
    }
    R.N = P.cprefix[P.batch];
    const int64_t c0 = P.cprefix[R.b], c1 = P.cprefix[R.b + 1];
    R.i_lo = c1 > c0 ? chunk_owner(c0, R.N, P.n_ctas) : 0;
    const int64_t i_hi = c1 > c0 ? chunk_owner(c1 - 1, R.N, P.n_ctas) : -1;
    R.nwt = P.n_win_tiles;
    R.psh = P.par == 2 ? 1 : 0;                    // partial slots per (CTA, request) = 1 << psh
    R.nsl = (int)(i_hi - R.i_lo + 1) << R.psh;     // this request's partial slots: (i_lo << psh) + b·par + u
    R.sl0 = (R.i_lo << R.psh) + ((int64_t)R.b << R.psh);
    const int nslice = R.nsl > kCombSlice ? (R.nsl + kCombSlice - 1) / kCombSlice : 1;
    if ((int)blockIdx.z >= nslice) return;
    if (nslice > 1) {
        combine_sliced<D>(P, R, s_c, nslice);
        return;
    }
    uint8_t* sval = reinterpret_cast<uint8_t*>(s_c + (2 * R.gh * D + 4 * R.gh));   // [nsl]: slot's CTA had a chunk run
    for (int u = tid; u < R.nsl; u += kMergeThreads) sval[u] = comb_slot_valid(P, R, u);
    __syncthreads();
    combine_finish<D, false>(P, R, s_c, sval, R.nsl);
}

}  // namespace oscar

using namespace oscar;

static int decode_validate(const oscar_config* cfg, const oscar_layer_cache* cache, int32_t batch,
                           int32_t max_seq_len, int64_t pt_stride) {
    int rc = validate_config(cfg);
    if (rc) return rc;
    rc = validate_cache(cfg, cache);
    if (rc) return rc;
    if (batch < 0 || batch > kMaxDecodeBatch)
        return fail(OSCAR_ERR_ARG, "batch must be in [0, %d] (got %d)", kMaxDecodeBatch, batch);
    if (max_seq_len < 1) return fail(OSCAR_ERR_ARG, "max_seq_len must be >= 1");
    if (pt_stride < max_seq_len) return fail(OSCAR_ERR_ARG, "pt_stride (%lld) must be >= max_seq_len (%d)",
                                             (long long)pt_stride, max_seq_len);
    if ((int64_t)cfg->num_q_heads * cfg->head_dim > 16384)
        return fail(OSCAR_ERR_ARG, "num_q_heads * head_dim must be <= 16384");
    return OSCAR_OK;
}

extern "C" int oscar_decode_workspace_bytes(const oscar_config* cfg, int32_t batch, int32_t max_seq_len,
                                            size_t* bytes) {
    clear_error();
    int rc = validate_config(cfg);
    if (rc) return rc;
    if (!bytes) return fail(OSCAR_ERR_NULL, "bytes is NULL");
    if (batch < 0 || batch > kMaxDecodeBatch || max_seq_len < 1)
        return fail(OSCAR_ERR_ARG, "batch in [0, %d] and max_seq_len >= 1 required", kMaxDecodeBatch);
    const int nsm = sm_count();
    if (nsm <= 0) return OSCAR_ERR_CUDA;
    *bytes = make_plan(cfg, batch, max_seq_len, nsm).total;
    return OSCAR_OK;
}

namespace oscar {
int launch_history_mma(DecodeParams& P, int head_dim, cudaStream_t st, bool* launched);
}

template <int D>
static int launch_history_combine(DecodeParams& P, cudaStream_t st, int impl);

template <int D>
static int launch_decode(DecodeParams& P, cudaStream_t st, int impl) {
    // the window kernel's grid carries one more z-slice: the query preparation
    // of every (KV head, request)
    const int gq = prep_bucket(P.g);
    const size_t psmem = (size_t)prep_smem_floats(D, gq) * 4;
    int rc = OSCAR_OK;
    const dim3 wgrid(P.Hkv, P.batch, P.n_win_tiles + 1);
    if (D <= 128 && P.g <= 8) {
        // tensor-core window: one block of 4 warps per (KV head, request, 64-token tile)
        constexpr int DW = D <= 128 ? D : 128;
        const size_t wsmem = std::max((size_t)WinMmaCfg<DW>::SMEM_WORDS * 4, psmem);
        auto kern = gq == 4 ? window_mma_kernel<DW, 4> : window_mma_kernel<DW, 8>;
        if (const int rc_ = ensure_dynamic_smem((const void*)kern, wsmem, "cudaFuncSetAttribute(window_mma_kernel)"))
            return rc_;
        const int prof_k = prof_begin(4, st);
        launch_dependent(kern, wgrid, dim3(128), wsmem, st, P);
        prof_end(prof_k, st);
    } else {
        const size_t wsmem = std::max(((size_t)P.g * D + (size_t)P.g * kWinTile + 2 * P.g) * 4 +
                                          (size_t)2 * kWinTile * (D / 2 + 1) * 4, psmem);
        auto kern = gq == 4 ? window_kernel<D, 4> : gq == 8 ? window_kernel<D, 8> : window_kernel<D, 16>;
        if (const int rc_ = ensure_dynamic_smem((const void*)kern, wsmem, "cudaFuncSetAttribute(window_kernel)"))
            return rc_;
        const int prof_k = prof_begin(4, st);
        launch_dependent(kern, wgrid, dim3(kCombThreads), wsmem, st, P);
        prof_end(prof_k, st);
    }
    rc = check_cuda("window kernel launch");
    if (rc) return rc;
    return launch_history_combine<D>(P, st, impl);
}

// The history kernel (tensor cores when a variant fits, else CUDA cores) and
// the combine, after the window partials and the rotated queries are written.
template <int D>
static int launch_history_combine(DecodeParams& P, cudaStream_t st, int impl) {
    int rc = OSCAR_OK;
    const int gq = prep_bucket(P.g);
    bool done = false;
    const int prof = prof_begin(0, st);
    if (impl != 1) {
        rc = launch_history_mma(P, D, st, &done);
        if (rc) return rc;
    }
    if (!done) {
        const int nwarps = std::min(16, P.Hkv);
        const int threads = 32 * nwarps;
        const size_t smem = ((size_t)P.Hq * D + (size_t)nwarps * gq * 32) * 4;
        auto pick = [&](auto kern) -> int {
            if (const int rc_ = ensure_dynamic_smem((const void*)kern, smem, "cudaFuncSetAttribute(history_simt_kernel)"))
                return rc_;
            int per_sm = 0;
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
            const int grid = std::min(P.n_ctas, std::max(1, sm_count() * std::max(1, per_sm)));
            P.n_ctas = grid;
            launch_dependent(kern, dim3(grid), dim3(threads), smem, st, P);
            return check_cuda("history_simt_kernel launch");
        };
        if (gq == 4) rc = pick(history_simt_kernel<D, 4>);
        else if (gq == 8) rc = pick(history_simt_kernel<D, 8>);
        else rc = pick(history_simt_kernel<D, 16>);
        if (rc) return rc;
    }
    prof_end(prof, st);
    const int gh = std::min(P.g, kCombHeads);   // query heads per combine block
    const size_t csmem = ((size_t)gh * D * 2 + (size_t)gh * 4) * 4 + (size_t)P.n_ctas * P.par + 16;
    // blocks per (request, KV head) for slice merging: about the slices an even split
    // over the history grid gives each request (any count is correct)
    const int nz = std::max(1, std::min(16, (P.n_ctas * P.par / std::max(1, P.batch) + kCombSlice - 1) / kCombSlice));
    if (const int rc_ = ensure_dynamic_smem((const void*)combine_kernel<D>, csmem, "cudaFuncSetAttribute(combine_kernel)"))
        return rc_;
    {
        const int prof_k = prof_begin(5, st);
        launch_dependent(combine_kernel<D>, dim3(P.Hkv * ((P.g + kCombHeads - 1) / kCombHeads), P.batch, nz),
                         dim3(kMergeThreads), csmem, st, P);
        prof_end(prof_k, st);
    }
    return check_cuda("combine_kernel launch");
}

// The fused decode step: one launch for the append, the query preparation and
// the window tiles, then the history kernel and the combine.
template <int D>
static int launch_step(DecodeParams& P, const AppendParams& A, NewRowSrc nr, cudaStream_t st) {
    const int gq = prep_bucket(P.g);
    const size_t psmem = (size_t)prep_smem_floats(D, gq) * 4;
    const size_t asmem = (size_t)2 * D * 4;
    const dim3 grid(P.Hkv, P.batch, P.n_win_tiles + 3);
    auto go = [&](auto kern, size_t wsmem) -> int {
        const size_t smem = std::max(std::max(wsmem, psmem), asmem);
        if (const int rc_ = ensure_dynamic_smem((const void*)kern, smem, "cudaFuncSetAttribute(step_pre_kernel)"))
            return rc_;
        const int prof_k = prof_begin(7, st);
        launch_dependent(kern, grid, dim3(128), smem, st, P, A, nr);
        prof_end(prof_k, st);
        return check_cuda("step_pre_kernel launch");
    };
    int rc;
    if constexpr (D <= 128) {
        if (P.g <= 8) {
            const size_t wsmem = (size_t)WinMmaCfg<D>::SMEM_WORDS * 4;
            rc = gq == 4 ? go(step_pre_kernel<D, 4, true>, wsmem) : go(step_pre_kernel<D, 8, true>, wsmem);
            if (rc) return rc;
            return launch_history_combine<D>(P, st, 0);
        }
    }
    const size_t wsmem = ((size_t)P.g * D + (size_t)P.g * kWinTile + 2 * P.g) * 4 + (size_t)2 * kWinTile * (D / 2 + 1) * 4;
    rc = gq == 4 ? go(step_pre_kernel<D, 4, false>, wsmem)
       : gq == 8 ? go(step_pre_kernel<D, 8, false>, wsmem) : go(step_pre_kernel<D, 16, false>, wsmem);
    if (rc) return rc;
    return launch_history_combine<D>(P, st, 0);
}

// Validates a decode call and fills P (batch > 0).
static int decode_prepare(const oscar_config* cfg, const oscar_layer_cache* cache, const void* q,
                          const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                          const int32_t* req_idx, int32_t batch, int32_t max_seq_len, float* out,
                          void* workspace, size_t workspace_bytes, DecodeParams& P) {
    if (!q || !page_table || !seq_lens || !out) return fail(OSCAR_ERR_NULL, "q, page_table, seq_lens and out are required");
    const int nsm = sm_count();
    if (nsm <= 0) return OSCAR_ERR_CUDA;
    const DecodePlan plan = make_plan(cfg, batch, max_seq_len, nsm);
    if (!workspace) return fail(OSCAR_ERR_WORKSPACE, "workspace is NULL");
    if (workspace_bytes < plan.total)
        return fail(OSCAR_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", workspace_bytes, plan.total);
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return fail(OSCAR_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    P.q = q;
    P.q_dtype = cfg->q_dtype;
    P.page_table = page_table;
    P.pt_stride = pt_stride;
    P.seq_lens = seq_lens;
    P.req_idx = req_idx;
    P.batch = batch;
    P.max_seq_len = max_seq_len;
    P.out = out;
    P.records = cache->records;
    P.sink = cache->sink;
    P.recent = cache->recent;
    P.rot_k = cache->rot_k;
    P.rot_v = cache->rot_v;
    P.num_slots = cache->num_slots;
    P.max_reqs = cache->max_reqs;
    P.Hq = cfg->num_q_heads;
    P.Hkv = cfg->num_kv_heads;
    P.g = P.Hq / P.Hkv;
    P.S = cfg->sink;
    P.W = cfg->recent;
    P.G = cfg->group_size;
    P.ng = cfg->head_dim / cfg->group_size;
    const RecordLayout lay = record_layout(cfg->head_dim, cfg->group_size, cfg->scale_dtype);
    P.rec_bytes = lay.bytes;
    P.slot_bytes = slot_bytes(lay, cfg->num_kv_heads);
    P.fp8 = cfg->scale_dtype == OSCAR_SCALE_E4M3;
    P.chunk = plan.chunk;
    P.n_ctas = plan.max_ctas;          // set by the history launcher
    P.par = 1;                         // set by the tensor-core history launcher
    P.n_frag_tiles = plan.n_frag_tiles;
    P.n_win_tiles = plan.n_win_tiles;
    P.qscale = (float)(1.4426950408889634 / std::sqrt((double)cfg->head_dim));
    char* ws = reinterpret_cast<char*>(workspace);
    P.len = reinterpret_cast<int32_t*>(ws + plan.off_len);
    P.req = reinterpret_cast<int32_t*>(ws + plan.off_req);
    P.cprefix = reinterpret_cast<int32_t*>(ws + plan.off_cprefix);
    P.qt = reinterpret_cast<float*>(ws + plan.off_qt);
    P.qsum = reinterpret_cast<float2*>(ws + plan.off_qsum);
    P.qfrag = reinterpret_cast<uint2*>(ws + plan.off_qfrag);
    P.ml = reinterpret_cast<float2*>(ws + plan.off_ml);
    P.po = reinterpret_cast<float*>(ws + plan.off_o);
    P.comb_count = reinterpret_cast<int*>(ws + plan.off_cnt);
    P.wml = reinterpret_cast<float2*>(ws + plan.off_wml);
    P.wo = reinterpret_cast<float*>(ws + plan.off_wo);
    P.status = status_word();
    if (!P.status) return OSCAR_ERR_CUDA;
    return OSCAR_OK;
}

static int decode_impl(const oscar_config* cfg, const oscar_layer_cache* cache, const void* q,
                       const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                       const int32_t* req_idx, int32_t batch, int32_t max_seq_len, float* out,
                       void* workspace, size_t workspace_bytes, void* stream, int impl) {
    clear_error();
    int rc = decode_validate(cfg, cache, batch, max_seq_len, pt_stride);
    if (rc) return rc;
    if (batch == 0) return OSCAR_OK;
    DecodeParams P;
    rc = decode_prepare(cfg, cache, q, page_table, pt_stride, seq_lens, req_idx, batch, max_seq_len, out,
                        workspace, workspace_bytes, P);
    if (rc) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    switch (cfg->head_dim) {
        case 64: return launch_decode<64>(P, st, impl);
        case 128: return launch_decode<128>(P, st, impl);
        default: return launch_decode<256>(P, st, impl);
    }
}

extern "C" int oscar_decode_attention(const oscar_config* cfg, const oscar_layer_cache* cache, const void* q,
                                      const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                                      const int32_t* req_idx, int32_t batch, int32_t max_seq_len, float* out,
                                      void* workspace, size_t workspace_bytes, void* stream) {
    return decode_impl(cfg, cache, q, page_table, pt_stride, seq_lens, req_idx, batch, max_seq_len, out,
                       workspace, workspace_bytes, stream, 0);
}

extern "C" int oscar_decode_attention_simt(const oscar_config* cfg, const oscar_layer_cache* cache, const void* q,
                                           const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                                           const int32_t* req_idx, int32_t batch, int32_t max_seq_len, float* out,
                                           void* workspace, size_t workspace_bytes, void* stream) {
    return decode_impl(cfg, cache, q, page_table, pt_stride, seq_lens, req_idx, batch, max_seq_len, out,
                       workspace, workspace_bytes, stream, 1);
}

extern "C" int oscar_decode_step(const oscar_config* cfg, const oscar_layer_cache* cache, const void* k_new,
                                 const void* v_new, const void* q, const int32_t* page_table, int64_t pt_stride,
                                 const int32_t* seq_lens, const int32_t* req_idx, int32_t batch,
                                 int32_t max_seq_len, float* out, void* workspace, size_t workspace_bytes,
                                 void* stream) {
    clear_error();
    int rc = decode_validate(cfg, cache, batch, max_seq_len, pt_stride);
    if (rc) return rc;
    if (batch == 0) return OSCAR_OK;
    if (!k_new || !v_new) return fail(OSCAR_ERR_NULL, "k_new and v_new are required");
    DecodeParams P;
    rc = decode_prepare(cfg, cache, q, page_table, pt_stride, seq_lens, req_idx, batch, max_seq_len, out,
                        workspace, workspace_bytes, P);
    if (rc) return rc;
    // the append of row b (position seq_lens[b] - 1): the fields the per-vector
    // append reads; the request resolution is the fused kernel's
    AppendParams A = {};
    A.k = k_new;
    A.v = v_new;
    A.kv_dtype = cfg->kv_dtype;
    A.req_idx = req_idx;
    A.page_table = page_table;
    A.pt_stride = pt_stride;
    A.batch = batch;
    A.records = cache->records;
    A.sink = cache->sink;
    A.recent = cache->recent;
    A.rot_k = cache->rot_k;
    A.rot_v = cache->rot_v;
    A.num_slots = cache->num_slots;
    A.max_reqs = cache->max_reqs;
    A.Hkv = cfg->num_kv_heads;
    A.S = cfg->sink;
    A.W = cfg->recent;
    A.G = cfg->group_size;
    A.rec_bytes = P.rec_bytes;
    A.slot_bytes = P.slot_bytes;
    A.fp8 = P.fp8;
    A.clip = cfg->clip_ratio;
    A.total_new = batch;
    A.status = P.status;
    const NewRowSrc nr{k_new, v_new, cfg->kv_dtype, 1};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    switch (cfg->head_dim) {
        case 64: return launch_step<64>(P, A, nr, st);
        case 128: return launch_step<128>(P, A, nr, st);
        default: return launch_step<256>(P, A, nr, st);
    }
}

// ---------------------------------------------------------------------------
// Allocation-free decode.  Some callers cannot allocate device memory for a
// workspace: host runtimes that reserve nearly all of the GPU for their own
// pool at start-up and hand plug-in kernels no allocation rights, and code
// paths where a cudaMalloc, which may synchronise the device, is not allowed.
// For them the decode below uses a fixed scratch area compiled into the
// library instead of a caller-provided workspace.  Every GPU that loads the
// library holds this array until the process exits.
// ---------------------------------------------------------------------------
namespace oscar {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;   // 16 MiB per device
__device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

// Device address of the scratch array in the current context.  Host code may
// not use g_decode_scratch's name as an address (it is a host-side stand-in),
// so the address is asked for on every call, with the caller's device current:
// the lookup allocates nothing, and a context created after a device reset
// (which loads the module again, possibly elsewhere) gets its own address.
static int static_scratch(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p)
        return fail(OSCAR_ERR_CUDA, "cudaGetSymbolAddress(decode scratch): %s", cudaGetErrorString(e));
    *out = p;
    return OSCAR_OK;
}

}  // namespace oscar

extern "C" int oscar_decode_attention_noalloc(const oscar_config* cfg, const oscar_layer_cache* cache,
                                              const void* q, const int32_t* page_table, int64_t pt_stride,
                                              const int32_t* seq_lens, const int32_t* req_idx, int32_t batch,
                                              int32_t max_seq_len, float* out, void* stream) {
    clear_error();
    int rc = decode_validate(cfg, cache, batch, max_seq_len, pt_stride);
    if (rc) return rc;
    const int nsm = sm_count();
    if (nsm <= 0) return OSCAR_ERR_CUDA;
    const size_t need = make_plan(cfg, batch, max_seq_len, nsm).total;
    if (need > kStaticScratchBytes)
        return fail(OSCAR_ERR_WORKSPACE,
                    "batch %d with max_seq_len %d needs %zu bytes of scratch; the built-in scratch holds %zu "
                    "(use oscar_decode_attention with a caller workspace)",
                    batch, max_seq_len, need, kStaticScratchBytes);
    void* ws = nullptr;
    rc = static_scratch(&ws);
    if (rc) return rc;
    return decode_impl(cfg, cache, q, page_table, pt_stride, seq_lens, req_idx, batch, max_seq_len, out, ws,
                       kStaticScratchBytes, stream, 0);
}
