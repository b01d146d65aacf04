// Prefill attention of a chunk over the mixed-precision cache, with no
// dequantised copy of the prefix.
//
// [Prefix log] "KVプールが上限だった — hybrid GDN の長文キャッシュ…": the INT2
// prefill path of the integration expands the cached prefix to fp16 in a
// workspace that grows with the sequence (dequantize_prefix_kv) and then runs
// ordinary attention.  Here the chunk's queries read the INT2 records directly.
// [OSCAR news] "サービングシステム：混合精度キャッシュレイアウト": the prefix is 64
// BF16 sink tokens, INT2 history (rotated), 256 BF16 recent tokens.
//
// Query i of request b's chunk (position L0 + i) attends over the prefix as
// stored (positions < L0) and over the chunk's own keys at positions L0 .. L0+i
// (bf16), one softmax, scale 1/sqrt(d); query head h reads KV head h/(Hq/Hkv).
//
// Everything runs in the rotated domain.  An INT2 key or value of group g is
// k̂ = s_g·c + z_g with c an integer in 0..3, exact as an fp16 tensor-core
// operand, so
//    q̃·k̂ = Σ_g s_g·(q̃_g·c_g) + z_g·Σ_{c∈g} q̃_c      and      Σ_t p_t v̂_t = Σ_t (p_t s_g)·c_t + Σ_t p_t z_g
// take the codes as operands (per-group accumulators for the logits, per-group
// weights w_g = p·s_g for the value sum; q̃ and w as fp16 hi + lo parts, about
// 22 bits) and apply the scales and zero points in the epilogues.  The BF16
// tokens (prefix windows and the chunk itself) are rotated first (k·R_K, v·R_V
// in fp32, kept as fp16 hi + lo parts): q̃·(k R_K) = q·k and Σ p (v R_V) R_Vᵀ =
// Σ p v for orthogonal R, so one online softmax and one accumulator cover every
// token, and R_Vᵀ is applied once per output row at the end.
//
// Kernels, in stream order: prefill_q_kernel (q̃ = q·R_K·log2(e)/√d, its fp16
// parts and group sums), prefill_dense_kernel (rotated BF16 tokens),
// prefill_attn_kernel (flash-attention style over mma.sync m16n8k16 tiles: a
// CTA takes 64 (query, head) rows of one KV head, history tiles then BF16
// tiles), rotate_back_kernel (out ← out·R_Vᵀ).
#include <algorithm>
#include <cmath>

#include "oscar_internal.h"
#include "oscar_device.cuh"

namespace oscar {

namespace {

// (query, head) rows of an attention CTA: 16 per warp, 8 warps for d <= 128 (the
// expanded history tile is shared by 128 rows), 4 for d = 256 (register budget)
__host__ __device__ constexpr int pf_warps(int D) { return D <= 128 ? 8 : 4; }
constexpr int kPfMaxRows = 128;
constexpr int kMaxPrefillBatch = 4096;

struct PrefillParams {
    const void* q;
    int q_dtype;
    const void* k;
    const void* v;
    int kv_dtype;
    int64_t total_q;
    const int32_t* cu_q;
    const int32_t* start_pos;
    const int32_t* req_idx;
    const int32_t* page_table;
    int64_t pt_stride;
    int batch;
    float* out;
    const uint8_t* records;
    const uint16_t* sink;
    const uint16_t* recent;
    const float* rot_k;
    const float* rot_v;
    int64_t num_slots;
    int max_reqs;
    int Hq, Hkv, g, S, W, G, ng, rec_bytes;
    int64_t slot_bytes;   // pool stride of one slot (all KV heads)
    int fp8;              // (s, z) stored as E4M3 pairs (else fp16 pairs)
    float qscale;
    // workspace
    __half* qh;       // [total_q][Hq][d] fp16 hi part of q̃
    __half* ql;       // lo part
    float* qsum;      // [total_q][Hq][ng] Σ over the group of (hi + lo)
    __half* dk;       // [dense slots][Hkv][2 parts][d] rotated BF16 keys (hi, lo)
    __half* dv;       // values
    int* status;
};

// Dense slots of request b start at cu_q[b] + b·(S + W): its prefix windows
// (at most S + W tokens) and then its chunk tokens.
__device__ __forceinline__ int64_t dense_base(const PrefillParams& P, int b) {
    return (int64_t)P.cu_q[b] + (int64_t)b * (P.S + P.W);
}

// Validated prefix length of request b (0 when the request is invalid; the
// status word records why).
__device__ __forceinline__ int prefix_len(const PrefillParams& P, int b, int* rq_out) {
    const int L0 = P.start_pos[b];
    const int rq = P.req_idx ? P.req_idx[b] : b;
    *rq_out = rq;
    if (L0 < 0 || L0 > P.pt_stride) return -1;
    if (L0 > 0 && (rq < 0 || rq >= P.max_reqs)) return -2;
    return L0;
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// fp16 hi part of (a, b) and the lo parts (x - fp16(x)).
__device__ __forceinline__ void split_h2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(a, b);
    const float2 f = __half22float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = pack_h2(a - f.x, b - f.y);
}

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}

// ---------------------------------------------------------------------------
// q̃ = q·R_K·qscale for every (query, head): fp16 hi and lo parts and, per
// group, Σ (hi + lo).  Block (query, head block of 8), 128 threads.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128) prefill_q_kernel(PrefillParams P) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    __shared__ float sq[8][D];
    __shared__ float sqt[8][D];
    const int64_t tq = blockIdx.x;
    const int h0 = blockIdx.y * 8, nh = min(8, P.Hq - h0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < 8 * D; i += 128)
        sq[i / D][i % D] = i / D < nh ? load_elem(P.q, (tq * P.Hq + h0 + i / D) * D + i % D, P.q_dtype) : 0.f;
    __syncthreads();
    for (int col = tid; col < D; col += 128) {
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.f;
        for (int k0 = 0; k0 < D; k0 += 32) {
            float r[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) r[u] = __ldg(P.rot_k + (int64_t)(k0 + u) * D + col);
#pragma unroll
            for (int u = 0; u < 32; ++u)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = fmaf(sq[j][k0 + u], r[u], acc[j]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) sqt[j][col] = acc[j] * P.qscale;
    }
    __syncthreads();
    for (int i = tid; i < nh * D; i += 128) {
        const int j = i / D, c = i % D;
        const float x = sqt[j][c];
        const __half hi = __float2half_rn(x);
        const int64_t o = (tq * P.Hq + h0 + j) * D + c;
        P.qh[o] = hi;
        P.ql[o] = __float2half_rn(x - __half2float(hi));
    }
    for (int i = warp; i < nh * P.ng; i += 4) {
        const int j = i / P.ng, gi = i % P.ng;
        float s = 0.f;
        for (int c = gi * P.G + lane; c < (gi + 1) * P.G; c += 32) {
            const float x = sqt[j][c];
            const __half hi = __float2half_rn(x);
            const __half lo = __float2half_rn(x - __half2float(hi));
            s += __half2float(hi) + __half2float(lo);
        }
        for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) P.qsum[(tq * P.Hq + h0 + j) * P.ng + gi] = s;
    }
}

// ---------------------------------------------------------------------------
// The BF16 tokens, rotated: for dense slot e of request b, its prefix window
// token (sink or recent ring) or chunk token, every KV head, K·R_K and V·R_V
// in fp32 (sequential FMA), kept as fp16 hi and lo parts.  Block of D threads
// per dense slot; thread c forms channel c.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(D) prefill_dense_kernel(PrefillParams P) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    __shared__ float sx[D];
    const int tid = threadIdx.x;
    const int64_t e = blockIdx.x;
    int lo = 0, hi = P.batch - 1;                     // request: largest b with dense_base(b) <= e
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (dense_base(P, mid) <= e) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    int rq;
    const int L0 = prefix_len(P, b, &rq);
    if (L0 < 0) return;                               // flagged by the attention kernel
    const int C = P.cu_q[b + 1] - P.cu_q[b];
    const int sink_end = min(P.S, L0), rec_lo = max(P.S, L0 - P.W);
    const int nwin = sink_end + max(0, L0 - rec_lo);
    const int td = (int)(e - dense_base(P, b));
    if (td >= nwin + C) return;                       // an unused slot
    for (int hk = 0; hk < P.Hkv; ++hk) {
        for (int mat = 0; mat < 2; ++mat) {
            float x;
            if (td < sink_end) {
                x = bf16_bits_to_f32(P.sink[((((int64_t)rq * P.S + td) * P.Hkv + hk) * 2 + mat) * D + tid]);
            } else if (td < nwin) {
                const int p = rec_lo + (td - sink_end);
                x = bf16_bits_to_f32(P.recent[((((int64_t)rq * P.W + p % P.W) * P.Hkv + hk) * 2 + mat) * D + tid]);
            } else {
                const int64_t t = (int64_t)P.cu_q[b] + (td - nwin);
                x = bf16_bits_to_f32(f32_to_bf16_bits(load_elem(mat ? P.v : P.k, (t * P.Hkv + hk) * D + tid,
                                                                P.kv_dtype)));
            }
            __syncthreads();
            sx[tid] = x;
            __syncthreads();
            const float* R = (mat ? P.rot_v : P.rot_k) + tid;
            float y = 0.f;
            for (int k0 = 0; k0 < D; k0 += 32) {
                float r[32];
#pragma unroll
                for (int u = 0; u < 32; ++u) r[u] = __ldg(R + (int64_t)(k0 + u) * D);
#pragma unroll
                for (int u = 0; u < 32; ++u) y = fmaf(sx[k0 + u], r[u], y);
            }
            const __half yh = __float2half_rn(y);
            __half* dst = (mat ? P.dv : P.dk) + ((e * P.Hkv + hk) * 2) * D;
            dst[tid] = yh;
            dst[D + tid] = __float2half_rn(y - __half2float(yh));
        }
    }
}

// ---------------------------------------------------------------------------
// Attention.  CTA (row block, KV head, request): rows r = 64·rb .. of the
// request's C·g (query, head) rows of KV head hk, row r ↔ (query r / g, head
// hk·g + r % g); warp w owns rows 16w .. 16w + 15.  Token tiles of TT:
//  * history tiles: the codes c (exact small integers in fp16) of K and V in
//    shared memory with their per-token (s, z); S_g = q̃·c_g per group
//    (q̃ hi and lo parts), logit = Σ_g s_g·S_g + z_g·Σ_g q̃; P·V per group with
//    w_g = p·s_g (hi and lo parts) against the V codes, plus Σ p·z_g;
//  * BF16 tiles: rotated rows as fp16 hi and lo parts (three products per
//    pair), the chunk's own tokens under the causal mask.
// One online softmax (log2 units: q̃ carries log2(e)/√d) over all tiles.
// ---------------------------------------------------------------------------
template <int D, int TT>
struct PfCfg {
    static constexpr int WARPS = pf_warps(D);
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int ROWS = 16 * WARPS;            // (query, head) rows per CTA
    static constexpr int RS = D + 8;                   // halves per staged row (16-byte pad: conflict-free ldmatrix)
    static constexpr int Q_HALVES = 2 * ROWS * RS;     // q̃ hi, lo
    static constexpr int T_HALVES = 4 * TT * RS;       // history: K codes, V codes; BF16: K hi, K lo, V hi, V lo
    // shared bytes: q̃, tile, (s, z) [4][TT][ng], token validity [TT], slots [3][TT],
    // raw records of two tiles [2][TT][rec_bytes]
    static size_t smem(int ng, int rec_bytes) {
        return (size_t)(Q_HALVES + T_HALVES) * 2 + (size_t)4 * TT * ng * 4 + (size_t)TT * 4 + (size_t)3 * TT * 4 +
               (size_t)2 * TT * rec_bytes;
    }
};

// Two blocks share an SM: at d <= 128 (about 111 KB of shared memory each)
// registers are bounded to 128 per thread, 16 warps per SM instead of 8; at d =
// 256 the key tiles hold 16 tokens (about 104 KB per block), 8 warps instead of 4.
template <int D, int G, int TT>
__global__ void __launch_bounds__(PfCfg<D, TT>::THREADS, 2) prefill_attn_kernel(PrefillParams P) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    using C_ = PfCfg<D, TT>;
    constexpr int RS = C_::RS, KS = D / 16, NTO = D / 8, NTT = TT / 8, KT = TT / 16, NG = D / G;
    constexpr int kPfRows = C_::ROWS, kPfThreads = C_::THREADS;
    constexpr int NTG = G / 8;                         // output n-tiles per group
    extern __shared__ __align__(16) unsigned char smem[];
    __half* sQh = reinterpret_cast<__half*>(smem);
    __half* sQl = sQh + kPfRows * RS;
    __half* sT = sQl + kPfRows * RS;                   // 4 tiles of TT rows
    float* sSZ = reinterpret_cast<float*>(sT + 4 * TT * RS);   // [4][TT][NG]: s_K, z_K, s_V, z_V
    int* sOk = reinterpret_cast<int*>(sSZ + 4 * TT * NG);      // [TT] token valid
    int* sSlot = sOk + TT;                                     // [3][TT] slots of history tiles i, i+1, i+2 (mod 3)
    unsigned char* sRaw = reinterpret_cast<unsigned char*>(sSlot + 3 * TT);   // [2][TT][rec_bytes] records
    const int rb = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = lane >> 2, j = lane & 3;
    const int g = P.g;
    const int c0 = P.cu_q[b], C = P.cu_q[b + 1] - c0;
    const int rows_total = C * g, r0 = rb * kPfRows;
    if (r0 >= rows_total) return;
    int rq;
    int L0 = prefix_len(P, b, &rq);
    if (L0 < 0) {
        if (tid == 0 && hk == 0 && rb == 0) set_status(P.status, L0 == -1 ? OSCAR_DEV_BAD_LEN : OSCAR_DEV_BAD_REQ);
        L0 = 0;                                        // attend over the chunk alone
    }
    const int S = P.S, W = P.W;
    const int hist_hi = max(S, L0 - W);
    const int sink_end = min(S, L0), rec_lo = max(S, L0 - W);
    const int nwin = sink_end + max(0, L0 - rec_lo);
    const int rows_here = min(kPfRows, rows_total - r0);
    const int q_last = (r0 + rows_here - 1) / g;       // last chunk query of the CTA

    // ---- q̃ rows (hi, lo) and this thread's two rows' metadata ----
    for (int i = tid; i < kPfRows * (D / 8); i += kPfThreads) {
        const int rr = i / (D / 8), cc = i % (D / 8);
        const int lr = r0 + rr;
        uint4 vh = make_uint4(0u, 0u, 0u, 0u), vl = vh;
        if (lr < rows_total) {
            const int64_t o = (((int64_t)c0 + lr / g) * P.Hq + hk * g + lr % g) * D + 8 * cc;
            vh = *reinterpret_cast<const uint4*>(P.qh + o);
            vl = *reinterpret_cast<const uint4*>(P.ql + o);
        }
        *reinterpret_cast<uint4*>(sQh + rr * RS + 8 * cc) = vh;
        *reinterpret_cast<uint4*>(sQl + rr * RS + 8 * cc) = vl;
    }
    int qi[2];                                         // chunk query of rows r and r + 8 (-1: padding)
    float qs[2][NG];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        const int lr = r0 + 16 * warp + r + 8 * h2;
        qi[h2] = lr < rows_total ? lr / g : -1;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
            qs[h2][gi] = lr < rows_total ? P.qsum[(((int64_t)c0 + lr / g) * P.Hq + hk * g + lr % g) * P.ng + gi] : 0.f;
    }

    float o[NTO][4];
#pragma unroll
    for (int n = 0; n < NTO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float oz[2][NG];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) oz[h2][gi] = 0.f;
    float m_run[2] = {-1e30f, -1e30f}, l_run[2] = {0.f, 0.f};

    const uint32_t aQh = smem_addr(sQh + (16 * warp + (lane & 7) + 8 * ((lane >> 3) & 1)) * RS + 8 * (lane >> 4));
    const uint32_t aQl = aQh + (uint32_t)(kPfRows * RS * 2);
    // QK B (non-transposed) and P·V B (transposed) lane addresses within a tile
    const uint32_t offQK = (uint32_t)(((lane & 7) + 8 * (lane >> 4)) * RS + 8 * ((lane >> 3) & 1)) * 2;
    const uint32_t offPV = (uint32_t)(((lane & 7) + 8 * ((lane >> 3) & 1)) * RS + 8 * (lane >> 4)) * 2;
    const uint32_t sTa = smem_addr(sT);
    constexpr uint32_t TILE_B = (uint32_t)TT * RS * 2;

    // online softmax over the tile's logits sc (masked entries -inf): returns p in sc
    auto softmax = [&](float (&sc)[NTT][4]) {
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < NTT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) mx[e >> 1] = fmaxf(mx[e >> 1], sc[n][e]);
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 1));
            mx[h2] = fmaxf(mx[h2], __shfl_xor_sync(0xffffffffu, mx[h2], 2));
            const float mn = fmaxf(m_run[h2], mx[h2]);
            const float alpha = fast_exp2(m_run[h2] - mn);
            m_run[h2] = mn;
            l_run[h2] *= alpha;
#pragma unroll
            for (int n = 0; n < NTO; ++n) {
                o[n][2 * h2] *= alpha;
                o[n][2 * h2 + 1] *= alpha;
            }
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) oz[h2][gi] *= alpha;
        }
#pragma unroll
        for (int n = 0; n < NTT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float pv = fast_exp2(sc[n][e] - m_run[e >> 1]);   // masked: 2^-inf = 0
                sc[n][e] = pv;
                l_run[e >> 1] += pv;
            }
    };

    // ---- history tiles: INT2 records of KV head hk ----
    // Pipeline over tiles of TT tokens: the records of tile i + 1 are copied
    // (8-byte cp.async, slot ids from a shared table filled one tile earlier)
    // while tile i is expanded and multiplied; the page-table entries of tile
    // i + 2 are loaded at the start of iteration i.
    const bool fp8 = P.fp8 != 0;
    const int rb_ = P.rec_bytes;
    const int rec_v = D / 4, rec_ks = D / 2, rec_vs = D / 2 + (fp8 ? 2 : 4) * NG;
    const int nht = hist_hi > S ? (hist_hi - S + TT - 1) / TT : 0;
    auto tile_slot = [&](int i) -> int {               // slot of token tid of history tile i, or -1
        const int t = S + i * TT + tid;
        if (tid >= TT || i >= nht || t >= hist_hi) return -1;
        const int sl = P.page_table[(int64_t)b * P.pt_stride + t];
        if (sl >= 0 && sl < P.num_slots) return sl;
        set_status(P.status, OSCAR_DEV_BAD_SLOT);
        return -1;
    };
    auto issue = [&](int i) {                          // records of tile i into raw buffer i & 1
        const int nch = rb_ / 8;
        const int* sl_ = sSlot + (i % 3) * TT;
        unsigned char* dst = sRaw + (size_t)(i & 1) * TT * rb_;
        for (int c = tid; c < TT * nch; c += kPfThreads) {
            const int tt = c / nch, ch = c - tt * nch;
            const int sl = sl_[tt];
            if (sl >= 0)
                cp_async8(dst + tt * rb_ + 8 * ch, P.records + (int64_t)sl * P.slot_bytes + (int64_t)hk * rb_ + 8 * ch);
        }
        cp_async_commit();
    };
    if (nht > 0) {
        const int s0 = tile_slot(0), s1 = tile_slot(1);
        if (tid < TT) {
            sSlot[tid] = s0;
            sSlot[TT + tid] = s1;
        }
        __syncthreads();
        issue(0);
    }
    for (int i = 0; i < nht; ++i) {
        const int t0 = S + i * TT;
        const int nt = min(TT, hist_hi - t0);
        const int s2 = tile_slot(i + 2);               // in flight through the wait and the expansion
        cp_async_wait<0>();                            // this thread's copies of tile i
        __syncthreads();                               // tile i's records visible; the previous tile's readers are done
        if (i + 1 < nht) issue(i + 1);
        const unsigned char* raw = sRaw + (size_t)(i & 1) * TT * rb_;
        const int* slt = sSlot + (i % 3) * TT;
        // item (token, 8-channel chunk, K|V): 8 codes as fp16 values, one 16-byte store
        for (int it = tid; it < TT * (D / 8) * 2; it += kPfThreads) {
            const int mat = it / (TT * (D / 8));
            const int tt = (it / (D / 8)) % TT, cc = it % (D / 8);
            const bool okt = tt < nt && slt[tt] >= 0;
            const unsigned char* rec = raw + tt * rb_;
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (okt) {
                const uint32_t cw = *reinterpret_cast<const uint16_t*>(rec + (mat ? rec_v : 0) + 2 * cc);
                uint32_t w4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    w4[u] = pack_h2((float)((cw >> (4 * u)) & 3u), (float)((cw >> (4 * u + 2)) & 3u));
                val = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
            *reinterpret_cast<uint4*>(sT + (mat * TT + tt) * RS + 8 * cc) = val;
            if ((8 * cc) % G == 0) {                   // the group's (s, z): zero for invalid tokens
                const int gi = (8 * cc) / G;
                float2 sz = make_float2(0.f, 0.f);
                if (okt) sz = load_sz(rec + (mat ? rec_vs : rec_ks), gi, fp8);
                sSZ[(2 * mat) * TT * NG + tt * NG + gi] = sz.x;
                sSZ[(2 * mat + 1) * TT * NG + tt * NG + gi] = sz.y;
            }
            if (mat == 0 && cc == 0) sOk[tt] = okt;
        }
        if (tid < TT) sSlot[((i + 2) % 3) * TT + tid] = s2;   // read from the next iteration on
        __syncthreads();
        // S_g = q̃·c over group g's channels
        float sg[NG][NTT][4];
#pragma unroll
        for (int gi = 0; gi < NG; ++gi)
#pragma unroll
            for (int n = 0; n < NTT; ++n) sg[gi][n][0] = sg[gi][n][1] = sg[gi][n][2] = sg[gi][n][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int gi = (16 * ks) / G;
            uint32_t ah[4], al[4];
            ldsm4(ah, aQh + ks * 32);
            ldsm4(al, aQl + ks * 32);
#pragma unroll
            for (int n2 = 0; n2 < NTT / 2; ++n2) {
                uint32_t bk[4];
                ldsm4(bk, sTa + offQK + (uint32_t)(16 * n2 * RS * 2) + ks * 32);
                mma_f16(sg[gi][2 * n2], ah[0], ah[1], ah[2], ah[3], bk[0], bk[1]);
                mma_f16(sg[gi][2 * n2 + 1], ah[0], ah[1], ah[2], ah[3], bk[2], bk[3]);
                mma_f16(sg[gi][2 * n2], al[0], al[1], al[2], al[3], bk[0], bk[1]);
                mma_f16(sg[gi][2 * n2 + 1], al[0], al[1], al[2], al[3], bk[2], bk[3]);
            }
        }
        float sc[NTT][4];
#pragma unroll
        for (int n = 0; n < NTT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = 8 * n + 2 * j + (e & 1), h2 = e >> 1;
                float x = 0.f;
#pragma unroll
                for (int gi = 0; gi < NG; ++gi)
                    x = fmaf(sSZ[t * NG + gi], sg[gi][n][e], fmaf(sSZ[TT * NG + t * NG + gi], qs[h2][gi], x));
                sc[n][e] = (sOk[t] && qi[h2] >= 0) ? x : -INFINITY;
            }
        softmax(sc);
        // P·V per group: w_g = p·s_g against the V codes, and Σ p·z_g
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
                float w[2][4];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int t = 16 * kt + 8 * hf + 2 * j + (e & 1);
                        const float pv = sc[2 * kt + hf][e];
                        w[hf][e] = pv * sSZ[2 * TT * NG + t * NG + gi];
                        oz[e >> 1][gi] = fmaf(pv, sSZ[3 * TT * NG + t * NG + gi], oz[e >> 1][gi]);
                    }
                uint32_t ph[4], pl[4];
                split_h2(w[0][0], w[0][1], ph[0], pl[0]);   // row r, tokens 2j, 2j+1
                split_h2(w[0][2], w[0][3], ph[1], pl[1]);   // row r + 8
                split_h2(w[1][0], w[1][1], ph[2], pl[2]);   // row r, tokens 8 + 2j, 9 + 2j
                split_h2(w[1][2], w[1][3], ph[3], pl[3]);   // row r + 8
                const uint32_t vb = sTa + TILE_B + offPV + (uint32_t)(16 * kt * RS * 2);
#pragma unroll
                for (int n2 = 0; n2 < NTG / 2; ++n2) {
                    const int nb = gi * NTG + 2 * n2;
                    uint32_t bv[4];
                    ldsm4t(bv, vb + nb * 16);
                    mma_f16(o[nb], ph[0], ph[1], ph[2], ph[3], bv[0], bv[1]);
                    mma_f16(o[nb + 1], ph[0], ph[1], ph[2], ph[3], bv[2], bv[3]);
                    mma_f16(o[nb], pl[0], pl[1], pl[2], pl[3], bv[0], bv[1]);
                    mma_f16(o[nb + 1], pl[0], pl[1], pl[2], pl[3], bv[2], bv[3]);
                }
            }
        }
    }

    // ---- BF16 tiles: prefix windows, then the chunk up to the CTA's last query ----
    const int ndense = nwin + q_last + 1;
    const int64_t dbase = dense_base(P, b);
    for (int td0 = 0; td0 < ndense; td0 += TT) {
        const int nt = min(TT, ndense - td0);
        __syncthreads();
        for (int i = tid; i < TT * (D / 8) * 4; i += kPfThreads) {
            const int part = i / (TT * (D / 8));     // 0: K hi, 1: K lo, 2: V hi, 3: V lo
            const int tt = (i / (D / 8)) % TT, cc = i % (D / 8);
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (tt < nt) {
                const __half* src = (part < 2 ? P.dk : P.dv) + (((dbase + td0 + tt) * P.Hkv + hk) * 2 + (part & 1)) * D;
                val = *reinterpret_cast<const uint4*>(src + 8 * cc);
            }
            *reinterpret_cast<uint4*>(sT + (part * TT + tt) * RS + 8 * cc) = val;
            if (part == 0 && cc == 0) sOk[tt] = tt < nt;
        }
        __syncthreads();
        float sc[NTT][4];
#pragma unroll
        for (int n = 0; n < NTT; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t ah[4], al[4];
            ldsm4(ah, aQh + ks * 32);
            ldsm4(al, aQl + ks * 32);
#pragma unroll
            for (int n2 = 0; n2 < NTT / 2; ++n2) {
                uint32_t bk[4], bl[4];
                ldsm4(bk, sTa + offQK + (uint32_t)(16 * n2 * RS * 2) + ks * 32);
                ldsm4(bl, sTa + TILE_B + offQK + (uint32_t)(16 * n2 * RS * 2) + ks * 32);
                mma_f16(sc[2 * n2], ah[0], ah[1], ah[2], ah[3], bk[0], bk[1]);
                mma_f16(sc[2 * n2 + 1], ah[0], ah[1], ah[2], ah[3], bk[2], bk[3]);
                mma_f16(sc[2 * n2], al[0], al[1], al[2], al[3], bk[0], bk[1]);
                mma_f16(sc[2 * n2 + 1], al[0], al[1], al[2], al[3], bk[2], bk[3]);
                mma_f16(sc[2 * n2], ah[0], ah[1], ah[2], ah[3], bl[0], bl[1]);
                mma_f16(sc[2 * n2 + 1], ah[0], ah[1], ah[2], ah[3], bl[2], bl[3]);
            }
        }
#pragma unroll
        for (int n = 0; n < NTT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = 8 * n + 2 * j + (e & 1), h2 = e >> 1;
                const int td = td0 + t;
                const bool ok = sOk[t] && qi[h2] >= 0 && (td < nwin || td - nwin <= qi[h2]);
                sc[n][e] = ok ? sc[n][e] : -INFINITY;
            }
        softmax(sc);
#pragma unroll
        for (int kt = 0; kt < KT; ++kt) {
            uint32_t ph[4], pl[4];
            split_h2(sc[2 * kt][0], sc[2 * kt][1], ph[0], pl[0]);
            split_h2(sc[2 * kt][2], sc[2 * kt][3], ph[1], pl[1]);
            split_h2(sc[2 * kt + 1][0], sc[2 * kt + 1][1], ph[2], pl[2]);
            split_h2(sc[2 * kt + 1][2], sc[2 * kt + 1][3], ph[3], pl[3]);
            const uint32_t vb = sTa + 2 * TILE_B + offPV + (uint32_t)(16 * kt * RS * 2);
#pragma unroll
            for (int n2 = 0; n2 < NTO / 2; ++n2) {
                uint32_t bv[4], bw[4];
                ldsm4t(bv, vb + n2 * 32);
                ldsm4t(bw, vb + TILE_B + n2 * 32);
                mma_f16(o[2 * n2], ph[0], ph[1], ph[2], ph[3], bv[0], bv[1]);
                mma_f16(o[2 * n2 + 1], ph[0], ph[1], ph[2], ph[3], bv[2], bv[3]);
                mma_f16(o[2 * n2], pl[0], pl[1], pl[2], pl[3], bv[0], bv[1]);
                mma_f16(o[2 * n2 + 1], pl[0], pl[1], pl[2], pl[3], bv[2], bv[3]);
                mma_f16(o[2 * n2], ph[0], ph[1], ph[2], ph[3], bw[0], bw[1]);
                mma_f16(o[2 * n2 + 1], ph[0], ph[1], ph[2], ph[3], bw[2], bw[3]);
            }
        }
    }

    // ---- normalise and write the rotated-domain rows (R_Vᵀ follows) ----
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        l_run[h2] += __shfl_xor_sync(0xffffffffu, l_run[h2], 1);
        l_run[h2] += __shfl_xor_sync(0xffffffffu, l_run[h2], 2);
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            oz[h2][gi] += __shfl_xor_sync(0xffffffffu, oz[h2][gi], 1);
            oz[h2][gi] += __shfl_xor_sync(0xffffffffu, oz[h2][gi], 2);
        }
    }
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
        const int lr = r0 + 16 * warp + r + 8 * h2;
        if (lr >= rows_total) continue;
        const float inv = l_run[h2] > 0.f ? 1.f / l_run[h2] : 0.f;
        float* dst = P.out + (((int64_t)c0 + lr / g) * P.Hq + hk * g + lr % g) * D;
#pragma unroll
        for (int n = 0; n < NTO; ++n) {
            const int ch = 8 * n + 2 * j;
            const float z = oz[h2][ch / G];
            *reinterpret_cast<float2*>(dst + ch) =
                make_float2((o[n][2 * h2] + z) * inv, (o[n][2 * h2 + 1] + z) * inv);
        }
    }
}

// ---------------------------------------------------------------------------
// out ← out·R_Vᵀ per output row (in place): one block per row, thread c forms
// channel c from the row (shared memory) and row c of R_V.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(D) rotate_back_kernel(float* out, const float* rot_v) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    __shared__ float sr[D];
    float* row = out + (int64_t)blockIdx.x * D;
    const int c = threadIdx.x;
    sr[c] = row[c];
    __syncthreads();
    const float* rv = rot_v + (int64_t)c * D;
    float acc = 0.f;
    for (int k0 = 0; k0 < D; k0 += 4) {
        const float4 r4 = *reinterpret_cast<const float4*>(rv + k0);
        acc = fmaf(sr[k0], r4.x, acc);
        acc = fmaf(sr[k0 + 1], r4.y, acc);
        acc = fmaf(sr[k0 + 2], r4.z, acc);
        acc = fmaf(sr[k0 + 3], r4.w, acc);
    }
    row[c] = acc;
}

struct PfPlan {
    size_t off_qh, off_ql, off_qsum, off_dk, off_dv, total;
};

PfPlan pf_plan(const oscar_config* cfg, int batch, int64_t total_q) {
    const int d = cfg->head_dim, Hq = cfg->num_q_heads, Hkv = cfg->num_kv_heads;
    const int ng = d / cfg->group_size;
    const int64_t dense = total_q + (int64_t)batch * (cfg->sink + cfg->recent);
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    PfPlan p;
    size_t off = 0;
    p.off_qh = off;   off = al(off + (size_t)total_q * Hq * d * 2);
    p.off_ql = off;   off = al(off + (size_t)total_q * Hq * d * 2);
    p.off_qsum = off; off = al(off + (size_t)total_q * Hq * ng * 4);
    p.off_dk = off;   off = al(off + (size_t)dense * Hkv * 2 * d * 2);
    p.off_dv = off;   off = al(off + (size_t)dense * Hkv * 2 * d * 2);
    p.total = off;
    return p;
}

template <int D>
int launch_prefill(PrefillParams& P, int max_c, cudaStream_t st) {
    launch_dependent(prefill_q_kernel<D>, dim3((unsigned)P.total_q, (P.Hq + 7) / 8), dim3(128), 0, st, P);
    if (int rc = check_cuda("prefill_q_kernel launch")) return rc;
    const int64_t dense = P.total_q + (int64_t)P.batch * (P.S + P.W);
    launch_dependent(prefill_dense_kernel<D>, dim3((unsigned)dense), dim3(D), 0, st, P);
    if (int rc = check_cuda("prefill_dense_kernel launch")) return rc;
    constexpr int TT = D >= 256 ? 16 : 32;          // key tile: two blocks per SM at d = 256 too
    using C_ = PfCfg<D, TT>;
    const int rblocks = (int)(((int64_t)max_c * P.g + C_::ROWS - 1) / C_::ROWS);
    const int prof = prof_begin(6, st);
    auto go = [&](auto kern, size_t smem) -> int {
        if (const int rc = ensure_dynamic_smem((const void*)kern, smem, "cudaFuncSetAttribute(prefill_attn_kernel)"))
            return rc;
        launch_dependent(kern, dim3((unsigned)rblocks, P.Hkv, P.batch), dim3(C_::THREADS), smem, st, P);
        return check_cuda("prefill_attn_kernel launch");
    };
    auto smem_for = [&](int ng) { return C_::smem(ng, P.rec_bytes); };
    int rc;
    if (P.G == 32 && D >= 32) rc = go(prefill_attn_kernel<D, 32, TT>, smem_for(D / 32));
    else if (P.G == 64 && D >= 64) rc = go(prefill_attn_kernel<D, (D >= 64 ? 64 : 32), TT>, smem_for(D / 64));
    else if (P.G == 128 && D >= 128) rc = go(prefill_attn_kernel<D, (D >= 128 ? 128 : 32), TT>, smem_for(D / 128));
    else rc = go(prefill_attn_kernel<D, (D >= 256 ? 256 : 32), TT>, smem_for(1));
    prof_end(prof, st);
    if (rc) return rc;
    launch_dependent(rotate_back_kernel<D>, dim3((unsigned)(P.total_q * P.Hq)), dim3(D), 0, st, P.out, P.rot_v);
    return check_cuda("rotate_back_kernel launch");
}

}  // namespace

}  // namespace oscar

using namespace oscar;

extern "C" int oscar_prefill_workspace_bytes(const oscar_config* cfg, int32_t batch, int64_t total_q, size_t* bytes) {
    clear_error();
    int rc = validate_config(cfg);
    if (rc) return rc;
    if (!bytes) return fail(OSCAR_ERR_NULL, "bytes is NULL");
    if (batch < 0 || batch > kMaxPrefillBatch || total_q < 0)
        return fail(OSCAR_ERR_ARG, "batch in [0, %d] and total_q >= 0 required", kMaxPrefillBatch);
    *bytes = pf_plan(cfg, batch, total_q).total;
    return OSCAR_OK;
}

extern "C" int oscar_prefill_attention(const oscar_config* cfg, const oscar_layer_cache* cache, const void* q,
                                       const void* k, const void* v, int64_t total_q, const int32_t* cu_q,
                                       const int32_t* start_pos, const int32_t* req_idx, const int32_t* page_table,
                                       int64_t pt_stride, int32_t batch, int32_t max_chunk, float* out,
                                       void* workspace, size_t workspace_bytes, void* stream) {
    clear_error();
    int rc = validate_config(cfg);
    if (rc) return rc;
    rc = validate_cache(cfg, cache);
    if (rc) return rc;
    if (batch < 0 || batch > kMaxPrefillBatch) return fail(OSCAR_ERR_ARG, "batch must be in [0, %d]", kMaxPrefillBatch);
    if (total_q < 0 || max_chunk < 0) return fail(OSCAR_ERR_ARG, "total_q and max_chunk must be >= 0");
    if (batch == 0 || total_q == 0) return OSCAR_OK;
    if (!q || !k || !v || !cu_q || !start_pos || !page_table || !out)
        return fail(OSCAR_ERR_NULL, "q, k, v, cu_q, start_pos, page_table and out are required");
    if (pt_stride < 1) return fail(OSCAR_ERR_ARG, "pt_stride must be >= 1");
    if (max_chunk < 1 || max_chunk > total_q) return fail(OSCAR_ERR_ARG, "max_chunk must be in [1, total_q]");
    if ((int64_t)max_chunk * (cfg->num_q_heads / cfg->num_kv_heads) > (int64_t)kPfMaxRows * 65535 / 2)
        return fail(OSCAR_ERR_ARG, "max_chunk too large");
    const int64_t dense = total_q + (int64_t)batch * (cfg->sink + cfg->recent);
    if (dense > 0x7FFFFFFF || total_q * cfg->num_q_heads > 0x7FFFFFFF || total_q > 65535LL * 65535LL)
        return fail(OSCAR_ERR_ARG, "total_q too large");
    if ((int64_t)total_q > 0x7FFFFFFF) return fail(OSCAR_ERR_ARG, "total_q too large");
    const PfPlan plan = pf_plan(cfg, batch, total_q);
    if (!workspace || workspace_bytes < plan.total || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return fail(OSCAR_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold %zu bytes", plan.total);
    PrefillParams P;
    P.q = q;
    P.q_dtype = cfg->q_dtype;
    P.k = k;
    P.v = v;
    P.kv_dtype = cfg->kv_dtype;
    P.total_q = total_q;
    P.cu_q = cu_q;
    P.start_pos = start_pos;
    P.req_idx = req_idx;
    P.page_table = page_table;
    P.pt_stride = pt_stride;
    P.batch = batch;
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
    P.qscale = (float)(1.4426950408889634 / std::sqrt((double)cfg->head_dim));
    char* ws = static_cast<char*>(workspace);
    P.qh = reinterpret_cast<__half*>(ws + plan.off_qh);
    P.ql = reinterpret_cast<__half*>(ws + plan.off_ql);
    P.qsum = reinterpret_cast<float*>(ws + plan.off_qsum);
    P.dk = reinterpret_cast<__half*>(ws + plan.off_dk);
    P.dv = reinterpret_cast<__half*>(ws + plan.off_dv);
    P.status = status_word();
    if (!P.status) return OSCAR_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    switch (cfg->head_dim) {
        case 64: return launch_prefill<64>(P, max_chunk, st);
        case 128: return launch_prefill<128>(P, max_chunk, st);
        default: return launch_prefill<256>(P, max_chunk, st);
    }
}
