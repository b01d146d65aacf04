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
//  * the CTA walks its chunk run in stages of TTOK tokens (64, or 32 when a
//    warp carries two n8 column tiles).  With PAR = 2 two sets of warps (one
//    warp per KV head each) take the even and the odd stages: two independent
//    pipelines over a shared ring of 4 or 8 shared-memory stages, so each SM
//    scheduler has 4 warps to interleave.  The warps of a set copy the
//    records of their stages with 16-byte cp.async: all KV heads of a token
//    are one contiguous slot-major record (640 B at d 128 / 8 heads), and one
//    warp instruction moves 16-byte chunks of four records; every thread's
//    copies complete on the stage's full mbarrier (cp.async.mbarrier.arrive);
//    each warp fetches the slot ids of its tokens from the page table one
//    stage ahead;
//  * every warp consumes its own KV head of its stages (its channel half for
//    d = 256, where two warps share a head) and releases each stage on its
//    empty mbarrier;
//  * each 16-token sub-tile runs mma.sync.m16n8k16 f16 → f32.  One AND masks a
//    code position of both 16-bit halves of a word, after at most one shift of
//    the word, and the code enters the MMA as the exact fp16 subnormal
//    c·2^(bit-24) (see sub_bit / slot_pos), so neither sum carries an offset to
//    cancel.  The query operand of a channel is q̃·2^(kQkExp - bit); the per-group
//    scale s and zero z are applied in fp32:
//        logit    = 2^(24-kQkExp)·Σ_g s_g·Σ_ch (q̃ 2^(kQkExp-bit))(c 2^(bit-24)) + Σ_g z_g·Σ q̃
//        o_rot[ch] = 2^(24-bit_ch)·Σ_t w_t·c_t·2^(bit_ch-24) + Σ_t p_t z_t,   w = p·s
//    (group size 32 keeps the older 1 + α·c encoding of the K codes, α = 1/16,
//    1/4, with one funnel shift per word and Σ q̃/α subtracted);
//    the query operand and p·s are split into fp16 hi + lo parts that occupy the n8 columns
//    (head, part), so the products carry ~22 bits;
//  * online softmax in log2 units; the running max moves only when a logit
//    exceeds it (one warp vote per stage otherwise); partials (m, l, o) per
//    (CTA, request, stage parity).
#include <algorithm>
#include <cmath>

#include "oscar_internal.h"
#include "oscar_device.cuh"
#include "oscar_decode_common.cuh"

namespace oscar {

namespace mma_detail {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// (x & mask) | one as a single LOP3 (look-up table 0xEA = (a & b) | c).
__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t mask, uint32_t one) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "r"(mask), "r"(one));
    return d;
}

// From x (the word rotated so that code position m sits at bits 8-9 and
// m-1 at bits 6-7 of each half): half2 of 1 + c/4 for position m, and of
// 1 + c/16 for position m-1.  Both values are exact in fp16.
__device__ __forceinline__ uint32_t code_q4(uint32_t x) { return and_or(x, 0x03000300u, 0x3C003C00u); }
__device__ __forceinline__ uint32_t code_q16(uint32_t x) { return and_or(x, 0x00C000C0u, 0x3C003C00u); }
__device__ __forceinline__ uint32_t rotr(uint32_t w, uint32_t n) { return __funnelshift_r(w, w, n); }

// V side: the code enters the MMA as the exact fp16 subnormal c·2^(bit - 24)
// (exponent field 0), so P·V accumulates Σ w·c itself with no offset to cancel
// over thousands of tokens.  Position p of a 16-code word sits at bit 2p of each
// half for p <= 4 and at bit 2p - 6 of the word >> 6 for p = 5, 6, 7.
__host__ __device__ constexpr float sub_inv(int bit) {   // 2^(24 - bit)
    return (float)(1u << (24 - bit));
}
template <int POS>
__device__ __forceinline__ uint32_t code_sub(uint32_t yd, uint32_t yr) {
    constexpr int bit = sub_bit(POS);
    constexpr uint32_t mask = (3u << bit) | (3u << (bit + 16));
    return (POS <= 4 ? yd : yr) & mask;
}


__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// c = A·B (no accumulator input: the zero C operand needs no register moves).
__device__ __forceinline__ void mma16816_first(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
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

// Named barrier that also returns the OR of v over the participating threads.
__device__ __forceinline__ int named_bar_or(int id, int nthreads, int v) {
    int r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, %2, %3, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"(v), "r"(id), "r"(nthreads) : "memory");
    return r;
}

// (s, z) of groups g0 .. g0 + N - 1 from the pair array at p (fp16 pairs of
// 4 bytes or E4M3 pairs of 2 bytes): E4M3 pairs two groups per load when N is
// even (g0 even, p 4-byte aligned); fp16 pairs one group per load (measured:
// paired 8-byte loads made the fp16 kernel 0.6% slower).
template <int N, bool FP8>
__device__ __forceinline__ void load_sz_groups(const unsigned char* p, int g0, float2 (&out)[N]) {
    if constexpr (FP8 && N % 2 == 0) {
#pragma unroll
        for (int q = 0; q < N; q += 2) {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(p + 2 * (g0 + q));
            uint32_t h0, h1;
            asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
                "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
                : "=r"(h0), "=r"(h1) : "r"(w));
            out[q] = h2f(h0);
            out[q + 1] = h2f(h1);
        }
    } else {
#pragma unroll
        for (int q = 0; q < N; ++q) out[q] = load_sz(p, g0 + q, FP8);
    }
}

}  // namespace mma_detail

// Row stride of one token's record in shared memory: rounded up to an odd
// multiple of 16 bytes, so that 8 consecutive rows start in 8 different
// 4-bank groups.
__host__ __device__ constexpr int row_bytes(int bytes) {
    return ((bytes + 15) / 16) % 2 == 1 ? (bytes + 15) / 16 * 16 : (bytes + 15) / 16 * 16 + 16;
}

// Stage iterator over a CTA's chunk run [f, f1): stages of TT tokens that never
// cross a request boundary (the last stage of a segment may be partial).  Chunk
// indices fit in 32 bits (the chunk prefix is int32); f1 is held by the caller.
template <int TT>
struct StageIter {
    int f, fe;          // current chunk; end of the current segment's chunks
    int b, t0, t_end;   // request, first token of the stage, end of the segment's tokens

    __device__ bool valid(int f1) const { return f < f1; }
    __device__ void seg(const DecodeParams& P, int f1) {
        if (f >= f1) return;
        int lo = 0, hi = P.batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (P.cprefix[mid] <= f) lo = mid; else hi = mid - 1;
        }
        b = lo;
        fe = min(f1, P.cprefix[b + 1]);
        const int h_end = max(P.S, P.len[b] - P.W);
        t0 = P.S + (f - P.cprefix[b]) * P.chunk;
        t_end = min(h_end, P.S + (fe - P.cprefix[b]) * P.chunk);
    }
    __device__ void init(const DecodeParams& P, int f0, int f1) {
        f = f0;
        seg(P, f1);
    }
    __device__ bool seg_last() const { return t0 + TT >= t_end; }
    __device__ void next(const DecodeParams& P, int f1) {
        t0 += TT;
        if (t0 >= t_end) {
            f = fe;
            seg(P, f1);
        }
    }
};

// D: head_dim; G: group size; NT: n8 tiles of (head, hi/lo) columns; WPH:
// warps per head along channels (2 for d = 256); TTOK: tokens per stage; FP8:
// (s, z) stored as E4M3 pairs (2 bytes) instead of fp16 pairs (4 bytes).
template <int D, int G, int NT, int WPH, int TTOK, bool FP8>
struct MmaCfg {
    static constexpr int kSliceCh = D / WPH;        // channels per warp
    static constexpr int kKS = kSliceCh / 16;       // k-steps (words of 16 codes) per warp
    static constexpr int kGW = kSliceCh / G;        // groups per warp slice
    static constexpr int kMT = kSliceCh / 16;       // P·V m-tiles per warp
    static constexpr int kMTG = G / 16;             // m-tiles per group
    static constexpr int kMQ = TTOK / 16;           // 16-token sub-tiles per stage
    static constexpr int PB = FP8 ? 2 : 4;                              // bytes per (s, z) pair
    static constexpr int RAL = FP8 ? 8 : 16;                            // record alignment
    static constexpr int REC = (D / 2 + 2 * PB * (D / G) + RAL - 1) / RAL * RAL;   // record bytes per (slot, head)
    static constexpr int NG = D / G;
    static constexpr int NR = 2 * kMQ;              // token rows per thread per stage
    static constexpr int XCH = WPH == 2 ? 2 * 2 * 32 * NT * NR : 0;   // logit exchange floats per head
    // P·V operand table of a warp: w = p·s per (column head, token, group) as fp16,
    // one table of hi parts and one of lo parts.  A row (head) holds TT tokens of
    // kGW halves each; the row stride (words, ≡ 8 mod 32) and the lo-table offset
    // (≡ 16 mod 32) make both the owner stores and the fragment loads conflict-free.
    static constexpr int kWT = TTOK * kGW / 2;                       // words per table row
    static constexpr int kWS = kWT + ((8 - kWT % 32) + 32) % 32;      // row stride in words
    static constexpr int kWLO = NT * 4 * kWS + 16;                    // lo table offset in words
    static constexpr int TBL = (kWLO + NT * 4 * kWS) * 4;             // bytes per warp
    static_assert(G <= kSliceCh, "a warp's channel slice must hold whole groups");
    static_assert(G >= 32, "group size below 32 has no fast path");
    static_assert(TTOK == 32 || TTOK == 64, "stages of 32 or 64 tokens");
    static_assert(G >= 64 || REC % 16 == 0, "the group-32 K path reads 16-byte words of a record");
};

// Bytes of one pool slot (the records of all KV heads, padded to 16).
__host__ __device__ constexpr int slot_bytes_of(int hkv, int rec) { return (hkv * rec + 15) / 16 * 16; }

// Shared-memory layout (byte offsets): [0, 64) full[8] and [64, 128) empty[8]
// mbarriers; [128, 256) stage validity masks, two 64-bit words per ring slot;
// [256, 260) the abort flag; from 384 per warp its P·V operand table, per (head, parity) the logit exchange
// area (d = 256), and the stage ring at stages_off.
constexpr int kSmemMask = 128, kSmemAbort = 256, kSmemTab = 384;

// HKV > 0 fixes the KV head count (and so the stage row stride) at compile time.
// HP splits a KV head's query group over HP warps (query heads 4·NT·hp ..),
// each carrying NT n8 column tiles.
template <int D, int G, int NT, int WPH, int TTOK, int PAR, int HKV, int HP, bool FP8>
__global__ void __launch_bounds__(256 * PAR * HP, 1)
history_mma_kernel(DecodeParams P, int x_off, int stages_off, int trow, int ns_log2) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    using namespace mma_detail;
    using C = MmaCfg<D, G, NT, WPH, TTOK, FP8>;
    constexpr int KS = C::kKS, GW = C::kGW, MT = C::kMT, MTG = C::kMTG, MQ = C::kMQ;
    constexpr int REC = C::REC, NG = C::NG, TT = TTOK, NR = C::NR, PB = C::PB;
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int Hkv = HKV > 0 ? HKV : P.Hkv;
    const int nwarps = blockDim.x >> 5;
    const int pi = warp % PAR;                  // parity of the stages this warp consumes
    const int hw = warp / PAR;
    const int wsl = hw % WPH;                   // channel slice
    const int hp = (hw / WPH) % HP;             // query-head part: head tiles hp·NT .. hp·NT + NT - 1
    const int h = hw / (WPH * HP);              // KV head
    const int hpx = h * HP + hp;                // (KV head, part)
    const int r = lane >> 2, j = lane & 3;
    const int g = P.g;
    const uint32_t NS = 1u << ns_log2;
    const int row = HKV > 0 ? row_bytes(slot_bytes_of(HKV, REC)) : trow;   // stage row stride of one token (all heads)
    const int tok_bytes = slot_bytes_of(Hkv, REC);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + 8;
    uint64_t* vmw = reinterpret_cast<uint64_t*>(smem + kSmemMask);      // [8 slots][2] validity masks
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemAbort);
    uint32_t* wtab = reinterpret_cast<uint32_t*>(smem + kSmemTab + warp * C::TBL);
    float* xb = reinterpret_cast<float*>(smem + x_off) + (hpx * PAR + pi) * C::XCH;
    unsigned char* stages = smem + stages_off;
    const uint32_t stage_bytes = (uint32_t)TT * (uint32_t)row;
    const int bar_id = 1 + hpx * PAR + pi;

    const int64_t N = P.cprefix[P.batch];
    const int f0 = (int)((int64_t)blockIdx.x * N / gridDim.x);
    const int f1 = (int)((int64_t)(blockIdx.x + 1) * N / gridDim.x);
    if (f0 >= f1) return;

    // ---- stage pipeline shared by the whole CTA ----
    // Every warp of a set copies its share (tokens [tbeg, tend)) of the token
    // records of the stages it issues.
    long long budget = 4000000000LL;            // cycles per pipeline wait (~2 s); 0 after a timeout
    // The warps of one parity copy and consume the stages of that parity: two
    // independent pipelines over even and odd stages when PAR = 2.
    const int npw = nwarps / PAR;               // warps per parity
    const int tpw = (TT + npw - 1) / npw;       // tokens whose records this warp copies per stage
    const int tbeg = min(TT, hw * tpw), tend = min(TT, tbeg + tpw);
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < NS; ++s) {
            mbar_init(&full[s], npw * 32);
            mbar_init(&empty[s], npw);
        }
        fence_mbar_init();
    }
    // zero the stage ring once: rows of invalid tokens then always hold finite values
    for (uint32_t i = threadIdx.x; i < NS * stage_bytes / 16; i += blockDim.x)
        *reinterpret_cast<uint4*>(stages + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
    // Every warp fetches the page-table entries of its tokens of the next stage it
    // issues one iteration ahead (nsl0, nsl1: tokens tbeg + lane, tbeg + 32 + lane;
    // kNoTok when the position lies outside the history).  At issue it posts the
    // validity bits of its tokens into the stage's mask word: two words per ring
    // slot, alternating with the slot's use, the next one cleared by the set's
    // first warp once the slot's previous consumers are done with it.
    constexpr int kNoTok = -2147483647 - 1;
    int nsl0 = kNoTok, nsl1 = kNoTok;
    StageIter<TT> pit;                               // next stage of this parity to issue
    auto load_slots = [&]() {
        nsl0 = kNoTok;
        nsl1 = kNoTok;
        if (!pit.valid(f1)) return;
        const int32_t* pt = P.page_table + (int64_t)pit.b * P.pt_stride + pit.t0;
        const int ta = tbeg + lane, tc = tbeg + 32 + lane;
        if (ta < tend && pit.t0 + ta < pit.t_end) nsl0 = pt[ta];
        if (tc < tend && pit.t0 + tc < pit.t_end) nsl1 = pt[tc];
    };
    for (uint32_t i = threadIdx.x; i < 2 * NS; i += blockDim.x) vmw[i] = 0ull;
    if (threadIdx.x == 0) *abort_flag = 0;
    __syncthreads();

    // copies of stage k (the stage at pit) by this warp
    auto issue = [&](uint32_t k) {
        const uint32_t s = k & (NS - 1);
        const uint32_t use = k >> ns_log2;
        if (k >= NS && !mbar_wait_bounded(&empty[s], (use - 1) & 1, P.status, budget)) *abort_flag = 1;
        const bool ok0 = nsl0 >= 0 && nsl0 < P.num_slots;
        const bool ok1 = nsl1 >= 0 && nsl1 < P.num_slots;
        if ((nsl0 != kNoTok && !ok0) || (nsl1 != kNoTok && !ok1)) set_status(P.status, OSCAR_DEV_BAD_SLOT);
        const uint32_t b0 = __ballot_sync(0xffffffffu, ok0), b1 = __ballot_sync(0xffffffffu, ok1);
        if (lane == 0) {
            if (hw == 0) vmw[2 * s + ((use + 1) & 1)] = 0ull;
            const uint64_t bits = ((uint64_t)b0 | ((uint64_t)b1 << 32)) << tbeg;
            if (bits) atomicOr(reinterpret_cast<unsigned long long*>(&vmw[2 * s + (use & 1)]),
                               (unsigned long long)bits);
        }
        unsigned char* dst = stages + s * stage_bytes;
        // 16-byte cp.async of whole token records, completing on the stage's full
        // barrier through every thread's no-increment arrival
        if constexpr (HKV > 0 && TT == 64 && (TT + HKV * WPH * HP - 1) / (HKV * WPH * HP) <= 8) {
            // at most 8 tokens per warp: lane l copies chunks (l & 7) + 8u of tokens
            // tbeg + (l >> 3) and tbeg + 4 + (l >> 3) (4 records per instruction;
            // a slot of 16·kCh bytes with kCh not a multiple of 8 leaves lanes idle
            // in the last round)
            constexpr int kTB = slot_bytes_of(HKV, REC);
            constexpr int kCh = kTB / 16;
            const int sa = ok0 ? nsl0 : -1;
#pragma unroll
            for (int v = 0; v < 2; ++v) {
                const int tt = (lane >> 3) + 4 * v;
                const int sl = __shfl_sync(0xffffffffu, sa, tt);
                if (tbeg + tt < tend && sl >= 0) {
                    const uint8_t* src = P.records + (int64_t)sl * kTB + (lane & 7) * 16;
                    unsigned char* d = dst + (tbeg + tt) * row + (lane & 7) * 16;
#pragma unroll
                    for (int u = 0; u < (kCh + 7) / 8; ++u)
                        if (kCh % 8 == 0 || (lane & 7) + 8 * u < kCh) cp_async16(d + 128 * u, src + 128 * u);
                }
            }
        } else {
            // any shape: the warp's tokens one at a time, lanes over 16-byte chunks
            const int cpt = tok_bytes / 16;
            for (int q = 0; q < tend - tbeg; ++q) {
                const int sl = __shfl_sync(0xffffffffu, q < 32 ? nsl0 : nsl1, q & 31);
                const bool okq = q < 32 ? ((b0 >> q) & 1u) : ((b1 >> (q - 32)) & 1u);
                if (okq) {
                    const uint8_t* src = P.records + (int64_t)sl * tok_bytes;
                    unsigned char* d = dst + (tbeg + q) * row;
                    for (int pc = lane; pc < cpt; pc += 32) cp_async16(d + 16 * pc, src + 16 * pc);
                }
            }
        }
        cp_async_mbar_arrive(&full[s]);
    };
    // Stage k + NS - PAR is issued at iteration k by the warps of k's parity: it
    // reuses the slot of stage k - PAR, which those warps released one round ago.
    pit.init(P, f0, f1);
    uint32_t pk = pi;
    for (int q = 0; q < pi; ++q)
        if (pit.valid(f1)) pit.next(P, f1);
    auto pit_step = [&]() {
        pk += PAR;
        for (int q = 0; q < PAR; ++q)
            if (pit.valid(f1)) pit.next(P, f1);
        load_slots();
    };
    load_slots();
    for (; pk < NS - PAR && pit.valid(f1); pit_step()) issue(pk);

    // funnel shift for the K extraction: code position 2j+1 to bits 8-9 (2j to 6-7)
    const uint32_t rotK = (uint32_t)(4 * j - 6) & 31u;   // (group size 32)
    int xpar = 0;   // logit-exchange buffer parity; continuous across segments
    uint32_t k = 0; // stages consumed

    // A pipeline wait that runs out of time sets the abort flag (and the device
    // status).  Every warp checks the flag before each of its stages, the two
    // channel-slice warps of a head agreeing on it through their named barrier;
    // it then waits (bounded) for the copies it has issued and returns.
    bool aborted = false;
    StageIter<TT> it;
    it.init(P, f0, f1);
    while (it.valid(f1) && !aborted) {
        const int b = it.b;
        // ---- per-segment query state ----
        uint32_t bq[NT][KS][2];
        {
            const uint2* qf = P.qfrag + (((int64_t)b * Hkv + h) * P.n_frag_tiles) * (D / 16) * 32;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const uint2 v = qf[((int64_t)(hp * NT + nt) * (D / 16) + wsl * KS + kk) * 32 + lane];
                    bq[nt][kk][0] = v.x;
                    bq[nt][kk][1] = v.y;
                }
        }
        float2 qs[NT][GW];          // (Σ q̃, Σ q̃/α) per group, head 4(hp·NT + nt) + j
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hh = 4 * (hp * NT + nt) + j;
#pragma unroll
            for (int gi = 0; gi < GW; ++gi)
                qs[nt][gi] = hh < g ? P.qsum[((int64_t)b * P.Hq + h * g + hh) * P.ng + wsl * GW + gi]
                                    : make_float2(0.f, 0.f);
        }
        float m_run[NT], l_run[NT];
        float acc[NT][MT][4];
        float Zsum[NT][GW];                 // Σ p·z for head 4nt + j over this thread's tokens
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m_run[nt] = -1e30f;     // finite: 2^(m_run - m) never sees -inf - -inf
            l_run[nt] = 0.f;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[nt][mt][e] = 0.f;
#pragma unroll
            for (int gi = 0; gi < GW; ++gi) Zsum[nt][gi] = 0.f;
        }

        bool seg_done = false;
        for (; !seg_done; ++k) {
            seg_done = it.seg_last();
            if ((k & (PAR - 1)) != (uint32_t)pi) {   // a stage of the other parity
                it.next(P, f1);
                continue;
            }
            int ab = *abort_flag;
            if (WPH == 2) ab = named_bar_or(bar_id, 64, ab);
            if (ab) {
                aborted = true;
                break;
            }
            if (pit.valid(f1)) {                 // stage k + NS - PAR (this parity)
                issue(pk);
                pit_step();
            }
            const uint32_t s = k & (NS - 1);
            if (!mbar_wait_bounded(&full[s], (k >> ns_log2) & 1, P.status, budget)) *abort_flag = 1;
            const uint64_t vmask = vmw[2 * s + ((k >> ns_log2) & 1)];
            const unsigned char* tb = stages + s * stage_bytes + h * REC;
            // ---------------- QK: MQ m16 tiles ----------------
            float lg[NT][NR];        // logits (log2 units) of head 4nt + j, token 8i + r
#pragma unroll
            for (int mh = 0; mh < MQ; mh += 2) {   // two m16 tiles at a time (register budget)
                constexpr int MB = MQ < 2 ? MQ : 2;
                float sc[MB][GW][NT][4];     // set by the first k-step of each group
#pragma unroll
                for (int k4 = 0; k4 < KS; k4 += 4) {
#pragma unroll
                    for (int mb = 0; mb < MB; ++mb) {
                        const int mq = mh + mb;
                        const uint32_t* w_r = reinterpret_cast<const uint32_t*>(tb + (16 * mq + r) * row) + wsl * KS + k4;
                        const uint32_t* w_r8 = reinterpret_cast<const uint32_t*>(tb + (16 * mq + r + 8) * row) + wsl * KS + k4;
                        if constexpr (G >= 64) {
                            // lane j owns word k4 + j of its rows: k-step k4 + q takes its
                            // slot q, (k 2j, 2j+1) <- first position of both halves and
                            // (2j+8, 2j+9) <- second position; all 4 words in one group
                            const int gi = (k4 * 16) / G;
                            const uint32_t u0 = w_r[j], u1 = w_r8[j];
                            const uint32_t d0 = u0, r0 = u0 >> 6;
                            const uint32_t d1 = u1, r1 = u1 >> 6;
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint32_t x0, x1, x2, x3;
                                if (q == 0) {
                                    x0 = code_sub<slot_pos(0, 0)>(d0, r0); x1 = code_sub<slot_pos(0, 0)>(d1, r1);
                                    x2 = code_sub<slot_pos(0, 1)>(d0, r0); x3 = code_sub<slot_pos(0, 1)>(d1, r1);
                                } else if (q == 1) {
                                    x0 = code_sub<slot_pos(1, 0)>(d0, r0); x1 = code_sub<slot_pos(1, 0)>(d1, r1);
                                    x2 = code_sub<slot_pos(1, 1)>(d0, r0); x3 = code_sub<slot_pos(1, 1)>(d1, r1);
                                } else if (q == 2) {
                                    x0 = code_sub<slot_pos(2, 0)>(d0, r0); x1 = code_sub<slot_pos(2, 0)>(d1, r1);
                                    x2 = code_sub<slot_pos(2, 1)>(d0, r0); x3 = code_sub<slot_pos(2, 1)>(d1, r1);
                                } else {
                                    x0 = code_sub<slot_pos(3, 0)>(d0, r0); x1 = code_sub<slot_pos(3, 0)>(d1, r1);
                                    x2 = code_sub<slot_pos(3, 1)>(d0, r0); x3 = code_sub<slot_pos(3, 1)>(d1, r1);
                                }
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    if ((k4 + q) * 16 % G == 0)
                                        mma16816_first(sc[mb][gi][nt], x0, x1, x2, x3, bq[nt][k4 + q][0], bq[nt][k4 + q][1]);
                                    else
                                        mma16816(sc[mb][gi][nt], x0, x1, x2, x3, bq[nt][k4 + q][0], bq[nt][k4 + q][1]);
                                }
                            }
                        } else {
                            const uint4 w0 = *reinterpret_cast<const uint4*>(w_r);
                            const uint4 w1 = *reinterpret_cast<const uint4*>(w_r8);
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
                                for (int nt = 0; nt < NT; ++nt) {
                                    if (kk * 16 % G == 0)
                                        mma16816_first(sc[mb][gi][nt], x0, x1, x2, x3, bq[nt][kk][0], bq[nt][kk][1]);
                                    else
                                        mma16816(sc[mb][gi][nt], x0, x1, x2, x3, bq[nt][kk][0], bq[nt][kk][1]);
                                }
                            }
                        }
                    }
                }
#pragma unroll
                for (int ib = 0; ib < 2 * MB; ++ib) {
                    const int i = 2 * mh + ib;       // token row 8i + r = 16·mq + 8·half + r
                    const int t = 8 * i + r;
                    const int mb = ib >> 1, hf = ib & 1;
                    if constexpr (G >= 64) {
                        // lg = 2^(24 - kQkExp) Σ_g s_g·acc_g + Σ_g z_g·Σ q̃  (subnormal K codes)
                        float ts[NT], tz[NT];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) { ts[nt] = 0.f; tz[nt] = 0.f; }
                        float2 szk[GW];
                        load_sz_groups<GW, FP8>(tb + t * row + D / 2, wsl * GW, szk);
#pragma unroll
                        for (int gi = 0; gi < GW; ++gi) {
                            const float2 sz = szk[gi];
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                ts[nt] = fmaf(sz.x, sc[mb][gi][nt][2 * hf] + sc[mb][gi][nt][2 * hf + 1], ts[nt]);
                                tz[nt] = fmaf(sz.y, qs[nt][gi].x, tz[nt]);
                            }
                        }
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) lg[nt][i] = fmaf(ts[nt], (float)(1u << (24 - kQkExp)), tz[nt]);
                    } else {
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) lg[nt][i] = 0.f;
                        float2 szk[GW];
                        load_sz_groups<GW, FP8>(tb + t * row + D / 2, wsl * GW, szk);
#pragma unroll
                        for (int gi = 0; gi < GW; ++gi) {
                            const float2 sz = szk[gi];
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const float2 Q = qs[nt][gi];       // (Σ q̃, Σ q̃/α)
                                lg[nt][i] += sz.x * (sc[mb][gi][nt][2 * hf] + sc[mb][gi][nt][2 * hf + 1] - Q.y) + sz.y * Q.x;
                            }
                        }
                    }
                }
            }
            if (WPH == 2) {   // add the other channel slice's partial logits
                float* my = xb + xpar * (2 * 32 * NT * NR) + wsl * (32 * NT * NR);
                float* ot = xb + xpar * (2 * 32 * NT * NR) + (1 - wsl) * (32 * NT * NR);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < NR; ++i) my[(nt * NR + i) * 32 + lane] = lg[nt][i];
                named_bar(bar_id, 64);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < NR; ++i) lg[nt][i] += ot[(nt * NR + i) * 32 + lane];
                xpar ^= 1;
            }
            // ---------------- online softmax over the stage ----------------
            // The running max moves only when a logit exceeds it (rare after the first
            // stages), so the common path is one vote and no max reduction.
            float x[NT][NR];
            bool over = false;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint64_t need = TT == 64 ? ~0ull : 0xffffffffull;
                const uint64_t vm = (4 * (hp * NT + nt) + j) < g ? vmask : 0ull;
#pragma unroll
                for (int i = 0; i < NR; ++i) x[nt][i] = lg[nt][i];
                if (vm != need) {
#pragma unroll
                    for (int i = 0; i < NR; ++i)
                        if (!((vm >> (8 * i + r)) & 1u)) x[nt][i] = -INFINITY;
                }
#pragma unroll
                for (int i = 0; i < NR; ++i) over |= x[nt][i] > m_run[nt];
            }
            if (__any_sync(0xffffffffu, over)) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float tm = -INFINITY;
#pragma unroll
                    for (int i = 0; i < NR; ++i) tm = fmaxf(tm, x[nt][i]);
                    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
                    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
                    tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
                    const float mn = fmaxf(m_run[nt], tm);
                    const float alpha = fast_exp2(m_run[nt] - mn);
                    m_run[nt] = mn;
                    l_run[nt] *= alpha;
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[nt][mt][e] *= alpha;
#pragma unroll
                    for (int gi = 0; gi < GW; ++gi) Zsum[nt][gi] *= alpha;
                }
            }
            // p, w = p·s of the V groups, and the fp16 hi / lo parts of w into the
            // operand table (row = head 4nt + j, this thread's tokens 8i + r)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                uint32_t* th = wtab + (4 * nt + j) * C::kWS;
#pragma unroll
                for (int i = 0; i < NR; ++i) {
                    const int t = 8 * i + r;
                    const float pv = fast_exp2(x[nt][i] - m_run[nt]);   // masked tokens: 2^-inf = 0
                    l_run[nt] += pv;
                    float w[GW];
                    float2 szv[GW];   // rows of invalid tokens hold finite stale data and get p = 0
                    load_sz_groups<GW, FP8>(tb + t * row + D / 2 + PB * NG, wsl * GW, szv);
#pragma unroll
                    for (int gi = 0; gi < GW; ++gi) {
                        const float2 sz = szv[gi];
                        w[gi] = pv * sz.x;
                        Zsum[nt][gi] = fmaf(pv, sz.y, Zsum[nt][gi]);
                    }
                    if constexpr (GW == 1) {
                        const __half hh = __float2half_rn(w[0]);
                        const __half hl = __float2half_rn(w[0] - __half2float(hh));
                        reinterpret_cast<__half*>(th)[t] = hh;
                        reinterpret_cast<__half*>(th + C::kWLO)[t] = hl;
                    } else {
#pragma unroll
                        for (int gp = 0; gp < GW / 2; ++gp) {
                            const uint32_t hi = pack_part(w[2 * gp], w[2 * gp + 1], false);
                            const float2 f = h2f(hi);
                            const uint32_t lo = pack_part(w[2 * gp] - f.x, w[2 * gp + 1] - f.y, false);
                            th[t * (GW / 2) + gp] = hi;
                            th[C::kWLO + t * (GW / 2) + gp] = lo;
                        }
                    }
                }
            }
            __syncwarp();
            // ---------------- P·V: MQ k16 steps ----------------
            // B fragment of column r (head 4nt + r/2, part r&1): tokens 16ks + {2j, 2j+1} and {2j+8, 2j+9}
            const uint32_t* tr = wtab + (r & 1) * C::kWLO + (r >> 1) * C::kWS;
#pragma unroll
            for (int ks = 0; ks < MQ; ++ks) {
                uint32_t bvg[NT][GW][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint32_t* tn = tr + 4 * nt * C::kWS;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int t0 = 16 * ks + 2 * j + 8 * hf;   // even
                        if constexpr (GW == 1) {
                            bvg[nt][0][hf] = tn[t0 / 2];
                        } else if constexpr (GW == 2) {
                            const uint2 u = *reinterpret_cast<const uint2*>(tn + t0);
                            bvg[nt][0][hf] = prmt(u.x, u.y, 0x5410u);
                            bvg[nt][1][hf] = prmt(u.x, u.y, 0x7632u);
                        } else {
#pragma unroll
                            for (int gp = 0; gp < GW / 2; ++gp) {
                                const uint32_t u0 = tn[t0 * (GW / 2) + gp], u1 = tn[(t0 + 1) * (GW / 2) + gp];
                                bvg[nt][2 * gp][hf] = prmt(u0, u1, 0x5410u);
                                bvg[nt][2 * gp + 1][hf] = prmt(u0, u1, 0x7632u);
                            }
                        }
                    }
                }
                const int tk[4] = {16 * ks + 2 * j, 16 * ks + 2 * j + 1, 16 * ks + 2 * j + 8, 16 * ks + 2 * j + 9};
#pragma unroll
                for (int gi = 0; gi < GW; ++gi) {
                    const int gg = wsl * GW + gi;
                    // this thread's V code slice of group gg: G/32 bytes per token
                    const int vb = D / 4 + gg * (G / 4) + r * (G / 32);   // byte offset in the record
                    if constexpr (G == 32) {
                        const int wo = vb & ~3;
                        const uint32_t bsel = (uint32_t)(vb & 3);
                        const uint32_t sel = bsel | ((4u + bsel) << 8) | (bsel << 4) | ((4u + bsel) << 12);
                        const uint32_t u01 = prmt(*reinterpret_cast<const uint32_t*>(tb + tk[0] * row + wo),
                                                  *reinterpret_cast<const uint32_t*>(tb + tk[1] * row + wo), sel);
                        const uint32_t u23 = prmt(*reinterpret_cast<const uint32_t*>(tb + tk[2] * row + wo),
                                                  *reinterpret_cast<const uint32_t*>(tb + tk[3] * row + wo), sel);
#pragma unroll
                        for (int mu = 0; mu < 2; ++mu) {   // rows r / r+8: positions 2mu / 2mu+1 of the byte
                            const int mt = gi * MTG + mu;
                            const uint32_t m0 = (3u << (4 * mu)) | (3u << (4 * mu + 16));
                            const uint32_t m1 = m0 << 2;
                            const uint32_t a0 = u01 & m0, a1 = u01 & m1;
                            const uint32_t a2 = u23 & m0, a3 = u23 & m1;
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                mma16816(acc[nt][mt], a0, a1, a2, a3, bvg[nt][gi][0], bvg[nt][gi][1]);
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
                            // m-tile slot mu: row r <- first, row r+8 <- second position of slot mu
                            const uint32_t d01 = u01, r01 = u01 >> 6;
                            const uint32_t d23 = u23, r23 = u23 >> 6;
#pragma unroll
                            for (int mu = 0; mu < 4; ++mu) {
                                const int mt = gi * MTG + hw * 4 + mu;
                                uint32_t a0, a1, a2, a3;
                                if (mu == 0) {
                                    a0 = code_sub<slot_pos(0, 0)>(d01, r01); a1 = code_sub<slot_pos(0, 1)>(d01, r01);
                                    a2 = code_sub<slot_pos(0, 0)>(d23, r23); a3 = code_sub<slot_pos(0, 1)>(d23, r23);
                                } else if (mu == 1) {
                                    a0 = code_sub<slot_pos(1, 0)>(d01, r01); a1 = code_sub<slot_pos(1, 1)>(d01, r01);
                                    a2 = code_sub<slot_pos(1, 0)>(d23, r23); a3 = code_sub<slot_pos(1, 1)>(d23, r23);
                                } else if (mu == 2) {
                                    a0 = code_sub<slot_pos(2, 0)>(d01, r01); a1 = code_sub<slot_pos(2, 1)>(d01, r01);
                                    a2 = code_sub<slot_pos(2, 0)>(d23, r23); a3 = code_sub<slot_pos(2, 1)>(d23, r23);
                                } else {
                                    a0 = code_sub<slot_pos(3, 0)>(d01, r01); a1 = code_sub<slot_pos(3, 1)>(d01, r01);
                                    a2 = code_sub<slot_pos(3, 0)>(d23, r23); a3 = code_sub<slot_pos(3, 1)>(d23, r23);
                                }
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
                                    mma16816(acc[nt][mt], a0, a1, a2, a3, bvg[nt][gi][0], bvg[nt][gi][1]);
                            }
                        }
                    }
                }
            }
            __syncwarp();                       // this warp is done with stage k and its scale table
            if (lane == 0) mbar_arrive(&empty[s]);
            it.next(P, f1);
        }

        if (aborted) break;
        // ---------------- segment end: reduce and write the partial ----------------
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 4);
            l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 8);
            l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 16);
#pragma unroll
            for (int gi = 0; gi < GW; ++gi) {
#pragma unroll
                for (int sh = 4; sh < 32; sh <<= 1) {
                    Zsum[nt][gi] += __shfl_xor_sync(0xffffffffu, Zsum[nt][gi], sh);
                }
            }
        }
        // out[head 4nt+j][ch] = (acc_hi + acc_lo − W)/α_ch + Z, with α = 1/16 on the
        // rows r (even code positions) and 1/4 on the rows r+8
        const int64_t slot = ((int64_t)blockIdx.x + b) * PAR + pi;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hh = 4 * (hp * NT + nt) + j;
            const int hq = h * g + hh;
            float* o = P.po + (slot * P.Hq + hq) * D;
            if (r == 0 && wsl == 0 && hh < g) P.ml[slot * P.Hq + hq] = make_float2(m_run[nt], l_run[nt]);
#pragma unroll
            for (int gi = 0; gi < GW; ++gi) {
                const float Zh = Zsum[nt][gi];
                const int gg = wsl * GW + gi;
#pragma unroll
                for (int mu = 0; mu < MTG; ++mu) {
                    const int mt = gi * MTG + mu;
                    if (hh >= g) continue;
                    const float v0 = acc[nt][mt][0] + acc[nt][mt][1];   // row r  (hi + lo columns)
                    const float v1 = acc[nt][mt][2] + acc[nt][mt][3];   // row r + 8
                    if constexpr (G == 32) {
                        // rows r / r+8: positions 2mu / 2mu+1 of the byte r (bits 4mu, 4mu+2)
                        const int ch0 = gg * G + 4 * r + 2 * mu;
                        o[ch0] = (mu == 0 ? sub_inv(0) : sub_inv(4)) * v0 + Zh;
                        o[ch0 + 1] = (mu == 0 ? sub_inv(2) : sub_inv(6)) * v1 + Zh;
                    } else {
                        // the 16-bit chunk r (and half-word mu / 4) of the group; slot mu % 4
                        const int base = gg * G + r * (G / 8) + 8 * (mu / 4);
                        const int s4 = mu % 4;
                        const int p0 = s4 == 0 ? slot_pos(0, 0) : s4 == 1 ? slot_pos(1, 0) : s4 == 2 ? slot_pos(2, 0) : slot_pos(3, 0);
                        const int p1 = s4 == 0 ? slot_pos(0, 1) : s4 == 1 ? slot_pos(1, 1) : s4 == 2 ? slot_pos(2, 1) : slot_pos(3, 1);
                        o[base + p0] = sub_inv(sub_bit(p0)) * v0 + Zh;
                        o[base + p1] = sub_inv(sub_bit(p1)) * v1 + Zh;
                    }
                }
            }
        }
    }
    if (aborted) {   // stages this warp issued but did not consume: k, k + PAR, ..., pk - PAR
        long long drain = 2000000000LL;
        for (uint32_t kk = k; kk < pk; kk += PAR)
            mbar_wait_bounded(&full[kk & (NS - 1)], (kk >> ns_log2) & 1, P.status, drain);
    }
}

// Shared-memory plan: (x_off, stages_off, ring depth log2, total bytes); false if it
// does not fit.  Two stage parities need at least 4 stages (2 in flight).
template <int D, int G, int NT, int WPH, int TTOK, int PAR, int HP, bool FP8>
static bool mma_smem_plan(int Hkv, int* x_off, int* stages_off, int* ns_log2, size_t* total) {
    using C = MmaCfg<D, G, NT, WPH, TTOK, FP8>;
    const int nwarps = Hkv * WPH * PAR * HP;
    // named barriers 1 .. Hkv·HP·PAR pair the channel-slice warps (ids up to 15)
    if (WPH == 2 && Hkv * HP * PAR > 15) return false;
    *x_off = kSmemTab + nwarps * C::TBL;
    *stages_off = (*x_off + Hkv * HP * PAR * C::XCH * 4 + 127) / 128 * 128;
    const size_t stage = (size_t)TTOK * row_bytes(slot_bytes_of(Hkv, C::REC));
    int lg = 3;                                  // 8 stages when they fit, else 4, else 2
    while (lg > PAR && *stages_off + (stage << lg) > 224 * 1024) --lg;
    *ns_log2 = lg;
    *total = *stages_off + (stage << lg);
    return *total <= 225 * 1024;
}

template <int D, int G, int NT, int WPH, int TTOK, int PAR, int HKV, int HP, bool FP8>
static int launch_mma(DecodeParams P, cudaStream_t st) {
    const int threads = 32 * P.Hkv * WPH * PAR * HP;
    int x_off, stages_off, ns_log2;
    size_t smem;
    if (!mma_smem_plan<D, G, NT, WPH, TTOK, PAR, HP, FP8>(P.Hkv, &x_off, &stages_off, &ns_log2, &smem))
        return OSCAR_ERR_ARG;
    auto kern = history_mma_kernel<D, G, NT, WPH, TTOK, PAR, HKV, HP, FP8>;
    if (const int rc_ = ensure_dynamic_smem((const void*)kern, smem, "cudaFuncSetAttribute(history_mma_kernel)"))
        return rc_;
    const int grid = std::min(P.n_ctas, sm_count());
    const int trow = row_bytes(slot_bytes_of(P.Hkv, MmaCfg<D, G, NT, WPH, TTOK, FP8>::REC));
    launch_dependent(kern, dim3(grid), dim3(threads), smem, st, P, x_off, stages_off, trow, ns_log2);
    return check_cuda("history_mma_kernel launch");
}

// Chooses the tensor-core kernel for the shape and (s, z) format, or reports
// that none fits (the caller then runs the CUDA-core kernel).  P.n_ctas is
// updated to the grid that was launched.
template <bool FP8>
static int launch_history_mma_fmt(DecodeParams& P, int head_dim, cudaStream_t st, bool* launched) {
    *launched = false;
    if (P.Hkv > (head_dim == 256 ? 4 : 8) || P.g > 8) return OSCAR_OK;
    const int nt = (2 * P.g + 7) / 8;
    int rc = OSCAR_OK;
    // a variant is taken when its shared-memory plan fits; otherwise the next one is tried
    auto go = [&](auto plan, auto fn, int par, int hkv, int warps_per_head) {
        if (*launched || (hkv > 0 && hkv != P.Hkv)) return;
        if (P.Hkv * warps_per_head > 32) return;     // at most 1,024 threads
        int xo, so, lg;
        size_t smem;
        if (!plan(P.Hkv, &xo, &so, &lg, &smem)) return;
        P.par = par;
        rc = fn(P, st);
        *launched = true;
    };
#define OSCAR_MMA_X(D_, G_, NT_, WPH_, TT_, PAR_, HKV_, HP_) \
    go(mma_smem_plan<D_, G_, NT_, WPH_, TT_, PAR_, HP_, FP8>, launch_mma<D_, G_, NT_, WPH_, TT_, PAR_, HKV_, HP_, FP8>, \
       PAR_, HKV_, \
       WPH_ * PAR_ * HP_)
#define OSCAR_MMA_H(D_, G_, NT_, WPH_, TT_, PAR_, HKV_) OSCAR_MMA_X(D_, G_, NT_, WPH_, TT_, PAR_, HKV_, 1)
#define OSCAR_MMA(D_, G_, NT_, WPH_, TT_, PAR_) OSCAR_MMA_H(D_, G_, NT_, WPH_, TT_, PAR_, 0)
#define OSCAR_MMA_HP(D_, G_, WPH_, HKV_) OSCAR_MMA_X(D_, G_, 1, WPH_, 64, 1, HKV_, 2)
    // one n8 column tile (g <= 4): two warps per (head, slice) on alternate stages;
    // two tiles (g = 5..8): two warps per (head, slice), each with four of the
    // query heads, on every stage; failing that, one warp with both tiles and
    // 32-token stages (register budget)
    if (head_dim == 128) {
        if (P.G == 64) {
            // 8 KV heads (Qwen3-8B-like layers): compile-time stage row stride
            if (nt == 1) { OSCAR_MMA_H(128, 64, 1, 1, 64, 2, 8); OSCAR_MMA(128, 64, 1, 1, 64, 2); OSCAR_MMA(128, 64, 1, 1, 64, 1); }
            else { OSCAR_MMA_HP(128, 64, 1, 8); OSCAR_MMA_HP(128, 64, 1, 0); OSCAR_MMA(128, 64, 2, 1, 32, 1); }
        } else if (P.G == 128) {
            if (nt == 1) { OSCAR_MMA(128, 128, 1, 1, 64, 2); OSCAR_MMA(128, 128, 1, 1, 64, 1); }
            else { OSCAR_MMA_HP(128, 128, 1, 0); OSCAR_MMA(128, 128, 2, 1, 32, 1); }
        } else if (P.G == 32) {
            if (nt == 1) OSCAR_MMA(128, 32, 1, 1, 64, 1);   // two sets would spill registers
            else OSCAR_MMA(128, 32, 2, 1, 32, 1);
        }
    } else if (head_dim == 256) {
        if (P.G == 128) {
            if (nt == 1) { OSCAR_MMA(256, 128, 1, 2, 64, 2); OSCAR_MMA(256, 128, 1, 2, 64, 1); }
            else { OSCAR_MMA_HP(256, 128, 2, 0); OSCAR_MMA(256, 128, 2, 2, 32, 1); }
        } else if (P.G == 64) {
            if (nt == 1) { OSCAR_MMA(256, 64, 1, 2, 64, 2); OSCAR_MMA(256, 64, 1, 2, 64, 1); }
            else { OSCAR_MMA_HP(256, 64, 2, 0); OSCAR_MMA(256, 64, 2, 2, 32, 1); }
        }
    }
#undef OSCAR_MMA
#undef OSCAR_MMA_H
#undef OSCAR_MMA_HP
#undef OSCAR_MMA_X
    if (*launched) P.n_ctas = std::min(P.n_ctas, sm_count());
    return rc;
}

int launch_history_mma(DecodeParams& P, int head_dim, cudaStream_t st, bool* launched) {
    return P.fp8 ? launch_history_mma_fmt<true>(P, head_dim, st, launched)
                 : launch_history_mma_fmt<false>(P, head_dim, st, launched);
}

}  // namespace oscar
