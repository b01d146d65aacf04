// Tensor-core rotation and quantisation of large appends (prefill chunks).
//
// [OSCAR news] "OSCARの違い" / "サービングシステム：混合精度キャッシュレイアウト":
// every head vector entering the INT2 history is rotated, y = x·R, then
// clipped and quantised per group (lo = r·min, hi = r·max, s = fp16((hi-lo)/3),
// z = fp16(lo), c = clamp(rint((y-z)/s), 0, 3)).
//
// y = x·R is a dense (vectors × d) · (d × d) contraction, so it runs on the
// fifth-generation tensor cores (tcgen05.mma, kind::f16, bf16 operands, fp32
// accumulators in tensor memory).  x is exactly bf16 (every input is rounded
// to bf16 first), and R (fp32) is split into three bf16 parts hi + mid + lo,
// which hold its 24-bit significand, so every product is exact.  One
// accumulator takes the lo parts of all k-steps first, then the mid parts,
// then the hi parts.  Measured against the exact product this is more
// accurate than a sequential fp32 FMA chain (largest error about 5.5e-7 of
// the row's largest |y|, against 1.2e-6), which matters because a code
// decided near a rounding boundary must agree with the oracle.
//
// One CTA per SM, persistent over tiles of 128 vectors of one matrix (K or V:
// blockIdx.y).  R's three parts stay in shared memory as the B operand (N = d
// output channels × K = d, K-major, 128-byte swizzle).  Three warpgroups take
// the tiles in turn, each with its own x tile (the A operand, M = 128
// vectors), its own accumulator in tensor memory and its own mbarrier; one
// thread of the group issues the group's MMAs.  A group's flow per tile: wait for its
// rows, issue the MMAs, finish resolving the next tile's vectors and start the
// page-table loads of the one after, wait for the MMAs, start the next tile's
// rows (one tensor-map TMA load when they are a contiguous block of the bf16
// input, else 16-byte cp.async per chunk), then quantise: thread
// i of the group owns tensor-memory lane i, that is vector i of the tile and
// all its d channels, so a group's min / max is a reduction in registers.
//
// The code decision uses the correctly rounded reciprocal of 3s: q = 3·sat(a ·
// (1/3s)) with a = y - z is within 2^-21 of the correctly rounded quotient a/s
// for q in [0, 3] (three roundings).  The tensor cores' y differs from x·R
// rounded to fp32 by at most e = kTcBound·‖y‖₂, so rint(q) is the code of the
// exact y unless q lies within e/s + 2^-19 + 2^-21 of a half-integer; a warp
// in which some thread meets such a q in a group decides that group again with
// correctly rounded division, forming y exactly (compensated dot product of
// the input row with R's column) wherever y ± e straddles a boundary.  The
// group's (s, z) are checked the same way at its extremes ± e first.  A vector
// whose (s, z) could change copies its bf16 row from the x tile into a small
// per-warpgroup stash before the next tile's rows overwrite the tile, so its
// exact products read x from shared memory (others read their row in global
// memory).
// Tensor-memory loads (tcgen05.ld) are warp-collective, so every branch around
// them is warp-uniform.
#include <algorithm>
#include <cstring>

#include <cuda.h>

#include "oscar_append_tc_common.cuh"

namespace oscar {

namespace {

using namespace tcq;

constexpr int kSlots = 3;                  // warpgroups, each with its own tile in flight
constexpr int kTcThreads = 128 * kSlots;
constexpr uint32_t kTmemCols = 512;        // slot e's accumulator: columns 128·e .. 128·e + d
constexpr int kXCap = 16;                  // stashed rows per warpgroup and tile, at most


__device__ __forceinline__ void group_bar(int e) {
    asm volatile("bar.sync %0, 128;" :: "r"(1 + e) : "memory");
}

// Group barrier that also returns the OR of v over the group.
__device__ __forceinline__ bool group_bar_or(int e, bool v) {
    int r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, %2, 128, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((int)v), "r"(1 + e) : "memory");
    return r != 0;
}


// fl(x·R[:, ch]) (compensated, faithful to the exact product) for the vector of
// lane L, by the whole warp: lane l takes k = l·D/32 .. + D/32 - 1, x from the
// vector's bf16 row stashed in shared memory (xrow, the same in every lane) or,
// without one, from its row in global memory, R exactly as hi + mid + lo from
// the bf16 parts in shared memory (B operand layout), then a compensated sum
// over the warp.
template <int D>
__device__ __forceinline__ float tc_dot2(const unsigned char* sB, const ExactSrc& src, const uint16_t* xrow, int L,
                                         int ch, int lane) {
    constexpr int KPL = D / 32;                       // k per lane: 4 (d 128) or 2 (d 64)
    constexpr int B_PART = D * D * 2;
    float x[KPL];
    if (xrow) {
#pragma unroll
        for (int i = 0; i < KPL; ++i) x[i] = bf16_bits_to_f32(xrow[lane * KPL + i]);
    } else {
        const int kd = __shfl_sync(0xffffffffu, src.kind, L);
        const uint32_t olo = __shfl_sync(0xffffffffu, (uint32_t)(uint64_t)src.off, L);
        const uint32_t ohi = __shfl_sync(0xffffffffu, (uint32_t)((uint64_t)src.off >> 32), L);
        const int64_t o = (int64_t)(((uint64_t)ohi << 32) | olo) + lane * KPL;
#pragma unroll
        for (int i = 0; i < KPL; ++i) {
            x[i] = kd == 1 ? bf16_bits_to_f32(src.recent[o + i])
                 : kd == 2 ? bf16_bits_to_f32(f32_to_bf16_bits(load_elem(src.src_new, o + i, src.kv_dtype)))
                           : 0.0f;
        }
    }
    const int k0 = lane * KPL;
    const uint32_t boff = tc5::sw128_offset(D, ch, k0 / 8) + (uint32_t)(k0 % 8) * 2;
    float s = 0.0f, c = 0.0f;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
        float r = 0.0f;
#pragma unroll
        for (int p = 0; p < 3; ++p)                   // hi + mid + lo: exact in fp32
            r += bf16_bits_to_f32(*reinterpret_cast<const uint16_t*>(sB + p * B_PART + boff + 2 * i));
        const float pr = __fmul_rn(x[i], r);
        const float pe = __fmaf_rn(x[i], r, -pr);
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
// (warp-collective; out of line, so the common path stays compact): the
// extremes lie among the channels within 2e of the computed ones (y reloaded
// from the group's tensor-memory columns tgrp), which are formed exactly.
// Returns (min, max) over the exact values of the candidates; meaningful for
// the uncertain lanes.
template <int D, int G>
__device__ __noinline__ float2 tc_exact_extremes(uint32_t tgrp, const unsigned char* sB, ExactSrc src,
                                                 const uint16_t* xs, int xslot, bool unc, float mn, float mx,
                                                 float e2, int ch0, int lane) {
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
            const int xl = __shfl_sync(0xffffffffu, xslot, L);
            const float ye = tc_dot2<D>(sB, src, xl >= 0 ? xs + xl * (D + 8) : nullptr, L, ch0 + 32 * c + q, lane);
            if (lane == L) {
                cm &= cm - 1u;
                mne = fminf(mne, ye);
                mxe = fmaxf(mxe, ye);
            }
        }
    }
    return make_float2(mne, mxe);
}

// Re-decides the codes of one 32-channel chunk whose reciprocal-path quotient
// lies near a half-integer (warp-collective; out of line): such a channel is
// decided by correctly rounded division, on the exact y where y ± e straddles
// a boundary, and patched into the chunk's two code words w.
template <int D>
__device__ __noinline__ uint2 tc_exact_codes(uint32_t tchunk, const unsigned char* sB, ExactSrc src,
                                             const uint16_t* xs, int xslot, float zc, float sc, float r3, float nb2,
                                             float be, uint2 w, int ch0, int lane) {
    float y[32];
    load_y(tchunk, y);
    uint32_t cm = 0;                              // channels to re-decide (the fast path's test)
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
        const float yq = load_col(tchunk + q);    // every lane's y of channel q; lane L's is the one used
        float u = sc != 0.0f ? __fdiv_rn(__fsub_rn(yq, zc), sc) : 0.0f;
        if (__shfl_sync(0xffffffffu, (int)(sc != 0.0f && code_near_boundary(u, be)), L)) {
            const int xl = __shfl_sync(0xffffffffu, xslot, L);
            const float ye = tc_dot2<D>(sB, src, xl >= 0 ? xs + xl * (D + 8) : nullptr, L, ch0 + q, lane);
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

template <int D>
struct TcCfg {
    static constexpr int KS = D / 16;               // k-steps of 16
    static constexpr int A_BYTES = kTcRows * D * 2; // one x tile
    static constexpr int B_PART = D * D * 2;        // one part of R
    static constexpr int CPR = D / 8;               // 16-byte chunks per row
    static constexpr int RPI = 32 / CPR;            // rows per warp instruction in the copy
    static constexpr size_t SMEM = 1024 + 3 * (size_t)B_PART + kSlots * (size_t)A_BYTES +
                                   (size_t)kSlots * 2 * kTcRows * kMetaInts * 4 + 128;   // + prefix, scratch
};

}  // namespace

template <int D, int G>
__global__ void __launch_bounds__(kTcThreads, 1)
quantize_tc_kernel(AppendParams P, const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   int use_tma, int xcap) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    using C = TcCfg<D>;
    constexpr int ng = D / G;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sB = smem;                                               // [3 parts][D rows][D] swizzled
    unsigned char* sA = smem + 3 * C::B_PART;                               // [slots][128 rows][D] swizzled
    int* meta = reinterpret_cast<int*>(sA + kSlots * C::A_BYTES);          // [slots][2 buffers][128][4]
    uint64_t* bars = reinterpret_cast<uint64_t*>(meta + kSlots * 2 * kTcRows * kMetaInts);   // [slots] MMAs done
    uint64_t* fulls = bars + kSlots;                                        // [slots] TMA rows landed
    uint32_t* tslot = reinterpret_cast<uint32_t*>(fulls + kSlots);
    int* prefix = reinterpret_cast<int*>(tslot + 2);                       // batch + 1
    int* scratch = prefix + P.batch + 1;                                    // kTcThreads
    int* nxs = scratch + kTcThreads;                                        // [slots] rows stashed (4 ints)
    uint16_t* xs_all = reinterpret_cast<uint16_t*>((reinterpret_cast<uintptr_t>(nxs + 4) + 15) & ~uintptr_t(15));
    constexpr int XS = D + 8;                                               // stashed row stride (bf16 elements)

    const int mat = blockIdx.y;
    const float* R = mat ? P.rot_v : P.rot_k;
    const void* src_new = mat ? P.v : P.k;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int e = warp >> 2;           // warpgroup = tile slot
    const int gw = warp & 3;           // warp of the group = tensor-memory lane quarter
    const int gt = tid & 127;          // thread of the group = tile row of the epilogue

    build_prefix(P, prefix, scratch);
    const int64_t total_vec = (int64_t)prefix[P.batch] * P.Hkv;
    const int64_t ntiles = (total_vec + kTcRows - 1) / kTcRows;
    if ((int64_t)blockIdx.x >= ntiles) return;    // uniform over the CTA, before any allocation

    if (tid == 0) {
        for (int q = 0; q < kSlots; ++q) {
            mbar_init(&bars[q], 1);
            mbar_init(&fulls[q], 1);
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        tc5::alloc(tslot, kTmemCols);
        tc5::relinquish();
    }
    // B: the three parts of R as D rows n (column n of R) × D k.  Item (n, j)
    // reads R[8j .. 8j+7][n] once and stores its 16-byte chunk of every part;
    // consecutive threads take consecutive n (coalesced reads; the swizzle
    // spreads the stores), two items in flight per thread.
    constexpr int NB = D * C::CPR;
#pragma unroll 1
    for (int i0 = tid; i0 < NB; i0 += 2 * kTcThreads) {
        float v[2][8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = i0 + u * kTcThreads;
            const int n = i % D, j = i / D;
#pragma unroll
            for (int q = 0; q < 8; ++q) v[u][q] = i < NB ? R[(int64_t)(8 * j + q) * D + n] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int i = i0 + u * kTcThreads;
            if (i >= NB) continue;
            const int n = i % D, j = i / D;
#pragma unroll
            for (int p = 0; p < 3; ++p) {
                uint32_t w[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) w[q] = pack_bf16(bf16_part(v[u][2 * q], p), bf16_part(v[u][2 * q + 1], p));
                *reinterpret_cast<uint4*>(sB + p * C::B_PART + tc5::sw128_offset(D, n, j)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
    tc5::fence_proxy_async();
    tc5::fence_before();
    __syncthreads();
    tc5::fence_after();
    const uint32_t tmem = *tslot;

    const bool vec_in = (reinterpret_cast<uintptr_t>(src_new) & 15) == 0;
    const float rclip = P.clip;
    const int rec_off_codes = mat ? D / 4 : 0;
    const bool fp8 = P.fp8 != 0;
    const int rec_off_sz = D / 2 + (mat ? (fp8 ? 2 : 4) * ng : 0);
    unsigned char* A = sA + e * C::A_BYTES;
    int* gmeta = meta + e * 2 * kTcRows * kMetaInts;
    int* nx = nxs + e;                              // this group's stash: xcap rows of XS
    const uint16_t* xs = xs_all + (int64_t)e * xcap * XS;
    uint64_t* bar = &bars[e];
    uint64_t* full = &fulls[e];
    const CUtensorMap* tmap = mat ? &tm_v : &tm_k;
    const uint32_t tacc = tmem + (uint32_t)(128 * e) + ((uint32_t)(32 * gw) << 16);

    // Vector gt of a tile is resolved in two stages one loop iteration apart, so
    // that its page-table load is in flight while the group quantises: locate()
    // finds the request and position and starts that load; publish() checks the
    // slot and writes the entry (slot, -1 when there is nothing to write; head;
    // source kind, 1 recent ring, 2 new input; element offset of the row).
    struct Loc {
        int b, p, h, sl;
        bool valid;
    };
    auto locate = [&](int64_t tile) {
        Loc L{0, 0, 0, -1, false};
        const int64_t ev = tile * kTcRows + gt;
        if (tile < ntiles && ev < total_vec) {
            int u;
            if (total_vec <= 0x7FFFFFFF) {       // 32-bit index arithmetic (uniform branch)
                u = (int)((uint32_t)ev / (uint32_t)P.Hkv);
                L.h = (int)((uint32_t)ev - (uint32_t)u * (uint32_t)P.Hkv);
            } else {
                u = (int)(ev / P.Hkv);
                L.h = (int)(ev % P.Hkv);
            }
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
                    off = ((((int64_t)rq * P.W + p % P.W) * P.Hkv + h) * 2 + mat) * D;
                } else {
                    kind = 2;
                    off = ((int64_t)(P.cu_new[b] + (p - L0)) * P.Hkv + h) * D;
                }
            }
        }
        int* m = gmeta + (buf * kTcRows + gt) * kMetaInts;
        m[0] = slot;
        m[1] = L.h | (kind << 16);
        *reinterpret_cast<int64_t*>(m + 2) = off;
    };
    // rows 32·gw .. +31 of a tile into the group's x tile; RPI rows per warp instruction
    auto gather = [&](int buf) {
#pragma unroll 4
        for (int rr = 0; rr < 32; rr += C::RPI) {
            const int row = 32 * gw + rr + lane / C::CPR, j = lane % C::CPR;
            unsigned char* dst = A + tc5::sw128_offset(kTcRows, row, j);
            const int4 m = *reinterpret_cast<const int4*>(gmeta + (buf * kTcRows + row) * kMetaInts);
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

    // A tile whose valid rows are all new input, row r at row 0's offset + r·d,
    // is one 128 × d block of the input: a tensor-map (TMA) load of two 64-wide
    // boxes lands it in the swizzled layout directly.  Called after the group
    // barrier that follows publish(buf); uniform over the group.
    auto contiguous = [&](int buf) -> bool {
        const int4 m0 = *reinterpret_cast<const int4*>(gmeta + buf * kTcRows * kMetaInts);
        const int4 m = *reinterpret_cast<const int4*>(gmeta + (buf * kTcRows + gt) * kMetaInts);
        const int64_t off0 = (int64_t)(((uint64_t)(uint32_t)m0.w << 32) | (uint32_t)m0.z);
        const int64_t off = (int64_t)(((uint64_t)(uint32_t)m.w << 32) | (uint32_t)m.z);
        const bool row_ok = m.x < 0 || ((m.y >> 16) == 2 && off == off0 + (int64_t)gt * D);
        const bool head_ok = m0.x >= 0 && (m0.y >> 16) == 2;
        return !group_bar_or(e, !(row_ok && head_ok));
    };
    auto issue_tma = [&](int buf) {
        if (gt == 0) {
            const int4 m0 = *reinterpret_cast<const int4*>(gmeta + buf * kTcRows * kMetaInts);
            const int64_t off0 = (int64_t)(((uint64_t)(uint32_t)m0.w << 32) | (uint32_t)m0.z);
            mbar_arrive_expect_tx(full, (uint32_t)C::A_BYTES);
#pragma unroll
            for (int xb = 0; xb < D / 64; ++xb)
                tc5::tma_load_2d(A + xb * kTcRows * 128, tmap, 64 * xb, (int)(off0 / D), full);
        }
    };

    long long budget = 2000000000LL;            // cycles per MMA wait (~1 s); 0 after a timeout
    bool aborted = false;
    uint32_t it = 0;
    const int64_t step = kSlots * (int64_t)gridDim.x;
    int64_t tile = blockIdx.x + (int64_t)e * gridDim.x;
    uint32_t tma_n = 0;                         // TMA tiles of this slot so far (parity of `full`)
    bool cur_tma = false;                       // the current tile's rows come by TMA
    int drain_full = -1, drain_mma = -1;        // parities still to wait for after an abort
    publish(locate(tile), 0);
    group_bar(e);
    if (tile < ntiles) {
        cur_tma = use_tma && contiguous(0);
        if (cur_tma) issue_tma(0);
        else gather(0);
    }
    Loc pend = locate(tile + step);             // the tile after the current one
    for (; tile < ntiles; tile += step, ++it) {
        const int buf = it & 1;
        bool to = false;
        if (cur_tma) {
            if (gt == 0 && !mbar_wait_bounded(full, tma_n & 1, P.status, budget)) {
                to = true;
                drain_full = (int)(tma_n & 1);
            }
            ++tma_n;
        } else {
            cp_async_wait<0>();
            tc5::fence_proxy_async();
        }
        tc5::fence_before();
        if (group_bar_or(e, to)) {              // the tile's rows are in place; last epilogue's loads done
            aborted = true;
            break;
        }
        if (gt == 0) {
            tc5::fence_after();
            constexpr uint32_t idesc = tc5::idesc_bf16_f32(kTcRows, D);
            const uint64_t ad0 = tc5::sw128_desc(smem_addr(A)), bd0 = tc5::sw128_desc(smem_addr(sB));
            const uint32_t dcol = tmem + (uint32_t)(128 * e);
#pragma unroll
            for (int p = 2; p >= 0; --p)          // lo parts first, hi parts last
#pragma unroll
                for (int kk = 0; kk < C::KS; ++kk) {
                    // the start address (bits 0-13, in 16-byte units) advances by the
                    // k-step's byte offset; it stays below 2^14, so no carry leaves the field
                    const uint32_t ao = (uint32_t)((kk >> 2) * kTcRows * 128 + (kk & 3) * 32);
                    const uint32_t bo = (uint32_t)(p * C::B_PART + (kk >> 2) * D * 128 + (kk & 3) * 32);
                    tc5::mma_bf16(dcol, ad0 + (ao >> 4), bd0 + (bo >> 4), idesc, !(p == 2 && kk == 0));
                }
            tc5::commit(bar);
            *nx = 0;                              // the last tile's stashed rows are done with (group barrier above)
        }
        const int64_t nxt = tile + step;
        publish(pend, buf ^ 1);                 // tile nxt: its page-table load was started one iteration ago
        pend = locate(nxt + step);
        // one thread observes the MMAs' completion; the group barrier passes it on
        to = false;
        if (gt == 0 && !mbar_wait_bounded(bar, it & 1, P.status, budget)) {
            to = true;
            drain_mma = (int)(it & 1);
        }
        if (group_bar_or(e, to)) {              // MMAs done (A free); next tile's vectors resolved
            aborted = true;
            break;
        }
        tc5::fence_after();
        constexpr int NC = G / 32;                // 32-channel chunks per group
        constexpr bool kKeep = G <= 64;           // the group's y stays in registers between the passes
        // err bounds |y - fl(x·R)| on every channel of the vector (kTcBound·‖y‖₂);
        // with it, which (s, z) of the vector y ± err could change (umask)
        float err;
        uint32_t umask = 0;
        {
            float2 q2 = make_float2(0.0f, 0.0f);
            float mn = INFINITY, mx = -INFINITY;
            float gmn[ng], gmx[ng];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float yy[32];
                load_y(tacc + 32 * c, yy);
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const float2 v = make_float2(yy[2 * q], yy[2 * q + 1]);
                    q2 = __ffma2_rn(v, v, q2);
                }
                minmax32(yy, mn, mx);
                if ((32 * (c + 1)) % G == 0) {    // the last chunk of group 32·c / G
                    gmn[32 * c / G] = mn;
                    gmx[32 * c / G] = mx;
                    mn = INFINITY;
                    mx = -INFINITY;
                }
            }
            err = kTcBound * sqrtf(q2.x + q2.y);
#pragma unroll
            for (int gi = 0; gi < ng; ++gi) umask |= sz_uncertain(gmn[gi], gmx[gi], rclip, err, fp8) ? (1u << gi) : 0u;
        }
        const float e2 = __fmul_ru(2.0f, err);
        // the vector's bf16 row into the group's stash when some (s, z) is
        // uncertain, before the next tile's rows overwrite the x tile
        int xslot = -1;
        if (umask) {
            const int sl = atomicAdd(nx, 1);
            if (sl < xcap) {
                xslot = sl;
                uint4* dst = reinterpret_cast<uint4*>(const_cast<uint16_t*>(xs) + sl * XS);
#pragma unroll
                for (int j = 0; j < C::CPR; ++j) dst[j] = *reinterpret_cast<const uint4*>(A + tc5::sw128_offset(kTcRows, gt, j));
            }
        }
        group_bar(e);                             // rows stashed: the x tile may be overwritten
        cur_tma = false;
        if (nxt < ntiles) {
            cur_tma = use_tma && contiguous(buf ^ 1);
            if (cur_tma) issue_tma(buf ^ 1);
            else gather(buf ^ 1);
        }

        // ---- quantise vector gt of the tile ----
        const int* m = gmeta + (buf * kTcRows + gt) * kMetaInts;
        const int slot = m[0];
        const ExactSrc xsrc{P.recent, src_new, P.kv_dtype, m[1] >> 16, *reinterpret_cast<const int64_t*>(m + 2)};
        uint8_t* rec = P.records + (int64_t)(slot < 0 ? 0 : slot) * P.slot_bytes + (int64_t)(m[1] & 0xFFFF) * P.rec_bytes;
        // one group at a time (not unrolled: the loop body stays small in the
        // instruction cache); its codes and (s, z) go to the record at its end
#pragma unroll 1
        for (int gi = 0; gi < ng; ++gi) {
            float yk[kKeep ? NC : 1][32];
            uint32_t words[G / 16];
            float mn = INFINITY, mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                float (&y)[32] = yk[kKeep ? c : 0];
                load_y(tacc + gi * G + 32 * c, y);
                minmax32(y, mn, mx);
            }
            // (s, z) that y ± err could change: the extremes formed exactly (out of line)
            const bool unc = (umask >> gi) & 1u;
            if (__any_sync(0xffffffffu, unc)) {
                const float2 ex = tc_exact_extremes<D, G>(tacc + gi * G, sB, xsrc, xs, xslot, unc, mn, mx, e2, gi * G,
                                                          lane);
                if (unc) {
                    mn = ex.x;
                    mx = ex.y;
                }
            }
            const SZ sz = sz_decide(mn, mx, rclip, fp8);
            const float sc = sz.s, zc = sz.z;
            // tcgen05.ld is warp-collective: every lane runs the same loads.  A flat
            // group (s = 0) takes r3 = 0, so its fast-path codes are all 0.
            const float r3 = sc != 0.0f ? __frcp_rn(3.0f * sc) : 0.0f;   // 3·sc is exact (≤ 11-bit significand × 3)
            // a code is certain when its quotient is farther from a half-integer than
            // err/s plus the reciprocal path's 2^-21
            const float be = code_band(err, r3);
            const float hb = 0.5f - (be + 1.0f / 2097152.0f);
            const float nb2 = hb > 0.0f ? -hb * hb : 0.0f;
            uint32_t tie = 0xFFFFFFFFu;
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                if (!kKeep) load_y(tacc + gi * G + 32 * c, yk[0]);
                codes32(yk[kKeep ? c : 0], zc, r3, nb2, words[2 * c], words[2 * c + 1], tie);
            }
            if (__any_sync(0xffffffffu, !(tie >> 31))) {
                // a quotient near a tie: re-decide those channels by correctly rounded
                // division, on the exact y where y ± err straddles a boundary
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    const uint2 w = tc_exact_codes<D>(tacc + gi * G + 32 * c, sB, xsrc, xs, xslot, zc, sc, r3, nb2, be,
                                                      make_uint2(words[2 * c], words[2 * c + 1]), gi * G + 32 * c,
                                                      lane);
                    words[2 * c] = w.x;
                    words[2 * c + 1] = w.y;
                }
            }
            if (slot >= 0) {
                store_sz(rec, rec_off_sz, gi, sz, fp8);
                uint8_t* dst = rec + rec_off_codes + gi * (G / 4);
                if (fp8) {   // E4M3 records start on 8-byte boundaries
#pragma unroll
                    for (int q = 0; q < G / 32; ++q)
                        *reinterpret_cast<uint2*>(dst + 8 * q) = make_uint2(words[2 * q], words[2 * q + 1]);
                } else if constexpr (G >= 64) {
#pragma unroll
                    for (int q = 0; q < G / 64; ++q)
                        *reinterpret_cast<uint4*>(dst + 16 * q) =
                            make_uint4(words[4 * q], words[4 * q + 1], words[4 * q + 2], words[4 * q + 3]);
                } else {
                    *reinterpret_cast<uint2*>(dst) = make_uint2(words[0], words[1]);
                }
            }
        }
    }
    if (aborted && gt == 0) {                     // copies or MMAs of the slot may still run: bounded drain
        long long drain = 2000000000LL;
        if (drain_full >= 0) mbar_wait_bounded(full, (uint32_t)drain_full, P.status, drain);
        if (drain_mma >= 0) mbar_wait_bounded(bar, (uint32_t)drain_mma, P.status, drain);
    }
    cp_async_wait<0>();
    tc5::fence_before();
    __syncthreads();
    if (warp == 0) {
        tc5::fence_after();
        tc5::dealloc(tmem, kTmemCols);
    }
}

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, fetched through the runtime (null if absent).
EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return (EncodeTiledFn) nullptr;
        }
        return (EncodeTiledFn)p;
    }();
    return fn;
}

// 2-D map of a [rows][d] bf16 input: boxes of 64 channels × 128 rows with the
// 128-byte swizzle (the MMA's operand layout); rows past the end read as zero.
bool encode_rows(CUtensorMap* m, const void* base, int64_t rows, int d) {
    const EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kTcRows};
    const cuuint32_t es[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

template <int D, int G>
static int launch_tc(const AppendParams& P, int64_t max_vec, cudaStream_t stream) {
    using C = TcCfg<D>;
    // prefix, scratch, the stash counters and 16 bytes of alignment, then each
    // warpgroup's stash (up to kXCap rows of d + 8 bf16) as far as the block's
    // shared memory holds it; at least 116 KB, so that one CTA (and one
    // tensor-memory allocation) sits on each SM
    const size_t fixed = C::SMEM + (size_t)(P.batch + 1 + kTcThreads + 4) * 4 + 16;
    const int lim = max_dynamic_smem();
    if (lim <= 0) return OSCAR_ERR_CUDA;
    const int64_t row_bytes = (int64_t)kSlots * (D + 8) * 2;
    const int xcap = (int)std::min<int64_t>(kXCap, std::max<int64_t>(0, ((int64_t)lim - (int64_t)fixed) / row_bytes));
    const size_t smem = std::max<size_t>(fixed + (size_t)xcap * row_bytes, 116 * 1024);
    auto kern = quantize_tc_kernel<D, G>;
    if (const int rc_ = ensure_dynamic_smem((const void*)kern, smem, "cudaFuncSetAttribute(quantize_tc_kernel)"))
        return rc_;
    const int64_t tiles = (max_vec + kTcRows - 1) / kTcRows;
    const int64_t grid_x = std::max<int64_t>(1, std::min<int64_t>((tiles + kSlots - 1) / kSlots, (int64_t)sm_count() / 2));
    // bf16 inputs on 16-byte boundaries: contiguous tiles arrive by TMA
    CUtensorMap tk, tv;
    memset(&tk, 0, sizeof tk);
    memset(&tv, 0, sizeof tv);
    const int64_t rows = P.total_new * P.Hkv;
    const int use_tma = P.kv_dtype == OSCAR_DTYPE_BF16 && rows > 0 && rows < 0x7FFFFFFF &&
                        (reinterpret_cast<uintptr_t>(P.k) & 15) == 0 && (reinterpret_cast<uintptr_t>(P.v) & 15) == 0 &&
                        encode_rows(&tk, P.k, rows, D) && encode_rows(&tv, P.v, rows, D);
    launch_dependent(kern, dim3((unsigned)grid_x, 2), dim3(kTcThreads), smem, stream, P, tk, tv, use_tma, xcap);
    return check_cuda("quantize_tc_kernel launch");
}

template <int D>
int launch_quantize_tc(const AppendParams& P, int64_t max_vec, cudaStream_t stream) {
    if (P.G == 32) return launch_tc<D, 32>(P, max_vec, stream);
    if (P.G == 64) return launch_tc<D, 64>(P, max_vec, stream);
    if (D >= 128 && P.G == 128) return launch_tc<D, (D >= 128 ? 128 : 64)>(P, max_vec, stream);
    return OSCAR_ERR_ARG;
}

bool tc_encode_rows(CUtensorMap* m, const void* base, int64_t rows, int d) { return encode_rows(m, base, rows, d); }

template int launch_quantize_tc<64>(const AppendParams&, int64_t, cudaStream_t);
template int launch_quantize_tc<128>(const AppendParams&, int64_t, cudaStream_t);

}  // namespace oscar
