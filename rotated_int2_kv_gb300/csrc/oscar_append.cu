// Quantise-on-append: rotate, clip, quantise and pack new K/V head vectors
// into the INT2 pool, and write the BF16 sink / recent windows.
//
// [OSCAR news] "サービングシステム：混合精度キャッシュレイアウト": the first 64
// tokens and the last 256 tokens of a request stay BF16; every token in between
// is stored as INT2 after the OSCAR rotation and clipping.  [Escha log] part 2,
// settings table: one (scale, zero) per group of 64 channels; fix 1: 0.25 byte
// per code.
//
// Two kernels, in stream order:
//  1. quantize_kernel: every position entering the history in this call
//     ([max(S, L0-W), max(S, L1-W)) of each request) -- read from the recent
//     ring if it was cached before, else from the new input -- is rotated
//     y = x·R in fp32 (FFMA, R staged in shared memory), then per group:
//     lo = r·min, hi = r·max, s = fp16((hi-lo)/3), z = fp16(lo),
//     c = clamp(rint((y - z)/s), 0, 3); codes are packed 4 per byte.
//  2. window_copy_kernel: new positions below S go to the sink, new positions at
//     or after max(S, L1-W) to the ring slot p % W.  Running it second keeps
//     the spill reads of kernel 1 ahead of the ring overwrites.
#include <algorithm>

#include "oscar_append_step.cuh"

namespace oscar {


template <int D>
__global__ void __launch_bounds__(kAppendThreads)
quantize_kernel(AppendParams P) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    constexpr bool kResidentR = (D * D * 4 <= 64 * 1024);
    constexpr int kNB = D / kColBlock;           // column blocks of R
    constexpr int kYStride = D + 4;
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int kRCols = kResidentR ? D : kColBlock;
    constexpr int kXT = D * kTileVec;                   // transposed X tile, floats
    constexpr int kY = kTileVec * kYStride;             // Y tile, floats
    constexpr int kXY = kXT + kY;                       // x stays in place for the exact re-decisions
    float* sR = reinterpret_cast<float*>(smem);         // D x kRCols
    float* sXT = sR + D * kRCols;                       // D x 64
    float* sY = sXT + kXT;                              // 64 x (D + 4)
    int* prefix = reinterpret_cast<int*>(sR + D * kRCols + kXY);   // batch + 1
    int* scratch = prefix + P.batch + 1;                // blockDim.x
    __shared__ int s_meta[kTileVec][4];                               // b, p, h, slot (-1: skip)

    const int mat = blockIdx.y;                                       // 0: K, 1: V
    const float* R = mat ? P.rot_v : P.rot_k;
    const void* src_new = mat ? P.v : P.k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    build_prefix(P, prefix, scratch);
    const int64_t total_vec = (int64_t)prefix[P.batch] * P.Hkv;
    const int64_t ntiles = (total_vec + kTileVec - 1) / kTileVec;
    if ((int64_t)blockIdx.x >= ntiles) return;

    if (kResidentR) {
        for (int i = tid * 4; i < D * D; i += kAppendThreads * 4)
            *reinterpret_cast<float4*>(sR + i) = *reinterpret_cast<const float4*>(R + i);
    }
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t e0 = tile * kTileVec;
        const int nvec = (int)(total_vec - e0 < kTileVec ? total_vec - e0 : kTileVec);
        // ---- resolve vectors of the tile ---------------------------------
        if (tid < kTileVec) {
            int b = -1, p = 0, h = 0, slot = -1;
            if (tid < nvec) {
                const int64_t e = e0 + tid;
                const int u = (int)(e / P.Hkv);
                h = (int)(e % P.Hkv);
                b = find_request(prefix, P.batch, u);
                const int L0 = P.start_pos[b];
                p = hist_hi(L0, P.S, P.W) + (u - prefix[b]);
                if (p >= P.pt_stride) {
                    set_status(P.status, OSCAR_DEV_BAD_LEN);
                } else {
                    const int s = P.page_table[(int64_t)b * P.pt_stride + p];
                    if (s < 0 || s >= P.num_slots) set_status(P.status, OSCAR_DEV_BAD_SLOT);
                    else slot = s;
                }
                const int rq = P.req_idx ? P.req_idx[b] : b;
                if (p < L0 && (rq < 0 || rq >= P.max_reqs)) {
                    set_status(P.status, OSCAR_DEV_BAD_REQ);
                    slot = -1;
                }
                if (p >= L0 && (int64_t)P.cu_new[b] + (p - L0) >= P.total_new) {
                    set_status(P.status, OSCAR_DEV_BAD_LEN);
                    slot = -1;
                }
            }
            s_meta[tid][0] = b;
            s_meta[tid][1] = p;
            s_meta[tid][2] = h;
            s_meta[tid][3] = slot;
        }
        __syncthreads();
        // ---- gather X (bf16-rounded) into sXT[k][v] ------------------------
        for (int idx = tid; idx < kTileVec * (D / 8); idx += kAppendThreads) {
            const int v = idx % kTileVec, c8 = idx / kTileVec;
            float x[8];
            if (v < nvec && s_meta[v][3] >= 0) {
                const int b = s_meta[v][0], p = s_meta[v][1], h = s_meta[v][2];
                const int L0 = P.start_pos[b];
                if (p < L0) {
                    const int rq = P.req_idx ? P.req_idx[b] : b;
                    const uint16_t* row = P.recent + ((((int64_t)rq * P.W + p % P.W) * P.Hkv + h) * 2 + mat) * D;
                    const uint4 raw = *reinterpret_cast<const uint4*>(row + c8 * 8);
                    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        x[2 * j] = __uint_as_float(w4[j] << 16);
                        x[2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
                    }
                } else {
                    const int64_t t = P.cu_new[b] + (p - L0);
                    const int64_t base = (t * P.Hkv + h) * D + c8 * 8;
                    if (t < P.total_new) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            x[j] = bf16_bits_to_f32(f32_to_bf16_bits(load_elem(src_new, base + j, P.kv_dtype)));
                    } else {                 // cu_new disagrees with total_new: flagged, row skipped
                        set_status(P.status, OSCAR_DEV_BAD_LEN);
#pragma unroll
                        for (int j = 0; j < 8; ++j) x[j] = 0.f;
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) x[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) sXT[(c8 * 8 + j) * kTileVec + v] = x[j];
        }
        __syncthreads();
        // ---- Y = X · R, 4x4 register tile per thread per column block -------
        const int tv = warp * 2 + (lane >> 4), tc = lane & 15;
        float acc_all[kResidentR ? kNB : 1][4][4];
#pragma unroll
        for (int cb = 0; cb < kNB; ++cb) {
            const float* Rb;
            if (kResidentR) {
                Rb = sR + cb * kColBlock;
            } else {
                __syncthreads();
                for (int i = tid * 4; i < D * kColBlock; i += kAppendThreads * 4) {
                    const int row = i / kColBlock, col = i % kColBlock;
                    *reinterpret_cast<float4*>(sR + i) =
                        *reinterpret_cast<const float4*>(R + (int64_t)row * D + cb * kColBlock + col);
                }
                __syncthreads();
                Rb = sR;
            }
            const int ldr = kResidentR ? D : kColBlock;
            float acc[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 4
            for (int kk = 0; kk < D; ++kk) {
                const float4 xv = *reinterpret_cast<const float4*>(sXT + kk * kTileVec + 4 * tv);
                const float4 rv = *reinterpret_cast<const float4*>(Rb + kk * ldr + 4 * tc);
                const float xs[4] = {xv.x, xv.y, xv.z, xv.w};
                const float rs[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xs[i], rs[j], acc[i][j]);
            }
            if (kResidentR) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc_all[kResidentR ? cb : 0][i][j] = acc[i][j];
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    *reinterpret_cast<float4*>(sY + (4 * tv + i) * kYStride + cb * kColBlock + 4 * tc) =
                        make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            }
        }
        if (kResidentR) {
#pragma unroll
            for (int cb = 0; cb < kNB; ++cb)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    *reinterpret_cast<float4*>(sY + (4 * tv + i) * kYStride + cb * kColBlock + 4 * tc) =
                        make_float4(acc_all[kResidentR ? cb : 0][i][0], acc_all[kResidentR ? cb : 0][i][1],
                                    acc_all[kResidentR ? cb : 0][i][2], acc_all[kResidentR ? cb : 0][i][3]);
        }
        __syncthreads();
        // ---- quantise: one warp per vector, D/32 contiguous channels per lane ----
        constexpr int CPL = D / 32;
        for (int v = warp; v < nvec; v += kAppendThreads / 32) {
            const int slot = s_meta[v][3];
            if (slot < 0) continue;      // warp-uniform
            const int h = s_meta[v][2];
            float y[CPL], xv[CPL];
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                y[j] = sY[v * kYStride + lane * CPL + j];
                xv[j] = sXT[(lane * CPL + j) * kTileVec + v];
            }
            const float e = fma_chain_bound<D>(warp_sum_sq<CPL>(xv));
            quantize_store<D>(P, y, slot, h, mat, lane, e, [&](int k) { return sXT[k * kTileVec + v]; }, R);
        }
        __syncthreads();
    }
}

// Small appends (decode steps): one warp per head vector entering the history,
// 8 per block, so that a few hundred vectors still spread over many SMs.  The
// warp rotates its vector with the same sequential fp32 FMA order over k as
// quantize_kernel (bit-identical y), reading R through the L1 cache.
constexpr int kSmallVec = kAppendThreads / 32;

template <int D>
__global__ void __launch_bounds__(kAppendThreads)
quantize_small_kernel(AppendParams P) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    // R is staged in shared memory when it fits in 64 KB (d <= 128): every
    // thread issues all of its loads at once, ahead of the request prefix
    constexpr bool kResidentR = (D * D * 4 <= 64 * 1024);
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float sx[kSmallVec][D];
    float* sR = reinterpret_cast<float*>(smem);
    int* prefix = reinterpret_cast<int*>(smem + (kResidentR ? D * D * 4 : 0));
    int* scratch = prefix + P.batch + 1;
    constexpr int CPL = D / 32;
    const int mat = blockIdx.y;
    const float* R = mat ? P.rot_v : P.rot_k;
    const void* src_new = mat ? P.v : P.k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (kResidentR) {
        constexpr int NU = D * D / 4 / kAppendThreads;   // 16-byte copies per thread
#pragma unroll
        for (int u = 0; u < NU; ++u)
            cp_async16(sR + 4 * (tid + kAppendThreads * u), R + 4 * (tid + kAppendThreads * u));
        cp_async_commit();
    }
    build_prefix(P, prefix, scratch);
    if (kResidentR) {
        cp_async_wait<0>();
        __syncthreads();
    }
    const float* Rs = kResidentR ? sR : R;
    const int64_t total_vec = (int64_t)prefix[P.batch] * P.Hkv;
    for (int64_t e = (int64_t)blockIdx.x * kSmallVec + warp; e < total_vec; e += (int64_t)gridDim.x * kSmallVec) {
        // ---- resolve the vector (every lane, warp-uniform) ----
        const int u = (int)(e / P.Hkv), h = (int)(e % P.Hkv);
        const int b = find_request(prefix, P.batch, u);
        const int L0 = P.start_pos[b];
        const int p = hist_hi(L0, P.S, P.W) + (u - prefix[b]);
        const int rq = P.req_idx ? P.req_idx[b] : b;
        const int64_t t = (int64_t)P.cu_new[b] + (p - L0);
        // ---- x (bf16-rounded): lane holds channels lane·CPL ..; loaded when its
        // address is valid, in the same round as the page-table entry ----
        const bool from_ring = p < L0;
        const bool src_ok = from_ring ? (rq >= 0 && rq < P.max_reqs) : (t < P.total_new);
        float x[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) x[j] = 0.f;
        if (src_ok) {
            if (from_ring) {
                const uint16_t* rowp =
                    P.recent + ((((int64_t)rq * P.W + p % P.W) * P.Hkv + h) * 2 + mat) * D + lane * CPL;
#pragma unroll
                for (int j = 0; j < CPL; ++j) x[j] = bf16_bits_to_f32(rowp[j]);
            } else {
                const int64_t base = (t * P.Hkv + h) * D + lane * CPL;
#pragma unroll
                for (int j = 0; j < CPL; ++j)
                    x[j] = bf16_bits_to_f32(f32_to_bf16_bits(load_elem(src_new, base + j, P.kv_dtype)));
            }
        }
        int slot = -1;
        int bits = 0;
        if (p >= P.pt_stride) {
            bits |= OSCAR_DEV_BAD_LEN;
        } else {
            const int sl = P.page_table[(int64_t)b * P.pt_stride + p];
            if (sl < 0 || sl >= P.num_slots) bits |= OSCAR_DEV_BAD_SLOT;
            else slot = sl;
        }
        if (!src_ok) {
            bits |= from_ring ? OSCAR_DEV_BAD_REQ : OSCAR_DEV_BAD_LEN;
            slot = -1;
        }
        if (bits && lane == 0) set_status(P.status, bits);
        if (slot < 0) continue;
#pragma unroll
        for (int j = 0; j < CPL; ++j) sx[warp][lane * CPL + j] = x[j];
        __syncwarp();
        // ---- y = x · R, sequential over k ----
        float y[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) y[j] = 0.f;
#pragma unroll 8
        for (int k = 0; k < D; ++k) {
            const float xk = sx[warp][k];
            const float* rr = Rs + (int64_t)k * D + lane * CPL;
#pragma unroll
            for (int j = 0; j < CPL; ++j) y[j] = fmaf(xk, rr[j], y[j]);
        }
        __syncwarp();
        const float eb = fma_chain_bound<D>(warp_sum_sq<CPL>(x));
        const float* xw = sx[warp];
        quantize_store<D>(P, y, slot, h, mat, lane, eb, [&](int k) { return xw[k]; }, Rs);
        __syncwarp();   // sx[warp] is rewritten by the warp's next vector
    }
}


// Decode-step appends at d = 256, where R (256 KB) does not fit the shared-memory
// staging: one block of D threads per head vector, thread c forming output
// channel c with the same sequential fp32 FMA order over k as the other
// kernels (bit-identical y).  A warp reads rows of R as coalesced 128-byte
// lines, 32 of them in flight, and the few vectors of a decode step spread
// over as many SMs, instead of a warp streaming all of R for its vector.
template <int D>
__global__ void __launch_bounds__(D, 2)   // a minimum residency, so that the 32 loads stay in flight
quantize_vec_kernel(AppendParams P) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    constexpr int CPL = D / 32;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float sx[D];
    __shared__ float sy[D];
    int* prefix = reinterpret_cast<int*>(smem);
    int* scratch = prefix + P.batch + 1;
    const int mat = blockIdx.y;
    const float* R = mat ? P.rot_v : P.rot_k;
    const void* src_new = mat ? P.v : P.k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    build_prefix(P, prefix, scratch);
    const int64_t total_vec = (int64_t)prefix[P.batch] * P.Hkv;
    for (int64_t e = blockIdx.x; e < total_vec; e += gridDim.x) {
        // ---- resolve the vector (every thread, block-uniform) ----
        const int u = (int)(e / P.Hkv), h = (int)(e % P.Hkv);
        const int b = find_request(prefix, P.batch, u);
        const int L0 = P.start_pos[b];
        const int p = hist_hi(L0, P.S, P.W) + (u - prefix[b]);
        const int rq = P.req_idx ? P.req_idx[b] : b;
        const int64_t t = (int64_t)P.cu_new[b] + (p - L0);
        const bool from_ring = p < L0;
        const bool src_ok = from_ring ? (rq >= 0 && rq < P.max_reqs) : (t < P.total_new);
        // x (bf16-rounded), channel tid, loaded in the page-table entry's round
        float x = 0.f;
        if (src_ok) {
            if (from_ring)
                x = bf16_bits_to_f32(P.recent[((((int64_t)rq * P.W + p % P.W) * P.Hkv + h) * 2 + mat) * D + tid]);
            else
                x = bf16_bits_to_f32(f32_to_bf16_bits(load_elem(src_new, (t * P.Hkv + h) * D + tid, P.kv_dtype)));
        }
        int slot = -1;
        int bits = 0;
        if (p >= P.pt_stride) {
            bits |= OSCAR_DEV_BAD_LEN;
        } else {
            const int sl = P.page_table[(int64_t)b * P.pt_stride + p];
            if (sl < 0 || sl >= P.num_slots) bits |= OSCAR_DEV_BAD_SLOT;
            else slot = sl;
        }
        if (!src_ok) {
            bits |= from_ring ? OSCAR_DEV_BAD_REQ : OSCAR_DEV_BAD_LEN;
            slot = -1;
        }
        if (bits && tid == 0) set_status(P.status, bits);
        if (slot < 0) continue;                    // the same decision in every thread
        sx[tid] = x;
        __syncthreads();
        // ---- y[c] = Σ_k x_k·R[k][c], k sequential ----
        float y = 0.f;
        const float* rc = R + tid;
        for (int k0 = 0; k0 < D; k0 += 32) {      // 32 rows of R in flight, then their FMAs in order
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
        sy[tid] = y;
        __syncthreads();
        if (warp == 0) {                           // lane: channels lane·CPL .. + CPL - 1
            float yv[CPL], xv[CPL];
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                yv[j] = sy[lane * CPL + j];
                xv[j] = sx[lane * CPL + j];
            }
            const float e = fma_chain_bound<D>(warp_sum_sq<CPL>(xv));
            quantize_store<D>(P, yv, slot, h, mat, lane, e, [&](int k) { return sx[k]; }, R);
        }
        __syncthreads();                           // sx and sy are reused by the next vector
    }
}


// d <= 128: one warp per (new token, KV head), R staged in shared memory.
template <int D>
__global__ void __launch_bounds__(kAppendThreads)
append_step_kernel(AppendParams P) {
    static_assert(D * D * 4 <= 64 * 1024, "R staged in shared memory");
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ float sx[kSmallVec][D];
    float* sR = reinterpret_cast<float*>(smem);
    constexpr int CPL = D / 32;
    const int mat = blockIdx.y;
    const float* R = mat ? P.rot_v : P.rot_k;
    const void* src_new = mat ? P.v : P.k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // R is no kernel's output, so its staging may start while the previous grid
    // of the stream drains; everything else waits for that grid
    constexpr int NU = D * D / 4 / kAppendThreads;   // 16-byte copies of R per thread
#pragma unroll
    for (int u = 0; u < NU; ++u)
        cp_async16(sR + 4 * (tid + kAppendThreads * u), R + 4 * (tid + kAppendThreads * u));
    cp_async_commit();
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    cp_async_wait<0>();
    __syncthreads();
    const int64_t total = P.total_new * P.Hkv;
    for (int64_t e = (int64_t)blockIdx.x * kSmallVec + warp; e < total; e += (int64_t)gridDim.x * kSmallVec) {
        const int64_t t = e / P.Hkv;
        const int h = (int)(e % P.Hkv);
        int b, p, rq, bits;
        const bool ok = resolve_new_row(P, t, b, p, rq, bits);
        const int q = p - P.W;                       // the position leaving the window, if any
        const bool spill = ok && q >= P.S;
        int slot = spill ? history_slot(P, b, q, bits) : -1;
        float xs[CPL], xn[CPL];
        if (spill) {
            const uint16_t* row = P.recent + window_row(P, rq, q, h, mat, D) + lane * CPL;
#pragma unroll
            for (int j = 0; j < CPL; ++j) xs[j] = bf16_bits_to_f32(row[j]);
        }
        const int64_t base = (t * P.Hkv + h) * D + lane * CPL;
#pragma unroll
        for (int j = 0; j < CPL; ++j) xn[j] = ok ? load_elem(src_new, base + j, P.kv_dtype) : 0.f;
        if (ok) {   // the new row over the leaving one (this lane read its elements above)
            uint16_t* dst = (p < P.S ? P.sink : P.recent) + window_row(P, rq, p, h, mat, D) + lane * CPL;
#pragma unroll
            for (int j = 0; j < CPL; ++j) dst[j] = f32_to_bf16_bits(xn[j]);
        }
        if (bits && lane == 0) set_status(P.status, bits);
        if (slot < 0) continue;                      // warp-uniform
#pragma unroll
        for (int j = 0; j < CPL; ++j) sx[warp][lane * CPL + j] = xs[j];
        __syncwarp();
        // ---- y = x · R, sequential over k (the order of the other CUDA-core kernels) ----
        float y[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) y[j] = 0.f;
#pragma unroll 8
        for (int k = 0; k < D; ++k) {
            const float xk = sx[warp][k];
            const float* rr = sR + k * D + lane * CPL;
#pragma unroll
            for (int j = 0; j < CPL; ++j) y[j] = fmaf(xk, rr[j], y[j]);
        }
        const float eb = fma_chain_bound<D>(warp_sum_sq<CPL>(xs));
        const float* xw = sx[warp];
        quantize_store<D>(P, y, slot, h, mat, lane, eb, [&](int k) { return xw[k]; }, sR);
        __syncwarp();   // sx[warp] is rewritten by the warp's next item
    }
}

// d = 256 (R does not fit in shared memory): one block of D threads per (new
// token, KV head); thread c owns element c of the rows and output channel c.
template <int D>
__global__ void __launch_bounds__(D, 2)
append_step_vec_kernel(AppendParams P) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    __shared__ float sx[D];
    __shared__ float sy[D];
    const int mat = blockIdx.y;
    const int64_t total = P.total_new * P.Hkv;
    for (int64_t e = blockIdx.x; e < total; e += gridDim.x)
        append_vec_item<D>(P, e / P.Hkv, (int)(e % P.Hkv), mat, sx, sy);
}

// Copies the new rows that land in a BF16 window: positions below S go to the
// sink, positions at or after max(S, L1 - W) to the ring slot p % W; the rows in
// between enter the history and are the quantise kernel's.  Block (b, y)
// takes window rows y, y + gridDim.y, ... of request b (sink rows first), so a
// 32K-token prefill visits its 320 window rows, not all of its rows.  bf16
// inputs on 16-byte boundaries move in 16-byte chunks (8 channels).
template <int D>
__global__ void __launch_bounds__(128)
window_copy_kernel(AppendParams P) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    const int b = blockIdx.x;
    const int L0 = P.start_pos[b];
    const int c0 = P.cu_new[b], c1 = P.cu_new[b + 1];
    const int n = c1 - c0;
    if (L0 < 0 || n <= 0) return;
    const int rq = P.req_idx ? P.req_idx[b] : b;
    if (rq < 0 || rq >= P.max_reqs) {
        if (threadIdx.x == 0 && blockIdx.y == 0) set_status(P.status, OSCAR_DEV_BAD_REQ);
        return;
    }
    const int L1 = L0 + n;
    const int hh = hist_hi(L1, P.S, P.W);
    const int s_end = min(n, max(0, P.S - L0));        // rows [0, s_end): sink
    const int r_beg = min(n, max(s_end, hh - L0));     // rows [r_beg, n): ring
    const int nwin = s_end + (n - r_beg);
    const int nel = P.Hkv * 2 * D;                      // one position: [Hkv][K|V][d]
    const bool vec = P.kv_dtype == OSCAR_DTYPE_BF16 &&
                     ((reinterpret_cast<uintptr_t>(P.k) | reinterpret_cast<uintptr_t>(P.v)) & 15) == 0;
    for (int w = blockIdx.y; w < nwin; w += gridDim.y) {
        const int r = w < s_end ? w : r_beg + (w - s_end);
        const int64_t t = (int64_t)c0 + r;
        if (t >= P.total_new) {
            if (threadIdx.x == 0) set_status(P.status, OSCAR_DEV_BAD_LEN);
            break;
        }
        const int p = L0 + r;
        uint16_t* dst = p < P.S ? P.sink + ((int64_t)rq * P.S + p) * nel
                                : P.recent + ((int64_t)rq * P.W + p % P.W) * nel;
        if (vec) {
            for (int ci = threadIdx.x; ci < nel / 8; ci += blockDim.x) {
                const int h = ci / (D / 4), mat = (ci / (D / 8)) & 1, c8 = ci % (D / 8);
                const uint16_t* src = reinterpret_cast<const uint16_t*>(mat ? P.v : P.k) + (t * P.Hkv + h) * D + 8 * c8;
                *reinterpret_cast<uint4*>(dst + 8 * ci) = *reinterpret_cast<const uint4*>(src);
            }
        } else {
            for (int i = threadIdx.x; i < nel; i += blockDim.x) {
                const int h = i / (2 * D), mat = (i / D) & 1, c = i % D;
                dst[i] = f32_to_bf16_bits(load_elem(mat ? P.v : P.k, (t * P.Hkv + h) * D + c, P.kv_dtype));
            }
        }
    }
}

template <int D>
static int launch_append(const AppendParams& P, int64_t total_new, cudaStream_t stream) {
    constexpr bool kResidentR = (D * D * 4 <= 64 * 1024);
    const int r_cols = kResidentR ? D : kColBlock;
    size_t smem = (size_t)D * r_cols * 4;  // must match the carve-up in quantize_kernel
    const size_t xt = (size_t)D * kTileVec * 4, y = (size_t)kTileVec * (D + 4) * 4;
    smem += xt + y;
    smem += (size_t)(P.batch + 1 + kAppendThreads) * 4;
    auto kern = quantize_kernel<D>;
    if (const int rc_ = ensure_dynamic_smem((const void*)kern, smem, "cudaFuncSetAttribute(quantize_kernel)"))
        return rc_;
    // Upper bound of the vectors entering the history: a request of L0 cached
    // and n new tokens moves max(S, L0+n-W) - max(S, L0-W) <= n positions.
    const int64_t max_units = total_new;
    const int64_t max_tiles = (max_units * P.Hkv + kTileVec - 1) / kTileVec;
    // blockIdx.y selects K or V, so the two halves together fill every SM
    // with its resident CTAs (2 per SM when R stays in shared memory).
    const int per_sm = kResidentR ? 2 : 1;
    const int64_t grid_x = std::max<int64_t>(1, std::min<int64_t>(max_tiles, (int64_t)sm_count() * per_sm / 2));
    const int64_t max_vec = max_units * P.Hkv;
    // at most W new tokens in the call: every new row lands in a window, and the
    // rows leaving the ring are quantised by the same launch (see append_step_kernel)
    const bool step = total_new > 0 && total_new <= P.W &&
                      (D * D * 4 > 64 * 1024 ? max_vec <= 2 * (int64_t)sm_count()
                                             : max_vec <= (int64_t)sm_count() * kTileVec);
    if (step) {
        const int prof = prof_begin(1, stream);
        if constexpr (D * D * 4 > 64 * 1024) {
            launch_dependent(append_step_vec_kernel<D>, dim3((unsigned)max_vec, 2), dim3(D), 0, stream, P);
        } else {
            const size_t ssmem = (size_t)D * D * 4;
            if (const int rc_ = ensure_dynamic_smem((const void*)append_step_kernel<D>, ssmem,
                                                    "cudaFuncSetAttribute(append_step_kernel)"))
                return rc_;
            const int64_t gs = std::min<int64_t>((max_vec + kSmallVec - 1) / kSmallVec, (int64_t)sm_count() * 4);
            launch_dependent(append_step_kernel<D>, dim3((unsigned)gs, 2), dim3(kAppendThreads), ssmem, stream, P);
        }
        prof_end(prof, stream);
        return check_cuda("append_step_kernel launch");
    }
    if (D * D * 4 > 64 * 1024 && max_vec > 0 && max_vec <= 2 * (int64_t)sm_count()) {
        // few vectors with R too large for shared memory (d 256): one block per vector
        const size_t vsmem = (size_t)(P.batch + 1 + D) * 4;
        if (const int rc_ = ensure_dynamic_smem((const void*)quantize_vec_kernel<D>, vsmem,
                                                "cudaFuncSetAttribute(quantize_vec_kernel)"))
            return rc_;
        const int prof = prof_begin(1, stream);
        launch_dependent(quantize_vec_kernel<D>, dim3((unsigned)max_vec, 2), dim3(D), vsmem, stream, P);
        prof_end(prof, stream);
        int rc = check_cuda("quantize_vec_kernel launch");
        if (rc) return rc;
    } else if (max_vec > 0 && max_vec <= (int64_t)sm_count() * kTileVec) {
        // few vectors (decode steps): one warp per vector over many blocks
        const size_t ssmem = (size_t)(P.batch + 1 + kAppendThreads) * 4 + (D * D * 4 <= 64 * 1024 ? D * D * 4 : 0);
        if (const int rc_ = ensure_dynamic_smem((const void*)quantize_small_kernel<D>, ssmem, "cudaFuncSetAttribute(quantize_small_kernel)"))
            return rc_;
        const int64_t gs = std::min<int64_t>((max_vec + kSmallVec - 1) / kSmallVec, (int64_t)sm_count() * 4);
        const int prof = prof_begin(1, stream);
        launch_dependent(quantize_small_kernel<D>, dim3((unsigned)gs, 2), dim3(kAppendThreads), ssmem, stream, P);
        prof_end(prof, stream);
        int rc = check_cuda("quantize_small_kernel launch");
        if (rc) return rc;
    } else if (max_tiles > 0) {
        const int prof = prof_begin(1, stream);
        int rc;
        if constexpr (D <= 128) {
            // large appends, d <= 128: rotation on the tensor cores
            rc = launch_quantize_tc<D>(P, max_vec, stream);
        } else if (P.G <= 128) {
            // d = 256: tensor cores, one half of the output channels per CTA
            rc = launch_quantize_tc256(P, max_vec, stream);
        } else {
            // group 256 spans both halves: fp32 FMA tiles
            launch_dependent(kern, dim3((unsigned)grid_x, 2), dim3(kAppendThreads), smem, stream, P);
            rc = check_cuda("quantize_kernel launch");
        }
        prof_end(prof, stream);
        if (rc) return rc;
    }
    if (total_new > 0) {
        // window rows per request (at most S + W; one per new token for decode
        // steps) are not known on the host: up to one block per window row
        const int64_t win = std::min<int64_t>((int64_t)P.S + P.W, (total_new + P.batch - 1) / P.batch);
        const int64_t gy = std::max<int64_t>(1, win);
        const int prof = prof_begin(2, stream);
        launch_dependent(window_copy_kernel<D>, dim3((unsigned)P.batch, (unsigned)gy), dim3(128), 0, stream, P);
        prof_end(prof, stream);
        int rc = check_cuda("window_copy_kernel launch");
        if (rc) return rc;
    }
    return OSCAR_OK;
}

}  // namespace oscar

using namespace oscar;

extern "C" int oscar_quantize_append(const oscar_config* cfg, const oscar_layer_cache* cache,
                                     const void* k, const void* v, int64_t total_new,
                                     const int32_t* cu_new, const int32_t* start_pos,
                                     const int32_t* req_idx, const int32_t* page_table,
                                     int64_t pt_stride, int32_t batch, void* stream) {
    clear_error();
    int rc = validate_config(cfg);
    if (rc) return rc;
    rc = validate_cache(cfg, cache);
    if (rc) return rc;
    if (batch < 0 || batch > kMaxAppendBatch)
        return fail(OSCAR_ERR_ARG, "batch must be in [0, %d] (got %d)", kMaxAppendBatch, batch);
    if (total_new < 0) return fail(OSCAR_ERR_ARG, "total_new must be >= 0");
    if (batch == 0) return OSCAR_OK;
    if (!cu_new || !start_pos || !page_table) return fail(OSCAR_ERR_NULL, "cu_new, start_pos and page_table are required");
    if (total_new > 0 && (!k || !v)) return fail(OSCAR_ERR_NULL, "k and v are required when total_new > 0");
    if (pt_stride < 1) return fail(OSCAR_ERR_ARG, "pt_stride must be >= 1");
    AppendParams P;
    P.k = k;
    P.v = v;
    P.kv_dtype = cfg->kv_dtype;
    P.cu_new = cu_new;
    P.start_pos = start_pos;
    P.req_idx = req_idx;
    P.page_table = page_table;
    P.pt_stride = pt_stride;
    P.batch = batch;
    P.records = cache->records;
    P.sink = cache->sink;
    P.recent = cache->recent;
    P.rot_k = cache->rot_k;
    P.rot_v = cache->rot_v;
    P.num_slots = cache->num_slots;
    P.max_reqs = cache->max_reqs;
    P.Hkv = cfg->num_kv_heads;
    P.S = cfg->sink;
    P.W = cfg->recent;
    P.G = cfg->group_size;
    const RecordLayout lay = record_layout(cfg->head_dim, cfg->group_size, cfg->scale_dtype);
    P.rec_bytes = lay.bytes;
    P.slot_bytes = slot_bytes(lay, cfg->num_kv_heads);
    P.fp8 = cfg->scale_dtype == OSCAR_SCALE_E4M3;
    P.clip = cfg->clip_ratio;
    P.total_new = total_new;
    P.status = status_word();
    if (!P.status) return OSCAR_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    switch (cfg->head_dim) {
        case 64: return launch_append<64>(P, total_new, st);
        case 128: return launch_append<128>(P, total_new, st);
        default: return launch_append<256>(P, total_new, st);
    }
}
