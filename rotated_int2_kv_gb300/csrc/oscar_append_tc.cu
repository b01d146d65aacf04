// Tensor-core rotation and quantisation of large appends (prefill chunks).
//
// [OSCAR news] "OSCARの違い" / "サービングシステム：混合精度キャッシュレイアウト":
// every head vector entering the INT2 history is rotated, y = x·R, then
// clipped and quantised per group (lo = r·min, hi = r·max, s = fp16((hi-lo)/3),
// z = fp16(lo), c = clamp(rint((y-z)/s), 0, 3)).
//
// y = x·R is a dense (vectors × d) · (d × d) contraction, so it runs on the
// tensor cores with mma.sync.m16n8k16 in bf16: x is exactly bf16 (every input
// is rounded to bf16 first), and R (fp32) is split into three bf16 parts
// hi + mid + lo, which hold its 24-bit significand.  Products are exact; for
// every k-step of 16 channels the three parts are chained from lo to hi from a
// zero accumulator, and the k-steps are summed in fp32 registers (round to
// nearest).  Measured against the exact product this is more accurate than a
// sequential fp32 FMA chain, which matters because a code decided near a
// rounding boundary must agree with the oracle.  The quantisation then uses
// the same IEEE fp32 operations as the CUDA-core kernels.
//
// One CTA of 8 warps takes tiles of 128 vectors of one matrix (K or V:
// blockIdx.y); warp w owns vectors 16w .. 16w+15 of the tile and all d output
// channels, so a group's min / max is a reduction over its own registers and 4
// lanes.  The B fragments of the three parts of R are built once per CTA in
// shared memory.
#include <algorithm>

#include "oscar_append_common.cuh"

namespace oscar {

namespace {

constexpr int kTcVec = 128;          // vectors per tile (8 warps x 16 rows)
constexpr int kTcThreads = 256;

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

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

}  // namespace

template <int D, int G>
__global__ void __launch_bounds__(kTcThreads, 1) quantize_tc_kernel(AppendParams P) {
    constexpr int KS = D / 16;           // k-steps
    constexpr int NTL = D / 8;           // n8 tiles of output channels
    constexpr int XS = D + 8;            // bf16 row stride of the X tile (≡ 4 words mod 32)
    constexpr int CB = D / 4;            // code bytes per vector
    extern __shared__ __align__(16) unsigned char smem[];
    uint2* fragB = reinterpret_cast<uint2*>(smem);                                   // [3][KS][NTL][32]
    uint16_t* sX = reinterpret_cast<uint16_t*>(smem + 3 * KS * NTL * 32 * 8);        // [2][kTcVec][XS]
    uint8_t* sC = reinterpret_cast<uint8_t*>(sX + 2 * kTcVec * XS);                  // [kTcVec][CB]
    int* prefix = reinterpret_cast<int*>(sC + kTcVec * CB);                          // batch + 1
    int* scratch = prefix + P.batch + 1;                                              // blockDim.x
    __shared__ int s_meta[2][kTcVec][4];                                              // b, p, h, slot

    const int mat = blockIdx.y;
    const float* R = mat ? P.rot_v : P.rot_k;
    const void* src_new = mat ? P.v : P.k;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = lane >> 2, j = lane & 3;

    build_prefix(P, prefix, scratch);
    const int64_t total_vec = (int64_t)prefix[P.batch] * P.Hkv;
    const int64_t ntiles = (total_vec + kTcVec - 1) / kTcVec;
    if ((int64_t)blockIdx.x >= ntiles) return;

    // B fragments of R's three parts: lane (n, j) of k-step kk, n-tile nt holds
    // (R[16kk+2j][8nt+n], R[16kk+2j+1][8nt+n]) and (R[16kk+2j+8][..], R[16kk+2j+9][..])
    for (int i = tid; i < 3 * KS * NTL * 32; i += kTcThreads) {
        const int ln = i & 31, nt = (i >> 5) % NTL, kk = (i / (32 * NTL)) % KS, p = i / (32 * NTL * KS);
        const int n = ln >> 2, jj = ln & 3;
        const int col = 8 * nt + n, k0 = 16 * kk + 2 * jj;
        const float* Rc = R + col;
        fragB[i] = make_uint2(pack_bf16(bf16_part(Rc[(int64_t)k0 * D], p), bf16_part(Rc[(int64_t)(k0 + 1) * D], p)),
                              pack_bf16(bf16_part(Rc[(int64_t)(k0 + 8) * D], p), bf16_part(Rc[(int64_t)(k0 + 9) * D], p)));
    }
    constexpr int ng = D / G;
    constexpr int lpg = G / 8;           // n-tiles per group
    const float rclip = P.clip;
    // 16-byte loads of the new rows when the input is 16-byte aligned (rows of d
    // elements then stay aligned: d·2 and d·4 bytes are multiples of 16)
    const bool vec_in = (reinterpret_cast<uintptr_t>(src_new) & 15) == 0;
    const int rec_off_codes = mat ? D / 4 : 0;
    const int rec_off_sz = D / 2 + (mat ? 4 * ng : 0);

    // Tiles are pipelined over two buffers: while the warps multiply tile t, the
    // vectors of tile t + gridDim.x are resolved and their rows copied (16-byte
    // cp.async for bf16 sources) into the other buffer.
    auto resolve = [&](int64_t tile, int buf) {
        const int64_t e0 = tile * kTcVec;
        const int nvec = (int)(total_vec - e0 < kTcVec ? total_vec - e0 : kTcVec);
        if (tid < kTcVec) {
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
                    const int sl = P.page_table[(int64_t)b * P.pt_stride + p];
                    if (sl < 0 || sl >= P.num_slots) set_status(P.status, OSCAR_DEV_BAD_SLOT);
                    else slot = sl;
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
            s_meta[buf][tid][0] = b;
            s_meta[buf][tid][1] = p;
            s_meta[buf][tid][2] = h;
            s_meta[buf][tid][3] = slot;
        }
    };
    auto gather = [&](int64_t tile, int buf) {
        const int64_t e0 = tile * kTcVec;
        const int nvec = (int)(total_vec - e0 < kTcVec ? total_vec - e0 : kTcVec);
        uint16_t* xb = sX + buf * kTcVec * XS;
        for (int idx = tid; idx < kTcVec * (D / 8); idx += kTcThreads) {
            const int v = idx / (D / 8), c8 = idx % (D / 8);
            uint32_t* dst = reinterpret_cast<uint32_t*>(xb + v * XS + c8 * 8);   // 16-byte aligned: XS·2 ≡ 0 mod 16
            if (v < nvec && s_meta[buf][v][3] >= 0) {
                const int b = s_meta[buf][v][0], p = s_meta[buf][v][1], h = s_meta[buf][v][2];
                const int L0 = P.start_pos[b];
                if (p < L0) {
                    const int rq = P.req_idx ? P.req_idx[b] : b;
                    const uint16_t* rowp = P.recent + ((((int64_t)rq * P.W + p % P.W) * P.Hkv + h) * 2 + mat) * D;
                    cp_async16(dst, rowp + c8 * 8);
                } else {
                    const int64_t t = P.cu_new[b] + (p - L0);
                    const int64_t base = (t * P.Hkv + h) * D + c8 * 8;
                    if (vec_in && P.kv_dtype == OSCAR_DTYPE_BF16) {
                        cp_async16(dst, reinterpret_cast<const uint16_t*>(src_new) + base);
                    } else if (vec_in) {
                        const float4 f0 = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src_new) + base);
                        const float4 f1 = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src_new) + base + 4);
                        *reinterpret_cast<uint4*>(dst) =
                            make_uint4(pack_bf16(f0.x, f0.y), pack_bf16(f0.z, f0.w), pack_bf16(f1.x, f1.y), pack_bf16(f1.z, f1.w));
                    } else {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = (uint32_t)f32_to_bf16_bits(load_elem(src_new, base + 2 * e, P.kv_dtype)) |
                                   ((uint32_t)f32_to_bf16_bits(load_elem(src_new, base + 2 * e + 1, P.kv_dtype)) << 16);
                        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            } else {
                *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        cp_async_commit();
    };
    int buf = 0;
    resolve(blockIdx.x, 0);
    __syncthreads();
    gather(blockIdx.x, 0);
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, buf ^= 1) {
        const int64_t e0 = tile * kTcVec;
        const int nvec = (int)(total_vec - e0 < kTcVec ? total_vec - e0 : kTcVec);
        const int64_t nxt = tile + gridDim.x;
        if (nxt < ntiles) resolve(nxt, buf ^ 1);
        cp_async_wait<0>();
        __syncthreads();                 // tile's rows landed; next tile's vectors resolved
        if (nxt < ntiles) gather(nxt, buf ^ 1);
        const uint16_t* sXb = sX + buf * kTcVec * XS;
        int (*meta)[4] = s_meta[buf];
        // ---- y = x·R for rows 16·warp .. +15: per k-step the parts lo, mid, hi ----
        const int row0 = 16 * warp;
        uint32_t a[KS][4];
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            const uint32_t* x0 = reinterpret_cast<const uint32_t*>(sXb + (row0 + r) * XS + 16 * kk);
            const uint32_t* x8 = reinterpret_cast<const uint32_t*>(sXb + (row0 + r + 8) * XS + 16 * kk);
            a[kk][0] = x0[j];
            a[kk][1] = x8[j];
            a[kk][2] = x0[j + 4];
            a[kk][3] = x8[j + 4];
        }
        // one group of output channels at a time keeps only its G/8 n-tiles live
        const int v0 = row0 + r;
        const int slot0 = v0 < nvec ? meta[v0][3] : -1;
        const int slot1 = v0 + 8 < nvec ? meta[v0 + 8][3] : -1;
#pragma unroll 1
        for (int gi = 0; gi < ng; ++gi) {
            float y[lpg][4];
#pragma unroll
            for (int t = 0; t < lpg; ++t) {
                const int nt = gi * lpg + t;
#pragma unroll
                for (int e = 0; e < 4; ++e) y[t][e] = 0.f;
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int p = 2; p >= 0; --p) {
                        const uint2 bb = fragB[((p * KS + kk) * NTL + nt) * 32 + lane];
                        mma_bf16(d, a[kk][0], a[kk][1], a[kk][2], a[kk][3], bb.x, bb.y);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) y[t][e] += d[e];
                }
            }
            // ---- quantise rows r (values y[.][0..1]) and r + 8 (y[.][2..3]) ----
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int v = v0 + 8 * hf;
                const int slot = hf ? slot1 : slot0;
                float mn = INFINITY, mx = -INFINITY;
#pragma unroll
                for (int t = 0; t < lpg; ++t) {
                    mn = fminf(mn, fminf(y[t][2 * hf], y[t][2 * hf + 1]));
                    mx = fmaxf(mx, fmaxf(y[t][2 * hf], y[t][2 * hf + 1]));
                }
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 2));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float lo = __fmul_rn(rclip, mn);
                const float hi = __fmul_rn(rclip, mx);
                const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 3.0f));
                const __half z16 = __float2half_rn(lo);
                const float sc = __half2float(s16), zc = __half2float(z16);
#pragma unroll
                for (int t = 0; t < lpg; ++t) {
                    uint32_t nib = 0;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        uint32_t c = 0;
                        if (sc != 0.0f) {
                            const float u = __fdiv_rn(__fsub_rn(y[t][2 * hf + e], zc), sc);
                            c = (uint32_t)fminf(fmaxf(rintf(u), 0.0f), 3.0f);
                        }
                        nib |= c << (2 * e);
                    }
                    // channels 8nt + 2j, +1: bits 4·(j & 1) of byte 2nt + j/2
                    const uint32_t other = __shfl_xor_sync(0xffffffffu, nib, 1);
                    if ((j & 1) == 0) sC[v * CB + 2 * (gi * lpg + t) + (j >> 1)] = (uint8_t)(nib | (other << 4));
                }
                if (j == 0 && slot >= 0) {
                    uint8_t* rec = P.records + ((int64_t)slot * P.Hkv + meta[v][2]) * P.rec_bytes;
                    *reinterpret_cast<__half2*>(rec + rec_off_sz + 4 * gi) = __halves2half2(s16, z16);
                }
            }
        }
        __syncwarp();
        // ---- codes of the warp's 16 rows: 16-byte stores ----
        for (int i = lane; i < 16 * (CB / 16); i += 32) {
            const int v = row0 + i / (CB / 16), q = i % (CB / 16);
            const int slot = v < nvec ? meta[v][3] : -1;
            if (slot >= 0) {
                uint8_t* rec = P.records + ((int64_t)slot * P.Hkv + meta[v][2]) * P.rec_bytes;
                *reinterpret_cast<uint4*>(rec + rec_off_codes + 16 * q) = *reinterpret_cast<const uint4*>(sC + v * CB + 16 * q);
            }
        }
        __syncthreads();
    }
}

template <int D, int G>
static int launch_tc(const AppendParams& P, int64_t max_vec, cudaStream_t stream) {
    constexpr int KS = D / 16, NTL = D / 8, XS = D + 8, CB = D / 4;
    const size_t smem = (size_t)3 * KS * NTL * 32 * 8 + (size_t)2 * kTcVec * XS * 2 + (size_t)kTcVec * CB +
                        (size_t)(P.batch + 1 + kTcThreads) * 4;
    auto kern = quantize_tc_kernel<D, G>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return check_cuda("cudaFuncSetAttribute(quantize_tc_kernel)");
    const int64_t tiles = (max_vec + kTcVec - 1) / kTcVec;
    const int64_t grid_x = std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)sm_count() / 2));
    kern<<<dim3((unsigned)grid_x, 2), kTcThreads, smem, stream>>>(P);
    return check_cuda("quantize_tc_kernel launch");
}

template <int D>
int launch_quantize_tc(const AppendParams& P, int64_t max_vec, cudaStream_t stream) {
    if (P.G == 32) return launch_tc<D, 32>(P, max_vec, stream);
    if (P.G == 64) return launch_tc<D, 64>(P, max_vec, stream);
    if (D >= 128 && P.G == 128) return launch_tc<D, (D >= 128 ? 128 : 64)>(P, max_vec, stream);
    return OSCAR_ERR_ARG;
}

template int launch_quantize_tc<64>(const AppendParams&, int64_t, cudaStream_t);
template int launch_quantize_tc<128>(const AppendParams&, int64_t, cudaStream_t);

}  // namespace oscar
