// Calibration statistics on the device: the query covariance C_Q and the
// score-weighted value covariance C_S that the rotation is built from.
//
// [OSCAR news] "OSCARの違い": the logit error of a rotated, quantised key is
// governed by C_Q = (1/N) Σ_n q_nᵀ q_n, and the output error of a quantised
// value by C_S = (1/N) Vᵀ Sᵀ S V (S the attention scores of the calibration
// queries); R = U·H·P takes U from the eigenvectors of such a covariance.
//
// Both are second moments of rows: C_Q of the query rows, C_S of the rows of
// Y = S·V.  They are accumulated in fp64 on the CUDA cores (every bf16 or fp32
// input is exact in fp64, so each product is exact and only the additions
// round), split over the rows in slices whose partial d×d sums land in the
// workspace and are added in slice order by a second kernel: the result does
// not depend on scheduling.  C is symmetric, so only tile pairs (i <= j) are
// formed and the reduction mirrors them.  Y = S·V is split the same way over
// ranges of keys when its tiles alone would leave SMs idle, the ranges' partial
// Y added in range order.
#include <algorithm>

#include "oscar_internal.h"
#include "oscar_device.cuh"

namespace oscar {

namespace {

constexpr int kCT = 64;           // C tile: 64 × 64 outputs per block
constexpr int kCRows = 32;        // rows staged per step
constexpr int kCThreads = 256;    // 4 × 4 outputs per thread
constexpr int kMaxSplits = 256;
constexpr int64_t kMaxYPartBytes = 64ll << 20;   // partial sums of Y over key ranges, at most

__device__ __forceinline__ double load_act(const void* base, int64_t i, int dtype) {
    if (dtype == OSCAR_DTYPE_BF16) return (double)bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(base)[i]);
    if (dtype == OSCAR_DTYPE_F32) return (double)reinterpret_cast<const float*>(base)[i];
    return reinterpret_cast<const double*>(base)[i];
}

// Upper-triangular tile pair k (row-major over i <= j) of an nt × nt tiling.
__device__ __forceinline__ void tile_pair(int k, int nt, int& ti, int& tj) {
    ti = 0;
    int row = nt;
    while (k >= row) {
        k -= row;
        ++ti;
        --row;
    }
    tj = ti + k;
}

// Partial Σ_rows x_i x_j over rows [r0, r1) of slice blockIdx.y, for tile pair
// blockIdx.x, into part[slice][d][d] (fp64).
__global__ void __launch_bounds__(kCThreads) cov_partial_kernel(const void* x, int dtype, int64_t n, int d,
                                                                int64_t rows_per_slice, double* part) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    __shared__ double sa[kCRows][kCT];
    __shared__ double sb[kCRows][kCT];
    const int nt = (d + kCT - 1) / kCT;
    int ti, tj;
    tile_pair(blockIdx.x, nt, ti, tj);
    const int64_t r0 = (int64_t)blockIdx.y * rows_per_slice;
    const int64_t r1 = min(n, r0 + rows_per_slice);
    const int tid = threadIdx.x;
    const int tr = (tid / 16) * 4, tc = (tid % 16) * 4;   // this thread's 4 × 4 outputs in the tile
    double acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.0;
    for (int64_t rb = r0; rb < r1; rb += kCRows) {
        __syncthreads();
        for (int i = tid; i < kCRows * kCT; i += kCThreads) {
            const int rr = i / kCT, c = i % kCT;
            const int64_t row = rb + rr;
            const int ca = ti * kCT + c, cb = tj * kCT + c;
            sa[rr][c] = (row < r1 && ca < d) ? load_act(x, row * d + ca, dtype) : 0.0;
            sb[rr][c] = (row < r1 && cb < d) ? load_act(x, row * d + cb, dtype) : 0.0;
        }
        __syncthreads();
#pragma unroll 4
        for (int rr = 0; rr < kCRows; ++rr) {
            double va[4], vb[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                va[a] = sa[rr][tr + a];
                vb[a] = sb[rr][tc + a];
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = fma(va[a], vb[b], acc[a][b]);
        }
    }
    double* out = part + (int64_t)blockIdx.y * d * d;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int i = ti * kCT + tr + a;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int j = tj * kCT + tc + b;
            if (i < d && j < d) out[(int64_t)i * d + j] = acc[a][b];
        }
    }
}

// C[i][j] = C[j][i] = (Σ_slices part[s][i][j]) / n for i <= j, slices in order.
__global__ void __launch_bounds__(256) cov_reduce_kernel(const double* part, int nslices, int64_t n, int d,
                                                         double* cov) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= (int64_t)d * d) return;
    const int i = (int)(e / d), j = (int)(e % d);
    const int64_t src = i <= j ? e : (int64_t)j * d + i;     // the upper-triangle element
    double s = 0.0;
    for (int k = 0; k < nslices; ++k) s += part[(int64_t)k * d * d + src];
    cov[e] = s / (double)n;
}

// Y = S·V (fp64 accumulation): one block per 64 × 64 tile of Y and range of
// k_chunk keys (blockIdx.z), written to slab z of Y (n_q × d each); a range past
// n_k writes zeros.
__global__ void __launch_bounds__(kCThreads) score_values_kernel(const float* S, const void* V, int v_dtype,
                                                                 int64_t n_q, int64_t n_k, int d, int64_t k_chunk,
                                                                 double* Y) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    __shared__ double ss[kCT][kCRows + 1];   // S tile: [query][k]
    __shared__ double sv[kCRows][kCT];       // V tile: [k][channel]
    const int64_t q0 = (int64_t)blockIdx.y * kCT;
    const int c0 = blockIdx.x * kCT;
    const int64_t kb = (int64_t)blockIdx.z * k_chunk, ke = min(n_k, kb + k_chunk);
    Y += (int64_t)blockIdx.z * n_q * d;
    const int tid = threadIdx.x;
    const int tr = (tid / 16) * 4, tc = (tid % 16) * 4;
    double acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = 0.0;
    for (int64_t k0 = kb; k0 < ke; k0 += kCRows) {
        __syncthreads();
        for (int i = tid; i < kCT * kCRows; i += kCThreads) {
            const int qq = i / kCRows, kk = i % kCRows;
            const int64_t q = q0 + qq, k = k0 + kk;
            ss[qq][kk] = (q < n_q && k < ke) ? (double)S[q * n_k + k] : 0.0;
            const int kv = i / kCT, c = i % kCT;
            const int64_t k2 = k0 + kv;
            sv[kv][c] = (k2 < ke && c0 + c < d) ? load_act(V, k2 * d + c0 + c, v_dtype) : 0.0;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < kCRows; ++kk) {
            double va[4], vb[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                va[a] = ss[tr + a][kk];
                vb[a] = sv[kk][tc + a];
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) acc[a][b] = fma(va[a], vb[b], acc[a][b]);
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int64_t q = q0 + tr + a;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int c = c0 + tc + b;
            if (q < n_q && c < d) Y[q * d + c] = acc[a][b];
        }
    }
}

// Y[e] = Σ_z part[z][e] over the key ranges, in range order (a fixed summation
// order, so repeated calls agree bit for bit).
__global__ void __launch_bounds__(256) sum_splits_kernel(const double* part, int nsplit, int64_t nel, double* Y) {
    grid_dep_sync();   // previous grid of the stream done (programmatic launch)
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= nel) return;
    double s = part[e];
    for (int z = 1; z < nsplit; ++z) s += part[(int64_t)z * nel + e];
    Y[e] = s;
}

// Key ranges of Y = S·V.  The fp64 FMA rate bounds the product, so every SM
// needs an equal share: when the 64 × 64 tiles of Y alone make less than
// about 16 blocks per SM, the keys are split into ranges (multiples of 32
// keys) until they do, within kMaxYPartBytes of partial sums.
int score_splits(int64_t n_q, int64_t n_k, int d, int nsm) {
    const int64_t tiles = (int64_t)((d + kCT - 1) / kCT) * ((n_q + kCT - 1) / kCT);
    int64_t s = ((int64_t)std::max(1, nsm) * 16 + tiles - 1) / tiles;
    s = std::min<int64_t>(s, (n_k + kCRows - 1) / kCRows);
    s = std::min<int64_t>(s, std::max<int64_t>(1, kMaxYPartBytes / (n_q * d * (int64_t)sizeof(double))));
    return (int)std::max<int64_t>(1, s);
}

// Keys per range for s ranges: a multiple of the 32-key staging step.
int64_t score_chunk(int64_t n_k, int s) {
    const int64_t per = (n_k + s - 1) / s;
    return (per + kCRows - 1) / kCRows * kCRows;
}

size_t aligned256(size_t b) { return (b + 255) / 256 * 256; }

// Blocks of cov_partial_kernel that one SM holds at once (4 at 64 registers
// per thread).
int cov_resident() {
    static const int r = [] {
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, cov_partial_kernel, kCThreads, 0) != cudaSuccess ||
            nb < 1) {
            (void)cudaGetLastError();
            nb = 4;
        }
        return nb;
    }();
    return r;
}

// Row slices of the covariance, at least 32 rows each: tile pairs × slices
// fill the SMs' resident blocks once, rounded down (the fp64 FMA rate bounds
// the kernel, so a block past a whole wave would run alone after it).
int cov_slices(int64_t n, int d, int nsm) {
    const int nt = (d + kCT - 1) / kCT;
    const int pairs = nt * (nt + 1) / 2;
    int64_t s = (int64_t)std::max(1, nsm) * cov_resident() / pairs;
    s = std::min<int64_t>(s, (n + kCRows - 1) / kCRows);
    return (int)std::max<int64_t>(1, std::min<int64_t>(s, kMaxSplits));
}

int validate_dims(int64_t n, int d) {
    if (n < 1 || d < 1 || d > 4096) return fail(OSCAR_ERR_ARG, "need n >= 1 and 1 <= d <= 4096");
    return OSCAR_OK;
}

// Launches the two covariance kernels over x (n × d rows); part: nslices·d·d doubles.
int launch_cov(const void* x, int dtype, int64_t n, int d, double* cov, double* part, int nslices,
               cudaStream_t st) {
    const int nt = (d + kCT - 1) / kCT;
    const int64_t per = (n + nslices - 1) / nslices;
    launch_dependent(cov_partial_kernel, dim3(nt * (nt + 1) / 2, nslices), dim3(kCThreads), 0, st, x, dtype, n, d,
                     per, part);
    if (int rc = check_cuda("cov_partial_kernel launch")) return rc;
    const int64_t nel = (int64_t)d * d;
    launch_dependent(cov_reduce_kernel, dim3((unsigned)((nel + 255) / 256)), dim3(256), 0, st, (const double*)part,
                     nslices, n, d, cov);
    return check_cuda("cov_reduce_kernel launch");
}

}  // namespace

}  // namespace oscar

using namespace oscar;

extern "C" int oscar_covariance_workspace_bytes(int64_t n, int32_t d, size_t* bytes) {
    clear_error();
    if (!bytes) return fail(OSCAR_ERR_NULL, "bytes is NULL");
    if (int rc = validate_dims(n, d)) return rc;
    const int nsm = sm_count();
    if (nsm <= 0) return OSCAR_ERR_CUDA;
    *bytes = (size_t)cov_slices(n, d, nsm) * d * d * sizeof(double);
    return OSCAR_OK;
}

extern "C" int oscar_covariance_device(const void* x, int32_t x_dtype, int64_t n, int32_t d, double* cov,
                                       void* workspace, size_t workspace_bytes, void* stream) {
    clear_error();
    if (!x || !cov) return fail(OSCAR_ERR_NULL, "x and cov are required");
    if (int rc = validate_dims(n, d)) return rc;
    if (x_dtype != OSCAR_DTYPE_BF16 && x_dtype != OSCAR_DTYPE_F32)
        return fail(OSCAR_ERR_ARG, "x_dtype must be OSCAR_DTYPE_BF16 or OSCAR_DTYPE_F32");
    const int nsm = sm_count();
    if (nsm <= 0) return OSCAR_ERR_CUDA;
    const int ns = cov_slices(n, d, nsm);
    const size_t need = (size_t)ns * d * d * sizeof(double);
    if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return fail(OSCAR_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold %zu bytes", need);
    return launch_cov(x, x_dtype, n, d, cov, static_cast<double*>(workspace), ns,
                      reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int oscar_value_covariance_workspace_bytes(int64_t n_q, int64_t n_k, int32_t d, size_t* bytes) {
    clear_error();
    if (!bytes) return fail(OSCAR_ERR_NULL, "bytes is NULL");
    if (n_k < 1) return fail(OSCAR_ERR_ARG, "need n_k >= 1");
    if (int rc = validate_dims(n_q, d)) return rc;
    const int nsm = sm_count();
    if (nsm <= 0) return OSCAR_ERR_CUDA;
    const size_t y = aligned256((size_t)n_q * d * sizeof(double));
    const int sk = score_splits(n_q, n_k, d, nsm);
    *bytes = y + (sk > 1 ? sk * y : 0) + (size_t)cov_slices(n_q, d, nsm) * d * d * sizeof(double);
    return OSCAR_OK;
}

extern "C" int oscar_value_covariance_device(const float* scores, const void* values, int32_t v_dtype, int64_t n_q,
                                             int64_t n_k, int32_t d, double* cov, void* workspace,
                                             size_t workspace_bytes, void* stream) {
    clear_error();
    if (!scores || !values || !cov) return fail(OSCAR_ERR_NULL, "scores, values and cov are required");
    if (n_k < 1) return fail(OSCAR_ERR_ARG, "need n_k >= 1");
    if (int rc = validate_dims(n_q, d)) return rc;
    if (v_dtype != OSCAR_DTYPE_BF16 && v_dtype != OSCAR_DTYPE_F32)
        return fail(OSCAR_ERR_ARG, "v_dtype must be OSCAR_DTYPE_BF16 or OSCAR_DTYPE_F32");
    if (n_q > (int64_t)65535 * kCT) return fail(OSCAR_ERR_ARG, "n_q must be <= %lld", (long long)65535 * kCT);
    const int nsm = sm_count();
    if (nsm <= 0) return OSCAR_ERR_CUDA;
    const int ns = cov_slices(n_q, d, nsm);
    const int sk = score_splits(n_q, n_k, d, nsm);
    const size_t y = aligned256((size_t)n_q * d * sizeof(double));
    const size_t yparts = sk > 1 ? sk * y : 0;
    const size_t need = y + yparts + (size_t)ns * d * d * sizeof(double);
    if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return fail(OSCAR_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold %zu bytes", need);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    double* Y = reinterpret_cast<double*>(ws);
    double* Yp = reinterpret_cast<double*>(ws + y);              // sk slabs of nel doubles (sk > 1)
    double* part = reinterpret_cast<double*>(ws + y + yparts);
    const int64_t nel = n_q * d;
    launch_dependent(score_values_kernel,
                     dim3((unsigned)((d + kCT - 1) / kCT), (unsigned)((n_q + kCT - 1) / kCT), (unsigned)sk),
                     dim3(kCThreads), 0, st, scores, values, v_dtype, n_q, n_k, (int)d, score_chunk(n_k, sk),
                     sk > 1 ? Yp : Y);
    if (int rc = check_cuda("score_values_kernel launch")) return rc;
    if (sk > 1) {
        // slab z of the partial sums starts nel doubles after slab z - 1 (sk·nel·8 <= yparts bytes)
        launch_dependent(sum_splits_kernel, dim3((unsigned)((nel + 255) / 256)), dim3(256), 0, st, (const double*)Yp,
                         sk, nel, Y);
        if (int rc = check_cuda("sum_splits_kernel launch")) return rc;
    }
    return launch_cov(Y, 2 /* fp64 rows */, n_q, d, cov, part, ns, st);
}
