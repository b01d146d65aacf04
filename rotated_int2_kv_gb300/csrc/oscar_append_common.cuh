// Shared declarations of the append kernels (quantise-on-append).
#pragma once

#include "oscar_internal.h"
#include "oscar_device.cuh"

namespace oscar {

constexpr int kMaxAppendBatch = 4096;
constexpr int kTileVec = 64;        // head vectors per tile (one matrix: K or V)
constexpr int kColBlock = 64;       // columns of R per GEMM pass
constexpr int kAppendThreads = 256;

struct AppendParams {
    const void* k;
    const void* v;
    int kv_dtype;
    const int32_t* cu_new;
    const int32_t* start_pos;
    const int32_t* req_idx;
    const int32_t* page_table;
    int64_t pt_stride;
    int batch;
    uint8_t* records;
    uint16_t* sink;
    uint16_t* recent;
    const float* rot_k;
    const float* rot_v;
    int64_t num_slots;
    int max_reqs;
    int Hkv, S, W, G, rec_bytes;
    float clip;
    int64_t total_new;
    int* status;
};

__device__ __forceinline__ int hist_hi(int L, int S, int W) { return max(S, L - W); }

// Exclusive prefix over requests of the number of positions entering the
// history; prefix[batch] is the total.  All threads of the block participate.
__device__ __forceinline__ void build_prefix(const AppendParams& P, int* prefix, int* scratch) {
    const int tid = threadIdx.x;
    const int per = (P.batch + blockDim.x - 1) / blockDim.x;
    const int b0 = min(P.batch, tid * per), b1 = min(P.batch, b0 + per);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
        const int L0 = P.start_pos[b];
        const int n = P.cu_new[b + 1] - P.cu_new[b];
        int cnt = 0;
        if (L0 < 0 || n < 0) {
            set_status(P.status, OSCAR_DEV_BAD_LEN);
        } else {
            cnt = hist_hi(L0 + n, P.S, P.W) - hist_hi(L0, P.S, P.W);
        }
        prefix[b] = cnt;  // temporarily the count
        local += cnt;
    }
    int total;
    int run = block_exclusive_scan(local, scratch, &total);
    for (int b = b0; b < b1; ++b) {
        const int c = prefix[b];
        prefix[b] = run;
        run += c;
    }
    if (tid == 0) prefix[P.batch] = total;
    __syncthreads();
}

// Largest b with prefix[b] <= u (prefix non-decreasing, prefix[0] = 0).
__device__ __forceinline__ int find_request(const int* prefix, int batch, int u) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Tensor-core rotation + quantisation of large appends (head_dim 64 or 128);
// returns OSCAR_OK after launching, or a negative status.
template <int D>
int launch_quantize_tc(const AppendParams& P, int64_t max_vec, cudaStream_t stream);

}  // namespace oscar
