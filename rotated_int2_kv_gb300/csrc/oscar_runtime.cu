// Runtime helpers of liboscar.so: the per-device status word written by the
// kernels' bounds checks, the SM count used to size persistent grids, and the
// mapping of CUDA runtime errors to OSCAR_ERR_CUDA.
#include <atomic>
#include <mutex>
#include <unordered_map>

#include <cuda_runtime.h>

#include "oscar_internal.h"
#include "oscar_device.cuh"

namespace oscar {

// OR of OSCAR_DEV_* bits; one instance per device (module-scope variable).
__device__ int g_status_word;

static constexpr int kMaxDevices = 64;
// SM count per device (a property of the device, not of a context); written
// with relaxed atomics, so threads making their first call concurrently race
// only to store the same value.
static std::atomic<int> g_sm_count[kMaxDevices];
// Largest dynamic shared memory a block may opt into, per device (same scheme).
static std::atomic<int> g_max_smem[kMaxDevices];

static int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

// Largest dynamic shared-memory size already granted per (device, kernel): the
// attribute is set only when a launch needs more, not on every call.
int ensure_dynamic_smem(const void* kernel, size_t bytes, const char* what) {
    const int dev = current_device();
    if (dev < 0) return fail(OSCAR_ERR_CUDA, "no current CUDA device");
    static std::mutex mu;
    static std::unordered_map<const void*, size_t> granted[kMaxDevices];
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = granted[dev].find(kernel);
        if (it != granted[dev].end() && it->second >= bytes) return OSCAR_OK;
    }
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return check_cuda(what);
    std::lock_guard<std::mutex> lock(mu);
    size_t& g = granted[dev][kernel];
    if (bytes > g) g = bytes;
    return OSCAR_OK;
}

// Device address of the status word in the current context, asked for on
// every call: the lookup allocates nothing and stays right after a device
// reset reloads the module.
int* status_word() {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess || !p) {
        fail(OSCAR_ERR_CUDA, "cudaGetSymbolAddress(status word): %s", cudaGetErrorString(e));
        return nullptr;
    }
    return static_cast<int*>(p);
}

int sm_count() {
    const int dev = current_device();
    if (dev < 0) {
        fail(OSCAR_ERR_CUDA, "no current CUDA device");
        return 0;
    }
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            fail(OSCAR_ERR_CUDA, "cannot query the SM count");
            return 0;
        }
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

int max_dynamic_smem() {
    const int dev = current_device();
    if (dev < 0) {
        fail(OSCAR_ERR_CUDA, "no current CUDA device");
        return 0;
    }
    int n = g_max_smem[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || n <= 0) {
            fail(OSCAR_ERR_CUDA, "cannot query the shared-memory limit");
            return 0;
        }
        g_max_smem[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

int check_cuda(const char* what) {
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return OSCAR_OK;
    return fail(OSCAR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace oscar

extern "C" int oscar_device_status(int32_t* flags, int32_t clear) {
    using namespace oscar;
    clear_error();
    if (!flags) return fail(OSCAR_ERR_NULL, "flags is NULL");
    int v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int));
    if (e == cudaSuccess && clear) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int));
    }
    if (e != cudaSuccess) return fail(OSCAR_ERR_CUDA, "reading the device status: %s", cudaGetErrorString(e));
    *flags = v;
    return OSCAR_OK;
}

// ---------------------------------------------------------------------------
// Kernel timing for benchmarks: when enabled, the entry points record a CUDA
// event pair around their dominant kernel on the call's stream (kind 0: the
// decode history kernel, kind 1: the append quantise kernel).
// ---------------------------------------------------------------------------
#include <vector>
#include <atomic>
#include <mutex>

namespace oscar {

struct ProfSlot { cudaEvent_t a, b; int kind; };
static std::mutex g_prof_mu;
static uint32_t g_prof_mask = 0;   // bit k: time launches of kind k
static std::vector<ProfSlot> g_prof_slots;
static size_t g_prof_used = 0;

int prof_begin(int kind, cudaStream_t st) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (kind < 0 || kind > 31 || !((g_prof_mask >> kind) & 1u)) return -1;
    if (g_prof_used == g_prof_slots.size()) {
        if (g_prof_slots.size() >= 65536) return -1;
        ProfSlot s;
        if (cudaEventCreate(&s.a) != cudaSuccess) return -1;
        if (cudaEventCreate(&s.b) != cudaSuccess) { cudaEventDestroy(s.a); return -1; }
        g_prof_slots.push_back(s);
    }
    const int idx = (int)g_prof_used++;
    g_prof_slots[idx].kind = kind;
    cudaEventRecord(g_prof_slots[idx].a, st);
    return idx;
}

void prof_end(int idx, cudaStream_t st) {
    if (idx < 0) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    cudaEventRecord(g_prof_slots[idx].b, st);
}

}  // namespace oscar

extern "C" int oscar_profile_enable(int32_t enable) {
    using namespace oscar;
    clear_error();
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_mask = (uint32_t)enable;
    g_prof_used = 0;
    return OSCAR_OK;
}

extern "C" int oscar_profile_read(int32_t kind, double* total_ms, int64_t* launches) {
    using namespace oscar;
    clear_error();
    if (!total_ms || !launches) return fail(OSCAR_ERR_NULL, "outputs must be non-NULL");
    std::lock_guard<std::mutex> lk(g_prof_mu);
    double ms = 0.0;
    int64_t n = 0;
    for (size_t i = 0; i < g_prof_used; ++i) {
        if (g_prof_slots[i].kind != kind) continue;
        float t = 0.f;
        cudaError_t e = cudaEventSynchronize(g_prof_slots[i].b);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&t, g_prof_slots[i].a, g_prof_slots[i].b);
        if (e != cudaSuccess) return fail(OSCAR_ERR_CUDA, "event timing: %s", cudaGetErrorString(e));
        ms += t;
        ++n;
    }
    *total_ms = ms;
    *launches = n;
    return OSCAR_OK;
}

namespace oscar {

// One warp waits (bounded) for phase 0 of an mbarrier that receives its single
// arrival only when `complete` is set.
__global__ void __launch_bounds__(32) selftest_wait_kernel(int* status, long long budget, int complete) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (complete && threadIdx.x == 0) mbar_arrive(&bar);
    __syncwarp();
    long long b = budget;
    mbar_wait_bounded(&bar, 0, status, b);
}

}  // namespace oscar

extern "C" int oscar_selftest_bounded_wait(int64_t budget_cycles, int32_t complete, void* stream) {
    using namespace oscar;
    clear_error();
    int* st = status_word();
    if (!st) return OSCAR_ERR_CUDA;
    const long long budget = budget_cycles < 1000 ? 1000 : (budget_cycles > 4000000000LL ? 4000000000LL : budget_cycles);
    selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(st, budget, complete ? 1 : 0);
    return check_cuda("selftest_wait_kernel launch");
}
