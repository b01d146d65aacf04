// Internal declarations shared by the host and CUDA translation units of
// liboscar.so.  Not part of the public ABI (include/oscar.h is).
#pragma once

#include <stdint.h>
#include <stddef.h>

#include <cuda_runtime.h>

#include "oscar.h"

namespace oscar {

// Record geometry of one (slot, KV head) entry of the INT2 pool:
// [K codes d/4][V codes d/4][K (s,z) pairs x d/G][V (s,z) x d/G]; fp16 pairs
// (4 B) padded to 16 bytes, E4M3 pairs (2 B) padded to 8.  A slot holds the
// records of all KV heads back to back (head h at h·bytes), padded to 16.
struct RecordLayout {
    int d, G, ng, pair;
    int k_codes, v_codes, k_sz, v_sz, bytes;
};

inline RecordLayout record_layout(int d, int G, int scale_dtype) {
    RecordLayout r;
    r.d = d;
    r.G = G;
    r.ng = d / G;
    r.pair = scale_dtype == OSCAR_SCALE_E4M3 ? 2 : 4;
    r.k_codes = 0;
    r.v_codes = d / 4;
    r.k_sz = d / 2;
    r.v_sz = d / 2 + r.pair * r.ng;
    const int al = scale_dtype == OSCAR_SCALE_E4M3 ? 8 : 16;
    r.bytes = (d / 2 + 2 * r.pair * r.ng + al - 1) / al * al;
    return r;
}

inline int64_t slot_bytes(const RecordLayout& r, int Hkv) { return ((int64_t)Hkv * r.bytes + 15) / 16 * 16; }

// Thread-local error message; returns `code` for convenient `return fail(...)`.
int fail(int code, const char* fmt, ...);
void clear_error();

// Host-side validation of a layer configuration (sets the error message).
int validate_config(const oscar_config* cfg);
int validate_cache(const oscar_config* cfg, const oscar_layer_cache* cache);

// Per-device address of the device status word (OSCAR_DEV_* bits).
int* status_word();

// Number of SMs of the current device (cached).
int sm_count();
// Largest dynamic shared memory per block (opt-in) of the current device; 0 on error.
int max_dynamic_smem();

// Converts the pending CUDA error (if any) into OSCAR_ERR_CUDA.
int check_cuda(const char* what);
// Sets the kernel's dynamic shared-memory limit to at least `bytes` (once per
// device and size); OSCAR_OK or the CUDA error, reported as `what`.
int ensure_dynamic_smem(const void* kernel, size_t bytes, const char* what);

// Launches `kern` on `st` as a programmatic dependent of the stream's previous
// kernel: the grid may be scheduled while that kernel drains.  Every kernel of
// the library begins with grid_dep_wait() (griddepcontrol.wait) before it
// touches global memory, which waits for the previous grid to complete and its
// writes to be visible, so the relaxed launch changes timing, not results.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Benchmark timing of the dominant kernels (see oscar_profile_enable).
int prof_begin(int kind, cudaStream_t st);   // returns a slot or -1 when disabled
void prof_end(int slot, cudaStream_t st);

}  // namespace oscar
