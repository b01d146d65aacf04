// Tensor-core (mma.sync m16n8k16) history kernel: placeholder until written.
#include "oscar_internal.h"
#include "oscar_device.cuh"
#include "oscar_decode_common.cuh"

namespace oscar {
int launch_history_mma(const DecodeParams& P, int head_dim, cudaStream_t st, bool* launched) {
    (void)P; (void)head_dim; (void)st;
    *launched = false;
    return OSCAR_OK;
}
}  // namespace oscar
