// Internal interface between the host-side C ABI (api.cpp) and the kernel
// translation units.  Plain C++; no device code.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "shardstep.h"

namespace shardstep {

// fp32 per-step scalars of the AdamW update (derived on the host in double).
struct AdamScalars {
    float lr_wd, beta1, omb1, beta2, omb2, step_size, sqrt_bc2, eps;
};

// How the reduce turns the N_d rank slices into a mean: the slices are summed
// in groups of `group` consecutive ranks (group == N_d: one rank-order sum;
// 1 < group < N_d: hybrid sharding, group sums first, then across groups),
// then the total is multiplied by the exact reciprocal when N_d is a power of
// two (identical to dividing) or divided by N_d.
struct MeanOp {
    float inv_nd;
    float nd;
    int pow2;
    int group;
};

struct PtrTable {
    const void* p[SHARDSTEP_MAX_ND];
};

// One contiguous byte range to copy (src == nullptr: fill with zeros).
constexpr int kMaxCopySegs = 64;
struct CopySeg {
    const char* src;
    char* dst;
    int64_t bytes;
    int64_t chunk0;  // first chunk index of this segment in the launch
    int64_t body;    // vectors of `width` bytes after the head
    int32_t width;   // 16, 8, 4, 2 or 1
    int32_t head;    // bytes before dst is `width`-aligned
};
struct CopyTable {
    CopySeg s[kMaxCopySegs];
    int32_t n;
    int64_t total_chunks;
};
constexpr int kCopyVecsPerChunk = 1024;  // 256 threads x 4

// Launch bookkeeping (api.cpp).
void note_launch();
int device_sms();                                   // SMs of the current device (cached)
int resident_blocks(const void* kernel, int threads);  // per SM, cached per kernel

// Launchers (return the CUDA error of the launch).
cudaError_t launch_rs_adamw_cast(const PtrTable& tab, int nd, bool f32_grads, int64_t S,
                                 float* master, float* m, float* v, uint16_t* out,
                                 const AdamScalars& c, const MeanOp& mo, bool vec,
                                 cudaStream_t stream);
// TMA-staged fused step (step_tma.cu): dynamic shared memory it needs, the
// launch, and the device watchdog status word.
size_t tma_step_smem_bytes(int nd, bool f32_grads);
cudaError_t launch_rs_adamw_cast_tma(const PtrTable& tab, int nd, bool f32_grads, int64_t S,
                                     float* master, float* m, float* v, uint16_t* out,
                                     const AdamScalars& c, const MeanOp& mo,
                                     cudaStream_t stream);
cudaError_t read_device_status(unsigned int* status, bool clear);
int device_smem_optin();  // max dynamic shared memory per block (cached)
constexpr int64_t kTmaMinElements = 4096;

cudaError_t launch_allreduce_avg(const PtrTable& tab, int nd, int64_t n, uint16_t* out,
                                 const MeanOp& mo, bool vec, cudaStream_t stream);
cudaError_t launch_copy(const CopyTable& t, cudaStream_t stream);
cudaError_t launch_accumulate(const uint16_t* g, float* acc, int64_t n, float scale, bool first,
                              bool vec, cudaStream_t stream);

}  // namespace shardstep
