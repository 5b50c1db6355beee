// Internal interface between the host-side C ABI (api.cpp) and the kernel
// translation units.  Plain C++; no device code.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "shardstep.h"

namespace shardstep {

// fp32 per-step scalars of the AdamW update (derived in double, on the host
// or by the state-advance kernel).  With `dev` set, each kernel replaces the
// eight values at its start by the eight floats at dev (the scalars of a
// device-resident step state, in this field order).
struct AdamScalars {
    float lr_wd, beta1, omb1, beta2, omb2, step_size, sqrt_bc2, eps;
    const float* dev;
};
static_assert(offsetof(shardstep_adamw_state_t, scalars) == 24, "state layout");

// The device-resident step state (api.cpp / step.cu): init writes step t's
// powers (and scalars for t >= 1), advance moves t to t + 1.
cudaError_t launch_adamw_state_set(shardstep_adamw_state_t* state, int64_t step, double b1p,
                                   double b2p, double lr, double beta1, double beta2, double eps,
                                   double wd, cudaStream_t stream);
cudaError_t launch_adamw_state_advance(shardstep_adamw_state_t* state, double lr, double beta1,
                                       double beta2, double eps, double wd,
                                       const unsigned int* skip, cudaStream_t stream);

// How the reduce turns the N_d rank slices into a mean: the slices are summed
// in groups of `group` consecutive ranks (group == N_d: one rank-order sum;
// 1 < group < N_d: hybrid sharding, group sums first, then across groups),
// then the total is divided by N_d, correctly rounded (div_nd: a multiply by
// the exact reciprocal when N_d is a power of two, else a multiply by
// inv_nd = RN(1/N_d) and one fma correction).
// With `scaled` set, the mean is then multiplied by inv_scale, the gradient
// scaler's 1/s, which each kernel computes at start from the device word
// *scale (resolve_scale).
struct MeanOp {
    float inv_nd;
    float nd;
    int pow2;
    int group;
    float inv_scale;
    int scaled;
    const float* scale;
};

// Gradient element types the fused kernels read (the C ABI's dtype codes).
constexpr int kGradBF16 = SHARDSTEP_DTYPE_BF16;
constexpr int kGradF32 = SHARDSTEP_DTYPE_F32;
constexpr int kGradF16 = SHARDSTEP_DTYPE_F16;

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

// Byte ranges for the aligned copy: source, destination and size all
// multiples of 16 bytes; cut into chunks of kAlignedChunk bytes, one block
// each.
constexpr int kAlignedChunk = 16384;
struct AlignedSeg {
    const char* src;
    char* dst;
    int64_t bytes;
    int64_t chunk0;  // first chunk index of this range in the launch
};
struct AlignedTable {
    AlignedSeg s[kMaxCopySegs];
    int32_t n;
    int64_t total_chunks;
};

// Launches `kernel` as a programmatic dependent of the previous kernel in
// `stream`: it may start while that kernel drains.  Only for launches whose
// kernel neither reads nor writes anything the previous kernel writes, and
// which wait (pdl_wait) for it before they end.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Whether kernels go out as programmatic dependent launches
// (shardstep_set_dependent_launch; api.cpp).
bool dependent_launches();

// Launches `kernel` as a programmatic dependent of the previous kernel in the
// stream when dependent launches are on, else as an ordinary launch.  The
// kernel must begin with pdl_enter() (it waits for its predecessor before it
// touches memory), so stream order holds whatever the predecessor is.
template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent_launches() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Launch bookkeeping (api.cpp).
void note_launch();
int device_sms();                                   // SMs of the current device (cached)
int resident_blocks(const void* kernel, int threads);  // per SM, cached per kernel

// Launchers (return the CUDA error of the launch).
// `skip` (may be null): a device word; when it holds a non-zero value at
// launch the kernel changes nothing (the gradient scaler's skipped step).
cudaError_t launch_rs_adamw_cast(const PtrTable& tab, int nd, int grad_type, int64_t S,
                                 float* master, float* m, float* v, uint16_t* out,
                                 const AdamScalars& c, const MeanOp& mo,
                                 const unsigned int* skip, bool vec, cudaStream_t stream);
// TMA-staged kernels (step_tma.cu).  Each needs every source 16-byte aligned,
// at least kTmaMinElements elements and two stages in shared memory (the
// *_fits checks: the fused step's stage holds N_d slices + 3 state arrays,
// the all-reduce's and the check's N_d slices).  set_tma_stage_limit fixes
// the stages per launch (0: about 128 KB of tiles in flight per SM; returns
// the previous setting).
bool tma_step_fits(int nd, int grad_type);
bool tma_reduce_fits(int nd, int grad_type);
int set_tma_stage_limit(int stages);
// The TMA-staged kernels' wait limit in ns (0: the default of two seconds);
// read at each launch.  Returns the previous limit.
int64_t set_tma_wait_ns(int64_t ns);
cudaError_t launch_rs_adamw_cast_tma(const PtrTable& tab, int nd, int grad_type, int64_t S,
                                     float* master, float* m, float* v, uint16_t* out,
                                     const AdamScalars& c, const MeanOp& mo,
                                     const unsigned int* skip, cudaStream_t stream);
cudaError_t launch_accumulate_tma(const uint16_t* g, float* acc, int64_t n, float scale,
                                  bool first, cudaStream_t stream);
// pdl: launch as a programmatic dependent of the previous bucket's kernel
// (later buckets of one ddp_bucket_allreduce_avg call).
cudaError_t launch_allreduce_avg_tma(const PtrTable& tab, int nd, int64_t n, uint16_t* out,
                                     const MeanOp& mo, bool pdl, cudaStream_t stream);
cudaError_t launch_nonfinite_check_tma(const PtrTable& tab, int nd, int grad_type, int64_t S,
                                       const MeanOp& mo, unsigned int* found,
                                       cudaStream_t stream);
// Gradient scaler (step.cu): the non-finite check of the unscaled mean and
// the scale update.
cudaError_t launch_nonfinite_check(const PtrTable& tab, int nd, int grad_type, int64_t S,
                                   const MeanOp& mo, unsigned int* found, bool vec,
                                   cudaStream_t stream);
cudaError_t launch_scaler_update(float* scale, int* tracker, unsigned int* found,
                                 float growth, float backoff, int interval, cudaStream_t stream);
cudaError_t read_device_status(unsigned int* status, bool clear);
int device_smem_optin();  // max dynamic shared memory per block (cached)
constexpr int64_t kTmaMinElements = 4096;

cudaError_t launch_allreduce_avg(const PtrTable& tab, int nd, int64_t n, uint16_t* out,
                                 const MeanOp& mo, bool vec, bool pdl, cudaStream_t stream);
// The segments of one FSDP2 step launch (launch_rs_adamw_cast_segs): segment
// s covers local elements [lo[s], lo[s] + n[s]) and reads the N_d slices
// p[po[s] + q] (po[s] < 0: padding rows, every contribution +0, no
// pointers); b0[s] is its first block, b0[ns] the launch's block count.
// About 2.9 KB as a kernel parameter.
constexpr int kSegMax = 32;
constexpr int kSegPtrMax = 256;
struct SegTable {
    const void* p[kSegPtrMax];
    int64_t lo[kSegMax];
    int64_t n[kSegMax];
    int64_t b0[kSegMax + 1];
    int32_t po[kSegMax];
    int ns;
};
// Blocks one segment of n elements takes in launch_rs_adamw_cast_segs.
int64_t seg_blocks(int64_t n);
// One launch over the table's segments: the fused step's reduce (rank
// order), mean, AdamW and cast; every segment 16-byte aligned in the state
// and 8-byte (16-bit slices) or 16-byte (fp32 slices) in its slices.
cudaError_t launch_rs_adamw_cast_segs(const SegTable& st, int nd, int grad_type, float* master,
                                      float* m, float* v, uint16_t* out, const AdamScalars& c,
                                      const MeanOp& mo, cudaStream_t stream);
// AdamW with a zero gradient over n elements (FSDP2 padding rows).
cudaError_t launch_adamw_zero_grad(int64_t n, float* master, float* m, float* v, uint16_t* out,
                                   const AdamScalars& c, cudaStream_t stream);
// The DDP all-reduce average fused with the replicated AdamW + cast over n
// bucketed elements (step.cu); mean_out may be null.  `vec`: state 16-byte,
// gradients, mean_out and out 8-byte aligned.
cudaError_t launch_ddp_allreduce_adamw_cast(const PtrTable& tab, int nd, int64_t n,
                                            uint16_t* mean_out, float* master, float* m,
                                            float* v, uint16_t* out, const AdamScalars& c,
                                            const MeanOp& mo, bool vec, cudaStream_t stream);
// Division self-check (step.cu): counts into *mismatches the fp32 patterns
// for which the reduce's division by N_d differs from IEEE division and
// lowers *first_bad to the smallest of them.
cudaError_t launch_mean_division_check(const MeanOp& mo, unsigned long long* mismatches,
                                       unsigned int* first_bad, cudaStream_t stream);
// The copy launchers' `pdl`: launch as a programmatic dependent of the
// previous kernel in the stream.  `wait_first`: the kernel waits for that
// predecessor before it touches memory (the first launch of a call, whose
// predecessor is unknown); without it the kernel waits only before it ends
// (a later launch of the same batch of disjoint copies, so that it overlaps
// the previous one's drain; the batch's last kernel still completes after
// all of them).
cudaError_t launch_copy(const CopyTable& t, bool pdl, bool wait_first, cudaStream_t stream);
// Aligned copy (copy.cu): one block per 16 KB chunk of 16-byte vectors.
cudaError_t launch_copy16(const AlignedTable& t, bool pdl, bool wait_first, cudaStream_t stream);
// Realigning copy (copy.cu): like copy16, but every source starts 1..15
// bytes past a 16-byte boundary (destinations and sizes 16-byte multiples).
cudaError_t launch_copy16_shift(const AlignedTable& t, bool pdl, bool wait_first,
                                cudaStream_t stream);
cudaError_t launch_accumulate(const uint16_t* g, float* acc, int64_t n, float scale, bool first,
                              bool vec, cudaStream_t stream);
// The last micro-batch's accumulation fused into the step (accum_step.cu):
// fp32 accumulator slices `acc`, bf16 last micro-batch slices `last`; `vec`:
// accumulators and state 16-byte aligned, bf16 slices and output 8-byte.
cudaError_t launch_accum_rs_adamw_cast(const PtrTable& acc, const PtrTable& last, int nd,
                                       int64_t S, float scale, float* master, float* m,
                                       float* v, uint16_t* out, const AdamScalars& c,
                                       const MeanOp& mo, bool vec, cudaStream_t stream);

}  // namespace shardstep
