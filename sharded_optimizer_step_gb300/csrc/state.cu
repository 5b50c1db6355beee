// The device-resident AdamW step state (shardstep_adamw_state_t): a
// one-thread kernel that sets it to a given step and one that advances it by
// a step, deriving the step's fp32 scalars on the device with the double
// operations the host uses for the same step.  The fused kernels read the
// scalars at their start (resolve_adam).
#include "common.cuh"

namespace shardstep {
namespace {

// Step t's fp32 scalars from the powers beta1^t, beta2^t, in AdamScalars'
// field order: every value formed in double (IEEE round to nearest) and
// rounded once to fp32, the operations the host performs for hp->step = t.
__device__ void derive_adam_scalars(float* out, double b1p, double b2p, double lr, double beta1,
                                    double beta2, double eps, double wd) {
    out[0] = __double2float_rn(__dmul_rn(lr, wd));
    out[1] = __double2float_rn(beta1);
    out[2] = __double2float_rn(__dsub_rn(1.0, beta1));
    out[3] = __double2float_rn(beta2);
    out[4] = __double2float_rn(__dsub_rn(1.0, beta2));
    out[5] = __double2float_rn(__ddiv_rn(lr, __dsub_rn(1.0, b1p)));
    out[6] = __double2float_rn(__dsqrt_rn(__dsub_rn(1.0, b2p)));
    out[7] = __double2float_rn(eps);
}

__global__ void adamw_state_set_kernel(shardstep_adamw_state_t* st, int64_t step, double b1p,
                                       double b2p, double lr, double beta1, double beta2,
                                       double eps, double wd) {
    pdl_enter();
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    st->step = step;
    st->beta1_pow = b1p;
    st->beta2_pow = b2p;
    if (step >= 1) {
        derive_adam_scalars(st->scalars, b1p, b2p, lr, beta1, beta2, eps, wd);
    } else {
        for (int k = 0; k < 8; ++k) st->scalars[k] = 0.0f;
    }
}

// t -> t + 1: each power times its beta (the next factor of the host's
// running product), then step t + 1's scalars; nothing when *skip is set.
__global__ void adamw_state_advance_kernel(shardstep_adamw_state_t* st, double lr, double beta1,
                                           double beta2, double eps, double wd,
                                           const unsigned int* skip) {
    pdl_enter();
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    if (skip_step(skip)) return;
    const double b1p = __dmul_rn(st->beta1_pow, beta1);
    const double b2p = __dmul_rn(st->beta2_pow, beta2);
    st->step += 1;
    st->beta1_pow = b1p;
    st->beta2_pow = b2p;
    derive_adam_scalars(st->scalars, b1p, b2p, lr, beta1, beta2, eps, wd);
}

}  // namespace

cudaError_t launch_adamw_state_set(shardstep_adamw_state_t* state, int64_t step, double b1p,
                                   double b2p, double lr, double beta1, double beta2, double eps,
                                   double wd, cudaStream_t stream) {
    const cudaError_t e = launch_after(adamw_state_set_kernel, dim3(1), dim3(32), 0, stream,
                                       state, step, b1p, b2p, lr, beta1, beta2, eps, wd);
    note_launch();
    return e;
}

cudaError_t launch_adamw_state_advance(shardstep_adamw_state_t* state, double lr, double beta1,
                                       double beta2, double eps, double wd,
                                       const unsigned int* skip, cudaStream_t stream) {
    const cudaError_t e = launch_after(adamw_state_advance_kernel, dim3(1), dim3(32), 0, stream,
                                       state, lr, beta1, beta2, eps, wd, skip);
    note_launch();
    return e;
}

}  // namespace shardstep
