// Shared device helpers of libshardstep: streaming 16-byte loads and stores,
// bf16 packing, and the per-element AdamW update.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "shardstep.h"

namespace shardstep {

constexpr int kThreads = 256;  // threads per block of every kernel here

// ---------------------------------------------------------------- memory

// Read-only stream, touched once: bypass L1, ask L2 for 256-byte fills.
__device__ __forceinline__ uint4 ld_once(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// 8-byte variant of ld_once.
__device__ __forceinline__ uint2 ld_once8(const void* p) {
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0,%1}, [%2];"
        : "=r"(r.x), "=r"(r.y)
        : "l"(p));
    return r;
}

// Read of data the same thread writes back later in the kernel (coherent
// path).  Each address is read once, before the store that depends on it.
__device__ __forceinline__ uint4 ld_rw(const void* p) {
    uint4 r;
    asm("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Streaming store (evict-first in L2).
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_stream8(void* p, uint2 v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// Streaming (evict-first) accesses through the compiler's own intrinsics:
// unlike volatile asm with a memory clobber, these let the scheduler overlap
// one iteration's stores with the next iteration's loads.
__device__ __forceinline__ uint2 ldcs8(const void* p) {
    return __ldcs(reinterpret_cast<const uint2*>(p));
}
__device__ __forceinline__ uint4 ldcs16(const void* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void stcs8(void* p, uint2 v) { __stcs(reinterpret_cast<uint2*>(p), v); }
__device__ __forceinline__ void stcs16(void* p, uint4 v) { __stcs(reinterpret_cast<uint4*>(p), v); }

// ------------------------------------------------- dependent launches

// Programmatic dependent launch: let the next grid of the stream, if it was
// launched as a dependent, be scheduled once every CTA of this grid has
// started; and wait for the grid this one depends on (if any) to complete
// and its memory to be visible.  Both return at once for ordinary launches.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// The start of a kernel that may be launched as a programmatic dependent of
// whatever kernel precedes it in the stream (the first kernel of a call, see
// launch_after): it waits for the preceding grid to complete, with that
// grid's memory visible, before it touches any memory, and only then lets
// its own dependents be scheduled.  The order matters: a dependent that
// waits only at its end (a later copy of the same call) starts its work as
// soon as every block of this grid has triggered, so triggering before the
// wait would let it read what the predecessor is still writing.  Only the
// launch latency overlaps; for an ordinary launch both return at once.
__device__ __forceinline__ void pdl_enter() {
    pdl_wait();
    pdl_trigger();
}

// ------------------------------------------------------------------- bf16

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Two fp32 -> packed bf16x2 (a in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint16_t f32_to_bf16(float a) {
    __nv_bfloat16 h = __float2bfloat16_rn(a);
    return *reinterpret_cast<uint16_t*>(&h);
}

// 16 bytes of bf16 -> 8 floats.
__device__ __forceinline__ void unpack8(const uint4& r, float* f) {
    f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x);
    f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
    f[4] = bf16_lo(r.z); f[5] = bf16_hi(r.z);
    f[6] = bf16_lo(r.w); f[7] = bf16_hi(r.w);
}
__device__ __forceinline__ void unpack4f(const uint4& r, float* f) {
    f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
}
__device__ __forceinline__ uint4 pack4f(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
}

// ------------------------------------------------------------- arithmetic

// Reduction of rank slices in the fixed order the method uses: slices arrive
// in rank order; every `group` consecutive slices are summed first, then the
// group sums are added in order.  With group == N_d this is the plain
// left-to-right rank-order sum (the compare below never fires).
template <int W>
struct GroupSum {
    float s[W], tot[W];
    int c;
    bool have;
    __device__ __forceinline__ void first(const float* t) {
#pragma unroll
        for (int k = 0; k < W; ++k) s[k] = t[k];
        c = 1;
        have = false;
    }
    __device__ __forceinline__ void add(const float* t, int group) {
        if (c == group) {
#pragma unroll
            for (int k = 0; k < W; ++k) {
                tot[k] = have ? __fadd_rn(tot[k], s[k]) : s[k];
                s[k] = t[k];
            }
            have = true;
            c = 1;
        } else {
#pragma unroll
            for (int k = 0; k < W; ++k) s[k] = __fadd_rn(s[k], t[k]);
            ++c;
        }
    }
    __device__ __forceinline__ void result(float* g) const {
#pragma unroll
        for (int k = 0; k < W; ++k) g[k] = have ? __fadd_rn(tot[k], s[k]) : s[k];
    }
};

// x / N_d, correctly rounded (the same bits as IEEE division).  A power of
// two multiplies by its exact reciprocal.  Any other N_d is divided with
// Markstein's correction step (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990), the divisor being known in advance: with r = RN(1/N_d) from the
// host, q0 = RN(x * r) is within one ulp of x / N_d, the residual
// x - q0 * N_d is exact in one fma (N_d is a small integer, so it fits in a
// few bits above q0's last place), and RN(q0 + residual * r) is the
// correctly rounded quotient.  Those exactness arguments need q0 and the
// residual well inside the normal range, so a sum whose biased exponent is
// below kDivFastMinExp (zero, subnormals, |x| < 2^-63) or 255 (inf, NaN)
// takes the IEEE division instead.  shardstep_check_mean_division compares
// this with IEEE division on all 2^32 fp32 inputs, for every N_d.
constexpr uint32_t kDivFastMinExp = 64u;
__device__ __forceinline__ float div_nd(float x, const MeanOp& mo) {
    if (mo.pow2) return __fmul_rn(x, mo.inv_nd);
    const uint32_t ex = (__float_as_uint(x) >> 23) & 0xFFu;
    if (ex >= kDivFastMinExp && ex != 0xFFu) {
        const float q0 = __fmul_rn(x, mo.inv_nd);
        const float res = __fmaf_rn(-q0, mo.nd, x);
        return __fmaf_rn(res, mo.inv_nd, q0);
    }
    return __fdiv_rn(x, mo.nd);
}

__device__ __forceinline__ float mean_of(float sum, const MeanOp& mo) {
    const float g = div_nd(sum, mo);
    return mo.scaled ? __fmul_rn(g, mo.inv_scale) : g;
}

// Reads the loss scale of a scaled reduction: inv_scale = 1 / *scale (IEEE
// division, fp32).
__device__ __forceinline__ MeanOp resolve_scale(MeanOp mo) {
    if (mo.scaled) mo.inv_scale = __fdiv_rn(1.0f, __ldcg(mo.scale));
    return mo;
}

// For fp16 slices the scaler's check can be decided on the input bits alone.
// A finite fp16 value is at most 65504 in magnitude, so the fp32 sum of at
// most SHARDSTEP_MAX_ND = 64 of them (in any grouping) stays below 2^22, so
// does the mean, and the mean times inv_scale stays finite while
// |inv_scale| <= 2^100.  An inf or NaN input makes the sum inf or NaN, and
// neither the division by N_d nor the multiplication by any inv_scale makes
// it finite again (inf * 0 is NaN).  So when |inv_scale| <= 2^100 (false for
// a NaN inv_scale) the unscaled mean is non-finite exactly where some slice
// holds an inf or NaN, i.e. an all-ones exponent field: no conversion and
// no arithmetic is needed.
__device__ __forceinline__ bool f16_check_on_bits(const MeanOp& mo) {
    return fabsf(mo.inv_scale) <= 0x1p100f;
}
__device__ __forceinline__ bool f16x2_nonfinite(uint32_t w) {
    return ((w & 0x7C00u) == 0x7C00u) | ((w & 0x7C000000u) == 0x7C000000u);
}
__device__ __forceinline__ bool f16_nonfinite(uint16_t h) { return (h & 0x7C00u) == 0x7C00u; }

// A gradient scaler's skip word: non-zero means this step changes nothing.
__device__ __forceinline__ bool skip_step(const unsigned int* skip) {
    return skip != nullptr && __ldcg(skip) != 0u;
}

// fp16 bits -> fp32 (exact).
__device__ __forceinline__ float f16_to_f32(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

// One AdamW element update, one IEEE rounding per operation, no contraction:
//   p = p - (lr*wd)*p ; m = b1*m + (1-b1)*g ; v = b2*v + ((1-b2)*g)*g ;
//   p = p - ((lr/bc1)*m) / (sqrt(v)/sqrt(bc2) + eps)
// The scalars a kernel computes with: the host's, or those of a device-
// resident step state.  The state's eight floats are read once per block
// (eight lanes of warp 0, through L1) and shared through shared memory: read
// by every thread, the one 32-byte line became a hot spot in L2 that more
// than doubled the 7B-shard step's time.  Every thread of the block must
// call it (it synchronises the block when c.dev is set; c.dev is the same
// for the whole grid).
__device__ __forceinline__ AdamScalars resolve_adam(AdamScalars c) {
    if (c.dev != nullptr) {
        __shared__ float sc[8];
        if (threadIdx.x < 8) sc[threadIdx.x] = __ldg(c.dev + threadIdx.x);
        __syncthreads();
        c.lr_wd = sc[0];
        c.beta1 = sc[1];
        c.omb1 = sc[2];
        c.beta2 = sc[3];
        c.omb2 = sc[4];
        c.step_size = sc[5];
        c.sqrt_bc2 = sc[6];
        c.eps = sc[7];
    }
    return c;
}

__device__ __forceinline__ void adamw_elem(float g, float& p, float& m, float& v,
                                           const AdamScalars& c) {
    p = __fsub_rn(p, __fmul_rn(c.lr_wd, p));
    m = __fadd_rn(__fmul_rn(c.beta1, m), __fmul_rn(c.omb1, g));
    v = __fadd_rn(__fmul_rn(c.beta2, v), __fmul_rn(__fmul_rn(c.omb2, g), g));
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), c.sqrt_bc2), c.eps);
    p = __fsub_rn(p, __fdiv_rn(__fmul_rn(c.step_size, m), den));
}

}  // namespace shardstep
