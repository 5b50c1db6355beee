// Register-staged kernels: the fused sharded optimizer step (reduce-scatter
// average + AdamW + bf16 cast in one pass over the shard) for the cases the
// TMA-staged kernel does not take, the DDP bucket all-reduce average, and
// the gradient scaler's non-finite check and scale update.
//
// All are HBM-bound streams: per shard element the fused kernel reads N_d
// gradient slices (2 B each for bf16 / fp16, 4 B for fp32) and the fp32
// master/m/v (12 B), and writes master/m/v (12 B) and the bf16 parameter
// (2 B), each byte touched once.  Each thread owns 4 consecutive elements:
// one 8-byte load per 16-bit slice (16 bytes for fp32 slices), one 16-byte
// load per fp32 state array, every load issued before any arithmetic; all
// accesses are streaming (evict-first) loads and stores.  Blocks of 128
// threads are capped at 64 registers so that 8 of them (32 warps) fit on an
// SM, and the grid covers the whole range in one pass (one 4-element vector
// per thread; the loop only strides if the range needs more than 2^31 - 1
// blocks), so the blocks resident at any time work on neighbouring
// addresses.  Measured on GB300 at 842M elements and N_d = 8: a one-pass grid
// of 512-thread blocks took 4.85 ms where a grid-stride loop over three waves
// of the same blocks took 5.32 ms (same GPU); 128-thread blocks took 1% less
// again, and the TMA-staged kernel 4% more (4.88 vs 5.08 ms, same GPU).
#include "common.cuh"

namespace shardstep {
namespace {

constexpr int kRuntimeND = 0;
constexpr int kStepThreads = 128;  // block of the fused / all-reduce / check kernels
constexpr int kStepMinBlocks = 8;  // 8 x 128 threads per SM -> <= 64 registers

// ----------------------------------------------------------------- loads

template <int GT>
struct GradVec;  // 4 gradient elements of one slice

template <>
struct GradVec<kGradBF16> {
    uint2 r;
    __device__ __forceinline__ void load(const void* base, int64_t i) {
        r = ldcs8(static_cast<const uint16_t*>(base) + 4 * i);
    }
    __device__ __forceinline__ void to_f32(float* f) const {
        f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x);
        f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
    }
};

template <>
struct GradVec<kGradF16> {
    uint2 r;
    __device__ __forceinline__ void load(const void* base, int64_t i) {
        r = ldcs8(static_cast<const uint16_t*>(base) + 4 * i);
    }
    __device__ __forceinline__ void to_f32(float* f) const {
        f[0] = f16_to_f32(static_cast<uint16_t>(r.x & 0xFFFFu));
        f[1] = f16_to_f32(static_cast<uint16_t>(r.x >> 16));
        f[2] = f16_to_f32(static_cast<uint16_t>(r.y & 0xFFFFu));
        f[3] = f16_to_f32(static_cast<uint16_t>(r.y >> 16));
    }
};

template <>
struct GradVec<kGradF32> {
    uint4 a;
    __device__ __forceinline__ void load(const void* base, int64_t i) {
        a = ldcs16(static_cast<const float*>(base) + 4 * i);
    }
    __device__ __forceinline__ void to_f32(float* f) const { unpack4f(a, f); }
};

template <int GT>
__device__ __forceinline__ float grad_scalar(const void* base, int64_t j) {
    if (GT == kGradF32) return static_cast<const float*>(base)[j];
    if (GT == kGradF16) return f16_to_f32(static_cast<const uint16_t*>(base)[j]);
    return bf16_to_f32(static_cast<const uint16_t*>(base)[j]);
}

// Sum of the N_d slices at 4 consecutive elements, in the order GroupSum
// fixes (rank order; grouped for hybrid sharding).
template <int ND, int GT>
__device__ __forceinline__ void reduce4(const PtrTable& tab, int nd, int group, int64_t i,
                                        float* g) {
    GroupSum<4> acc;
    if constexpr (ND < 0) {
        // up to -ND slices, every load in flight at once, the first nd used
        // (N_d = 5 and 7 on the 8-slice kernel: 6.6 and 6.7 TB/s where the
        // loop below moved 5.8 and 6.1 and the TMA-staged kernel 6.2 and 6.5)
        constexpr int NM = -ND;
        GradVec<GT> gv[NM];
#pragma unroll
        for (int q = 0; q < NM; ++q)
            if (q < nd) gv[q].load(tab.p[q], i);
        {
            float t[4];
            gv[0].to_f32(t);
            acc.first(t);
        }
#pragma unroll
        for (int q = 1; q < NM; ++q) {
            if (q < nd) {
                float t[4];
                gv[q].to_f32(t);
                acc.add(t, group);
            }
        }
    } else if constexpr (ND != kRuntimeND) {
        GradVec<GT> gv[ND];
#pragma unroll
        for (int q = 0; q < ND; ++q) gv[q].load(tab.p[q], i);
        {
            float t[4];
            gv[0].to_f32(t);
            acc.first(t);
        }
#pragma unroll
        for (int q = 1; q < ND; ++q) {
            float t[4];
            gv[q].to_f32(t);
            acc.add(t, group);
        }
    } else {
        // any N_d: batches of eight 16-bit slices (four fp32 slices) in
        // flight at a time.  Against batches of four, on GB300 at N_d = 24 /
        // 32 / 64 this moved 6.5 / 6.6 / 6.7 instead of 5.4 / 5.7 / 6.0 TB/s.
        constexpr int B = GT == kGradF32 ? 4 : 8;
        for (int q = 0; q < nd; q += B) {
            const int cnt = nd - q < B ? nd - q : B;
            GradVec<GT> gv[B];
#pragma unroll
            for (int u = 0; u < B; ++u)
                if (u < cnt) gv[u].load(tab.p[q + u], i);
#pragma unroll
            for (int u = 0; u < B; ++u) {
                if (u < cnt) {
                    float t[4];
                    gv[u].to_f32(t);
                    if (q + u == 0) acc.first(t);
                    else acc.add(t, group);
                }
            }
        }
    }
    acc.result(g);
}

// The sum of ND slices already loaded, in reduce4's order.
template <int ND, int GT>
__device__ __forceinline__ void sum_loaded(const GradVec<GT>* gv, int group, float* g) {
    GroupSum<4> acc;
    {
        float t[4];
        gv[0].to_f32(t);
        acc.first(t);
    }
#pragma unroll
    for (int q = 1; q < ND; ++q) {
        float t[4];
        gv[q].to_f32(t);
        acc.add(t, group);
    }
    acc.result(g);
}

// The all-reduce and the check read 2 bytes per slice element, so with one
// vector per thread in flight a thread has only 8 x N_d bytes outstanding:
// at N_d < 8 too little to cover the latency of HBM.  A thread therefore
// issues the loads of light_u<ND>() vectors before summing any of them (at
// least 64 bytes in flight per thread).  On GB300 (200M elements) this took
// the fp16 check at N_d = 1 / 2 / 4 from 1.4 / 2.5 / 6.1 to 5.0 / 6.0 / 6.7
// TB/s and the all-reduce on 25 MiB buckets from 4.7 / 5.2 / 6.0 to 5.8 /
// 6.3 / 6.6 TB/s.
template <int ND>
__host__ __device__ constexpr int light_u() {
    return ND <= 3 ? 4 : 2;
}
template <int ND>
__host__ __device__ constexpr bool light_nd() {
    return ND >= 1 && ND <= 7;
}

template <int GT>
__device__ __forceinline__ float reduce1(const PtrTable& tab, int nd, int group, int64_t j) {
    GroupSum<1> acc;
    float t = grad_scalar<GT>(tab.p[0], j);
    acc.first(&t);
    for (int q = 1; q < nd; ++q) {
        t = grad_scalar<GT>(tab.p[q], j);
        acc.add(&t, group);
    }
    float g;
    acc.result(&g);
    return g;
}

// --------------------------------------------------- fused step kernels

template <int GT>
__device__ __forceinline__ void step_scalar(const PtrTable& tab, int nd, int64_t j,
                                            float* __restrict__ P, float* __restrict__ M,
                                            float* __restrict__ V, uint16_t* __restrict__ out,
                                            const AdamScalars& c, const MeanOp& mo) {
    const float g = mean_of(reduce1<GT>(tab, nd, mo.group, j), mo);
    float p = P[j], m = M[j], v = V[j];
    adamw_elem(g, p, m, v, c);
    P[j] = p;
    M[j] = m;
    V[j] = v;
    out[j] = f32_to_bf16(p);
}

// Aligned operands (16-bit gradient slices and the bf16 output 8-byte
// aligned, fp32 slices and the state 16-byte aligned): 4 elements per thread
// per iteration, then the (< 4 element) tail by block 0.
template <int ND, int GT>
__global__ void __launch_bounds__(kStepThreads, kStepMinBlocks)
    rs_adamw_cast_vec4(PtrTable tab, int nd, int64_t S, float* __restrict__ P,
                       float* __restrict__ M, float* __restrict__ V, uint16_t* __restrict__ out,
                       AdamScalars c, MeanOp mo, const unsigned int* skip) {
    pdl_enter();
    if (skip_step(skip)) return;
    mo = resolve_scale(mo);
    c = resolve_adam(c);
    const int64_t nvec = S >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kStepThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kStepThreads + threadIdx.x; i < nvec;
         i += stride) {
        // all loads of the iteration first
        const uint4 p0 = ldcs16(P + 4 * i);
        const uint4 m0 = ldcs16(M + 4 * i);
        const uint4 v0 = ldcs16(V + 4 * i);
        float g[4];
        reduce4<ND, GT>(tab, nd, mo.group, i, g);
        float p[4], m[4], v[4];
        unpack4f(p0, p);
        unpack4f(m0, m);
        unpack4f(v0, v);
#pragma unroll
        for (int k = 0; k < 4; ++k) adamw_elem(mean_of(g[k], mo), p[k], m[k], v[k], c);
        stcs16(P + 4 * i, pack4f(p));
        stcs16(M + 4 * i, pack4f(m));
        stcs16(V + 4 * i, pack4f(v));
        stcs8(out + 4 * i, make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3])));
    }
    if (blockIdx.x == 0 && threadIdx.x < (S & 3))
        step_scalar<GT>(tab, nd, (nvec << 2) + threadIdx.x, P, M, V, out, c, mo);
}

// Any alignment: one element per thread per iteration.
template <int GT>
__global__ void __launch_bounds__(kThreads)
    rs_adamw_cast_scalar(PtrTable tab, int nd, int64_t S, float* __restrict__ P,
                         float* __restrict__ M, float* __restrict__ V,
                         uint16_t* __restrict__ out, AdamScalars c, MeanOp mo,
                         const unsigned int* skip) {
    pdl_enter();
    if (skip_step(skip)) return;
    c = resolve_adam(c);
    mo = resolve_scale(mo);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < S;
         j += stride)
        step_scalar<GT>(tab, nd, j, P, M, V, out, c, mo);
}

// ------------------------------------- DDP all-reduce avg + AdamW, fused

// The replicated update of DDP in one pass over bucketed elements: the N_d
// bf16 gradients summed in rank order and divided by N_d, the mean rounded
// to bf16 once (the all-reduce keeps the gradient's dtype), optionally
// stored, upcast, then AdamW and the bf16 cast -- the bits of the bucket
// all-reduce followed by the fused step at N_d = 1 on its output.
__device__ __forceinline__ void ddp_elem(float sum, float& p, float& m, float& v,
                                         uint16_t* mean_out, int64_t j, const AdamScalars& c,
                                         const MeanOp& mo) {
    const uint16_t h = f32_to_bf16(mean_of(sum, mo));
    if (mean_out != nullptr) mean_out[j] = h;
    adamw_elem(bf16_to_f32(h), p, m, v, c);
}

template <int ND>
__global__ void __launch_bounds__(kStepThreads, kStepMinBlocks)
    ddp_allreduce_adamw_cast_vec4(PtrTable tab, int nd, int64_t n, uint16_t* __restrict__ mean_out,
                                  float* __restrict__ P, float* __restrict__ M,
                                  float* __restrict__ V, uint16_t* __restrict__ out,
                                  AdamScalars c, MeanOp mo) {
    pdl_enter();
    c = resolve_adam(c);
    const int64_t nvec = n >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kStepThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kStepThreads + threadIdx.x; i < nvec;
         i += stride) {
        const uint4 p0 = ldcs16(P + 4 * i);
        const uint4 m0 = ldcs16(M + 4 * i);
        const uint4 v0 = ldcs16(V + 4 * i);
        float g[4];
        reduce4<ND, kGradBF16>(tab, nd, mo.group, i, g);
        const uint2 h = make_uint2(pack_bf16x2(mean_of(g[0], mo), mean_of(g[1], mo)),
                                   pack_bf16x2(mean_of(g[2], mo), mean_of(g[3], mo)));
        if (mean_out != nullptr) stcs8(mean_out + 4 * i, h);
        g[0] = bf16_lo(h.x);
        g[1] = bf16_hi(h.x);
        g[2] = bf16_lo(h.y);
        g[3] = bf16_hi(h.y);
        float p[4], m[4], v[4];
        unpack4f(p0, p);
        unpack4f(m0, m);
        unpack4f(v0, v);
#pragma unroll
        for (int k = 0; k < 4; ++k) adamw_elem(g[k], p[k], m[k], v[k], c);
        stcs16(P + 4 * i, pack4f(p));
        stcs16(M + 4 * i, pack4f(m));
        stcs16(V + 4 * i, pack4f(v));
        stcs8(out + 4 * i, make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3])));
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
        const int64_t j = (nvec << 2) + threadIdx.x;
        float p = P[j], m = M[j], v = V[j];
        ddp_elem(reduce1<kGradBF16>(tab, nd, mo.group, j), p, m, v, mean_out, j, c, mo);
        P[j] = p;
        M[j] = m;
        V[j] = v;
        out[j] = f32_to_bf16(p);
    }
}

__global__ void __launch_bounds__(kThreads)
    ddp_allreduce_adamw_cast_scalar(PtrTable tab, int nd, int64_t n,
                                    uint16_t* __restrict__ mean_out, float* __restrict__ P,
                                    float* __restrict__ M, float* __restrict__ V,
                                    uint16_t* __restrict__ out, AdamScalars c, MeanOp mo) {
    pdl_enter();
    c = resolve_adam(c);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < n;
         j += stride) {
        float p = P[j], m = M[j], v = V[j];
        ddp_elem(reduce1<kGradBF16>(tab, nd, mo.group, j), p, m, v, mean_out, j, c, mo);
        P[j] = p;
        M[j] = m;
        V[j] = v;
        out[j] = f32_to_bf16(p);
    }
}

// ------------------------------------------------ bucket all-reduce avg

// Both all-reduce kernels may run as programmatic dependents of the previous
// bucket's kernel: they trigger their own dependents at start and wait for
// the grid they depend on before they end (no-ops for ordinary launches).
// The all-reduce and the check move few bytes per 4-element vector (6 B per
// element at N_d = 2), so each block takes `vpt` rows of kStepThreads vectors
// (a contiguous run of vpt x kStepThreads vectors) to keep the rate of block
// launches per SM down; the launcher picks vpt from the bytes per vector.
template <int ND>
__global__ void __launch_bounds__(kStepThreads, kStepMinBlocks)
    allreduce_avg_vec4(PtrTable tab, int nd, int64_t n, uint16_t* __restrict__ out, MeanOp mo,
                       int vpt) {
    pdl_trigger();
    const int64_t nvec = n >> 2;
    const int64_t run = static_cast<int64_t>(kStepThreads) * vpt;
    for (int64_t b0 = static_cast<int64_t>(blockIdx.x) * run; b0 < nvec;
         b0 += static_cast<int64_t>(gridDim.x) * run) {
        if constexpr (light_nd<ND>()) {
            constexpr int kLightU = light_u<ND>();
            for (int k = 0; k < vpt; k += kLightU) {
                GradVec<kGradBF16> gv[kLightU][ND];
                int64_t iv[kLightU];
#pragma unroll
                for (int u = 0; u < kLightU; ++u) {
                    iv[u] = b0 + static_cast<int64_t>(k + u) * kStepThreads + threadIdx.x;
                    if (k + u < vpt && iv[u] < nvec) {
#pragma unroll
                        for (int q = 0; q < ND; ++q) gv[u][q].load(tab.p[q], iv[u]);
                    }
                }
#pragma unroll
                for (int u = 0; u < kLightU; ++u) {
                    if (k + u < vpt && iv[u] < nvec) {
                        float g[4];
                        sum_loaded<ND, kGradBF16>(gv[u], mo.group, g);
#pragma unroll
                        for (int e = 0; e < 4; ++e) g[e] = mean_of(g[e], mo);
                        stcs8(out + 4 * iv[u],
                              make_uint2(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3])));
                    }
                }
            }
        } else {
            for (int k = 0; k < vpt; ++k) {
                const int64_t i = b0 + static_cast<int64_t>(k) * kStepThreads + threadIdx.x;
                if (i >= nvec) break;
                float g[4];
                reduce4<ND, kGradBF16>(tab, nd, mo.group, i, g);
#pragma unroll
                for (int e = 0; e < 4; ++e) g[e] = mean_of(g[e], mo);
                stcs8(out + 4 * i, make_uint2(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3])));
            }
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
        const int64_t j = (nvec << 2) + threadIdx.x;
        out[j] = f32_to_bf16(mean_of(reduce1<kGradBF16>(tab, nd, mo.group, j), mo));
    }
    pdl_wait();
}

__global__ void __launch_bounds__(kThreads)
    allreduce_avg_scalar(PtrTable tab, int nd, int64_t n, uint16_t* __restrict__ out,
                         MeanOp mo) {
    pdl_trigger();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < n;
         j += stride)
        out[j] = f32_to_bf16(mean_of(reduce1<kGradBF16>(tab, nd, mo.group, j), mo));
    pdl_wait();
}

// ------------------------------------------------------ gradient scaler

__device__ __forceinline__ bool not_finite(float x) {
    return (__float_as_uint(x) & 0x7F800000u) == 0x7F800000u;
}

// The fp16 check decided on the input bits (f16_check_on_bits): whether any
// slice holds an inf or NaN in this thread's vectors, with the loads of
// light_u<ND>() vectors (a batch of 8 slices at a time for any N_d) in
// flight before any test.
template <int ND>
__device__ __forceinline__ bool f16_bits_scan(const PtrTable& tab, int nd, int64_t nvec,
                                              int64_t b0, int vpt) {
    bool bad = false;
    if constexpr (light_nd<ND>()) {
        constexpr int kLightU = light_u<ND>();
        for (int k = 0; k < vpt; k += kLightU) {
            GradVec<kGradF16> gv[kLightU][ND];
#pragma unroll
            for (int u = 0; u < kLightU; ++u) {
                const int64_t i = b0 + static_cast<int64_t>(k + u) * kStepThreads + threadIdx.x;
                if (k + u < vpt && i < nvec) {
#pragma unroll
                    for (int q = 0; q < ND; ++q) gv[u][q].load(tab.p[q], i);
                } else {
#pragma unroll
                    for (int q = 0; q < ND; ++q) gv[u][q].r = make_uint2(0u, 0u);
                }
            }
#pragma unroll
            for (int u = 0; u < kLightU; ++u)
#pragma unroll
                for (int q = 0; q < ND; ++q)
                    bad |= f16x2_nonfinite(gv[u][q].r.x) | f16x2_nonfinite(gv[u][q].r.y);
        }
    } else {
        for (int k = 0; k < vpt; ++k) {
            const int64_t i = b0 + static_cast<int64_t>(k) * kStepThreads + threadIdx.x;
            if (i >= nvec) break;
            const int n = ND == kRuntimeND ? nd : (ND < 0 ? nd : ND);
            for (int q = 0; q < n; q += 8) {
                GradVec<kGradF16> gv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (q + u < n) gv[u].load(tab.p[q + u], i);
                    else gv[u].r = make_uint2(0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    bad |= f16x2_nonfinite(gv[u].r.x) | f16x2_nonfinite(gv[u].r.y);
            }
        }
    }
    return bad;
}

// Sets *found when any unscaled mean gradient is inf or NaN.  Reads the
// slices only (2 B per fp16 slice element); one atomic per warp that saw one.
template <int ND, int GT>
__global__ void __launch_bounds__(kStepThreads, kStepMinBlocks)
    nonfinite_check_vec4(PtrTable tab, int nd, int64_t S, MeanOp mo, unsigned int* found,
                         int vpt) {
    mo = resolve_scale(mo);
    bool bad = false;
    const int64_t nvec = S >> 2;
    const int64_t run = static_cast<int64_t>(kStepThreads) * vpt;
    if constexpr (GT == kGradF16) {
        if (f16_check_on_bits(mo)) {     // the same for the whole grid
            for (int64_t b0 = static_cast<int64_t>(blockIdx.x) * run; b0 < nvec;
                 b0 += static_cast<int64_t>(gridDim.x) * run)
                bad |= f16_bits_scan<ND>(tab, nd, nvec, b0, vpt);
            if (blockIdx.x == 0 && threadIdx.x < (S & 3))
                for (int q = 0; q < nd; ++q)
                    bad |= f16_nonfinite(static_cast<const uint16_t*>(
                        tab.p[q])[(nvec << 2) + threadIdx.x]);
            if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0) atomicOr(found, 1u);
            return;
        }
    }
    for (int64_t b0 = static_cast<int64_t>(blockIdx.x) * run; b0 < nvec;
         b0 += static_cast<int64_t>(gridDim.x) * run) {
        if constexpr (light_nd<ND>()) {
            constexpr int kLightU = light_u<ND>();
            for (int k = 0; k < vpt; k += kLightU) {
                GradVec<GT> gv[kLightU][ND];
                int64_t iv[kLightU];
#pragma unroll
                for (int u = 0; u < kLightU; ++u) {
                    iv[u] = b0 + static_cast<int64_t>(k + u) * kStepThreads + threadIdx.x;
                    if (k + u < vpt && iv[u] < nvec) {
#pragma unroll
                        for (int q = 0; q < ND; ++q) gv[u][q].load(tab.p[q], iv[u]);
                    }
                }
#pragma unroll
                for (int u = 0; u < kLightU; ++u) {
                    if (k + u < vpt && iv[u] < nvec) {
                        float g[4];
                        sum_loaded<ND, GT>(gv[u], mo.group, g);
#pragma unroll
                        for (int e = 0; e < 4; ++e) bad |= not_finite(mean_of(g[e], mo));
                    }
                }
            }
        } else {
            for (int k = 0; k < vpt; ++k) {
                const int64_t i = b0 + static_cast<int64_t>(k) * kStepThreads + threadIdx.x;
                if (i >= nvec) break;
                float g[4];
                reduce4<ND, GT>(tab, nd, mo.group, i, g);
#pragma unroll
                for (int e = 0; e < 4; ++e) bad |= not_finite(mean_of(g[e], mo));
            }
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < (S & 3))
        bad |= not_finite(mean_of(reduce1<GT>(tab, nd, mo.group, (nvec << 2) + threadIdx.x), mo));
    if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0) atomicOr(found, 1u);
}

template <int GT>
__global__ void __launch_bounds__(kThreads)
    nonfinite_check_scalar(PtrTable tab, int nd, int64_t S, MeanOp mo, unsigned int* found) {
    mo = resolve_scale(mo);
    bool bad = false;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < S;
         j += stride)
        bad |= not_finite(mean_of(reduce1<GT>(tab, nd, mo.group, j), mo));
    if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0) atomicOr(found, 1u);
}

// Dynamic loss-scale update, one thread: backoff on a found inf/NaN, growth
// after `interval` clean steps in a row (kept only when finite); the found
// word is consumed and reset for the next step.
__global__ void scaler_update_kernel(float* scale, int* tracker, unsigned int* found,
                                     float growth, float backoff, int interval) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    const float s = *scale;
    if (*found != 0u) {
        *scale = __fmul_rn(s, backoff);
        *tracker = 0;
    } else {
        const int t = *tracker + 1;
        if (t == interval) {
            const float grown = __fmul_rn(s, growth);
            if (!not_finite(grown)) *scale = grown;
            *tracker = 0;
        } else {
            *tracker = t;
        }
    }
    *found = 0u;
}

// ------------------------------------------------- division self-check

// Compares div_nd with IEEE division (__fdiv_rn) on every fp32 bit pattern:
// counts the patterns whose results differ in any bit and keeps the
// smallest such pattern.
__global__ void __launch_bounds__(kThreads)
    mean_division_check(MeanOp mo, unsigned long long* mismatches, unsigned int* first_bad) {
    unsigned long long bad = 0;
    unsigned int first = 0xFFFFFFFFu;
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
    for (uint64_t b = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x;
         b < (uint64_t{1} << 32); b += stride) {
        const float x = __uint_as_float(static_cast<uint32_t>(b));
        if (__float_as_uint(div_nd(x, mo)) != __float_as_uint(__fdiv_rn(x, mo.nd))) {
            ++bad;
            if (static_cast<uint32_t>(b) < first) first = static_cast<uint32_t>(b);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        bad += __shfl_xor_sync(0xFFFFFFFFu, bad, o);
        first = min(first, __shfl_xor_sync(0xFFFFFFFFu, first, o));
    }
    if ((threadIdx.x & 31) == 0 && bad != 0) {
        atomicAdd(mismatches, bad);
        atomicMin(first_bad, first);
    }
}

// --------------------------------------------------------------- launch

unsigned grid_for(const void* kernel, int64_t work_items, int threads = kThreads) {
    const int64_t want = (work_items + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(device_sms()) * resident_blocks(kernel, threads);
    const int64_t g = want < cap ? want : cap;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

// One pass: a block per vpt x kStepThreads vectors, at most 2^31 - 1 blocks.
unsigned grid_one_pass(int64_t vectors, int vpt = 1) {
    const int64_t run = static_cast<int64_t>(kStepThreads) * vpt;
    const int64_t want = (vectors + run - 1) / run;
    const int64_t cap = (int64_t{1} << 31) - 1;
    const int64_t g = want < cap ? want : cap;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

// Vectors per thread for a kernel that moves `bytes_per_vector` per 4-element
// vector: enough for a block to move about kBlockBytes, at most 8.  Measured
// on GB300 (400M elements, bf16): the N_d = 2 all-reduce moved 3.0 TB/s with
// one vector per thread, 5.5 / 5.7 / 5.7 TB/s with blocks of 8 / 16 / 32 KB;
// the N_d = 4 check 4.6 / 5.5 / 6.0 / 6.3 TB/s.
constexpr int kBlockBytes = 32768;
int vectors_per_thread(int bytes_per_vector) {
    const int per_row = kStepThreads * bytes_per_vector;
    const int v = (kBlockBytes + per_row - 1) / per_row;
    return v < 1 ? 1 : (v > 8 ? 8 : v);
}

struct StepArgs {
    PtrTable tab;
    int nd;
    int64_t S;
    float *P, *M, *V;
    uint16_t* out;
    AdamScalars c;
    MeanOp mo;
    const unsigned int* skip;
};

template <int ND, int GT>
cudaError_t go_vec(const StepArgs& a, cudaStream_t s) {
    const unsigned grid = grid_one_pass(a.S >> 2);
    const cudaError_t e = launch_after(rs_adamw_cast_vec4<ND, GT>, dim3(grid), dim3(kStepThreads),
                                       0, s, a.tab, a.nd, a.S, a.P, a.M, a.V, a.out, a.c, a.mo,
                                       a.skip);
    note_launch();
    return e;
}

template <int GT>
cudaError_t dispatch_vec(const StepArgs& a, cudaStream_t s) {
    switch (a.nd) {
        case 1: return go_vec<1, GT>(a, s);
        case 2: return go_vec<2, GT>(a, s);
        case 3: return go_vec<3, GT>(a, s);
        case 4: return go_vec<4, GT>(a, s);
        case 5: case 7:  // 8 fp32 slices would spill at 64 registers: the loop instead
            if constexpr (GT != kGradF32) return go_vec<-8, GT>(a, s);
            else return go_vec<kRuntimeND, GT>(a, s);
        case 6: return go_vec<6, GT>(a, s);
        case 8: return go_vec<8, GT>(a, s);
        default: break;
    }
    // 9..16 slices: compiled for 16-bit slices (54-62 registers, every load
    // in flight); as many fp32 slices would spill at 64 registers, so those
    // take the loop.  At 9..11 and 13..15 the compiled forms moved 7.15-7.35
    // TB/s where the TMA-staged kernel moved 6.80-7.09 on the same buffers.
    if constexpr (GT != kGradF32) {
        switch (a.nd) {
            case 9: return go_vec<9, GT>(a, s);
            case 10: return go_vec<10, GT>(a, s);
            case 11: return go_vec<11, GT>(a, s);
            case 12: return go_vec<12, GT>(a, s);
            case 13: return go_vec<13, GT>(a, s);
            case 14: return go_vec<14, GT>(a, s);
            case 15: return go_vec<15, GT>(a, s);
            case 16: return go_vec<16, GT>(a, s);
            default: break;
        }
    }
    return go_vec<kRuntimeND, GT>(a, s);
}

template <int GT>
cudaError_t go_scalar(const StepArgs& a, cudaStream_t s) {
    const unsigned grid = grid_for(reinterpret_cast<const void*>(rs_adamw_cast_scalar<GT>), a.S);
    const cudaError_t e = launch_after(rs_adamw_cast_scalar<GT>, dim3(grid), dim3(kThreads), 0, s,
                                       a.tab, a.nd, a.S, a.P, a.M, a.V, a.out, a.c, a.mo, a.skip);
    note_launch();
    return e;
}

template <int ND>
cudaError_t go_ar(const PtrTable& tab, int nd, int64_t n, uint16_t* out, const MeanOp& mo,
                  bool pdl, cudaStream_t s) {
    auto k = allreduce_avg_vec4<ND>;
    const int vpt = vectors_per_thread(4 * (2 * nd + 2));
    const unsigned grid = grid_one_pass(n >> 2, vpt);
    cudaError_t e;
    if (pdl) {
        e = launch_dependent(k, dim3(grid), dim3(kStepThreads), 0, s, tab, nd, n, out, mo, vpt);
    } else {
        k<<<grid, kStepThreads, 0, s>>>(tab, nd, n, out, mo, vpt);
        e = cudaGetLastError();
    }
    note_launch();
    return e;
}

template <int ND, int GT>
cudaError_t go_check(const PtrTable& tab, int nd, int64_t S, const MeanOp& mo,
                     unsigned int* found, cudaStream_t s) {
    auto k = nonfinite_check_vec4<ND, GT>;
    const int vpt = vectors_per_thread(4 * nd * (GT == kGradF32 ? 4 : 2));
    const unsigned grid = grid_one_pass(S >> 2, vpt);
    k<<<grid, kStepThreads, 0, s>>>(tab, nd, S, mo, found, vpt);
    note_launch();
    return cudaGetLastError();
}

template <int GT>
cudaError_t dispatch_check(const PtrTable& tab, int nd, int64_t S, const MeanOp& mo,
                           unsigned int* found, bool vec, cudaStream_t s) {
    if (!vec) {
        const unsigned grid =
            grid_for(reinterpret_cast<const void*>(nonfinite_check_scalar<GT>), S);
        nonfinite_check_scalar<GT><<<grid, kThreads, 0, s>>>(tab, nd, S, mo, found);
        note_launch();
        return cudaGetLastError();
    }
    // fp32 slices at N_d = 3..7 would hold too many registers of loads in
    // flight: they take the loop over any N_d
    switch (nd) {
        case 1: return go_check<1, GT>(tab, nd, S, mo, found, s);
        case 2: return go_check<2, GT>(tab, nd, S, mo, found, s);
        case 3:
            if constexpr (GT != kGradF32) return go_check<3, GT>(tab, nd, S, mo, found, s);
            else return go_check<kRuntimeND, GT>(tab, nd, S, mo, found, s);
        case 4: return go_check<4, GT>(tab, nd, S, mo, found, s);
        case 5:
            if constexpr (GT != kGradF32) return go_check<5, GT>(tab, nd, S, mo, found, s);
            else return go_check<kRuntimeND, GT>(tab, nd, S, mo, found, s);
        case 6:
            if constexpr (GT != kGradF32) return go_check<6, GT>(tab, nd, S, mo, found, s);
            else return go_check<kRuntimeND, GT>(tab, nd, S, mo, found, s);
        case 7:
            if constexpr (GT != kGradF32) return go_check<7, GT>(tab, nd, S, mo, found, s);
            else return go_check<kRuntimeND, GT>(tab, nd, S, mo, found, s);
        case 8: return go_check<8, GT>(tab, nd, S, mo, found, s);
        default: break;
    }
    // 9..16 16-bit slices: compiled for their count as well (7.1-7.4 TB/s,
    // where the TMA-staged check moved 6.1-6.9 on the same buffers)
    if constexpr (GT != kGradF32) {
        switch (nd) {
            case 9: return go_check<9, GT>(tab, nd, S, mo, found, s);
            case 10: return go_check<10, GT>(tab, nd, S, mo, found, s);
            case 11: return go_check<11, GT>(tab, nd, S, mo, found, s);
            case 12: return go_check<12, GT>(tab, nd, S, mo, found, s);
            case 13: return go_check<13, GT>(tab, nd, S, mo, found, s);
            case 14: return go_check<14, GT>(tab, nd, S, mo, found, s);
            case 15: return go_check<15, GT>(tab, nd, S, mo, found, s);
            case 16: return go_check<16, GT>(tab, nd, S, mo, found, s);
            default: break;
        }
    }
    return go_check<kRuntimeND, GT>(tab, nd, S, mo, found, s);
}

}  // namespace

cudaError_t launch_rs_adamw_cast(const PtrTable& tab, int nd, int grad_type, int64_t S,
                                 float* master, float* m, float* v, uint16_t* out,
                                 const AdamScalars& c, const MeanOp& mo,
                                 const unsigned int* skip, bool vec, cudaStream_t stream) {
    const StepArgs a{tab, nd, S, master, m, v, out, c, mo, skip};
    switch (grad_type) {
        case kGradF32: return vec ? dispatch_vec<kGradF32>(a, stream) : go_scalar<kGradF32>(a, stream);
        case kGradF16: return vec ? dispatch_vec<kGradF16>(a, stream) : go_scalar<kGradF16>(a, stream);
        default: return vec ? dispatch_vec<kGradBF16>(a, stream) : go_scalar<kGradBF16>(a, stream);
    }
}

cudaError_t launch_allreduce_avg(const PtrTable& tab, int nd, int64_t n, uint16_t* out,
                                 const MeanOp& mo, bool vec, bool pdl, cudaStream_t stream) {
    if (vec) {
        switch (nd) {
            case 1: return go_ar<1>(tab, nd, n, out, mo, pdl, stream);
            case 2: return go_ar<2>(tab, nd, n, out, mo, pdl, stream);
            case 3: return go_ar<3>(tab, nd, n, out, mo, pdl, stream);
            case 4: return go_ar<4>(tab, nd, n, out, mo, pdl, stream);
            case 5: return go_ar<5>(tab, nd, n, out, mo, pdl, stream);
            case 6: return go_ar<6>(tab, nd, n, out, mo, pdl, stream);
            case 7: return go_ar<7>(tab, nd, n, out, mo, pdl, stream);
            case 8: return go_ar<8>(tab, nd, n, out, mo, pdl, stream);
            case 9: return go_ar<9>(tab, nd, n, out, mo, pdl, stream);
            case 10: return go_ar<10>(tab, nd, n, out, mo, pdl, stream);
            case 11: return go_ar<11>(tab, nd, n, out, mo, pdl, stream);
            case 12: return go_ar<12>(tab, nd, n, out, mo, pdl, stream);
            case 13: return go_ar<13>(tab, nd, n, out, mo, pdl, stream);
            case 14: return go_ar<14>(tab, nd, n, out, mo, pdl, stream);
            case 15: return go_ar<15>(tab, nd, n, out, mo, pdl, stream);
            case 16: return go_ar<16>(tab, nd, n, out, mo, pdl, stream);
            default: return go_ar<kRuntimeND>(tab, nd, n, out, mo, pdl, stream);
        }
    }
    const unsigned grid = grid_for(reinterpret_cast<const void*>(allreduce_avg_scalar), n);
    cudaError_t e;
    if (pdl) {
        e = launch_dependent(allreduce_avg_scalar, dim3(grid), dim3(kThreads), 0, stream, tab, nd,
                             n, out, mo);
    } else {
        allreduce_avg_scalar<<<grid, kThreads, 0, stream>>>(tab, nd, n, out, mo);
        e = cudaGetLastError();
    }
    note_launch();
    return e;
}

cudaError_t launch_nonfinite_check(const PtrTable& tab, int nd, int grad_type, int64_t S,
                                   const MeanOp& mo, unsigned int* found, bool vec,
                                   cudaStream_t stream) {
    switch (grad_type) {
        case kGradF32: return dispatch_check<kGradF32>(tab, nd, S, mo, found, vec, stream);
        case kGradF16: return dispatch_check<kGradF16>(tab, nd, S, mo, found, vec, stream);
        default: return dispatch_check<kGradBF16>(tab, nd, S, mo, found, vec, stream);
    }
}

cudaError_t launch_scaler_update(float* scale, int* tracker, unsigned int* found, float growth,
                                 float backoff, int interval, cudaStream_t stream) {
    scaler_update_kernel<<<1, 32, 0, stream>>>(scale, tracker, found, growth, backoff, interval);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_ddp_allreduce_adamw_cast(const PtrTable& tab, int nd, int64_t n,
                                            uint16_t* mean_out, float* master, float* m,
                                            float* v, uint16_t* out, const AdamScalars& c,
                                            const MeanOp& mo, bool vec, cudaStream_t stream) {
    if (!vec) {
        const unsigned grid = grid_for(
            reinterpret_cast<const void*>(ddp_allreduce_adamw_cast_scalar), n);
        const cudaError_t e = launch_after(ddp_allreduce_adamw_cast_scalar, dim3(grid),
                                           dim3(kThreads), 0, stream, tab, nd, n, mean_out,
                                           master, m, v, out, c, mo);
        note_launch();
        return e;
    }
    const unsigned grid = grid_one_pass(n >> 2);
    cudaError_t e = cudaSuccess;
#define SHARDSTEP_DDP_GO(K)                                                                    \
    e = launch_after(ddp_allreduce_adamw_cast_vec4<K>, dim3(grid), dim3(kStepThreads), 0, stream, \
                     tab, nd, n, mean_out, master, m, v, out, c, mo)
    switch (nd) {
        case 1: SHARDSTEP_DDP_GO(1); break;
        case 2: SHARDSTEP_DDP_GO(2); break;
        case 3: SHARDSTEP_DDP_GO(3); break;
        case 4: SHARDSTEP_DDP_GO(4); break;
        case 5: case 7: SHARDSTEP_DDP_GO(-8); break;
        case 6: SHARDSTEP_DDP_GO(6); break;
        case 8: SHARDSTEP_DDP_GO(8); break;
        case 9: SHARDSTEP_DDP_GO(9); break;
        case 10: SHARDSTEP_DDP_GO(10); break;
        case 11: SHARDSTEP_DDP_GO(11); break;
        case 12: SHARDSTEP_DDP_GO(12); break;
        case 13: SHARDSTEP_DDP_GO(13); break;
        case 14: SHARDSTEP_DDP_GO(14); break;
        case 15: SHARDSTEP_DDP_GO(15); break;
        case 16: SHARDSTEP_DDP_GO(16); break;
        default: SHARDSTEP_DDP_GO(kRuntimeND); break;
    }
#undef SHARDSTEP_DDP_GO
    note_launch();
    return e;
}

cudaError_t launch_mean_division_check(const MeanOp& mo, unsigned long long* mismatches,
                                       unsigned int* first_bad, cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>(device_sms()) * 8u;
    mean_division_check<<<grid, kThreads, 0, stream>>>(mo, mismatches, first_bad);
    note_launch();
    return cudaGetLastError();
}

}  // namespace shardstep
