// The fused sharded optimizer step (reduce-scatter average + AdamW + bf16
// cast in one pass over the shard) and the DDP bucket all-reduce average.
//
// Both are HBM-bound streams: per shard element the fused kernel reads N_d
// gradient slices (2 B each, bf16) and the fp32 master/m/v (12 B), and writes
// master/m/v (12 B) and the bf16 parameter (2 B) -- 2*N_d + 26 bytes, each
// byte touched once.  Each thread owns 4 consecutive elements per iteration:
// one 8-byte load per bf16 slice (16 bytes for fp32 slices), one 16-byte load
// per fp32 state array, every load of the iteration issued before any
// arithmetic; all accesses are streaming (evict-first) loads and stores.  Blocks of 512 threads are capped at 64 registers so that 32
// warps per SM keep requests in flight; the grid is three times the resident
// capacity (SMs x 2 blocks) and strides over the shard.  Measured on GB300
// against 8-elements-per-thread blocks of 256 at 112 registers, this shape
// moves the same bytes about 6% faster.
#include "common.cuh"

namespace shardstep {
namespace {

constexpr int kRuntimeND = 0;

// ----------------------------------------------------------------- loads

constexpr int kStepThreads = 512;  // block of the fused / all-reduce kernels
constexpr int kStepMinBlocks = 2;   // 2 x 512 threads per SM -> <= 64 registers
constexpr int kGridOversub = 3;     // blocks launched per resident block slot

template <bool F32G>
struct GradVec;  // 4 gradient elements of one slice

template <>
struct GradVec<false> {
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
struct GradVec<true> {
    uint4 a;
    __device__ __forceinline__ void load(const void* base, int64_t i) {
        a = ldcs16(static_cast<const float*>(base) + 4 * i);
    }
    __device__ __forceinline__ void to_f32(float* f) const { unpack4f(a, f); }
};

template <bool F32G>
__device__ __forceinline__ float grad_scalar(const void* base, int64_t j) {
    if (F32G) return static_cast<const float*>(base)[j];
    return bf16_to_f32(static_cast<const uint16_t*>(base)[j]);
}

// Sum of the N_d slices at 4 consecutive elements, in the order GroupSum
// fixes (rank order; grouped for hybrid sharding).
template <int ND, bool F32G>
__device__ __forceinline__ void reduce4(const PtrTable& tab, int nd, int group, int64_t i,
                                        float* g) {
    GroupSum<4> acc;
    if constexpr (ND != kRuntimeND) {
        GradVec<F32G> gv[ND];
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
        // any N_d: groups of four slices in flight at a time
        {
            GradVec<F32G> g0;
            g0.load(tab.p[0], i);
            float t[4];
            g0.to_f32(t);
            acc.first(t);
        }
        int q = 1;
        for (; q + 4 <= nd; q += 4) {
            GradVec<F32G> gv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) gv[u].load(tab.p[q + u], i);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float t[4];
                gv[u].to_f32(t);
                acc.add(t, group);
            }
        }
        for (; q < nd; ++q) {
            GradVec<F32G> gq;
            gq.load(tab.p[q], i);
            float t[4];
            gq.to_f32(t);
            acc.add(t, group);
        }
    }
    acc.result(g);
}

template <bool F32G>
__device__ __forceinline__ float reduce1(const PtrTable& tab, int nd, int group, int64_t j) {
    GroupSum<1> acc;
    float t = grad_scalar<F32G>(tab.p[0], j);
    acc.first(&t);
    for (int q = 1; q < nd; ++q) {
        t = grad_scalar<F32G>(tab.p[q], j);
        acc.add(&t, group);
    }
    float g;
    acc.result(&g);
    return g;
}

// --------------------------------------------------- fused step kernels

template <bool F32G>
__device__ __forceinline__ void step_scalar(const PtrTable& tab, int nd, int64_t j,
                                            float* __restrict__ P, float* __restrict__ M,
                                            float* __restrict__ V, uint16_t* __restrict__ out,
                                            const AdamScalars& c, const MeanOp& mo) {
    const float g = mean_of(reduce1<F32G>(tab, nd, mo.group, j), mo);
    float p = P[j], m = M[j], v = V[j];
    adamw_elem(g, p, m, v, c);
    P[j] = p;
    M[j] = m;
    V[j] = v;
    out[j] = f32_to_bf16(p);
}

// Aligned operands (gradient slices and the bf16 output 8-byte aligned for
// bf16, 16-byte for fp32 slices; state 16-byte aligned): 4 elements per
// thread per iteration, then the (< 4 element) tail by block 0.
template <int ND, bool F32G>
__global__ void __launch_bounds__(kStepThreads, kStepMinBlocks)
    rs_adamw_cast_vec4(PtrTable tab, int nd, int64_t S, float* __restrict__ P,
                       float* __restrict__ M, float* __restrict__ V, uint16_t* __restrict__ out,
                       AdamScalars c, MeanOp mo) {
    const int64_t nvec = S >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kStepThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kStepThreads + threadIdx.x; i < nvec;
         i += stride) {
        // all loads of the iteration first
        const uint4 p0 = ldcs16(P + 4 * i);
        const uint4 m0 = ldcs16(M + 4 * i);
        const uint4 v0 = ldcs16(V + 4 * i);
        float g[4];
        reduce4<ND, F32G>(tab, nd, mo.group, i, g);
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
        step_scalar<F32G>(tab, nd, (nvec << 2) + threadIdx.x, P, M, V, out, c, mo);
}

// Any alignment: one element per thread per iteration.
template <bool F32G>
__global__ void __launch_bounds__(kThreads)
    rs_adamw_cast_scalar(PtrTable tab, int nd, int64_t S, float* __restrict__ P,
                         float* __restrict__ M, float* __restrict__ V,
                         uint16_t* __restrict__ out, AdamScalars c, MeanOp mo) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < S;
         j += stride)
        step_scalar<F32G>(tab, nd, j, P, M, V, out, c, mo);
}

// ------------------------------------------------ bucket all-reduce avg

template <int ND>
__global__ void __launch_bounds__(kStepThreads, kStepMinBlocks)
    allreduce_avg_vec4(PtrTable tab, int nd, int64_t n, uint16_t* __restrict__ out, MeanOp mo) {
    const int64_t nvec = n >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kStepThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kStepThreads + threadIdx.x; i < nvec;
         i += stride) {
        float g[4];
        reduce4<ND, false>(tab, nd, mo.group, i, g);
#pragma unroll
        for (int k = 0; k < 4; ++k) g[k] = mean_of(g[k], mo);
        stcs8(out + 4 * i, make_uint2(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3])));
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
        const int64_t j = (nvec << 2) + threadIdx.x;
        out[j] = f32_to_bf16(mean_of(reduce1<false>(tab, nd, mo.group, j), mo));
    }
}

__global__ void __launch_bounds__(kThreads)
    allreduce_avg_scalar(PtrTable tab, int nd, int64_t n, uint16_t* __restrict__ out,
                         MeanOp mo) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < n;
         j += stride)
        out[j] = f32_to_bf16(mean_of(reduce1<false>(tab, nd, mo.group, j), mo));
}

// --------------------------------------------------------------- launch

unsigned grid_for(const void* kernel, int64_t work_items, int threads = kThreads,
                  int oversub = 1) {
    const int64_t want = (work_items + threads - 1) / threads;
    const int64_t cap =
        static_cast<int64_t>(device_sms()) * resident_blocks(kernel, threads) * oversub;
    const int64_t g = want < cap ? want : cap;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

template <int ND, bool F32G>
cudaError_t go_vec(const PtrTable& tab, int nd, int64_t S, float* P, float* M, float* V,
                   uint16_t* out, const AdamScalars& c, const MeanOp& mo, cudaStream_t s) {
    auto k = rs_adamw_cast_vec4<ND, F32G>;
    const unsigned grid = grid_for(reinterpret_cast<const void*>(k), (S >> 2) > 0 ? (S >> 2) : 1,
                                   kStepThreads, kGridOversub);
    k<<<grid, kStepThreads, 0, s>>>(tab, nd, S, P, M, V, out, c, mo);
    note_launch();
    return cudaGetLastError();
}

template <bool F32G>
cudaError_t dispatch_vec(const PtrTable& tab, int nd, int64_t S, float* P, float* M, float* V,
                         uint16_t* out, const AdamScalars& c, const MeanOp& mo,
                         cudaStream_t s) {
    switch (nd) {
        case 1: return go_vec<1, F32G>(tab, nd, S, P, M, V, out, c, mo, s);
        case 2: return go_vec<2, F32G>(tab, nd, S, P, M, V, out, c, mo, s);
        case 3: return go_vec<3, F32G>(tab, nd, S, P, M, V, out, c, mo, s);
        case 4: return go_vec<4, F32G>(tab, nd, S, P, M, V, out, c, mo, s);
        case 8: return go_vec<8, F32G>(tab, nd, S, P, M, V, out, c, mo, s);
        case 16: return go_vec<16, F32G>(tab, nd, S, P, M, V, out, c, mo, s);
        default: return go_vec<kRuntimeND, F32G>(tab, nd, S, P, M, V, out, c, mo, s);
    }
}

template <int ND>
cudaError_t go_ar(const PtrTable& tab, int nd, int64_t n, uint16_t* out, const MeanOp& mo,
                  cudaStream_t s) {
    auto k = allreduce_avg_vec4<ND>;
    const unsigned grid = grid_for(reinterpret_cast<const void*>(k), (n >> 2) > 0 ? (n >> 2) : 1,
                                   kStepThreads, kGridOversub);
    k<<<grid, kStepThreads, 0, s>>>(tab, nd, n, out, mo);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rs_adamw_cast(const PtrTable& tab, int nd, bool f32_grads, int64_t S,
                                 float* master, float* m, float* v, uint16_t* out,
                                 const AdamScalars& c, const MeanOp& mo, bool vec,
                                 cudaStream_t stream) {
    if (vec) {
        return f32_grads ? dispatch_vec<true>(tab, nd, S, master, m, v, out, c, mo, stream)
                         : dispatch_vec<false>(tab, nd, S, master, m, v, out, c, mo, stream);
    }
    const void* kp = f32_grads ? reinterpret_cast<const void*>(rs_adamw_cast_scalar<true>)
                               : reinterpret_cast<const void*>(rs_adamw_cast_scalar<false>);
    const unsigned grid = grid_for(kp, S);
    if (f32_grads)
        rs_adamw_cast_scalar<true><<<grid, kThreads, 0, stream>>>(tab, nd, S, master, m, v, out, c,
                                                                  mo);
    else
        rs_adamw_cast_scalar<false><<<grid, kThreads, 0, stream>>>(tab, nd, S, master, m, v, out,
                                                                   c, mo);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_allreduce_avg(const PtrTable& tab, int nd, int64_t n, uint16_t* out,
                                 const MeanOp& mo, bool vec, cudaStream_t stream) {
    if (vec) {
        switch (nd) {
            case 1: return go_ar<1>(tab, nd, n, out, mo, stream);
            case 2: return go_ar<2>(tab, nd, n, out, mo, stream);
            case 4: return go_ar<4>(tab, nd, n, out, mo, stream);
            case 8: return go_ar<8>(tab, nd, n, out, mo, stream);
            default: return go_ar<kRuntimeND>(tab, nd, n, out, mo, stream);
        }
    }
    const unsigned grid = grid_for(reinterpret_cast<const void*>(allreduce_avg_scalar), n);
    allreduce_avg_scalar<<<grid, kThreads, 0, stream>>>(tab, nd, n, out, mo);
    note_launch();
    return cudaGetLastError();
}

}  // namespace shardstep
