// The fused sharded optimizer step (reduce-scatter average + AdamW + bf16
// cast in one pass over the shard) and the DDP bucket all-reduce average.
//
// Both are HBM-bound streams: per shard element the fused kernel reads N_d
// gradient slices (2 B each, bf16) and the fp32 master/m/v (12 B), and writes
// master/m/v (12 B) and the bf16 parameter (2 B) -- 2*N_d + 26 bytes, each
// byte touched once.  Each thread owns 8 consecutive elements per iteration:
// one 16-byte load per bf16 slice, two per fp32 array, every load of the
// iteration issued before any arithmetic so that N_d + 6 independent 16-byte
// requests are in flight per thread.  Grids are sized to the resident
// capacity of the GPU (SMs x blocks per SM) and stride over the shard.
#include "common.cuh"

namespace shardstep {
namespace {

constexpr int kRuntimeND = 0;

// ----------------------------------------------------------------- loads

template <bool F32G>
struct GradVec;  // 8 gradient elements of one slice

template <>
struct GradVec<false> {
    uint4 r;
    __device__ __forceinline__ void load(const void* base, int64_t i) {
        r = ld_once(static_cast<const uint16_t*>(base) + 8 * i);
    }
    __device__ __forceinline__ void to_f32(float* f) const { unpack8(r, f); }
};

template <>
struct GradVec<true> {
    uint4 a, b;
    __device__ __forceinline__ void load(const void* base, int64_t i) {
        const float* p = static_cast<const float*>(base) + 8 * i;
        a = ld_once(p);
        b = ld_once(p + 4);
    }
    __device__ __forceinline__ void to_f32(float* f) const {
        unpack4f(a, f);
        unpack4f(b, f + 4);
    }
};

template <bool F32G>
__device__ __forceinline__ float grad_scalar(const void* base, int64_t j) {
    if (F32G) return static_cast<const float*>(base)[j];
    return bf16_to_f32(static_cast<const uint16_t*>(base)[j]);
}

// Sum of the N_d slices at 8 consecutive elements, in rank order.
template <int ND, bool F32G>
__device__ __forceinline__ void reduce8(const PtrTable& tab, int nd, int64_t i, float* g) {
    if constexpr (ND != kRuntimeND) {
        GradVec<F32G> gv[ND];
#pragma unroll
        for (int q = 0; q < ND; ++q) gv[q].load(tab.p[q], i);
        gv[0].to_f32(g);
#pragma unroll
        for (int q = 1; q < ND; ++q) {
            float t[8];
            gv[q].to_f32(t);
#pragma unroll
            for (int k = 0; k < 8; ++k) g[k] = __fadd_rn(g[k], t[k]);
        }
    } else {
        // any N_d: groups of four slices in flight at a time
        {
            GradVec<F32G> g0;
            g0.load(tab.p[0], i);
            g0.to_f32(g);
        }
        int q = 1;
        for (; q + 4 <= nd; q += 4) {
            GradVec<F32G> gv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) gv[u].load(tab.p[q + u], i);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float t[8];
                gv[u].to_f32(t);
#pragma unroll
                for (int k = 0; k < 8; ++k) g[k] = __fadd_rn(g[k], t[k]);
            }
        }
        for (; q < nd; ++q) {
            GradVec<F32G> gq;
            gq.load(tab.p[q], i);
            float t[8];
            gq.to_f32(t);
#pragma unroll
            for (int k = 0; k < 8; ++k) g[k] = __fadd_rn(g[k], t[k]);
        }
    }
}

template <bool F32G>
__device__ __forceinline__ float reduce1(const PtrTable& tab, int nd, int64_t j) {
    float s = grad_scalar<F32G>(tab.p[0], j);
    for (int q = 1; q < nd; ++q) s = __fadd_rn(s, grad_scalar<F32G>(tab.p[q], j));
    return s;
}

// --------------------------------------------------- fused step kernels

template <bool F32G>
__device__ __forceinline__ void step_scalar(const PtrTable& tab, int nd, int64_t j,
                                            float* __restrict__ P, float* __restrict__ M,
                                            float* __restrict__ V, uint16_t* __restrict__ out,
                                            const AdamScalars& c, const MeanOp& mo) {
    const float g = mean_of(reduce1<F32G>(tab, nd, j), mo);
    float p = P[j], m = M[j], v = V[j];
    adamw_elem(g, p, m, v, c);
    P[j] = p;
    M[j] = m;
    V[j] = v;
    out[j] = f32_to_bf16(p);
}

// 16-byte-aligned operands: 8 elements per thread per iteration, then the
// (< 8 element) tail by block 0.
template <int ND, bool F32G>
__global__ void __launch_bounds__(kThreads)
    rs_adamw_cast_vec8(PtrTable tab, int nd, int64_t S, float* __restrict__ P,
                       float* __restrict__ M, float* __restrict__ V, uint16_t* __restrict__ out,
                       AdamScalars c, MeanOp mo) {
    const int64_t nvec = S >> 3;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < nvec;
         i += stride) {
        // all loads of the iteration first
        const uint4 p0 = ld_rw(P + 8 * i), p1 = ld_rw(P + 8 * i + 4);
        const uint4 m0 = ld_rw(M + 8 * i), m1 = ld_rw(M + 8 * i + 4);
        const uint4 v0 = ld_rw(V + 8 * i), v1 = ld_rw(V + 8 * i + 4);
        float g[8];
        reduce8<ND, F32G>(tab, nd, i, g);
        float p[8], m[8], v[8];
        unpack4f(p0, p); unpack4f(p1, p + 4);
        unpack4f(m0, m); unpack4f(m1, m + 4);
        unpack4f(v0, v); unpack4f(v1, v + 4);
#pragma unroll
        for (int k = 0; k < 8; ++k) adamw_elem(mean_of(g[k], mo), p[k], m[k], v[k], c);
        st_stream(P + 8 * i, pack4f(p));
        st_stream(P + 8 * i + 4, pack4f(p + 4));
        st_stream(M + 8 * i, pack4f(m));
        st_stream(M + 8 * i + 4, pack4f(m + 4));
        st_stream(V + 8 * i, pack4f(v));
        st_stream(V + 8 * i + 4, pack4f(v + 4));
        st_stream(out + 8 * i, make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
                                          pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7])));
    }
    if (blockIdx.x == 0 && threadIdx.x < (S & 7))
        step_scalar<F32G>(tab, nd, (nvec << 3) + threadIdx.x, P, M, V, out, c, mo);
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
__global__ void __launch_bounds__(kThreads)
    allreduce_avg_vec8(PtrTable tab, int nd, int64_t n, uint16_t* __restrict__ out, MeanOp mo) {
    const int64_t nvec = n >> 3;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < nvec;
         i += stride) {
        float g[8];
        reduce8<ND, false>(tab, nd, i, g);
#pragma unroll
        for (int k = 0; k < 8; ++k) g[k] = mean_of(g[k], mo);
        st_stream(out + 8 * i, make_uint4(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3]),
                                          pack_bf16x2(g[4], g[5]), pack_bf16x2(g[6], g[7])));
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 7)) {
        const int64_t j = (nvec << 3) + threadIdx.x;
        out[j] = f32_to_bf16(mean_of(reduce1<false>(tab, nd, j), mo));
    }
}

__global__ void __launch_bounds__(kThreads)
    allreduce_avg_scalar(PtrTable tab, int nd, int64_t n, uint16_t* __restrict__ out,
                         MeanOp mo) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < n;
         j += stride)
        out[j] = f32_to_bf16(mean_of(reduce1<false>(tab, nd, j), mo));
}

// --------------------------------------------------------------- launch

unsigned grid_for(const void* kernel, int64_t work_items) {
    const int64_t want = (work_items + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(device_sms()) * resident_blocks(kernel, kThreads);
    const int64_t g = want < cap ? want : cap;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

template <int ND, bool F32G>
cudaError_t go_vec(const PtrTable& tab, int nd, int64_t S, float* P, float* M, float* V,
                   uint16_t* out, const AdamScalars& c, const MeanOp& mo, cudaStream_t s) {
    auto k = rs_adamw_cast_vec8<ND, F32G>;
    const unsigned grid = grid_for(reinterpret_cast<const void*>(k), (S >> 3) > 0 ? (S >> 3) : 1);
    k<<<grid, kThreads, 0, s>>>(tab, nd, S, P, M, V, out, c, mo);
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
    auto k = allreduce_avg_vec8<ND>;
    const unsigned grid = grid_for(reinterpret_cast<const void*>(k), (n >> 3) > 0 ? (n >> 3) : 1);
    k<<<grid, kThreads, 0, s>>>(tab, nd, n, out, mo);
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
