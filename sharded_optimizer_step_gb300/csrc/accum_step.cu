// The last micro-batch's gradient accumulation fused into the sharded step.
//
// With M micro-batches, every rank accumulates the bf16 gradient of each
// micro-batch into an fp32 accumulator (acc += fl(g * (1/M))) and reduce-
// scatters the accumulator after the last one.  Run as two passes, the last
// micro-batch costs, per shard element and slice, a read of g and of the
// accumulator and a write of the accumulator (10 B) before the fused step
// reads the accumulator again (4 B).  This kernel takes both at once: slice
// q's contribution is acc_q + fl(g_q * scale), computed in registers exactly
// as the accumulation would have stored it, then summed in rank order (in
// groups of F ranks under hybrid sharding), averaged, AdamW-updated and cast
// like the plain fused step.  The
// accumulators are only read.  Per shard element it moves 6 * N_d + 26 bytes
// where the two passes move 14 * N_d + 26 (74 against 138 at N_d = 8).
//
// Layout as in the plain fused kernel: 128-thread blocks, one 4-element
// vector per thread, a one-pass grid, every load of an iteration issued
// before any arithmetic (one 16-byte load per accumulator slice, one 8-byte
// load per bf16 slice, one 16-byte load per state array), streaming loads
// and stores.  With N_d = 8 that is 60 registers of loads per thread, so
// the register cap is raised to 80 (6 blocks per SM).  Compiled for N_d =
// 1, 2, 3, 4, 6 and 8, an up-to-8 form for 5 and 7, and a loop over batches
// of 4 slices for the rest.
#include "common.cuh"

namespace shardstep {
namespace {

constexpr int kAccThreads = 128;
constexpr int kAccRuntimeND = 0;  // any N_d: slices in batches of 4

// ND > 0: exactly ND slices; ND < 0: up to -ND slices, every load in flight
// at once and the first nd used; kAccRuntimeND: any N_d in batches of 4.
// Kernels holding the loads of 6 or more slices get 80 registers (6 blocks
// per SM); at a 64-register cap the 6- and 8-slice kernels spilled.
template <int ND>
constexpr int acc_min_blocks() {
    return ND >= 6 || ND < 0 || ND == kAccRuntimeND ? 6 : 8;
}

// Slice contributions at 4 consecutive elements, summed in rank order
// (GROUPED: in the order GroupSum fixes for hybrid sharding, groups of
// `group` ranks first; the plain sum keeps the 8-slice kernel unspilled).
template <int ND, bool GROUPED>
__device__ __forceinline__ void accum_reduce4(const PtrTable& acc, const PtrTable& last,
                                              int nd, int group, float scale, int64_t i,
                                              float* g) {
    constexpr int B = ND > 0 ? ND : (ND < 0 ? -ND : 4);
    constexpr bool kGuard = ND <= 0;
    float s[4];
    GroupSum<4> grouped;
    for (int q0 = 0; q0 < nd; q0 += B) {
        uint4 a[B];
        uint2 b[B];
#pragma unroll
        for (int u = 0; u < B; ++u) {
            if (!kGuard || q0 + u < nd) {
                a[u] = ldcs16(static_cast<const float*>(acc.p[q0 + u]) + 4 * i);
                b[u] = ldcs8(static_cast<const uint16_t*>(last.p[q0 + u]) + 4 * i);
            }
        }
#pragma unroll
        for (int u = 0; u < B; ++u) {
            if (!kGuard || q0 + u < nd) {
                float t[4];
                unpack4f(a[u], t);
                const float f[4] = {bf16_lo(b[u].x), bf16_hi(b[u].x), bf16_lo(b[u].y),
                                    bf16_hi(b[u].y)};
#pragma unroll
                for (int k = 0; k < 4; ++k) t[k] = __fadd_rn(t[k], __fmul_rn(f[k], scale));
                if constexpr (GROUPED) {
                    if (q0 + u == 0) grouped.first(t);
                    else grouped.add(t, group);
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) s[k] = q0 + u == 0 ? t[k] : __fadd_rn(s[k], t[k]);
                }
            }
        }
    }
    if constexpr (GROUPED) grouped.result(s);
#pragma unroll
    for (int k = 0; k < 4; ++k) g[k] = s[k];
}

template <bool GROUPED>
__device__ __forceinline__ void accum_step_elem(const PtrTable& acc, const PtrTable& last,
                                                int nd, float scale, int64_t j,
                                                float* __restrict__ P, float* __restrict__ M,
                                                float* __restrict__ V,
                                                uint16_t* __restrict__ out,
                                                const AdamScalars& c, const MeanOp& mo) {
    GroupSum<1> grouped;
    float s = 0.0f;
    for (int q = 0; q < nd; ++q) {
        const float a = static_cast<const float*>(acc.p[q])[j];
        const float g = bf16_to_f32(static_cast<const uint16_t*>(last.p[q])[j]);
        const float t = __fadd_rn(a, __fmul_rn(g, scale));
        if constexpr (GROUPED) {
            if (q == 0) grouped.first(&t);
            else grouped.add(&t, mo.group);
        } else {
            s = q == 0 ? t : __fadd_rn(s, t);
        }
    }
    if constexpr (GROUPED) grouped.result(&s);
    float p = P[j], m = M[j], v = V[j];
    adamw_elem(mean_of(s, mo), p, m, v, c);
    P[j] = p;
    M[j] = m;
    V[j] = v;
    out[j] = f32_to_bf16(p);
}

// Accumulator slices and state 16-byte aligned, bf16 slices and the output
// 8-byte aligned: 4 elements per thread, the (< 4 element) tail by block 0.
template <int ND, bool GROUPED>
__global__ void __launch_bounds__(kAccThreads, acc_min_blocks<ND>())
    accum_rs_adamw_cast_vec4(PtrTable acc, PtrTable last, int nd, int64_t S, float scale,
                             float* __restrict__ P, float* __restrict__ M,
                             float* __restrict__ V, uint16_t* __restrict__ out, AdamScalars c,
                             MeanOp mo) {
    pdl_enter();
    c = resolve_adam(c);
    const int64_t nvec = S >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kAccThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kAccThreads + threadIdx.x; i < nvec;
         i += stride) {
        const uint4 p0 = ldcs16(P + 4 * i);
        const uint4 m0 = ldcs16(M + 4 * i);
        const uint4 v0 = ldcs16(V + 4 * i);
        float g[4];
        accum_reduce4<ND, GROUPED>(acc, last, nd, mo.group, scale, i, g);
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
        accum_step_elem<GROUPED>(acc, last, nd, scale, (nvec << 2) + threadIdx.x, P, M, V, out,
                                 c, mo);
}

// Any alignment: one element per thread per iteration.
__global__ void __launch_bounds__(kThreads)
    accum_rs_adamw_cast_scalar(PtrTable acc, PtrTable last, int nd, int64_t S, float scale,
                               float* __restrict__ P, float* __restrict__ M,
                               float* __restrict__ V, uint16_t* __restrict__ out,
                               AdamScalars c, MeanOp mo) {
    pdl_enter();
    c = resolve_adam(c);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < S;
         j += stride)
        accum_step_elem<true>(acc, last, nd, scale, j, P, M, V, out, c, mo);
}

template <int ND, bool GROUPED = false>
cudaError_t go_accum(const PtrTable& acc, const PtrTable& last, int nd, int64_t S, float scale,
                     float* P, float* M, float* V, uint16_t* out, const AdamScalars& c,
                     const MeanOp& mo, cudaStream_t s) {
    const int64_t blocks = ((S >> 2) + kAccThreads - 1) / kAccThreads;
    const int64_t cap = (int64_t{1} << 31) - 1;
    const unsigned grid = static_cast<unsigned>(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
    const cudaError_t e = launch_after(accum_rs_adamw_cast_vec4<ND, GROUPED>, dim3(grid),
                                       dim3(kAccThreads), 0, s, acc, last, nd, S, scale, P, M, V,
                                       out, c, mo);
    note_launch();
    return e;
}

}  // namespace

cudaError_t launch_accum_rs_adamw_cast(const PtrTable& acc, const PtrTable& last, int nd,
                                       int64_t S, float scale, float* master, float* m,
                                       float* v, uint16_t* out, const AdamScalars& c,
                                       const MeanOp& mo, bool vec, cudaStream_t stream) {
    if (vec && mo.group != nd)  // hybrid sharding: grouped order, any N_d
        return go_accum<kAccRuntimeND, true>(acc, last, nd, S, scale, master, m, v, out, c, mo,
                                             stream);
    if (vec) {
        switch (nd) {
            case 1: return go_accum<1>(acc, last, nd, S, scale, master, m, v, out, c, mo, stream);
            case 2: return go_accum<2>(acc, last, nd, S, scale, master, m, v, out, c, mo, stream);
            case 3: return go_accum<3>(acc, last, nd, S, scale, master, m, v, out, c, mo, stream);
            case 4: return go_accum<4>(acc, last, nd, S, scale, master, m, v, out, c, mo, stream);
            case 5:
            case 7:
                return go_accum<-8>(acc, last, nd, S, scale, master, m, v, out, c, mo, stream);
            case 6: return go_accum<6>(acc, last, nd, S, scale, master, m, v, out, c, mo, stream);
            case 8: return go_accum<8>(acc, last, nd, S, scale, master, m, v, out, c, mo, stream);
            default:
                return go_accum<kAccRuntimeND>(acc, last, nd, S, scale, master, m, v, out, c, mo,
                                               stream);
        }
    }
    const int64_t want = (S + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(device_sms()) *
                        resident_blocks(reinterpret_cast<const void*>(accum_rs_adamw_cast_scalar),
                                        kThreads);
    const int64_t g = want < cap ? want : cap;
    const cudaError_t e = launch_after(accum_rs_adamw_cast_scalar,
                                       dim3(static_cast<unsigned>(g < 1 ? 1 : g)), dim3(kThreads),
                                       0, stream, acc, last, nd, S, scale, master, m, v, out, c,
                                       mo);
    note_launch();
    return e;
}

}  // namespace shardstep
