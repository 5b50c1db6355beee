// The FSDP2 optimizer step of one rank over all of its parameters in one
// launch, read straight from the ranks' per-parameter gradients.
//
// A rank's padded local buffer is a run of segments: for each parameter the
// rows the rank holds (N_d gradient slices, one per rank, each starting at
// row rank * chunk of that rank's gradient), then its padding rows (every
// contribution +0).  The host packs up to kSegMax segments (and at most
// kSegPtrMax slice pointers; padding rows take none) into one SegTable,
// passed as a __grid_constant__
// parameter so that a block can index its segment's pointers without a local
// copy of the table.  Each block serves one segment: 128 threads, one
// 4-element vector per thread, every load issued before any arithmetic, and
// the reduce, mean, AdamW and cast of the fused step (GroupSum in rank order,
// mean_of, adamw_elem), so the bits are the fused step's on a chunk-cat
// buffer.  One launch replaces one per parameter, whose ramps and tails, and
// the tiny launches of the norm vectors, cost the FSDP2 layer step about a
// tenth of its time.
#include "common.cuh"

namespace shardstep {
namespace {

constexpr int kSegThreads = 128;
constexpr int kSegMinBlocks = 8;   // 8 x 128 threads per SM -> <= 64 registers
constexpr int kAnyND = 0;

// 4 consecutive gradient elements of one slice, kept packed as loaded (8
// bytes of 16-bit values, 16 of fp32) until they are summed.
template <int GT>
struct Raw4 {
    uint2 r;
    __device__ __forceinline__ void load(const void* base, int64_t i) {
        r = ldcs8(static_cast<const uint16_t*>(base) + 4 * i);
    }
    __device__ __forceinline__ void to_f32(float* f) const {
        if constexpr (GT == kGradF16) {
            f[0] = f16_to_f32(static_cast<uint16_t>(r.x & 0xFFFFu));
            f[1] = f16_to_f32(static_cast<uint16_t>(r.x >> 16));
            f[2] = f16_to_f32(static_cast<uint16_t>(r.y & 0xFFFFu));
            f[3] = f16_to_f32(static_cast<uint16_t>(r.y >> 16));
        } else {
            f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x);
            f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
        }
    }
};
template <>
struct Raw4<kGradF32> {
    uint4 a;
    __device__ __forceinline__ void load(const void* base, int64_t i) {
        a = ldcs16(static_cast<const float*>(base) + 4 * i);
    }
    __device__ __forceinline__ void to_f32(float* f) const { unpack4f(a, f); }
};

template <int GT>
__device__ __forceinline__ float load1(const void* base, int64_t j) {
    if constexpr (GT == kGradF32) return static_cast<const float*>(base)[j];
    if constexpr (GT == kGradF16) return f16_to_f32(static_cast<const uint16_t*>(base)[j]);
    return bf16_to_f32(static_cast<const uint16_t*>(base)[j]);
}

// The N_d slices summed at 4 consecutive elements in rank order; ND > 0:
// all ND loads in flight first; kAnyND: batches of 8 16-bit (4 fp32) slices.
template <int ND, int GT>
__device__ __forceinline__ void sum4(const void* const* p, int nd, int64_t i, float* g) {
    GroupSum<4> acc;
    if constexpr (ND > 0) {
        Raw4<GT> r[ND];
#pragma unroll
        for (int q = 0; q < ND; ++q) r[q].load(p[q], i);
        float t[4];
        r[0].to_f32(t);
        acc.first(t);
#pragma unroll
        for (int q = 1; q < ND; ++q) {
            r[q].to_f32(t);
            acc.add(t, ND);
        }
    } else {
        constexpr int B = GT == kGradF32 ? 4 : 8;
        for (int q = 0; q < nd; q += B) {
            const int cnt = nd - q < B ? nd - q : B;
            Raw4<GT> r[B];
#pragma unroll
            for (int u = 0; u < B; ++u)
                if (u < cnt) r[u].load(p[q + u], i);
#pragma unroll
            for (int u = 0; u < B; ++u) {
                if (u < cnt) {
                    float t[4];
                    r[u].to_f32(t);
                    if (q + u == 0) acc.first(t);
                    else acc.add(t, nd);
                }
            }
        }
    }
    acc.result(g);
}

template <int GT>
__device__ __forceinline__ float sum1(const void* const* p, int nd, int64_t j) {
    GroupSum<1> acc;
    float t = load1<GT>(p[0], j);
    acc.first(&t);
    for (int q = 1; q < nd; ++q) {
        t = load1<GT>(p[q], j);
        acc.add(&t, nd);
    }
    float s;
    acc.result(&s);
    return s;
}

template <int ND, int GT>
__global__ void __launch_bounds__(kSegThreads, kSegMinBlocks)
    rs_adamw_cast_segs(const __grid_constant__ SegTable st, int nd, float* __restrict__ P,
                       float* __restrict__ M, float* __restrict__ V,
                       uint16_t* __restrict__ out, AdamScalars c, MeanOp mo) {
    pdl_enter();
    c = resolve_adam(c);
    int s = 0;
    while (s + 1 < st.ns && static_cast<int64_t>(blockIdx.x) >= st.b0[s + 1]) ++s;
    const int64_t n = st.n[s];
    const int64_t nvec = n >> 2;
    const int64_t i = (static_cast<int64_t>(blockIdx.x) - st.b0[s]) * kSegThreads + threadIdx.x;
    const bool zero = st.po[s] < 0;        // padding rows: every contribution is +0
    const void* const* p = st.p + (zero ? 0 : st.po[s]);
    float* Ps = P + st.lo[s];
    float* Ms = M + st.lo[s];
    float* Vs = V + st.lo[s];
    uint16_t* Os = out + st.lo[s];
    if (i < nvec) {
        const uint4 p0 = ldcs16(Ps + 4 * i);
        const uint4 m0 = ldcs16(Ms + 4 * i);
        const uint4 v0 = ldcs16(Vs + 4 * i);
        float g[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (!zero) sum4<ND, GT>(p, nd, i, g);
        float pp[4], mm[4], vv[4];
        unpack4f(p0, pp);
        unpack4f(m0, mm);
        unpack4f(v0, vv);
#pragma unroll
        for (int k = 0; k < 4; ++k) adamw_elem(mean_of(g[k], mo), pp[k], mm[k], vv[k], c);
        stcs16(Ps + 4 * i, pack4f(pp));
        stcs16(Ms + 4 * i, pack4f(mm));
        stcs16(Vs + 4 * i, pack4f(vv));
        stcs8(Os + 4 * i, make_uint2(pack_bf16x2(pp[0], pp[1]), pack_bf16x2(pp[2], pp[3])));
    } else if (i == nvec) {
        // the segment's last n % 4 elements, one at a time
        for (int64_t j = nvec << 2; j < n; ++j) {
            const float g = zero ? 0.0f : sum1<GT>(p, nd, j);
            float pp = Ps[j], mm = Ms[j], vv = Vs[j];
            adamw_elem(mean_of(g, mo), pp, mm, vv, c);
            Ps[j] = pp;
            Ms[j] = mm;
            Vs[j] = vv;
            Os[j] = f32_to_bf16(pp);
        }
    }
}

// AdamW on a zero gradient over n elements: padding rows the segment kernel
// does not take (a start that is not 16-byte aligned).  Every rank's
// reduce-scatter contribution there is +0, so their rank-order sum and its
// mean are +0 whatever N_d is: the fused step's update of those positions,
// without reading the zeros.
__global__ void __launch_bounds__(kSegThreads)
    adamw_zero_grad(int64_t n, float* __restrict__ P, float* __restrict__ M,
                    float* __restrict__ V, uint16_t* __restrict__ out, AdamScalars c) {
    pdl_enter();
    c = resolve_adam(c);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kSegThreads;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kSegThreads + threadIdx.x; j < n;
         j += stride) {
        float p = P[j], m = M[j], v = V[j];
        adamw_elem(0.0f, p, m, v, c);
        P[j] = p;
        M[j] = m;
        V[j] = v;
        out[j] = f32_to_bf16(p);
    }
}

template <int ND, int GT>
cudaError_t go_segs(const SegTable& st, int nd, float* P, float* M, float* V, uint16_t* out,
                    const AdamScalars& c, const MeanOp& mo, cudaStream_t s) {
    const cudaError_t e = launch_after(rs_adamw_cast_segs<ND, GT>,
                                       dim3(static_cast<unsigned>(st.b0[st.ns])),
                                       dim3(kSegThreads), 0, s, st, nd, P, M, V, out, c, mo);
    note_launch();
    return e;
}

template <int GT>
cudaError_t dispatch_segs(const SegTable& st, int nd, float* P, float* M, float* V,
                          uint16_t* out, const AdamScalars& c, const MeanOp& mo,
                          cudaStream_t s) {
    switch (nd) {
        case 1: return go_segs<1, GT>(st, nd, P, M, V, out, c, mo, s);
        case 2: return go_segs<2, GT>(st, nd, P, M, V, out, c, mo, s);
        case 3: return go_segs<3, GT>(st, nd, P, M, V, out, c, mo, s);
        case 4: return go_segs<4, GT>(st, nd, P, M, V, out, c, mo, s);
        case 5: return go_segs<5, GT>(st, nd, P, M, V, out, c, mo, s);
        case 6: return go_segs<6, GT>(st, nd, P, M, V, out, c, mo, s);
        case 7: return go_segs<7, GT>(st, nd, P, M, V, out, c, mo, s);
        case 8: return go_segs<8, GT>(st, nd, P, M, V, out, c, mo, s);
        default: break;
    }
    // 9..16 16-bit slices compiled for their count too (all loads in
    // flight); as many fp32 slices would spill at 64 registers: the loop
    if constexpr (GT != kGradF32) {
        switch (nd) {
            case 9: return go_segs<9, GT>(st, nd, P, M, V, out, c, mo, s);
            case 10: return go_segs<10, GT>(st, nd, P, M, V, out, c, mo, s);
            case 11: return go_segs<11, GT>(st, nd, P, M, V, out, c, mo, s);
            case 12: return go_segs<12, GT>(st, nd, P, M, V, out, c, mo, s);
            case 13: return go_segs<13, GT>(st, nd, P, M, V, out, c, mo, s);
            case 14: return go_segs<14, GT>(st, nd, P, M, V, out, c, mo, s);
            case 15: return go_segs<15, GT>(st, nd, P, M, V, out, c, mo, s);
            case 16: return go_segs<16, GT>(st, nd, P, M, V, out, c, mo, s);
            default: break;
        }
    }
    return go_segs<kAnyND, GT>(st, nd, P, M, V, out, c, mo, s);
}

}  // namespace

int64_t seg_blocks(int64_t n) {
    const int64_t slots = (n + 3) / 4;     // 4-element vectors, the last one partial
    return (slots + kSegThreads - 1) / kSegThreads;
}

cudaError_t launch_adamw_zero_grad(int64_t n, float* master, float* m, float* v, uint16_t* out,
                                   const AdamScalars& c, cudaStream_t stream) {
    // one pass (the loop strides only past 2^31 - 1 blocks)
    int64_t blocks = (n + kSegThreads - 1) / kSegThreads;
    if (blocks > (int64_t{1} << 31) - 1) blocks = (int64_t{1} << 31) - 1;
    const cudaError_t e = launch_after(adamw_zero_grad, dim3(static_cast<unsigned>(blocks)),
                                       dim3(kSegThreads), 0, stream, n, master, m, v, out, c);
    note_launch();
    return e;
}

cudaError_t launch_rs_adamw_cast_segs(const SegTable& st, int nd, int grad_type, float* master,
                                      float* m, float* v, uint16_t* out, const AdamScalars& c,
                                      const MeanOp& mo, cudaStream_t stream) {
    switch (grad_type) {
        case kGradF32: return dispatch_segs<kGradF32>(st, nd, master, m, v, out, c, mo, stream);
        case kGradF16: return dispatch_segs<kGradF16>(st, nd, master, m, v, out, c, mo, stream);
        default: return dispatch_segs<kGradBF16>(st, nd, master, m, v, out, c, mo, stream);
    }
}

}  // namespace shardstep
