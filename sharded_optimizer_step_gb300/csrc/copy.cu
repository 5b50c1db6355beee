// Copy-shaped kernels: the batched segment copies behind fsdp_flat_pack,
// fsdp_ag_unpack and the FSDP2 chunk-cat / copy-out, and the register-staged
// micro-batch gradient accumulation.
//
// Aligned copy (copy16): ranges whose source, destination and size are all
// multiples of 16 bytes, one block per 16 KB chunk (256 threads x 4
// vectors, streaming loads and stores), the chunks of every range in one
// grid that the hardware schedules at full occupancy (32 registers).  On
// GB300 it moved a 405 MB all-gather at 6.82 TB/s, against 6.19 TB/s for
// the same copy staged through shared memory by bulk copies (one persistent
// CTA per SM) and 6.67 TB/s for torch's device copy of the same size.
//
// Realigning copy (copy16_shift): ranges whose destination and size are
// multiples of 16 bytes but whose source is not, such as a tensor packed at
// an odd element offset.  Each destination vector takes 16 bytes that
// straddle two aligned source vectors: a lane loads both (the second is its
// neighbour lane's first, so DRAM sees each byte once and the repeat is
// served by L2), all of its loads before any store, and funnel-shifts the
// pair into place.  Every aligned vector it reads holds bytes of the source
// range, so no read leaves the 16-byte vectors around the range's ends.  On
// GB300, packing a 256 MB tensor at an odd bf16 offset moved 5.7-5.9 TB/s
// this way, 5.3-5.6 TB/s when the second vector came from the neighbour lane
// by warp shuffles, and 4.0 TB/s through the segment copy (2-byte vectors).
//
// Segment copy: one launch moves up to kMaxCopySegs byte ranges.  Each
// segment is cut into chunks of 1024 vectors; blocks stride over the chunks
// of all segments, so large and small tensors share one balanced grid.  The
// vector width of a segment is the widest of 16/8/4/2/1 bytes for which
// source and destination are congruent; a head of up to width-1 bytes brings
// the destination to that alignment and the tail is copied byte-wise, both by
// the lanes of the block that owns the segment's first / last chunk.
//
// Every launch of a call goes out as a programmatic dependent of the kernel
// before it (unless dependent launches are switched off).  The first one
// (wait_first) waits for that unknown predecessor before it touches memory
// and only then lets the next kernel be scheduled.  One call's copies are
// disjoint and read nothing the call writes, so the second and later ones
// let the next kernel be scheduled as soon as all of their own blocks have
// started and wait for the previous grid of the call only before they end
// (both no-ops for an ordinary launch): a call that mixes congruent and
// realigned ranges, heads and tails runs without an idle gap between its
// kernels.
#include "common.cuh"

namespace shardstep {
namespace {

template <typename T>
__device__ __forceinline__ T load_vec(const T* p) {
    return *p;
}
template <>
__device__ __forceinline__ uint4 load_vec<uint4>(const uint4* p) {
    return ld_once(p);
}
template <typename T>
__device__ __forceinline__ void store_vec(T* p, const T& v) {
    *p = v;
}
template <>
__device__ __forceinline__ void store_vec<uint4>(uint4* p, const uint4& v) {
    st_stream(p, v);
}

template <typename T>
__device__ __forceinline__ void copy_vecs(const char* src, char* dst, int64_t v0, int64_t v1) {
    const T* s = reinterpret_cast<const T*>(src);
    T* d = reinterpret_cast<T*>(dst);
    constexpr int U = kCopyVecsPerChunk / kThreads;
    if (src != nullptr) {
        T r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = v0 + u * kThreads + threadIdx.x;
            if (k < v1) r[u] = load_vec<T>(s + k);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = v0 + u * kThreads + threadIdx.x;
            if (k < v1) store_vec<T>(d + k, r[u]);
        }
    } else {
        T z;
        memset(&z, 0, sizeof(T));
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t k = v0 + u * kThreads + threadIdx.x;
            if (k < v1) store_vec<T>(d + k, z);
        }
    }
}

__global__ void __launch_bounds__(kThreads) copy_segments(CopyTable t, int wait_first) {
    if (wait_first) pdl_wait();   // before the trigger: see pdl_enter
    pdl_trigger();
    int seg = 0;
    for (int64_t c = blockIdx.x; c < t.total_chunks; c += gridDim.x) {
        while (seg + 1 < t.n && t.s[seg + 1].chunk0 <= c) ++seg;
        const CopySeg& sg = t.s[seg];
        const int64_t local = c - sg.chunk0;
        const int64_t nchunks =
            sg.body > 0 ? (sg.body + kCopyVecsPerChunk - 1) / kCopyVecsPerChunk : 1;
        const char* src = sg.src ? sg.src + sg.head : nullptr;
        char* dst = sg.dst + sg.head;
        const int64_t v0 = local * kCopyVecsPerChunk;
        const int64_t v1 = v0 + kCopyVecsPerChunk < sg.body ? v0 + kCopyVecsPerChunk : sg.body;
        switch (sg.width) {
            case 16: copy_vecs<uint4>(src, dst, v0, v1); break;
            case 8: copy_vecs<uint2>(src, dst, v0, v1); break;
            case 4: copy_vecs<uint32_t>(src, dst, v0, v1); break;
            case 2: copy_vecs<uint16_t>(src, dst, v0, v1); break;
            default: copy_vecs<uint8_t>(src, dst, v0, v1); break;
        }
        if (local == 0 && threadIdx.x < sg.head)
            sg.dst[threadIdx.x] = sg.src ? sg.src[threadIdx.x] : 0;
        if (local == nchunks - 1) {
            const int64_t done = sg.head + sg.body * sg.width;
            const int64_t tail = sg.bytes - done;
            if (threadIdx.x < tail)
                sg.dst[done + threadIdx.x] = sg.src ? sg.src[done + threadIdx.x] : 0;
        }
    }
    pdl_wait();
}

__global__ void __launch_bounds__(kThreads, 8) copy16(AlignedTable t, int wait_first) {
    if (wait_first) pdl_wait();   // before the trigger: see pdl_enter
    pdl_trigger();
    const int64_t c = blockIdx.x;
    int lo = 0, hi = t.n - 1;  // the range owning chunk c (chunk0 increasing)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (t.s[mid].chunk0 <= c) lo = mid;
        else hi = mid - 1;
    }
    const AlignedSeg& sg = t.s[lo];
    constexpr int kVecs = kAlignedChunk / 16;  // 1024 = 256 threads x 4
    const int64_t v0 = (c - sg.chunk0) * kVecs;
    const int64_t nv = sg.bytes / 16;
    const uint4* src = reinterpret_cast<const uint4*>(sg.src);
    uint4* dst = reinterpret_cast<uint4*>(sg.dst);
    uint4 r[kVecs / kThreads];
#pragma unroll
    for (int u = 0; u < kVecs / kThreads; ++u) {
        const int64_t k = v0 + u * kThreads + threadIdx.x;
        if (k < nv) r[u] = ld_once(src + k);
    }
#pragma unroll
    for (int u = 0; u < kVecs / kThreads; ++u) {
        const int64_t k = v0 + u * kThreads + threadIdx.x;
        if (k < nv) st_stream(dst + k, r[u]);
    }
    pdl_wait();
}

// Bytes [delta, delta + 16) of the 32-byte pair (a, b), delta = 4 * ws + sh / 8.
__device__ __forceinline__ uint4 shift_pair(const uint4& a, const uint4& b, int ws, int sh) {
    uint32_t w0, w1, w2, w3, w4;
    switch (ws) {
        case 0: w0 = a.x; w1 = a.y; w2 = a.z; w3 = a.w; w4 = b.x; break;
        case 1: w0 = a.y; w1 = a.z; w2 = a.w; w3 = b.x; w4 = b.y; break;
        case 2: w0 = a.z; w1 = a.w; w2 = b.x; w3 = b.y; w4 = b.z; break;
        default: w0 = a.w; w1 = b.x; w2 = b.y; w3 = b.z; w4 = b.w; break;
    }
    return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh),
                      __funnelshift_r(w2, w3, sh), __funnelshift_r(w3, w4, sh));
}

__global__ void __launch_bounds__(kThreads, 5) copy16_shift(AlignedTable t, int wait_first) {
    if (wait_first) pdl_wait();   // before the trigger: see pdl_enter
    pdl_trigger();
    const int64_t c = blockIdx.x;
    int lo = 0, hi = t.n - 1;  // the range owning chunk c (chunk0 increasing)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (t.s[mid].chunk0 <= c) lo = mid;
        else hi = mid - 1;
    }
    const AlignedSeg& sg = t.s[lo];
    constexpr int kVecs = kAlignedChunk / 16;  // 1024 = 256 threads x 4
    const int64_t v0 = (c - sg.chunk0) * kVecs;
    const int64_t nv = sg.bytes / 16;
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(sg.src);
    const int delta = static_cast<int>(s0 & 15u);  // 1..15
    const uint4* src = reinterpret_cast<const uint4*>(s0 - delta);
    uint4* dst = reinterpret_cast<uint4*>(sg.dst);
    const int ws = delta >> 2, sh = (delta & 3) * 8;
    constexpr int U = kVecs / kThreads;
    uint4 a[U], b[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t k = v0 + u * kThreads + threadIdx.x;
        if (k < nv) {
            a[u] = ld_once(src + k);
            b[u] = ld_once(src + k + 1);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t k = v0 + u * kThreads + threadIdx.x;
        if (k < nv) st_stream(dst + k, shift_pair(a[u], b[u], ws, sh));
    }
    pdl_wait();
}

// ------------------------------------------------------- accumulation

template <bool FIRST>
__device__ __forceinline__ void acc_scalar(const uint16_t* g, float* acc, int64_t j,
                                           float scale) {
    const float t = __fmul_rn(bf16_to_f32(g[j]), scale);
    acc[j] = FIRST ? t : __fadd_rn(acc[j], t);
}

// One 8-element vector per thread in a one-pass grid (the loop strides only
// past 2^31 - 1 blocks); 8 blocks per SM, at most 32 registers.  On GB300
// (1.2G elements) this moved 7.0 TB/s for the first micro-batch and 7.2 TB/s
// for the others, against 6.0 and 6.6 TB/s for the TMA-staged kernel; the
// same kernel with a grid-stride loop over one wave of blocks moved 5.7 TB/s
// over a whole accumulation.
template <bool FIRST>
__global__ void __launch_bounds__(kThreads, 8)
    accumulate_vec8(const uint16_t* __restrict__ g, float* __restrict__ acc, int64_t n,
                    float scale) {
    pdl_enter();
    const int64_t nvec = n >> 3;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < nvec;
         i += stride) {
        const uint4 gr = ld_once(g + 8 * i);
        float a[8];
        if (!FIRST) {
            unpack4f(ld_rw(acc + 8 * i), a);
            unpack4f(ld_rw(acc + 8 * i + 4), a + 4);
        }
        float f[8];
        unpack8(gr, f);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float t = __fmul_rn(f[k], scale);
            a[k] = FIRST ? t : __fadd_rn(a[k], t);
        }
        st_stream(acc + 8 * i, pack4f(a));
        st_stream(acc + 8 * i + 4, pack4f(a + 4));
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 7))
        acc_scalar<FIRST>(g, acc, (nvec << 3) + threadIdx.x, scale);
}

template <bool FIRST>
__global__ void __launch_bounds__(kThreads)
    accumulate_scalar(const uint16_t* __restrict__ g, float* __restrict__ acc, int64_t n,
                      float scale) {
    pdl_enter();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; j < n;
         j += stride)
        acc_scalar<FIRST>(g, acc, j, scale);
}

unsigned grid_for(const void* kernel, int64_t work_items) {
    const int64_t want = (work_items + kThreads - 1) / kThreads;
    const int64_t cap = static_cast<int64_t>(device_sms()) * resident_blocks(kernel, kThreads);
    const int64_t g = want < cap ? want : cap;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

unsigned grid_one_pass(int64_t vectors) {
    const int64_t want = (vectors + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t{1} << 31) - 1;
    const int64_t g = want < cap ? want : cap;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

template <typename Table>
cudaError_t launch_table(void (*kernel)(Table, int), unsigned grid, const Table& t, bool pdl,
                         bool wait_first, cudaStream_t stream) {
    cudaError_t e;
    if (pdl) {
        e = launch_dependent(kernel, dim3(grid), dim3(kThreads), 0, stream, t,
                             wait_first ? 1 : 0);
    } else {
        kernel<<<grid, kThreads, 0, stream>>>(t, 0);
        e = cudaGetLastError();
    }
    note_launch();
    return e;
}

}  // namespace

cudaError_t launch_copy(const CopyTable& t, bool pdl, bool wait_first, cudaStream_t stream) {
    const int64_t cap = static_cast<int64_t>(device_sms()) *
                        resident_blocks(reinterpret_cast<const void*>(copy_segments), kThreads);
    const int64_t g = t.total_chunks < cap ? t.total_chunks : cap;
    return launch_table(copy_segments, static_cast<unsigned>(g < 1 ? 1 : g), t, pdl, wait_first,
                        stream);
}

cudaError_t launch_copy16(const AlignedTable& t, bool pdl, bool wait_first, cudaStream_t stream) {
    return launch_table(copy16, static_cast<unsigned>(t.total_chunks), t, pdl, wait_first,
                        stream);
}

cudaError_t launch_copy16_shift(const AlignedTable& t, bool pdl, bool wait_first,
                                cudaStream_t stream) {
    return launch_table(copy16_shift, static_cast<unsigned>(t.total_chunks), t, pdl, wait_first,
                        stream);
}

cudaError_t launch_accumulate(const uint16_t* g, float* acc, int64_t n, float scale, bool first,
                              bool vec, cudaStream_t stream) {
    auto kernel = vec ? (first ? accumulate_vec8<true> : accumulate_vec8<false>)
                      : (first ? accumulate_scalar<true> : accumulate_scalar<false>);
    const unsigned grid = vec ? grid_one_pass(n >> 3)
                              : grid_for(reinterpret_cast<const void*>(kernel), n);
    const cudaError_t e = launch_after(kernel, dim3(grid), dim3(kThreads), 0, stream, g, acc, n,
                                       scale);
    note_launch();
    return e;
}

}  // namespace shardstep
