// TMA-staged streaming kernels: the fused sharded step (reduce-scatter
// average + AdamW + bf16 cast), the micro-batch gradient accumulation, the
// DDP bucket all-reduce average and the gradient scaler's non-finite check.
// They need every source 16-byte aligned and two stages in shared memory.
// The automatic kernel choice takes them where they measured faster than the
// one-pass register-staged kernels: the fused step and the check at the N_d
// those are not compiled for, the all-reduce on buckets of 32M elements and
// more at N_d >= 3.
//
// One skeleton serves all four.  One CTA per SM, 17 warps.  Warp 16's first
// lane is the producer: for each tile of 2048 elements it issues one
// cp.async.bulk per input array (a gradient slice, a state array, an
// accumulator) from HBM into a shared-memory stage and completes them on that
// stage's mbarrier (expect-tx).  Warps 0..15 consume: they wait on the
// stage's barrier, compute on 4 elements per thread from shared memory and
// write the results straight to HBM with streaming stores, then each warp
// arrives on the stage's "empty" barrier so the producer can refill it.
// Tiles are dealt round-robin over the grid.  The number of stages is chosen
// per launch so that about 128 KB of tiles are in flight per SM (2 stages of
// 57 KB for the fused step at N_d = 8 and bf16, 4 of 28 KB at N_d = 1, 8
// of 12 KB for an accumulation), at least 2 and at most 16, rounded down to
// one of the instantiated counts 2, 3, 4, 6, 8, 12, 16.
//
// Every wait is bounded (by default about two seconds of %globaltimer; a
// process-wide setting passed to each launch, shardstep_set_tma_wait_ns).  A
// wait that runs out sets a bit in the device status word
// (shardstep_device_status) and the waiting warp returns.  No CTA exits
// while a bulk copy it issued may still be writing its shared memory: before
// it returns, on every path, the producer lane waits for the copies of the
// last tiles it issued (the earlier ones were consumed, so they landed).
// That drain waits on copies from validated, in-bounds global memory, which
// always complete; its own limit (kDrainNs, two seconds) is fixed, so a short
// watchdog setting never cuts it short.  Nothing here spins on another CTA
// or on the host.
#include <atomic>

#include "common.cuh"

namespace shardstep {

// Watchdog status of this device's TMA-staged launches (0 = no wait ran out).
__device__ unsigned int g_device_status = 0;

namespace {

constexpr int kTile = 2048;
constexpr int kMaxStages = 16;
// Reads kept in flight per SM: the stage count is chosen so that about this
// many bytes of tiles are staged (at least 2 stages).  Measured on GB300 for
// the fused step at N_d = 8 (57 KB stages), N_d = 1 (28 KB), the bucket
// all-reduce (32 KB) and the accumulation (12 KB): each is fastest at 100 to
// 130 KB per SM; filling all 227 KB of shared memory is slower (5.51 vs
// 5.15 ms for the N_d = 8 step over 842M elements).
constexpr size_t kTargetInflight = 128 * 1024;
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;   // 512: 4 elements each per tile
constexpr int kTmaThreads = kConsumers + 32;      // + the producer warp
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;
constexpr unsigned long long kDrainNs = 2000000000ull;
constexpr size_t kBarrierBytes = 2 * kMaxStages * sizeof(uint64_t);
// Left for the kernels' static shared memory (the step scalars' broadcast).
constexpr size_t kStaticSmemReserve = 1024;

constexpr unsigned kStatusConsumerTimeout = 1u;
constexpr unsigned kStatusProducerTimeout = 2u;
constexpr unsigned kStatusDrainTimeout = 4u;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
// Non-blocking test of the phase of `parity`.
__device__ __forceinline__ bool mbar_test_now(uint64_t* b, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return done != 0;
}
// Limits below this are a test control: their waits poll without blocking
// and read the clock after every poll, so that they run out even when each
// blocking poll would have lasted until the copy landed.
constexpr unsigned long long kShortWaitNs = 1000000ull;
// Waits for the phase of `parity` to complete; false after limit_ns.  The
// usual limit polls with try_wait, which suspends the thread until the
// phase completes or a hardware time slice ends, and reads the clock every
// 256 polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity,
                                          unsigned long long limit_ns) {
    const unsigned long long t0 = now_ns();
    if (limit_ns < kShortWaitNs) {
        while (!mbar_test_now(b, parity))
            if (now_ns() - t0 > limit_ns) return false;
        return true;
    }
    for (uint32_t k = 1;; ++k) {
        if (mbar_test(b, parity)) return true;
        if ((k & 255u) == 0 && now_ns() - t0 > limit_ns) return false;
    }
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 4 consecutive gradient elements of type GT from shared memory, as fp32.
template <int GT>
__device__ __forceinline__ void load4_smem(const uint8_t* p, float* f) {
    if (GT == kGradF32) {
        const float4 x = *reinterpret_cast<const float4*>(p);
        f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
    } else if (GT == kGradF16) {
        const uint2 r = *reinterpret_cast<const uint2*>(p);
        f[0] = f16_to_f32(static_cast<uint16_t>(r.x & 0xFFFFu));
        f[1] = f16_to_f32(static_cast<uint16_t>(r.x >> 16));
        f[2] = f16_to_f32(static_cast<uint16_t>(r.y & 0xFFFFu));
        f[3] = f16_to_f32(static_cast<uint16_t>(r.y >> 16));
    } else {
        const uint2 r = *reinterpret_cast<const uint2*>(p);
        f[0] = bf16_lo(r.x); f[1] = bf16_hi(r.x);
        f[2] = bf16_lo(r.y); f[3] = bf16_hi(r.y);
    }
}

template <int GT>
__device__ __forceinline__ float grad1(const void* base, int64_t j) {
    if (GT == kGradF32) return static_cast<const float*>(base)[j];
    if (GT == kGradF16) return f16_to_f32(static_cast<const uint16_t*>(base)[j]);
    return bf16_to_f32(static_cast<const uint16_t*>(base)[j]);
}

template <int GT>
__host__ __device__ constexpr uint32_t grad_bytes() {
    return GT == kGradF32 ? 4u : 2u;
}

// The N_d slices of one tile reduced at 4 consecutive elements, in the order
// GroupSum fixes (rank order; grouped for hybrid sharding), from a stage that
// holds the slices back to back (kTile elements each).
template <int GT>
__device__ __forceinline__ void reduce4_smem(const uint8_t* st, int nd, int group, int e,
                                             float* g) {
    constexpr uint32_t gsz = grad_bytes<GT>();
    GroupSum<4> acc;
    {
        float t[4];
        load4_smem<GT>(st + e * gsz, t);
        acc.first(t);
    }
    for (int q = 1; q < nd; ++q) {
        float t[4];
        load4_smem<GT>(st + q * (kTile * gsz) + e * gsz, t);
        acc.add(t, group);
    }
    acc.result(g);
}

// The same sum at one element, read from global memory (the < 8 tail).
template <int GT>
__device__ __forceinline__ float reduce1_global(const PtrTable& tab, int nd, int group,
                                                int64_t j) {
    GroupSum<1> acc;
    float t = grad1<GT>(tab.p[0], j);
    acc.first(&t);
    for (int q = 1; q < nd; ++q) {
        t = grad1<GT>(tab.p[q], j);
        acc.add(&t, group);
    }
    float s;
    acc.result(&s);
    return s;
}

__device__ __forceinline__ bool not_finite(float x) {
    return (__float_as_uint(x) & 0x7F800000u) == 0x7F800000u;
}

// ------------------------------------------------------------ the skeleton
//
// An Op (passed by value as the kernel parameter, read-only) provides
//   State                                  per-thread mutable state
//   skipped()                              true: every thread returns at once
//   init()                                 the thread's State
//   stage_bytes()                          one stage (a multiple of 16 bytes)
//   tx_bytes(e0, n)                        bytes the copies of the n-element tile at e0 bring
//   issue(stage, e0, n, bar)               the producer lane's bulk copies of a tile
//   consume(stage, e0, e, state)           4 elements at tile offset e
//   tail(j, state)                         element j past the tiles, global loads
//   finish(state, lane)                    whole consumer warps, after the loop
//
// n_main = n rounded down to a multiple of 8 is covered by tiles (the last one
// possibly shorter, still a multiple of 8 elements, so every bulk copy is a
// multiple of 16 bytes); the final n - n_main < 8 elements go to block 0's
// first threads with ordinary loads.
static_assert(kConsumers * 4 == kTile, "one group of 4 elements per consumer thread per tile");

// NST, the number of stages, is a compile-time constant: with a runtime count
// the same kernel issued 24% more instructions and ran 1.4% slower (5.15 vs
// 5.08 ms for the N_d = 8 step over 842M elements).
template <class Op, int NST>
__device__ __forceinline__ void staged_body(const Op& op, int64_t n,
                                            unsigned long long wait_ns) {
    constexpr int nst = NST;
    if (op.skipped()) return;
    typename Op::State state = op.init();
    const uint32_t stage_bytes = op.stage_bytes();
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(nst) * stage_bytes);
    uint64_t* empty = full + nst;
    const int tid = threadIdx.x;
    const int64_t n_main = n & ~static_cast<int64_t>(7);
    const int64_t ntiles = (n_main + kTile - 1) / kTile;
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int64_t my_tiles =
        ntiles > blockIdx.x ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

    if (tid >= kConsumers) {  // producer warp
        if (tid != kConsumers) return;
        int64_t j = 0;
        int s = 0;
        uint32_t use = 0;
        bool ok = true;
        for (; j < my_tiles; ++j) {
            if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1u, wait_ns)) {
                ok = false;
                break;
            }
            const int64_t e0 = (static_cast<int64_t>(blockIdx.x) + j * gridDim.x) * kTile;
            const uint32_t cnt = static_cast<uint32_t>(n_main - e0 < kTile ? n_main - e0 : kTile);
            mbar_expect_tx(&full[s], op.tx_bytes(e0, cnt));
            op.issue(smem + static_cast<size_t>(s) * stage_bytes, e0, cnt, &full[s]);
            if (++s == nst) {
                s = 0;
                ++use;
            }
        }
        if (!ok) atomicOr(&g_device_status, kStatusProducerTimeout);
        // Tiles 0..j-1 were issued.  A stage was refilled only after its
        // consumers released it, so every tile before the last nst has
        // landed; the last nst (or fewer) land in this CTA's shared memory
        // and are waited for here, whether or not the consumers are still
        // there to see them, before the CTA may exit.
        bool drained = true;
        for (int64_t k = j > nst ? j - nst : 0; k < j; ++k)
            drained = mbar_wait(&full[k % nst], static_cast<uint32_t>(k / nst) & 1u, kDrainNs) &&
                      drained;
        if (!drained) atomicOr(&g_device_status, kStatusDrainTimeout);
        return;
    }

    // consumers: every lane waits (each gets the barrier's acquire), the
    // warp takes one decision
    const int lane = tid & 31;
    const int e = tid * 4;
    int s = 0;
    uint32_t use = 0;
    for (int64_t j = 0; j < my_tiles; ++j) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], use & 1u, wait_ns))) {
            if (lane == 0) atomicOr(&g_device_status, kStatusConsumerTimeout);
            return;
        }
        const int64_t e0 = (static_cast<int64_t>(blockIdx.x) + j * gridDim.x) * kTile;
        const int64_t cnt = n_main - e0 < kTile ? n_main - e0 : kTile;
        if (e < cnt) op.consume(smem + static_cast<size_t>(s) * stage_bytes, e0, e, state);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == nst) {
            s = 0;
            ++use;
        }
    }
    if (blockIdx.x == 0 && tid < n - n_main) op.tail(n_main + tid, state);
    op.finish(state, lane);
}

// The kernel lets a programmatically dependent launch (the next bucket of the
// same all-reduce call) start as soon as every CTA has begun, and does not
// end before the grid it depends on has ended, so that stream order still
// holds for whatever runs after the last launch.  Both are no-ops for an
// ordinary launch.
template <class Op, int NST>
__global__ void __launch_bounds__(kTmaThreads, 1)
    staged_stream(const Op op, int64_t n, unsigned long long wait_ns) {
    pdl_trigger();
    staged_body<Op, NST>(op, n, wait_ns);
    pdl_wait();
}

// ------------------------------------------------------------------ ops

// The fused sharded step: N_d gradient slices + master / m / v in; master /
// m / v and the bf16 parameter out.  Stage: the slices, then the 3 state
// arrays, kTile elements each.
template <int GT>
struct AdamOp {
    PtrTable tab;
    int nd;
    float* P;
    float* M;
    float* V;
    uint16_t* out;
    AdamScalars c;
    MeanOp mo;
    const unsigned int* skip;

    struct State {
        MeanOp mo;
        AdamScalars c;
    };
    static constexpr uint32_t gsz = grad_bytes<GT>();
    __device__ bool skipped() const { return skip_step(skip); }
    __device__ State init() const { return State{resolve_scale(mo), resolve_adam(c)}; }
    __host__ __device__ uint32_t stage_bytes() const {
        return static_cast<uint32_t>(nd) * kTile * gsz + 3u * kTile * 4u;
    }
    __device__ uint32_t tx_bytes(int64_t, uint32_t n) const { return nd * n * gsz + 3u * n * 4u; }
    __device__ void issue(uint8_t* st, int64_t e0, uint32_t n, uint64_t* bar) const {
        for (int q = 0; q < nd; ++q)
            bulk_load(st + q * (kTile * gsz), static_cast<const uint8_t*>(tab.p[q]) + e0 * gsz,
                      n * gsz, bar);
        uint8_t* sst = st + nd * (kTile * gsz);
        bulk_load(sst, P + e0, n * 4, bar);
        bulk_load(sst + kTile * 4, M + e0, n * 4, bar);
        bulk_load(sst + 2 * kTile * 4, V + e0, n * 4, bar);
    }
    __device__ void consume(const uint8_t* st, int64_t e0, int e, State& s) const {
        float g[4];
        reduce4_smem<GT>(st, nd, s.mo.group, e, g);
        const uint8_t* sst = st + nd * (kTile * gsz);
        const float4 pp = *reinterpret_cast<const float4*>(sst + e * 4);
        const float4 mm = *reinterpret_cast<const float4*>(sst + kTile * 4 + e * 4);
        const float4 vv = *reinterpret_cast<const float4*>(sst + 2 * kTile * 4 + e * 4);
        float p[4] = {pp.x, pp.y, pp.z, pp.w};
        float m[4] = {mm.x, mm.y, mm.z, mm.w};
        float v[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) adamw_elem(mean_of(g[k], s.mo), p[k], m[k], v[k], s.c);
        const int64_t ge = e0 + e;
        stcs16(P + ge, pack4f(p));
        stcs16(M + ge, pack4f(m));
        stcs16(V + ge, pack4f(v));
        stcs8(out + ge, make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3])));
    }
    __device__ void tail(int64_t j, State& s) const {
        float p = P[j], m = M[j], v = V[j];
        adamw_elem(mean_of(reduce1_global<GT>(tab, nd, s.mo.group, j), s.mo), p, m, v, s.c);
        P[j] = p;
        M[j] = m;
        V[j] = v;
        out[j] = f32_to_bf16(p);
    }
    __device__ void finish(State&, int) const {}
};

// Micro-batch accumulation: acc = g*scale (first) or acc + g*scale, one
// rounding per operation.  Stage: the bf16 gradient tile, then (not first)
// the fp32 accumulator tile.
template <bool FIRST>
struct AccumOp {
    const uint16_t* g;
    float* acc;
    float scale;

    struct State {};
    __device__ bool skipped() const { return false; }
    __device__ State init() const { return State{}; }
    __host__ __device__ uint32_t stage_bytes() const {
        return kTile * 2u + (FIRST ? 0u : kTile * 4u);
    }
    __device__ uint32_t tx_bytes(int64_t, uint32_t n) const { return n * 2u + (FIRST ? 0u : n * 4u); }
    __device__ void issue(uint8_t* st, int64_t e0, uint32_t n, uint64_t* bar) const {
        bulk_load(st, g + e0, n * 2, bar);
        if (!FIRST) bulk_load(st + kTile * 2, acc + e0, n * 4, bar);
    }
    __device__ void consume(const uint8_t* st, int64_t e0, int e, State&) const {
        float f[4], a[4];
        load4_smem<kGradBF16>(st + e * 2, f);
        if (!FIRST) {
            const float4 x = *reinterpret_cast<const float4*>(st + kTile * 2 + e * 4);
            a[0] = x.x; a[1] = x.y; a[2] = x.z; a[3] = x.w;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float t = __fmul_rn(f[k], scale);
            a[k] = FIRST ? t : __fadd_rn(a[k], t);
        }
        stcs16(acc + e0 + e, pack4f(a));
    }
    __device__ void tail(int64_t j, State&) const {
        const float t = __fmul_rn(bf16_to_f32(g[j]), scale);
        acc[j] = FIRST ? t : __fadd_rn(acc[j], t);
    }
    __device__ void finish(State&, int) const {}
};

// DDP bucket all-reduce average: N_d bf16 slices in, the bf16 mean out.
struct MeanOutOp {
    PtrTable tab;
    int nd;
    uint16_t* out;
    MeanOp mo;

    using State = MeanOp;
    __device__ bool skipped() const { return false; }
    __device__ State init() const { return mo; }
    __host__ __device__ uint32_t stage_bytes() const {
        return static_cast<uint32_t>(nd) * kTile * 2u;
    }
    __device__ uint32_t tx_bytes(int64_t, uint32_t n) const { return nd * n * 2u; }
    __device__ void issue(uint8_t* st, int64_t e0, uint32_t n, uint64_t* bar) const {
        for (int q = 0; q < nd; ++q)
            bulk_load(st + q * (kTile * 2), static_cast<const uint16_t*>(tab.p[q]) + e0, n * 2,
                      bar);
    }
    __device__ void consume(const uint8_t* st, int64_t e0, int e, State& m0) const {
        float g[4];
        reduce4_smem<kGradBF16>(st, nd, m0.group, e, g);
#pragma unroll
        for (int k = 0; k < 4; ++k) g[k] = mean_of(g[k], m0);
        stcs8(out + e0 + e, make_uint2(pack_bf16x2(g[0], g[1]), pack_bf16x2(g[2], g[3])));
    }
    __device__ void tail(int64_t j, State& m0) const {
        out[j] = f32_to_bf16(mean_of(reduce1_global<kGradBF16>(tab, nd, m0.group, j), m0));
    }
    __device__ void finish(State&, int) const {}
};

// Gradient scaler's check: sets *found when any unscaled mean gradient is
// inf or NaN.  Reads the slices only; one atomic per warp that saw one.
template <int GT>
struct CheckOp {
    PtrTable tab;
    int nd;
    MeanOp mo;
    unsigned int* found;

    struct State {
        MeanOp mo;
        bool bad;
        bool bits;   // fp16 slices decided on their bits (f16_check_on_bits)
    };
    static constexpr uint32_t gsz = grad_bytes<GT>();
    __device__ bool skipped() const { return false; }
    __device__ State init() const {
        const MeanOp m = resolve_scale(mo);
        return State{m, false, GT == kGradF16 && f16_check_on_bits(m)};
    }
    __host__ __device__ uint32_t stage_bytes() const {
        return static_cast<uint32_t>(nd) * kTile * gsz;
    }
    __device__ uint32_t tx_bytes(int64_t, uint32_t n) const { return nd * n * gsz; }
    __device__ void issue(uint8_t* st, int64_t e0, uint32_t n, uint64_t* bar) const {
        for (int q = 0; q < nd; ++q)
            bulk_load(st + q * (kTile * gsz), static_cast<const uint8_t*>(tab.p[q]) + e0 * gsz,
                      n * gsz, bar);
    }
    __device__ void consume(const uint8_t* st, int64_t, int e, State& s) const {
        if (GT == kGradF16 && s.bits) {
            for (int q = 0; q < nd; ++q) {
                const uint2 r = *reinterpret_cast<const uint2*>(st + q * (kTile * gsz) + e * gsz);
                s.bad |= f16x2_nonfinite(r.x) | f16x2_nonfinite(r.y);
            }
            return;
        }
        float g[4];
        reduce4_smem<GT>(st, nd, s.mo.group, e, g);
#pragma unroll
        for (int k = 0; k < 4; ++k) s.bad |= not_finite(mean_of(g[k], s.mo));
    }
    __device__ void tail(int64_t j, State& s) const {
        if (GT == kGradF16 && s.bits) {
            for (int q = 0; q < nd; ++q)
                s.bad |= f16_nonfinite(static_cast<const uint16_t*>(tab.p[q])[j]);
            return;
        }
        s.bad |= not_finite(mean_of(reduce1_global<GT>(tab, nd, s.mo.group, j), s.mo));
    }
    __device__ void finish(State& s, int lane) const {
        if (__any_sync(0xFFFFFFFFu, s.bad) && lane == 0) atomicOr(found, 1u);
    }
};

// --------------------------------------------------------------- launch

std::atomic<int> g_stage_limit{0};  // 0: about kTargetInflight bytes of stages
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};

// The stage counts instantiated; a launch takes the largest one not above
// what it asks for.
constexpr int kStageSet[] = {2, 3, 4, 6, 8, 12, 16};

int stages_for(size_t stage_bytes) {
    const size_t optin = static_cast<size_t>(device_smem_optin()) - kStaticSmemReserve;
    size_t fit = optin > kBarrierBytes ? (optin - kBarrierBytes) / stage_bytes : 0;
    if (fit > static_cast<size_t>(kMaxStages)) fit = kMaxStages;
    const int lim = g_stage_limit.load(std::memory_order_relaxed);
    size_t want = lim >= 2 ? static_cast<size_t>(lim) : kTargetInflight / stage_bytes;
    if (want > fit) want = fit;
    int nst = 2;
    for (int k : kStageSet)
        if (static_cast<size_t>(k) <= want) nst = k;
    return nst;
}

template <class Op, int NST>
cudaError_t launch_stages(const Op& op, int64_t n, cudaStream_t stream, bool pdl) {
    static int attr_set[256];  // per instantiation: dynamic shared memory opt-in applied
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 256 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(staged_stream<Op, NST>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 device_smem_optin() - static_cast<int>(kStaticSmemReserve));
        if (e != cudaSuccess) return e;
        attr_set[dev] = 1;
    }
    const size_t smem = static_cast<size_t>(NST) * op.stage_bytes() + kBarrierBytes;
    const int64_t ntiles = ((n & ~static_cast<int64_t>(7)) + kTile - 1) / kTile;
    int64_t grid = device_sms();
    if (grid > ntiles) grid = ntiles;
    if (grid < 1) grid = 1;
    const unsigned long long wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    if (pdl) {
        e = launch_dependent(staged_stream<Op, NST>, dim3(static_cast<unsigned>(grid)),
                             dim3(kTmaThreads), smem, stream, op, n, wait_ns);
    } else {
        staged_stream<Op, NST><<<static_cast<unsigned>(grid), kTmaThreads, smem, stream>>>(
            op, n, wait_ns);
        e = cudaGetLastError();
    }
    note_launch();
    return e;
}

template <class Op>
cudaError_t launch_staged(const Op& op, int64_t n, cudaStream_t stream, bool pdl = false) {
    switch (stages_for(op.stage_bytes())) {
        case 3: return launch_stages<Op, 3>(op, n, stream, pdl);
        case 4: return launch_stages<Op, 4>(op, n, stream, pdl);
        case 6: return launch_stages<Op, 6>(op, n, stream, pdl);
        case 8: return launch_stages<Op, 8>(op, n, stream, pdl);
        case 12: return launch_stages<Op, 12>(op, n, stream, pdl);
        case 16: return launch_stages<Op, 16>(op, n, stream, pdl);
        default: return launch_stages<Op, 2>(op, n, stream, pdl);
    }
}

bool fits_two_stages(size_t stage_bytes) {
    return 2 * stage_bytes + kBarrierBytes + kStaticSmemReserve <=
           static_cast<size_t>(device_smem_optin());
}

}  // namespace

bool tma_step_fits(int nd, int grad_type) {
    const size_t gsz = grad_type == kGradF32 ? 4 : 2;
    return fits_two_stages(static_cast<size_t>(kTile) * (nd * gsz + 12));
}

bool tma_reduce_fits(int nd, int grad_type) {
    const size_t gsz = grad_type == kGradF32 ? 4 : 2;
    return fits_two_stages(static_cast<size_t>(kTile) * nd * gsz);
}

int set_tma_stage_limit(int stages) { return g_stage_limit.exchange(stages); }

int64_t set_tma_wait_ns(int64_t ns) {
    const unsigned long long v = ns == 0 ? kDefaultWaitNs : static_cast<unsigned long long>(ns);
    return static_cast<int64_t>(g_wait_ns.exchange(v));
}

cudaError_t launch_rs_adamw_cast_tma(const PtrTable& tab, int nd, int grad_type, int64_t S,
                                     float* master, float* m, float* v, uint16_t* out,
                                     const AdamScalars& c, const MeanOp& mo,
                                     const unsigned int* skip, cudaStream_t stream) {
    switch (grad_type) {
        case kGradF32:
            return launch_staged(AdamOp<kGradF32>{tab, nd, master, m, v, out, c, mo, skip}, S,
                                 stream);
        case kGradF16:
            return launch_staged(AdamOp<kGradF16>{tab, nd, master, m, v, out, c, mo, skip}, S,
                                 stream);
        default:
            return launch_staged(AdamOp<kGradBF16>{tab, nd, master, m, v, out, c, mo, skip}, S,
                                 stream);
    }
}

cudaError_t launch_accumulate_tma(const uint16_t* g, float* acc, int64_t n, float scale,
                                  bool first, cudaStream_t stream) {
    if (first) return launch_staged(AccumOp<true>{g, acc, scale}, n, stream);
    return launch_staged(AccumOp<false>{g, acc, scale}, n, stream);
}

cudaError_t launch_allreduce_avg_tma(const PtrTable& tab, int nd, int64_t n, uint16_t* out,
                                     const MeanOp& mo, bool pdl, cudaStream_t stream) {
    return launch_staged(MeanOutOp{tab, nd, out, mo}, n, stream, pdl);
}

cudaError_t launch_nonfinite_check_tma(const PtrTable& tab, int nd, int grad_type, int64_t S,
                                       const MeanOp& mo, unsigned int* found,
                                       cudaStream_t stream) {
    switch (grad_type) {
        case kGradF32: return launch_staged(CheckOp<kGradF32>{tab, nd, mo, found}, S, stream);
        case kGradF16: return launch_staged(CheckOp<kGradF16>{tab, nd, mo, found}, S, stream);
        default: return launch_staged(CheckOp<kGradBF16>{tab, nd, mo, found}, S, stream);
    }
}

cudaError_t read_device_status(unsigned int* status, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_device_status, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
}

}  // namespace shardstep
