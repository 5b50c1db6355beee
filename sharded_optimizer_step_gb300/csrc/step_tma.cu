// The fused sharded step with TMA bulk staging (the default path when every
// pointer is 16-byte aligned and the stages fit in shared memory).
//
// One CTA per SM, 17 warps.  Warp 16's first lane is the producer: for each
// tile of 2048 shard elements it issues one cp.async.bulk per gradient slice
// and per state array (master, m, v) from HBM into a shared-memory stage and
// completes them on that stage's mbarrier (expect-tx).  Warps 0..15 consume:
// they wait on the stage's barrier, reduce the N_d slices in rank order from
// shared memory, run AdamW, and write master / m / v and the bf16 parameter
// straight to HBM with streaming stores; each warp then arrives on the
// stage's "empty" barrier so the producer can refill it.  The slices are
// summed in the order GroupSum fixes (rank order, grouped for hybrid
// sharding).  Two stages of
// 2048 x (N_d x grad bytes + 12) bytes are in flight per SM (114 KB at N_d =
// 8, bf16).  Tiles are dealt round-robin over the grid.  Measured on GB300
// against the register-staged kernel (4 elements / thread, 512-thread
// blocks) on the same GPU: 4.98 ms vs 5.43 ms for an 842M-element shard at
// N_d = 8.
//
// Every wait is bounded (about two seconds of %globaltimer).  A wait that
// runs out sets a bit in the device status word (shardstep_device_status),
// the producer then waits, again bounded, for the copies it already issued,
// and the CTA returns.  Nothing here spins on another CTA or on the host.
#include "common.cuh"

namespace shardstep {

// Watchdog status of this device's TMA-staged launches (0 = no wait ran out).
__device__ unsigned int g_device_status = 0;

namespace {

constexpr int kTile = 2048;
constexpr int kStages = 2;
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;   // 512: 4 elements each per tile
constexpr int kTmaThreads = kConsumers + 32;      // + the producer warp
constexpr unsigned long long kWaitNs = 2000000000ull;

constexpr unsigned kStatusConsumerTimeout = 1u;
constexpr unsigned kStatusProducerTimeout = 2u;

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
// Waits for the phase of `parity` to complete; false after kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity) {
    const unsigned long long t0 = now_ns();
    for (uint32_t k = 1;; ++k) {
        if (mbar_test(b, parity)) return true;
        if ((k & 255u) == 0 && now_ns() - t0 > kWaitNs) return false;
    }
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

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

// S_main = S rounded down to a multiple of 8 is covered by tiles (the last
// one possibly shorter, still a multiple of 8 elements, so every bulk copy is
// a multiple of 16 bytes); the final S - S_main < 8 elements are done by
// block 0 with ordinary loads.
template <int GT>
__global__ void __launch_bounds__(kTmaThreads, 1)
    rs_adamw_cast_tma(PtrTable tab, int nd, int64_t S, float* __restrict__ P,
                      float* __restrict__ M, float* __restrict__ V, uint16_t* __restrict__ out,
                      AdamScalars c, MeanOp mo, const unsigned int* skip) {
    // a skipped step (gradient scaler found inf/NaN): every thread returns
    // before any barrier or copy exists
    if (skip_step(skip)) return;
    mo = resolve_scale(mo);
    constexpr uint32_t gsz = GT == kGradF32 ? 4 : 2;
    const uint32_t slice_bytes = kTile * gsz;
    const uint32_t stage_bytes = nd * slice_bytes + 3 * kTile * 4;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * stage_bytes);
    uint64_t* empty = full + kStages;
    const int tid = threadIdx.x;
    const int64_t s_main = S & ~static_cast<int64_t>(7);
    const int64_t ntiles = (s_main + kTile - 1) / kTile;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
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
        bool ok = true;
        for (; j < my_tiles; ++j) {
            const int s = static_cast<int>(j % kStages);
            const uint32_t use = static_cast<uint32_t>(j / kStages);
            if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1u)) {
                ok = false;
                break;
            }
            const int64_t e0 = (static_cast<int64_t>(blockIdx.x) + j * gridDim.x) * kTile;
            const int64_t n = s_main - e0 < kTile ? s_main - e0 : kTile;
            const uint32_t gb = static_cast<uint32_t>(n) * gsz, sb = static_cast<uint32_t>(n) * 4;
            uint8_t* st = smem + s * stage_bytes;
            mbar_expect_tx(&full[s], nd * gb + 3 * sb);
            for (int q = 0; q < nd; ++q)
                bulk_load(st + q * slice_bytes, static_cast<const uint8_t*>(tab.p[q]) + e0 * gsz,
                          gb, &full[s]);
            uint8_t* sst = st + nd * slice_bytes;
            bulk_load(sst, P + e0, sb, &full[s]);
            bulk_load(sst + kTile * 4, M + e0, sb, &full[s]);
            bulk_load(sst + 2 * kTile * 4, V + e0, sb, &full[s]);
        }
        if (!ok) {
            atomicOr(&g_device_status, kStatusProducerTimeout);
            // the copies already issued land in this CTA's shared memory:
            // wait for them (bounded) before the CTA may exit
            for (int64_t k = j > kStages ? j - kStages : 0; k < j; ++k)
                mbar_wait(&full[k % kStages], static_cast<uint32_t>(k / kStages) & 1u);
        }
        return;
    }

    // consumers
    const int lane = tid & 31;
    for (int64_t j = 0; j < my_tiles; ++j) {
        const int s = static_cast<int>(j % kStages);
        const uint32_t use = static_cast<uint32_t>(j / kStages);
        if (!mbar_wait(&full[s], use & 1u)) {
            atomicOr(&g_device_status, kStatusConsumerTimeout);
            return;
        }
        const int64_t e0 = (static_cast<int64_t>(blockIdx.x) + j * gridDim.x) * kTile;
        const int64_t n = s_main - e0 < kTile ? s_main - e0 : kTile;
        const uint8_t* st = smem + s * stage_bytes;
        const uint8_t* sst = st + nd * slice_bytes;
        for (int e = tid * 4; e < n; e += kConsumers * 4) {
            GroupSum<4> acc;
            {
                float t[4];
                load4_smem<GT>(st + e * gsz, t);
                acc.first(t);
            }
            for (int q = 1; q < nd; ++q) {
                float t[4];
                load4_smem<GT>(st + q * slice_bytes + e * gsz, t);
                acc.add(t, mo.group);
            }
            float g[4];
            acc.result(g);
            const float4 pp = *reinterpret_cast<const float4*>(sst + e * 4);
            const float4 mm = *reinterpret_cast<const float4*>(sst + kTile * 4 + e * 4);
            const float4 vv = *reinterpret_cast<const float4*>(sst + 2 * kTile * 4 + e * 4);
            float p[4] = {pp.x, pp.y, pp.z, pp.w};
            float m[4] = {mm.x, mm.y, mm.z, mm.w};
            float v[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) adamw_elem(mean_of(g[k], mo), p[k], m[k], v[k], c);
            const int64_t ge = e0 + e;
            stcs16(P + ge, pack4f(p));
            stcs16(M + ge, pack4f(m));
            stcs16(V + ge, pack4f(v));
            stcs8(out + ge, make_uint2(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3])));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (blockIdx.x == 0 && tid < S - s_main) {
        const int64_t jx = s_main + tid;
        GroupSum<1> acc;
        float t = grad1<GT>(tab.p[0], jx);
        acc.first(&t);
        for (int q = 1; q < nd; ++q) {
            t = grad1<GT>(tab.p[q], jx);
            acc.add(&t, mo.group);
        }
        float sum;
        acc.result(&sum);
        float p = P[jx], m = M[jx], v = V[jx];
        adamw_elem(mean_of(sum, mo), p, m, v, c);
        P[jx] = p;
        M[jx] = m;
        V[jx] = v;
        out[jx] = f32_to_bf16(p);
    }
}

int g_smem_set[256];  // per device: dynamic shared memory attribute applied

}  // namespace

size_t tma_step_smem_bytes(int nd, int grad_type) {
    const size_t gsz = grad_type == kGradF32 ? 4 : 2;
    return static_cast<size_t>(kStages) * kTile * (nd * gsz + 12) + 2 * kStages * sizeof(uint64_t);
}

cudaError_t launch_rs_adamw_cast_tma(const PtrTable& tab, int nd, int grad_type, int64_t S,
                                     float* master, float* m, float* v, uint16_t* out,
                                     const AdamScalars& c, const MeanOp& mo,
                                     const unsigned int* skip, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const size_t smem = tma_step_smem_bytes(nd, grad_type);
    if (dev >= 0 && dev < 256 && !g_smem_set[dev]) {
        int optin = 0;
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(rs_adamw_cast_tma<kGradBF16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(rs_adamw_cast_tma<kGradF32>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(rs_adamw_cast_tma<kGradF16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        if (e != cudaSuccess) return e;
        g_smem_set[dev] = 1;
    }
    const int64_t ntiles = ((S & ~static_cast<int64_t>(7)) + kTile - 1) / kTile;
    int64_t grid = device_sms();
    if (grid > ntiles) grid = ntiles;
    if (grid < 1) grid = 1;
    const unsigned g = static_cast<unsigned>(grid);
    if (grad_type == kGradF32)
        rs_adamw_cast_tma<kGradF32><<<g, kTmaThreads, smem, stream>>>(tab, nd, S, master, m, v,
                                                                     out, c, mo, skip);
    else if (grad_type == kGradF16)
        rs_adamw_cast_tma<kGradF16><<<g, kTmaThreads, smem, stream>>>(tab, nd, S, master, m, v,
                                                                     out, c, mo, skip);
    else
        rs_adamw_cast_tma<kGradBF16><<<g, kTmaThreads, smem, stream>>>(tab, nd, S, master, m, v,
                                                                      out, c, mo, skip);
    note_launch();
    return cudaGetLastError();
}

cudaError_t read_device_status(unsigned int* status, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_device_status, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
}

}  // namespace shardstep
