// Host side of the C ABI declared in include/shardstep.h: argument checks,
// FlatParameter layout and bucket planning, the AdamW scalar derivation, and
// dispatch to the kernels.  Nothing here allocates device memory.
#include <atomic>
#include <initializer_list>
#include <cmath>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"
#include "shardstep.h"

namespace shardstep {
namespace {

thread_local std::string g_error;
thread_local char g_last_kernel[128] = "";

// Records which kernel the calling thread's last streaming call launched.
void note_kernel(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_kernel, sizeof g_last_kernel, fmt, ap);
    va_end(ap);
}

// Whether nd is one of the counts a register-staged kernel is compiled for
// (the others take its loop over any N_d).
bool compiled_nd(int nd, std::initializer_list<int> counts) {
    for (int c : counts)
        if (c == nd) return true;
    return false;
}

const char* dtype_name(int dtype) {
    return dtype == SHARDSTEP_DTYPE_F32 ? "f32" : dtype == SHARDSTEP_DTYPE_F16 ? "f16" : "bf16";
}
std::atomic<uint64_t> g_launches{0};

// The inter-rank bytes the emulated collectives of the accepted calls stand
// for (ring model; see shardstep_comm_counter in shardstep.h).
std::mutex g_comm_mu;
double g_comm_bytes = 0.0;
void count_comm(double bytes) {
    std::lock_guard<std::mutex> lock(g_comm_mu);
    g_comm_bytes += bytes;
}
// The reduce of a fused step over S shard positions of es-byte
// contributions: the reduce-scatter inside the group of `group` ranks, then,
// under hybrid sharding, the ring all-reduce of the shard across the
// nd / group groups.
double reduce_comm_bytes(int32_t nd, int32_t group, int64_t S, int es) {
    const double n = static_cast<double>(S) * es;
    const int32_t R = nd / group;
    double b = static_cast<double>(group - 1) * n;
    if (R > 1) b += 2.0 * (R - 1) / R * n;
    return b;
}
// One ring all-reduce of `bytes` over nd ranks: a reduce-scatter and an
// all-gather, each sending (nd - 1) / nd of the buffer.
double allreduce_comm_bytes(int32_t nd, double bytes) { return 2.0 * (nd - 1) / nd * bytes; }

std::atomic<int> g_fused_path{SHARDSTEP_PATH_AUTO};
std::atomic<int> g_dependent_launch{1};

// Whether a launch of n elements goes to a TMA-staged kernel (the caller
// still checks alignment and the stage size).  PATH_REGISTER: never;
// PATH_TMA: always; PATH_AUTO: where it measured faster on GB300 against the
// register-staged kernel of the same operation --
//   fused step: only at N_d > 16 and with fp32 slices at N_d = 5, 7 and
//     9..16, which the compiled register kernels do not take because they
//     would spill (where two stages do not fit, at 12..16 fp32 slices, the
//     register kernel's loop over any N_d runs: 7.22 TB/s at 16, against
//     6.57 for a spilling compiled form).  Elsewhere the register kernel
//     won: at N_d = 8 7.13 vs 6.88 TB/s; at 6, compiled, 6.8 vs 6.3; at 5
//     and 7 on the up-to-8 kernel 6.6 vs 6.2 and 6.7 vs 6.5; compiled for
//     9..16 16-bit slices 7.15-7.35 vs 6.80-7.15 (50M elements, the same
//     buffers in one process); at 1..4 it was faster as well;
//   bucket all-reduce: at N_d = 4 and 8 on buckets of at least 32M
//     elements (one 400M bucket at N_d = 4: 6.9 vs 6.4 TB/s; at N_d = 8:
//     7.05 vs 6.98) and at N_d > 16; never at N_d = 1..3 and 5..7, where the
//     register kernel is compiled with several vectors' loads in flight
//     (200M elements in 25 MiB buckets, register / TMA-staged: N_d = 3
//     6.1 / 3.7, 5 6.5 / 4.8, 6 6.5 / 5.4, 7 6.7 / 5.9 TB/s), nor at
//     9..16, where it is compiled for each count (50M elements in 25 MiB
//     buckets, same buffers: 6.8-7.0 vs 5.7-6.8 TB/s, the widest gap at
//     11..14);
//   non-finite check: with 16-bit slices at N_d > 16 only (at 9..16,
//     compiled for each count, 7.1-7.4 vs 6.1-6.9 TB/s; N_d = 3 / 5 / 6
//     / 7, 200M fp16 elements: 5.1 / 2.7, 6.4 / 4.1, 6.9 / 4.6, 6.9 / 5.1
//     TB/s; at N_d = 1 / 2 / 4 / 8: 5.0 vs 2.1, 6.0 vs 3.2, 6.7 vs 5.7,
//     7.4 vs 7.3), with fp32 slices at every N_d but 1, 2, 4 and 8;
//   accumulation: never (7.0 vs 6.0 TB/s for the first micro-batch, 7.2 vs
//     6.6 for the others).
enum class TmaOp { kStep, kAllReduce, kAccumulate, kCheck };
bool register_step_kernel(int nd, int grad_dtype) {
    switch (nd) {
        case 1: case 2: case 3: case 4: case 6: case 8: return true;
        case 5: case 7: case 9: case 10: case 11: case 12: case 13: case 14: case 15:
        case 16: return grad_dtype != SHARDSTEP_DTYPE_F32;
        default: return false;
    }
}
bool use_tma(TmaOp op, int64_t n, int nd = 0, int grad_dtype = SHARDSTEP_DTYPE_BF16) {
    const int path = g_fused_path.load(std::memory_order_relaxed);
    if (path == SHARDSTEP_PATH_REGISTER) return false;
    if (n < kTmaMinElements) return false;
    if (path == SHARDSTEP_PATH_TMA) return true;
    switch (op) {
        case TmaOp::kStep: return nd >= 3 && !register_step_kernel(nd, grad_dtype);
        case TmaOp::kAllReduce:
            if (nd == 4 || nd == 8) return n >= (int64_t{32} << 20);
            return nd > 16;
        case TmaOp::kCheck:
            if (grad_dtype == SHARDSTEP_DTYPE_F32) return nd != 1 && nd != 2 && nd != 4 && nd != 8;
            return nd > 16;
        default: return false;
    }
}

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_error = buf;
    return code;
}

int ok() {
    g_error.clear();
    return SHARDSTEP_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(SHARDSTEP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct Span {
    uintptr_t lo, hi;  // [lo, hi); empty spans never overlap anything
};
Span span(const void* p, int64_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Span{a, a + static_cast<uintptr_t>(bytes > 0 ? bytes : 0)};
}
bool overlap(Span a, Span b) {
    return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
}
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_size_of(int32_t dtype) {
    switch (dtype) {
        case SHARDSTEP_DTYPE_BF16:
        case SHARDSTEP_DTYPE_F16: return 2;
        case SHARDSTEP_DTYPE_F32: return 4;
        default: return 0;
    }
}

// RN(1/nd) in fp32, from integers: the significand is 2^k / nd rounded to
// the nearest integer for the k that puts it in [2^23, 2^24).  A tie cannot
// occur (2^(k+1) / nd is an integer only for a power of two, and then the
// quotient is exact), so rounding half up is round to nearest.
float reciprocal_rn(int nd) {
    int k = 0;
    while ((uint64_t{1} << k) / static_cast<uint64_t>(nd) < (uint64_t{1} << 23)) ++k;
    const uint64_t num = uint64_t{1} << k;
    const uint64_t q = num / static_cast<uint64_t>(nd);
    const uint64_t rem = num % static_cast<uint64_t>(nd);
    const uint64_t sig = q + (2 * rem >= static_cast<uint64_t>(nd) ? 1 : 0);
    return std::ldexp(static_cast<float>(sig), -k);
}

MeanOp mean_op(int nd, int group) {
    MeanOp mo;
    mo.nd = static_cast<float>(nd);
    mo.pow2 = (nd & (nd - 1)) == 0;
    mo.inv_nd = reciprocal_rn(nd);  // exact when nd is a power of two
    mo.group = group;
    mo.inv_scale = 1.0f;
    mo.scaled = 0;
    mo.scale = nullptr;
    return mo;
}

// Per-step scalars: double arithmetic, one rounding to fp32 each.  beta^t is
// the left-to-right product of t factors; once both products reach zero they
// stay zero, so the loop stops there.
AdamScalars adam_scalars(const shardstep_adamw_t& hp) {
    double b1t = 1.0, b2t = 1.0;
    for (int64_t k = 0; k < hp.step; ++k) {
        b1t *= hp.beta1;
        b2t *= hp.beta2;
        if (b1t == 0.0 && b2t == 0.0) break;
    }
    const double bc1 = 1.0 - b1t;
    const double bc2 = 1.0 - b2t;
    AdamScalars c{};
    c.lr_wd = static_cast<float>(hp.lr * hp.weight_decay);
    c.beta1 = static_cast<float>(hp.beta1);
    c.omb1 = static_cast<float>(1.0 - hp.beta1);
    c.beta2 = static_cast<float>(hp.beta2);
    c.omb2 = static_cast<float>(1.0 - hp.beta2);
    c.step_size = static_cast<float>(hp.lr / bc1);
    c.sqrt_bc2 = static_cast<float>(std::sqrt(bc2));
    c.eps = static_cast<float>(hp.eps);
    return c;
}

// Layout arithmetic shared by fsdp_layout / fsdp_flat_pack / fsdp_views.
int compute_layout(const int64_t* numels, int32_t n, int32_t nd, shardstep_layout_info_t* info,
                   int64_t* offsets) {
    if (n < 0) return fail(SHARDSTEP_ERR_INVALID, "n_tensors must be >= 0 (got %d)", n);
    if (nd < 1) return fail(SHARDSTEP_ERR_INVALID, "nd must be >= 1 (got %d)", nd);
    if (n > 0 && numels == nullptr) return fail(SHARDSTEP_ERR_INVALID, "numels is NULL");
    int64_t total = 0;
    for (int32_t t = 0; t < n; ++t) {
        if (numels[t] < 0)
            return fail(SHARDSTEP_ERR_INVALID, "numel of tensor %d is negative", t);
        if (numels[t] > INT64_MAX / 8 - total)
            return fail(SHARDSTEP_ERR_INVALID, "unit too large");
        if (offsets) offsets[t] = total;
        total += numels[t];
    }
    const int64_t padded = (total + nd - 1) / nd * nd;
    info->total = total;
    info->padded = padded;
    info->shard = padded / nd;
    info->n_tensors = n;
    info->nd = nd;
    return SHARDSTEP_OK;
}

std::mutex g_occ_mu;
struct OccEntry {
    int dev;
    const void* kernel;
    int threads;
    int blocks;
};
std::vector<OccEntry> g_occ;

}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

bool dependent_launches() { return g_dependent_launch.load(std::memory_order_relaxed) != 0; }

// Error reporting for ckpt.cpp: the message is fmt with one string and one
// integer argument (either may be unused).
int ckpt_fail(int code, const char* fmt, const char* a, long long b) {
    return fail(code, fmt, a, b);
}

// Error reporting for the host-only translation units (bucket readiness).
int ready_fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_error = buf;
    return code;
}

int ready_ok() { return ok(); }

int device_sms() {
    static std::atomic<int> cache[256];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 1;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return 1;
    cache[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

int device_smem_optin() {
    static std::atomic<int> cache[256];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 0;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        optin < 1)
        return 0;
    cache[dev].store(optin, std::memory_order_relaxed);
    return optin;
}

int resident_blocks(const void* kernel, int threads) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    {
        std::lock_guard<std::mutex> lk(g_occ_mu);
        for (const OccEntry& e : g_occ)
            if (e.dev == dev && e.kernel == kernel && e.threads == threads) return e.blocks;
    }
    int blocks = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, threads, 0) != cudaSuccess ||
        blocks < 1)
        blocks = 1;
    std::lock_guard<std::mutex> lk(g_occ_mu);
    g_occ.push_back(OccEntry{dev, kernel, threads, blocks});
    return blocks;
}

}  // namespace shardstep

using namespace shardstep;

extern "C" {

const char* shardstep_last_error(void) { return g_error.c_str(); }

const char* shardstep_last_kernel(void) { return g_last_kernel; }

uint64_t shardstep_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

double shardstep_comm_counter(int32_t reset) {
    std::lock_guard<std::mutex> lock(g_comm_mu);
    const double b = g_comm_bytes;
    if (reset != 0) g_comm_bytes = 0.0;
    return b;
}

int32_t shardstep_set_fused_path(int32_t path) {
    if (path != SHARDSTEP_PATH_AUTO && path != SHARDSTEP_PATH_REGISTER &&
        path != SHARDSTEP_PATH_TMA)
        return fail(SHARDSTEP_ERR_INVALID, "unknown path %d", path);
    return g_fused_path.exchange(path);
}

int32_t shardstep_set_dependent_launch(int32_t enable) {
    return g_dependent_launch.exchange(enable != 0 ? 1 : 0);
}

int32_t shardstep_set_tma_stages(int32_t stages) {
    if (stages != 0 && (stages < 2 || stages > 16))
        return fail(SHARDSTEP_ERR_INVALID, "stages must be 0 or 2..16 (got %d)", stages);
    return set_tma_stage_limit(stages);
}

int64_t shardstep_set_tma_wait_ns(int64_t ns) {
    if (ns < 0) return fail(SHARDSTEP_ERR_INVALID, "the wait limit must be >= 0 (got %lld)",
                            static_cast<long long>(ns));
    return set_tma_wait_ns(ns);
}

int shardstep_check_mean_division(int32_t nd, uint64_t* mismatches, uint32_t* first_bad,
                                  void* stream) {
    if (nd < 1 || nd > SHARDSTEP_MAX_ND)
        return fail(SHARDSTEP_ERR_INVALID, "nd must be 1..%d (got %d)", SHARDSTEP_MAX_ND, nd);
    if (mismatches == nullptr || first_bad == nullptr)
        return fail(SHARDSTEP_ERR_INVALID, "mismatches / first_bad is NULL");
    if (!aligned(mismatches, 8) || !aligned(first_bad, 4))
        return fail(SHARDSTEP_ERR_INVALID, "mismatches / first_bad misaligned");
    cudaError_t e = launch_mean_division_check(
        mean_op(nd, nd), reinterpret_cast<unsigned long long*>(mismatches), first_bad,
        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "division check kernel launch");
    return ok();
}

int shardstep_device_status(uint32_t* status, int32_t clear) {
    if (status == nullptr) return fail(SHARDSTEP_ERR_INVALID, "status is NULL");
    unsigned int s = 0;
    cudaError_t e = read_device_status(&s, clear != 0);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    *status = s;
    return ok();
}

int fsdp_layout(const int64_t* numels, int32_t n, int32_t nd, shardstep_layout_info_t* info,
                int64_t* offsets, int64_t* lo, int64_t* hi) {
    if (info == nullptr) return fail(SHARDSTEP_ERR_INVALID, "info is NULL");
    std::vector<int64_t> off(n > 0 ? n : 0);
    int rc = compute_layout(numels, n, nd, info, off.data());
    if (rc != SHARDSTEP_OK) return rc;
    if (offsets)
        for (int32_t t = 0; t < n; ++t) offsets[t] = off[t];
    const int64_t S = info->shard;
    for (int32_t r = 0; r < nd && (lo || hi); ++r) {
        const int64_t base = static_cast<int64_t>(r) * S;
        for (int32_t t = 0; t < n; ++t) {
            int64_t a = off[t] - base, b = off[t] + numels[t] - base;
            a = a < 0 ? 0 : (a > S ? S : a);
            b = b < 0 ? 0 : (b > S ? S : b);
            if (lo) lo[static_cast<int64_t>(r) * n + t] = a;
            if (hi) hi[static_cast<int64_t>(r) * n + t] = b;
        }
    }
    return ok();
}

int fsdp_shard_pieces(const int64_t* numels, int32_t n, int32_t nd, int32_t rank,
                      int64_t* shard_lo, int64_t* tensor_lo, int64_t* count) {
    shardstep_layout_info_t info;
    std::vector<int64_t> off(n > 0 ? n : 0);
    int rc = compute_layout(numels, n, nd, &info, off.data());
    if (rc != SHARDSTEP_OK) return rc;
    if (rank < 0 || rank >= nd)
        return fail(SHARDSTEP_ERR_INVALID, "rank %d out of 0..%d", rank, nd - 1);
    if (n > 0 && (shard_lo == nullptr || tensor_lo == nullptr || count == nullptr))
        return fail(SHARDSTEP_ERR_INVALID, "shard_lo / tensor_lo / count is NULL");
    const int64_t S = info.shard, r0 = static_cast<int64_t>(rank) * S;
    for (int32_t t = 0; t < n; ++t) {
        // the tensor's flat range [off, off + n_t) meets [r0, r0 + S)
        const int64_t a = off[t] > r0 ? off[t] : r0;
        const int64_t e = off[t] + numels[t] < r0 + S ? off[t] + numels[t] : r0 + S;
        if (a < e) {
            shard_lo[t] = a - r0;
            tensor_lo[t] = a - off[t];
            count[t] = e - a;
        } else {
            shard_lo[t] = 0;
            tensor_lo[t] = 0;
            count[t] = 0;
        }
    }
    return ok();
}

int fsdp_views(const int64_t* numels, int32_t n, int32_t nd, int32_t rank, void* base,
               int32_t elem_size, void** ptrs, int64_t* counts) {
    shardstep_layout_info_t info;
    std::vector<int64_t> off(n > 0 ? n : 0);
    int rc = compute_layout(numels, n, nd, &info, off.data());
    if (rc != SHARDSTEP_OK) return rc;
    if (rank >= nd) return fail(SHARDSTEP_ERR_INVALID, "rank %d >= nd %d", rank, nd);
    if (elem_size <= 0) return fail(SHARDSTEP_ERR_INVALID, "elem_size must be > 0");
    if (n > 0 && (ptrs == nullptr || counts == nullptr))
        return fail(SHARDSTEP_ERR_INVALID, "ptrs / counts is NULL");
    char* b = static_cast<char*>(base);
    for (int32_t t = 0; t < n; ++t) {
        if (rank < 0) {
            ptrs[t] = b + off[t] * elem_size;
            counts[t] = numels[t];
        } else {
            const int64_t S = info.shard, r0 = static_cast<int64_t>(rank) * S;
            int64_t a = off[t] - r0, e = off[t] + numels[t] - r0;
            a = a < 0 ? 0 : (a > S ? S : a);
            e = e < 0 ? 0 : (e > S ? S : e);
            ptrs[t] = b + a * elem_size;
            counts[t] = e - a;
        }
    }
    return ok();
}

// Turns (src, dst, bytes) triples into copy-kernel launches of <= kMaxCopySegs.
namespace {
// Whether the body of a copy range between its first and last 16-byte
// boundary of the destination goes to copy16 / copy16_shift (every kernel
// choice but PATH_REGISTER, which keeps all copies on copy_segments).
bool use_copy16() {
    return g_fused_path.load(std::memory_order_relaxed) != SHARDSTEP_PATH_REGISTER;
}

struct CopyBatcher {
    CopyTable t;
    AlignedTable bt;  // 16-byte aligned source and destination (copy16)
    AlignedTable st;  // aligned destination, unaligned source (copy16_shift)
    cudaStream_t stream;
    int rc = SHARDSTEP_OK;
    // whether this call has launched a kernel.  With dependent launches on
    // (the default) every launch goes out as a programmatic dependent of the
    // kernel before it in the stream: the first one of the call waits for
    // that unknown predecessor before it touches memory, the later ones
    // (disjoint copies of the same call) only before they end, so that each
    // overlaps the previous one's drain
    bool launched = false;
    const bool pdl_ok = g_dependent_launch.load(std::memory_order_relaxed) != 0;
    explicit CopyBatcher(cudaStream_t s) : stream(s) {
        t.n = 0;
        t.total_chunks = 0;
        bt.n = 0;
        bt.total_chunks = 0;
        st.n = 0;
        st.total_chunks = 0;
    }
    // The body of a range between its first and last 16-byte boundary of the
    // destination goes to copy16 when the source is congruent to the
    // destination modulo 16 bytes, else to copy16_shift (unless the register
    // path is forced); the head and tail bytes, zero fills and everything
    // under PATH_REGISTER go to copy_segments.
    void add(const void* src, void* dst, int64_t bytes) {
        if (bytes <= 0 || rc != SHARDSTEP_OK) return;
        const uintptr_t d = reinterpret_cast<uintptr_t>(dst);
        if (src != nullptr && use_copy16()) {
            const int64_t head = static_cast<int64_t>((16 - d % 16) % 16);
            const int64_t body = bytes > head ? ((bytes - head) & ~int64_t{15}) : 0;
            if (body > 0) {
                const char* s8 = static_cast<const char*>(src);
                char* d8 = static_cast<char*>(dst);
                const bool congruent = ((reinterpret_cast<uintptr_t>(src) ^ d) & 15u) == 0;
                add_vector(s8, d8, head);
                add_chunked(congruent ? bt : st, s8 + head, d8 + head, body);
                add_vector(s8 + head + body, d8 + head + body, bytes - head - body);
                return;
            }
        }
        add_vector(src, dst, bytes);
    }
    void add_chunked(AlignedTable& tab, const char* src, char* dst, int64_t bytes) {
        AlignedSeg& s = tab.s[tab.n];
        s.src = src;
        s.dst = dst;
        s.bytes = bytes;
        s.chunk0 = tab.total_chunks;
        tab.total_chunks += (bytes + kAlignedChunk - 1) / kAlignedChunk;
        if (++tab.n == kMaxCopySegs) flush_chunked(tab);
    }
    void add_vector(const void* src, void* dst, int64_t bytes) {
        if (bytes <= 0 || rc != SHARDSTEP_OK) return;
        CopySeg& s = t.s[t.n];
        s.src = static_cast<const char*>(src);
        s.dst = static_cast<char*>(dst);
        s.bytes = bytes;
        const uintptr_t d = reinterpret_cast<uintptr_t>(dst);
        const uintptr_t x = src ? (reinterpret_cast<uintptr_t>(src) ^ d) : 0;
        int w = 16;
        while (w > 1 && (x % w) != 0) w >>= 1;
        int64_t head = static_cast<int64_t>((w - d % w) % w);
        if (head > bytes) head = bytes;
        s.width = w;
        s.head = static_cast<int32_t>(head);
        s.body = (bytes - head) / w;
        s.chunk0 = t.total_chunks;
        t.total_chunks += s.body > 0 ? (s.body + kCopyVecsPerChunk - 1) / kCopyVecsPerChunk : 1;
        if (++t.n == kMaxCopySegs) flush_vector();
    }
    void flush_vector() {
        if (t.n == 0 || rc != SHARDSTEP_OK) return;
        cudaError_t e = launch_copy(t, pdl_ok, !launched, stream);
        if (e != cudaSuccess) rc = cuda_fail(e, "copy kernel launch");
        launched = true;
        t.n = 0;
        t.total_chunks = 0;
    }
    void flush_chunked(AlignedTable& tab) {
        if (tab.n == 0 || rc != SHARDSTEP_OK) return;
        cudaError_t e = &tab == &bt ? launch_copy16(tab, pdl_ok, !launched, stream)
                                    : launch_copy16_shift(tab, pdl_ok, !launched, stream);
        if (e != cudaSuccess) rc = cuda_fail(e, "aligned copy kernel launch");
        launched = true;
        tab.n = 0;
        tab.total_chunks = 0;
    }
    void flush() {
        flush_chunked(bt);
        flush_chunked(st);
        flush_vector();
    }
};
}  // namespace

int fsdp_flat_pack(const void* const* src, const int64_t* numels, int32_t n, int32_t nd,
                   int32_t dtype, void* flat, void* stream) {
    const int es = elem_size_of(dtype);
    if (es == 0) return fail(SHARDSTEP_ERR_INVALID, "unknown dtype %d", dtype);
    shardstep_layout_info_t info;
    std::vector<int64_t> off(n > 0 ? n : 0);
    int rc = compute_layout(numels, n, nd, &info, off.data());
    if (rc != SHARDSTEP_OK) return rc;
    if (info.padded == 0) return ok();
    if (flat == nullptr) return fail(SHARDSTEP_ERR_INVALID, "flat is NULL");
    if (n > 0 && src == nullptr) return fail(SHARDSTEP_ERR_INVALID, "src is NULL");
    if (!aligned(flat, es)) return fail(SHARDSTEP_ERR_INVALID, "flat is not %d-byte aligned", es);
    const Span fs = span(flat, info.padded * es);
    for (int32_t t = 0; t < n; ++t) {
        if (numels[t] == 0) continue;
        if (src[t] == nullptr) return fail(SHARDSTEP_ERR_INVALID, "src[%d] is NULL", t);
        if (!aligned(src[t], es))
            return fail(SHARDSTEP_ERR_INVALID, "src[%d] is not %d-byte aligned", t, es);
        if (overlap(span(src[t], numels[t] * es), fs))
            return fail(SHARDSTEP_ERR_INVALID, "src[%d] overlaps flat", t);
    }
    CopyBatcher cb(static_cast<cudaStream_t>(stream));
    char* f = static_cast<char*>(flat);
    for (int32_t t = 0; t < n; ++t) cb.add(src[t], f + off[t] * es, numels[t] * es);
    cb.add(nullptr, f + info.total * es, (info.padded - info.total) * es);
    cb.flush();
    return cb.rc == SHARDSTEP_OK ? ok() : cb.rc;
}

int fsdp_ag_unpack(const uint16_t* const* shards, int32_t nd, int64_t S, uint16_t* full,
                   void* stream) {
    if (nd < 1) return fail(SHARDSTEP_ERR_INVALID, "nd must be >= 1 (got %d)", nd);
    if (nd > SHARDSTEP_MAX_ND)
        return fail(SHARDSTEP_ERR_CAPACITY, "nd %d > %d", nd, SHARDSTEP_MAX_ND);
    if (S < 0) return fail(SHARDSTEP_ERR_INVALID, "S must be >= 0");
    if (S == 0) return ok();
    if (shards == nullptr || full == nullptr)
        return fail(SHARDSTEP_ERR_INVALID, "shards / full is NULL");
    if (!aligned(full, 2)) return fail(SHARDSTEP_ERR_INVALID, "full is not 2-byte aligned");
    const Span fs = span(full, static_cast<int64_t>(nd) * S * 2);
    for (int32_t q = 0; q < nd; ++q) {
        if (shards[q] == nullptr) return fail(SHARDSTEP_ERR_INVALID, "shards[%d] is NULL", q);
        if (!aligned(shards[q], 2))
            return fail(SHARDSTEP_ERR_INVALID, "shards[%d] is not 2-byte aligned", q);
        if (shards[q] == full + static_cast<int64_t>(q) * S) continue;
        if (overlap(span(shards[q], S * 2), fs))
            return fail(SHARDSTEP_ERR_INVALID, "shards[%d] overlaps full", q);
    }
    CopyBatcher cb(static_cast<cudaStream_t>(stream));
    for (int32_t q = 0; q < nd; ++q) {
        uint16_t* dst = full + static_cast<int64_t>(q) * S;
        if (shards[q] != dst) cb.add(shards[q], dst, S * 2);
    }
    cb.flush();
    if (cb.rc != SHARDSTEP_OK) return cb.rc;
    count_comm(static_cast<double>(nd - 1) * static_cast<double>(S) * 2.0);
    return ok();
}

int fsdp_grad_accumulate(const uint16_t* g, float* acc, int64_t n, float scale, int32_t first,
                         void* stream) {
    if (n < 0) return fail(SHARDSTEP_ERR_INVALID, "n must be >= 0");
    if (n == 0) return ok();
    if (g == nullptr || acc == nullptr) return fail(SHARDSTEP_ERR_INVALID, "g / acc is NULL");
    if (!aligned(g, 2) || !aligned(acc, 4))
        return fail(SHARDSTEP_ERR_INVALID, "g / acc misaligned for their element type");
    if (overlap(span(g, n * 2), span(acc, n * 4)))
        return fail(SHARDSTEP_ERR_INVALID, "g overlaps acc");
    const bool vec = aligned(g, 16) && aligned(acc, 16);
    const bool tma = vec && use_tma(TmaOp::kAccumulate, n);
    cudaError_t e = tma ? launch_accumulate_tma(g, acc, n, scale, first != 0,
                                                static_cast<cudaStream_t>(stream))
                        : launch_accumulate(g, acc, n, scale, first != 0, vec,
                                            static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "accumulate kernel launch");
    note_kernel(tma ? "staged_stream<AccumOp> (TMA-staged)"
                    : vec ? "accumulate_vec8 (register-staged)" : "accumulate_scalar");
    return ok();
}

}  // extern "C"

namespace {

// Validates N_d gradient slices of S elements, fills `tab`, and reports
// whether they suit the register-staged vector path (8-byte 16-bit slices,
// 16-byte fp32 slices) and the TMA-staged path (16-byte slices).
int take_slices(const void* const* grad_slices, int32_t grad_dtype, int32_t nd, int64_t S,
                const Span* outs, int n_outs, PtrTable* tab, bool* vec, bool* tma) {
    const int gs = elem_size_of(grad_dtype);
    if (gs == 0) return fail(SHARDSTEP_ERR_INVALID, "unknown grad dtype %d", grad_dtype);
    if (nd < 1) return fail(SHARDSTEP_ERR_INVALID, "nd must be >= 1 (got %d)", nd);
    if (nd > SHARDSTEP_MAX_ND)
        return fail(SHARDSTEP_ERR_CAPACITY, "nd %d > %d", nd, SHARDSTEP_MAX_ND);
    if (grad_slices == nullptr) return fail(SHARDSTEP_ERR_INVALID, "grad_slices is NULL");
    const uintptr_t gvec = grad_dtype == SHARDSTEP_DTYPE_F32 ? 16 : 8;
    *vec = true;
    *tma = true;
    for (int32_t q = 0; q < nd; ++q) {
        const void* p = grad_slices[q];
        if (p == nullptr) return fail(SHARDSTEP_ERR_INVALID, "grad_slices[%d] is NULL", q);
        if (!aligned(p, gs))
            return fail(SHARDSTEP_ERR_INVALID, "grad_slices[%d] misaligned for its dtype", q);
        const Span gsn = span(p, S * gs);
        for (int a = 0; a < n_outs; ++a)
            if (overlap(gsn, outs[a]))
                return fail(SHARDSTEP_ERR_INVALID, "grad_slices[%d] overlaps an output", q);
        *vec = *vec && aligned(p, gvec);
        *tma = *tma && aligned(p, 16);
        tab->p[q] = p;
    }
    for (int32_t q = nd; q < SHARDSTEP_MAX_ND; ++q) tab->p[q] = nullptr;
    return SHARDSTEP_OK;
}

// Shared argument checks of the hybrid / scaled entry points (INVALID with a
// message, or SHARDSTEP_OK).
int check_shard_group(int32_t nd, int32_t shard_group) {
    if (shard_group < 1 || nd < 1 || nd % shard_group != 0)
        return fail(SHARDSTEP_ERR_INVALID,
                    "the sharding factor %d must be >= 1 and divide nd = %d", shard_group, nd);
    return SHARDSTEP_OK;
}

// master / m / v (fp32) and out_bf16 of a step over S > 0 elements: present,
// aligned for their element type and pairwise disjoint; fills their spans.
int check_step_outputs(int64_t S, const float* master, const float* m, const float* v,
                       const uint16_t* out_bf16, Span* outs) {
    if (!master || !m || !v || !out_bf16)
        return fail(SHARDSTEP_ERR_INVALID, "master / m / v / out_bf16 is NULL");
    if (!aligned(master, 4) || !aligned(m, 4) || !aligned(v, 4) || !aligned(out_bf16, 2))
        return fail(SHARDSTEP_ERR_INVALID, "state or output misaligned for its element type");
    outs[0] = span(master, S * 4);
    outs[1] = span(m, S * 4);
    outs[2] = span(v, S * 4);
    outs[3] = span(out_bf16, S * 2);
    for (int a = 0; a < 4; ++a)
        for (int b = a + 1; b < 4; ++b)
            if (overlap(outs[a], outs[b]))
                return fail(SHARDSTEP_ERR_INVALID, "outputs %d and %d overlap", a, b);
    return SHARDSTEP_OK;
}

// The AdamW scalars of a step: from a device-resident step state (its device
// address; the host never reads it) when `state` is set, else from `hp`.
int adam_source(const shardstep_adamw_t* hp, const shardstep_adamw_state_t* state,
                AdamScalars* c) {
    if (state != nullptr) {
        if (!aligned(state, 8)) return fail(SHARDSTEP_ERR_INVALID, "state misaligned");
        c->dev = reinterpret_cast<const float*>(reinterpret_cast<const char*>(state) +
                                                offsetof(shardstep_adamw_state_t, scalars));
        return SHARDSTEP_OK;
    }
    if (hp == nullptr) return fail(SHARDSTEP_ERR_INVALID, "hp is NULL");
    if (hp->step < 1)
        return fail(SHARDSTEP_ERR_INVALID, "step must be >= 1 (got %lld)",
                    static_cast<long long>(hp->step));
    *c = adam_scalars(*hp);
    return SHARDSTEP_OK;
}

int check_scaler_words(const float* scale, const uint32_t* found_inf) {
    if (found_inf == nullptr || scale == nullptr)
        return fail(SHARDSTEP_ERR_INVALID, "found_inf / scale is NULL");
    if (!aligned(found_inf, 4) || !aligned(scale, 4))
        return fail(SHARDSTEP_ERR_INVALID, "found_inf / scale misaligned");
    return SHARDSTEP_OK;
}

// `hp` gives the AdamW scalars on the host; with `state` instead, the
// kernels read them from the device-resident step state.
// The fused step with the slices reduced in groups of `group` ranks
// (group == nd: plain rank order); with `scaled`, the mean is multiplied by
// inv_scale and a non-zero *skip at launch leaves everything unchanged.
int fused_step(const void* const* grad_slices, int32_t grad_dtype, int32_t nd, int32_t group,
               int64_t S, float* master, float* m, float* v, uint16_t* out_bf16,
               const shardstep_adamw_t* hp, void* stream, const float* scale = nullptr,
               const unsigned int* skip = nullptr,
               const shardstep_adamw_state_t* state = nullptr) {
    int rc = SHARDSTEP_OK;
    const int gs = elem_size_of(grad_dtype);
    if (gs == 0) return fail(SHARDSTEP_ERR_INVALID, "unknown grad dtype %d", grad_dtype);
    if (nd < 1) return fail(SHARDSTEP_ERR_INVALID, "nd must be >= 1 (got %d)", nd);
    if (nd > SHARDSTEP_MAX_ND)
        return fail(SHARDSTEP_ERR_CAPACITY, "nd %d > %d", nd, SHARDSTEP_MAX_ND);
    if (S < 0) return fail(SHARDSTEP_ERR_INVALID, "S must be >= 0");
    AdamScalars c{};
    if (int rc2 = adam_source(hp, state, &c); rc2 != SHARDSTEP_OK) return rc2;
    if (S == 0) return ok();
    Span outs[4];
    if (int rc2 = check_step_outputs(S, master, m, v, out_bf16, outs); rc2 != SHARDSTEP_OK)
        return rc2;
    // vector path: 4 elements per access -> 16-byte state, 8-byte 16-bit
    // (16-byte fp32) gradient slices, 8-byte bf16 output
    PtrTable tab;
    bool vec = false, tma = false;
    rc = take_slices(grad_slices, grad_dtype, nd, S, outs, 4, &tab, &vec, &tma);
    if (rc != SHARDSTEP_OK) return rc;
    vec = vec && aligned(master, 16) && aligned(m, 16) && aligned(v, 16) && aligned(out_bf16, 8);
    // TMA-staged path: bulk copies need 16-byte aligned sources; the two
    // stages must fit in shared memory
    tma = tma && use_tma(TmaOp::kStep, S, nd, grad_dtype) && aligned(master, 16) && aligned(m, 16) && aligned(v, 16) &&
          aligned(out_bf16, 8) && tma_step_fits(nd, grad_dtype);
    MeanOp mo = mean_op(nd, group);
    mo.scaled = scale != nullptr;
    mo.scale = scale;
    cudaError_t e =
        tma ? launch_rs_adamw_cast_tma(tab, nd, grad_dtype, S, master, m, v, out_bf16, c, mo,
                                       skip, static_cast<cudaStream_t>(stream))
            : launch_rs_adamw_cast(tab, nd, grad_dtype, S, master, m, v, out_bf16, c, mo, skip,
                                   vec, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fused step kernel launch");
    if (tma)
        note_kernel("staged_stream<AdamOp<%s>> (TMA-staged)", dtype_name(grad_dtype));
    else if (vec && (compiled_nd(nd, {1, 2, 3, 4, 6, 8}) ||
                     (nd >= 9 && nd <= 16 && grad_dtype != SHARDSTEP_DTYPE_F32)))
        note_kernel("rs_adamw_cast_vec4<%d, %s> (register-staged)", nd, dtype_name(grad_dtype));
    else if (vec && (nd == 5 || nd == 7) && grad_dtype != SHARDSTEP_DTYPE_F32)
        note_kernel("rs_adamw_cast_vec4<up to 8: %d, %s> (register-staged)", nd,
                    dtype_name(grad_dtype));
    else if (vec)
        note_kernel("rs_adamw_cast_vec4<any N_d = %d, %s> (register-staged)", nd,
                    dtype_name(grad_dtype));
    else
        note_kernel("rs_adamw_cast_scalar<%s>", dtype_name(grad_dtype));
    count_comm(reduce_comm_bytes(nd, group, S, elem_size_of(grad_dtype)));
    return ok();
}

// The last micro-batch accumulated inside the fused step; the AdamW scalars
// from `hp` on the host or from a device-resident step `state`.
int accum_step(const float* const* acc_slices, const uint16_t* const* last_slices, int32_t nd,
               int32_t shard_group, int64_t S, float scale, float* master, float* m, float* v,
               uint16_t* out_bf16, const shardstep_adamw_t* hp,
               const shardstep_adamw_state_t* state, void* stream) {
    if (nd < 1) return fail(SHARDSTEP_ERR_INVALID, "nd must be >= 1 (got %d)", nd);
    if (nd > SHARDSTEP_MAX_ND)
        return fail(SHARDSTEP_ERR_CAPACITY, "nd %d > %d", nd, SHARDSTEP_MAX_ND);
    if (int rc = check_shard_group(nd, shard_group); rc != SHARDSTEP_OK) return rc;
    if (S < 0) return fail(SHARDSTEP_ERR_INVALID, "S must be >= 0");
    AdamScalars c{};
    if (int rc = adam_source(hp, state, &c); rc != SHARDSTEP_OK) return rc;
    if (S == 0) return ok();
    Span outs[4];
    if (int rc = check_step_outputs(S, master, m, v, out_bf16, outs); rc != SHARDSTEP_OK)
        return rc;
    PtrTable acc, last;
    bool vec_a = false, vec_l = false, tma = false;
    int rc = take_slices(reinterpret_cast<const void* const*>(acc_slices), SHARDSTEP_DTYPE_F32,
                         nd, S, outs, 4, &acc, &vec_a, &tma);
    if (rc != SHARDSTEP_OK) return rc;
    rc = take_slices(reinterpret_cast<const void* const*>(last_slices), SHARDSTEP_DTYPE_BF16, nd,
                     S, outs, 4, &last, &vec_l, &tma);
    if (rc != SHARDSTEP_OK) return rc;
    const bool vec = vec_a && vec_l && aligned(master, 16) && aligned(m, 16) &&
                     aligned(v, 16) && aligned(out_bf16, 8);
    cudaError_t e = launch_accum_rs_adamw_cast(acc, last, nd, S, scale, master, m, v, out_bf16,
                                               c, mean_op(nd, shard_group), vec,
                                               static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fused accumulate + step kernel launch");
    if (vec && shard_group != nd)
        note_kernel("accum_rs_adamw_cast_vec4<any N_d = %d, groups of %d> (register-staged)", nd,
                    shard_group);
    else if (vec && compiled_nd(nd, {1, 2, 3, 4, 6, 8}))
        note_kernel("accum_rs_adamw_cast_vec4<%d> (register-staged)", nd);
    else if (vec && (nd == 5 || nd == 7))
        note_kernel("accum_rs_adamw_cast_vec4<up to 8: %d> (register-staged)", nd);
    else if (vec)
        note_kernel("accum_rs_adamw_cast_vec4<any N_d = %d> (register-staged)", nd);
    else
        note_kernel("accum_rs_adamw_cast_scalar");
    // the contributions reduced are the fp32 sums acc_q + g_q / M
    count_comm(reduce_comm_bytes(nd, shard_group, S, 4));
    return ok();
}

}  // namespace

extern "C" {

int fsdp_rs_avg_adamw_cast(const void* const* grad_slices, int32_t grad_dtype, int32_t nd,
                           int64_t S, float* master, float* m, float* v, uint16_t* out_bf16,
                           const shardstep_adamw_t* hp, void* stream) {
    return fused_step(grad_slices, grad_dtype, nd, nd, S, master, m, v, out_bf16, hp, stream);
}

int fsdp_accumulate_rs_avg_adamw_cast(const float* const* acc_slices,
                                      const uint16_t* const* last_slices, int32_t nd,
                                      int32_t shard_group, int64_t S, float scale, float* master,
                                      float* m, float* v, uint16_t* out_bf16,
                                      const shardstep_adamw_t* hp, void* stream) {
    if (hp == nullptr) return fail(SHARDSTEP_ERR_INVALID, "hp is NULL");
    return accum_step(acc_slices, last_slices, nd, shard_group, S, scale, master, m, v, out_bf16,
                      hp, nullptr, stream);
}

int fsdp_state_accumulate_rs_avg_adamw_cast(const float* const* acc_slices,
                                            const uint16_t* const* last_slices, int32_t nd,
                                            int32_t shard_group, int64_t S, float scale,
                                            float* master, float* m, float* v,
                                            uint16_t* out_bf16,
                                            const shardstep_adamw_state_t* state,
                                            void* stream) {
    if (state == nullptr) return fail(SHARDSTEP_ERR_INVALID, "state is NULL");
    return accum_step(acc_slices, last_slices, nd, shard_group, S, scale, master, m, v, out_bf16,
                      nullptr, state, stream);
}

int fsdp_hybrid_rs_avg_adamw_cast(const void* const* grad_slices, int32_t grad_dtype, int32_t nd,
                                  int32_t shard_group, int64_t S, float* master, float* m,
                                  float* v, uint16_t* out_bf16, const shardstep_adamw_t* hp,
                                  void* stream) {
    if (int rc = check_shard_group(nd, shard_group); rc != SHARDSTEP_OK) return rc;
    return fused_step(grad_slices, grad_dtype, nd, shard_group, S, master, m, v, out_bf16, hp,
                      stream);
}

int fsdp_state_rs_avg_adamw_cast(const void* const* grad_slices, int32_t grad_dtype, int32_t nd,
                                 int32_t shard_group, int64_t S, float* master, float* m,
                                 float* v, uint16_t* out_bf16,
                                 const shardstep_adamw_state_t* state, void* stream) {
    if (int rc = check_shard_group(nd, shard_group); rc != SHARDSTEP_OK) return rc;
    if (state == nullptr) return fail(SHARDSTEP_ERR_INVALID, "state is NULL");
    return fused_step(grad_slices, grad_dtype, nd, shard_group, S, master, m, v, out_bf16,
                      nullptr, stream, nullptr, nullptr, state);
}

int shardstep_adamw_state_init(shardstep_adamw_state_t* state, const shardstep_adamw_t* hp,
                               int64_t step, void* stream) {
    if (state == nullptr || hp == nullptr) return fail(SHARDSTEP_ERR_INVALID, "state / hp is NULL");
    if (!aligned(state, 8)) return fail(SHARDSTEP_ERR_INVALID, "state misaligned");
    if (step < 0) return fail(SHARDSTEP_ERR_INVALID, "step must be >= 0");
    // the running products of step factors, as adam_scalars forms them
    double b1p = 1.0, b2p = 1.0;
    for (int64_t k = 0; k < step; ++k) {
        b1p *= hp->beta1;
        b2p *= hp->beta2;
        if (b1p == 0.0 && b2p == 0.0) break;
    }
    cudaError_t e = launch_adamw_state_set(state, step, b1p, b2p, hp->lr, hp->beta1, hp->beta2,
                                           hp->eps, hp->weight_decay,
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "state init launch");
    return ok();
}

int shardstep_adamw_state_advance(shardstep_adamw_state_t* state, const shardstep_adamw_t* hp,
                                  const uint32_t* skip, void* stream) {
    if (state == nullptr || hp == nullptr) return fail(SHARDSTEP_ERR_INVALID, "state / hp is NULL");
    if (!aligned(state, 8)) return fail(SHARDSTEP_ERR_INVALID, "state misaligned");
    if (skip != nullptr && !aligned(skip, 4)) return fail(SHARDSTEP_ERR_INVALID, "skip misaligned");
    cudaError_t e = launch_adamw_state_advance(state, hp->lr, hp->beta1, hp->beta2, hp->eps,
                                               hp->weight_decay, skip,
                                               static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "state advance launch");
    return ok();
}

int fsdp_grad_unscale_check(const void* const* grad_slices, int32_t grad_dtype, int32_t nd,
                            int32_t shard_group, int64_t S, const float* scale,
                            uint32_t* found_inf, void* stream) {
    if (int rc = check_shard_group(nd, shard_group); rc != SHARDSTEP_OK) return rc;
    if (S < 0) return fail(SHARDSTEP_ERR_INVALID, "S must be >= 0");
    if (int rc = check_scaler_words(scale, found_inf); rc != SHARDSTEP_OK) return rc;
    if (S == 0) return ok();
    PtrTable tab;
    bool vec = false, tma = false;
    const Span fs = span(found_inf, 4);
    int rc = take_slices(grad_slices, grad_dtype, nd, S, &fs, 1, &tab, &vec, &tma);
    if (rc != SHARDSTEP_OK) return rc;
    MeanOp mo = mean_op(nd, shard_group);
    mo.scaled = 1;
    mo.scale = scale;
    tma = tma && use_tma(TmaOp::kCheck, S, nd, grad_dtype) && tma_reduce_fits(nd, grad_dtype);
    cudaError_t e = tma ? launch_nonfinite_check_tma(tab, nd, grad_dtype, S, mo, found_inf,
                                                     static_cast<cudaStream_t>(stream))
                        : launch_nonfinite_check(tab, nd, grad_dtype, S, mo, found_inf, vec,
                                                 static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "non-finite check launch");
    if (tma)
        note_kernel("staged_stream<CheckOp<%s>> (TMA-staged)", dtype_name(grad_dtype));
    else if (vec && (compiled_nd(nd, {1, 2, 4, 8}) ||
                     (grad_dtype != SHARDSTEP_DTYPE_F32 && nd >= 3 && nd <= 16)))
        note_kernel("nonfinite_check_vec4<%d, %s> (register-staged)", nd, dtype_name(grad_dtype));
    else if (vec)
        note_kernel("nonfinite_check_vec4<any N_d = %d, %s> (register-staged)", nd,
                    dtype_name(grad_dtype));
    else
        note_kernel("nonfinite_check_scalar<%s>", dtype_name(grad_dtype));
    // the reduce itself is the scaled step's; the ranks OR their flags
    count_comm(allreduce_comm_bytes(nd, 4.0));
    return ok();
}

int fsdp_state_scaled_rs_avg_adamw_cast(const void* const* grad_slices, int32_t grad_dtype,
                                        int32_t nd, int32_t shard_group, int64_t S,
                                        float* master, float* m, float* v, uint16_t* out_bf16,
                                        const shardstep_adamw_state_t* state, const float* scale,
                                        const uint32_t* found_inf, void* stream) {
    if (int rc = check_shard_group(nd, shard_group); rc != SHARDSTEP_OK) return rc;
    if (state == nullptr) return fail(SHARDSTEP_ERR_INVALID, "state is NULL");
    if (int rc = check_scaler_words(scale, found_inf); rc != SHARDSTEP_OK) return rc;
    return fused_step(grad_slices, grad_dtype, nd, shard_group, S, master, m, v, out_bf16,
                      nullptr, stream, scale, found_inf, state);
}

int fsdp_scaled_rs_avg_adamw_cast(const void* const* grad_slices, int32_t grad_dtype, int32_t nd,
                                  int32_t shard_group, int64_t S, float* master, float* m,
                                  float* v, uint16_t* out_bf16, const shardstep_adamw_t* hp,
                                  const float* scale, const uint32_t* found_inf, void* stream) {
    if (int rc = check_shard_group(nd, shard_group); rc != SHARDSTEP_OK) return rc;
    if (int rc = check_scaler_words(scale, found_inf); rc != SHARDSTEP_OK) return rc;
    return fused_step(grad_slices, grad_dtype, nd, shard_group, S, master, m, v, out_bf16, hp,
                      stream, scale, found_inf);
}

int fsdp_grad_scaler_update(float* scale, int32_t* growth_tracker, uint32_t* found_inf,
                            float growth_factor, float backoff_factor, int32_t growth_interval,
                            void* stream) {
    if (scale == nullptr || growth_tracker == nullptr || found_inf == nullptr)
        return fail(SHARDSTEP_ERR_INVALID, "scale / growth_tracker / found_inf is NULL");
    if (!aligned(scale, 4) || !aligned(growth_tracker, 4) || !aligned(found_inf, 4))
        return fail(SHARDSTEP_ERR_INVALID, "scaler words must be 4-byte aligned");
    if (growth_interval < 1) return fail(SHARDSTEP_ERR_INVALID, "growth_interval must be >= 1");
    cudaError_t e = launch_scaler_update(scale, growth_tracker, found_inf, growth_factor,
                                         backoff_factor, growth_interval,
                                         static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "scaler update launch");
    return ok();
}

double shardstep_hybrid_state_bytes(double psi, int32_t shard_group, double k) {
    if (shard_group < 1) return -1.0;
    return (2 * psi + 2 * psi + k * psi) / shard_group;
}

double shardstep_hybrid_comm_bytes(double psi, int32_t nd, int32_t shard_group, int32_t kind,
                                   int32_t exact) {
    if (shard_group < 1 || nd < 1 || nd % shard_group != 0) return -1.0;
    const int32_t R = nd / shard_group;
    if (kind == SHARDSTEP_HYBRID_INTRA) {
        if (shard_group == 1) return 0.0;
        const double f = exact ? static_cast<double>(shard_group - 1) / shard_group : 1.0;
        return 2 * (2 * psi * f);
    }
    if (kind == SHARDSTEP_HYBRID_INTER) {
        if (R == 1) return 0.0;
        const double f = exact ? static_cast<double>(R - 1) / R : 1.0;
        return 4 * (psi / shard_group) * f;
    }
    return -1.0;
}

// ------------------------------------------------------------- FSDP2

}  // extern "C"

namespace {

// Per-parameter dim-0 layout shared by the FSDP2 entry points.
struct Fsdp2Plan {
    std::vector<int64_t> chunk, offset;
    int64_t local = 0;
};

int fsdp2_plan(const int64_t* dim0, const int64_t* row, int32_t n, int32_t nd, Fsdp2Plan* plan) {
    if (n < 0) return fail(SHARDSTEP_ERR_INVALID, "n must be >= 0");
    if (nd < 1) return fail(SHARDSTEP_ERR_INVALID, "nd must be >= 1 (got %d)", nd);
    if (n > 0 && (dim0 == nullptr || row == nullptr))
        return fail(SHARDSTEP_ERR_INVALID, "dim0 / row is NULL");
    plan->chunk.assign(n, 0);
    plan->offset.assign(n, 0);
    int64_t pos = 0;
    for (int32_t t = 0; t < n; ++t) {
        if (dim0[t] < 0 || row[t] < 0)
            return fail(SHARDSTEP_ERR_INVALID, "parameter %d has a negative size", t);
        const int64_t c = (dim0[t] + nd - 1) / nd;
        if (row[t] > 0 && c > (INT64_MAX / 16 - pos) / row[t])
            return fail(SHARDSTEP_ERR_INVALID, "group too large");
        plan->chunk[t] = c;
        plan->offset[t] = pos;
        pos += c * row[t];
    }
    plan->local = pos;
    return SHARDSTEP_OK;
}

int64_t rows_of(const Fsdp2Plan& p, const int64_t* dim0, int32_t r, int32_t t) {
    const int64_t left = dim0[t] - static_cast<int64_t>(r) * p.chunk[t];
    return left < 0 ? 0 : (left < p.chunk[t] ? left : p.chunk[t]);
}

}  // namespace

extern "C" {

int fsdp2_layout(const int64_t* dim0, const int64_t* row, int32_t n, int32_t nd, int64_t* chunk,
                 int64_t* offset, int64_t* local) {
    if (local == nullptr) return fail(SHARDSTEP_ERR_INVALID, "local is NULL");
    Fsdp2Plan plan;
    int rc = fsdp2_plan(dim0, row, n, nd, &plan);
    if (rc != SHARDSTEP_OK) return rc;
    for (int32_t t = 0; t < n; ++t) {
        if (chunk) chunk[t] = plan.chunk[t];
        if (offset) offset[t] = plan.offset[t];
    }
    *local = plan.local;
    return ok();
}

int fsdp2_local_views(const int64_t* dim0, const int64_t* row, int32_t n, int32_t nd,
                      int32_t rank, void* base, int32_t elem_size, void** ptrs, int64_t* rows) {
    Fsdp2Plan plan;
    int rc = fsdp2_plan(dim0, row, n, nd, &plan);
    if (rc != SHARDSTEP_OK) return rc;
    if (rank < 0 || rank >= nd) return fail(SHARDSTEP_ERR_INVALID, "rank %d out of range", rank);
    if (elem_size <= 0) return fail(SHARDSTEP_ERR_INVALID, "elem_size must be > 0");
    if (n > 0 && (ptrs == nullptr || rows == nullptr))
        return fail(SHARDSTEP_ERR_INVALID, "ptrs / rows is NULL");
    for (int32_t t = 0; t < n; ++t) {
        ptrs[t] = static_cast<char*>(base) + plan.offset[t] * elem_size;
        rows[t] = rows_of(plan, dim0, rank, t);
    }
    return ok();
}

int fsdp2_chunk_cat(const void* const* grads, const int64_t* dim0, const int64_t* row, int32_t n,
                    int32_t nd, int32_t dtype, void* out, void* stream) {
    const int es = elem_size_of(dtype);
    if (es == 0) return fail(SHARDSTEP_ERR_INVALID, "unknown dtype %d", dtype);
    Fsdp2Plan plan;
    int rc = fsdp2_plan(dim0, row, n, nd, &plan);
    if (rc != SHARDSTEP_OK) return rc;
    if (plan.local == 0) return ok();
    if (out == nullptr || (n > 0 && grads == nullptr))
        return fail(SHARDSTEP_ERR_INVALID, "grads / out is NULL");
    if (!aligned(out, es)) return fail(SHARDSTEP_ERR_INVALID, "out is not %d-byte aligned", es);
    const Span os = span(out, static_cast<int64_t>(nd) * plan.local * es);
    for (int32_t t = 0; t < n; ++t) {
        const int64_t bytes = dim0[t] * row[t] * es;
        if (bytes == 0) continue;
        if (grads[t] == nullptr) return fail(SHARDSTEP_ERR_INVALID, "grads[%d] is NULL", t);
        if (!aligned(grads[t], es))
            return fail(SHARDSTEP_ERR_INVALID, "grads[%d] is not %d-byte aligned", t, es);
        if (overlap(span(grads[t], bytes), os))
            return fail(SHARDSTEP_ERR_INVALID, "grads[%d] overlaps out", t);
    }
    CopyBatcher cb(static_cast<cudaStream_t>(stream));
    char* o = static_cast<char*>(out);
    for (int32_t r = 0; r < nd; ++r)
        for (int32_t t = 0; t < n; ++t) {
            const int64_t rows = rows_of(plan, dim0, r, t), seg = plan.chunk[t] * row[t];
            char* dst = o + (static_cast<int64_t>(r) * plan.local + plan.offset[t]) * es;
            const int64_t have = rows * row[t];
            cb.add(static_cast<const char*>(grads[t]) +
                       static_cast<int64_t>(r) * plan.chunk[t] * row[t] * es,
                   dst, have * es);
            cb.add(nullptr, dst + have * es, (seg - have) * es);  // zero padding rows
        }
    cb.flush();
    return cb.rc == SHARDSTEP_OK ? ok() : cb.rc;
}

int fsdp2_all_gather_copy_out(const void* const* local_bufs, const int64_t* dim0,
                              const int64_t* row, int32_t n, int32_t nd, int32_t dtype,
                              void* const* params, void* stream) {
    const int es = elem_size_of(dtype);
    if (es == 0) return fail(SHARDSTEP_ERR_INVALID, "unknown dtype %d", dtype);
    Fsdp2Plan plan;
    int rc = fsdp2_plan(dim0, row, n, nd, &plan);
    if (rc != SHARDSTEP_OK) return rc;
    if (plan.local == 0) return ok();
    if (local_bufs == nullptr || (n > 0 && params == nullptr))
        return fail(SHARDSTEP_ERR_INVALID, "local_bufs / params is NULL");
    for (int32_t r = 0; r < nd; ++r) {
        if (local_bufs[r] == nullptr)
            return fail(SHARDSTEP_ERR_INVALID, "local_bufs[%d] is NULL", r);
        if (!aligned(local_bufs[r], es))
            return fail(SHARDSTEP_ERR_INVALID, "local_bufs[%d] is not %d-byte aligned", r, es);
    }
    for (int32_t t = 0; t < n; ++t) {
        const int64_t bytes = dim0[t] * row[t] * es;
        if (bytes == 0) continue;
        if (params[t] == nullptr) return fail(SHARDSTEP_ERR_INVALID, "params[%d] is NULL", t);
        if (!aligned(params[t], es))
            return fail(SHARDSTEP_ERR_INVALID, "params[%d] is not %d-byte aligned", t, es);
        for (int32_t r = 0; r < nd; ++r)
            if (overlap(span(params[t], bytes), span(local_bufs[r], plan.local * es)))
                return fail(SHARDSTEP_ERR_INVALID, "params[%d] overlaps local_bufs[%d]", t, r);
    }
    CopyBatcher cb(static_cast<cudaStream_t>(stream));
    for (int32_t t = 0; t < n; ++t)
        for (int32_t r = 0; r < nd; ++r) {
            const int64_t have = rows_of(plan, dim0, r, t) * row[t];
            cb.add(static_cast<const char*>(local_bufs[r]) + plan.offset[t] * es,
                   static_cast<char*>(params[t]) +
                       static_cast<int64_t>(r) * plan.chunk[t] * row[t] * es,
                   have * es);
        }
    cb.flush();
    if (cb.rc != SHARDSTEP_OK) return cb.rc;
    count_comm(static_cast<double>(nd - 1) * static_cast<double>(plan.local) * es);
    return ok();
}

namespace {

// The FSDP2 step of one rank; the AdamW scalars from `hp` on the host or
// from a device-resident step `state`.
int fsdp2_step(const void* const* grads, int32_t grad_dtype, const int64_t* dim0,
               const int64_t* row, int32_t n, int32_t nd, int32_t rank, float* master, float* m,
               float* v, uint16_t* out_bf16, const shardstep_adamw_t* hp,
               const shardstep_adamw_state_t* state, void* stream) {
    const int es = elem_size_of(grad_dtype);
    if (es == 0) return fail(SHARDSTEP_ERR_INVALID, "unknown grad dtype %d", grad_dtype);
    if (nd > SHARDSTEP_MAX_ND)
        return fail(SHARDSTEP_ERR_CAPACITY, "nd %d > %d", nd, SHARDSTEP_MAX_ND);
    Fsdp2Plan plan;
    int rc = fsdp2_plan(dim0, row, n, nd, &plan);
    if (rc != SHARDSTEP_OK) return rc;
    if (rank < 0 || rank >= nd) return fail(SHARDSTEP_ERR_INVALID, "rank %d not in [0, %d)", rank, nd);
    AdamScalars c{};
    if (int rc2 = adam_source(hp, state, &c); rc2 != SHARDSTEP_OK) return rc2;
    const int64_t L = plan.local;
    if (L == 0) return ok();
    Span outs[4];
    if (int rc2 = check_step_outputs(L, master, m, v, out_bf16, outs); rc2 != SHARDSTEP_OK)
        return rc2;
    if (n > 0 && grads == nullptr) return fail(SHARDSTEP_ERR_INVALID, "grads is NULL");
    // every gradient whole: present, aligned, and clear of the local buffers
    for (int32_t q = 0; q < nd; ++q)
        for (int32_t t = 0; t < n; ++t) {
            const int64_t bytes = dim0[t] * row[t] * es;
            if (bytes == 0) continue;
            const void* g = grads[static_cast<int64_t>(q) * n + t];
            if (g == nullptr) return fail(SHARDSTEP_ERR_INVALID, "grads[%d][%d] is NULL", q, t);
            if (!aligned(g, es))
                return fail(SHARDSTEP_ERR_INVALID, "grads[%d][%d] is not %d-byte aligned", q, t, es);
            for (const Span& o : outs)
                if (overlap(span(g, bytes), o))
                    return fail(SHARDSTEP_ERR_INVALID, "grads[%d][%d] overlaps an output", q, t);
        }
    // Segments: per parameter, the rank's rows (slice q = rank q's gradient
    // from row rank * chunk) and its padding rows (every contribution +0).
    // Aligned ones go into tables of one launch each (rs_adamw_cast_segs);
    // the others, and every one when the TMA path is forced, take the fused
    // step per parameter and the zero-gradient AdamW per padding run.
    const bool segs_ok = g_fused_path.load(std::memory_order_relaxed) != SHARDSTEP_PATH_TMA &&
                         aligned(master, 16) && aligned(m, 16) && aligned(v, 16) &&
                         aligned(out_bf16, 8);
    const uintptr_t slice_align = grad_dtype == SHARDSTEP_DTYPE_F32 ? 16 : 8;
    const MeanOp mo = mean_op(nd, nd);
    SegTable st{};
    st.ns = 0;
    st.b0[0] = 0;
    int tables = 0;
    int np = 0;  // slice pointers used in the current table
    auto flush = [&]() -> int {
        if (st.ns == 0) return SHARDSTEP_OK;
        cudaError_t e = launch_rs_adamw_cast_segs(st, nd, grad_dtype, master, m, v, out_bf16, c,
                                                  mo, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "FSDP2 step launch");
        ++tables;
        st.ns = 0;
        st.b0[0] = 0;
        np = 0;
        return SHARDSTEP_OK;
    };
    // p == nullptr: padding rows, which take no slice pointers
    auto add_seg = [&](int64_t lo, int64_t cnt, const void* const* p) -> int {
        if (st.ns == kSegMax || (p != nullptr && np + nd > kSegPtrMax))
            if (int r = flush(); r != SHARDSTEP_OK) return r;
        const int k = st.ns;
        st.lo[k] = lo;
        st.n[k] = cnt;
        st.po[k] = -1;
        if (p != nullptr) {
            st.po[k] = np;
            for (int32_t q = 0; q < nd; ++q) st.p[np + q] = p[q];
            np += nd;
        }
        st.b0[k + 1] = st.b0[k] + seg_blocks(cnt);
        st.ns = k + 1;
        return SHARDSTEP_OK;
    };
    std::vector<const void*> slices(nd);
    bool fused_launched = false, pad_launched = false;
    for (int32_t t = 0; t < n; ++t) {
        const int64_t off = plan.offset[t];
        const int64_t have = rows_of(plan, dim0, rank, t) * row[t];
        const int64_t pad = plan.chunk[t] * row[t] - have;
        if (have > 0) {
            const int64_t src = static_cast<int64_t>(rank) * plan.chunk[t] * row[t] * es;
            bool vec = segs_ok && off % 4 == 0;
            for (int32_t q = 0; q < nd; ++q) {
                slices[q] = static_cast<const char*>(grads[static_cast<int64_t>(q) * n + t]) + src;
                vec = vec && aligned(slices[q], slice_align);
            }
            if (vec) {
                if (int r = add_seg(off, have, slices.data()); r != SHARDSTEP_OK) return r;
                count_comm(reduce_comm_bytes(nd, nd, have, es));
            } else {
                rc = fused_step(slices.data(), grad_dtype, nd, nd, have, master + off, m + off,
                                v + off, out_bf16 + off, hp, stream, nullptr, nullptr, state);
                if (rc != SHARDSTEP_OK) return rc;
                fused_launched = true;
            }
        }
        if (pad > 0) {
            // the padding rows are in the reduce-scatter a real group sends
            count_comm(reduce_comm_bytes(nd, nd, pad, es));
            if (segs_ok && (off + have) % 4 == 0) {
                if (int r = add_seg(off + have, pad, nullptr); r != SHARDSTEP_OK) return r;
            } else {
                cudaError_t e = launch_adamw_zero_grad(pad, master + off + have, m + off + have,
                                                       v + off + have, out_bf16 + off + have, c,
                                                       static_cast<cudaStream_t>(stream));
                if (e != cudaSuccess) return cuda_fail(e, "zero-gradient AdamW launch");
                pad_launched = true;
            }
        }
    }
    if (int r = flush(); r != SHARDSTEP_OK) return r;
    // compiled for 1..8 slices and 9..16 16-bit slices; the loop over any
    // N_d otherwise
    const bool compiled = nd <= 8 || (nd <= 16 && grad_dtype != SHARDSTEP_DTYPE_F32);
    if (tables > 0)
        note_kernel("rs_adamw_cast_segs<%s%d, %s> (register-staged, %d launch%s)",
                    compiled ? "" : "any N_d = ", nd, dtype_name(grad_dtype), tables,
                    tables > 1 ? "es" : "");
    else if (pad_launched && !fused_launched)
        note_kernel("adamw_zero_grad");
    return ok();
}

}  // namespace

int fsdp2_rs_avg_adamw_cast(const void* const* grads, int32_t grad_dtype, const int64_t* dim0,
                            const int64_t* row, int32_t n, int32_t nd, int32_t rank,
                            float* master, float* m, float* v, uint16_t* out_bf16,
                            const shardstep_adamw_t* hp, void* stream) {
    if (hp == nullptr) return fail(SHARDSTEP_ERR_INVALID, "hp is NULL");
    return fsdp2_step(grads, grad_dtype, dim0, row, n, nd, rank, master, m, v, out_bf16, hp,
                      nullptr, stream);
}

int fsdp2_state_rs_avg_adamw_cast(const void* const* grads, int32_t grad_dtype,
                                  const int64_t* dim0, const int64_t* row, int32_t n, int32_t nd,
                                  int32_t rank, float* master, float* m, float* v,
                                  uint16_t* out_bf16, const shardstep_adamw_state_t* state,
                                  void* stream) {
    if (state == nullptr) return fail(SHARDSTEP_ERR_INVALID, "state is NULL");
    return fsdp2_step(grads, grad_dtype, dim0, row, n, nd, rank, master, m, v, out_bf16, nullptr,
                      state, stream);
}

int ddp_bucket_plan(const int64_t* numels, int32_t n, int32_t elem_size, int64_t cap_bytes,
                    int64_t* param_offset, int32_t* bucket_of_param, int64_t* bucket_offsets,
                    int32_t* n_buckets) {
    if (n < 0) return fail(SHARDSTEP_ERR_INVALID, "n must be >= 0");
    if (elem_size <= 0 || cap_bytes <= 0)
        return fail(SHARDSTEP_ERR_INVALID, "elem_size and cap_bytes must be > 0");
    if (n_buckets == nullptr || bucket_offsets == nullptr)
        return fail(SHARDSTEP_ERR_INVALID, "bucket_offsets / n_buckets is NULL");
    if (n > 0 && (numels == nullptr || param_offset == nullptr || bucket_of_param == nullptr))
        return fail(SHARDSTEP_ERR_INVALID, "numels / param_offset / bucket_of_param is NULL");
    for (int32_t i = 0; i < n; ++i)
        if (numels[i] < 0) return fail(SHARDSTEP_ERR_INVALID, "numel %d is negative", i);
    int32_t nb = 0;
    int64_t pos = 0, cur_bytes = 0;
    bool open = false;
    bucket_offsets[0] = 0;
    for (int32_t i = n - 1; i >= 0; --i) {
        const int64_t b = numels[i] * elem_size;
        if (open && cur_bytes + b > cap_bytes) {
            bucket_offsets[++nb] = pos;
            cur_bytes = 0;
            open = false;
        }
        open = true;
        bucket_of_param[i] = nb;
        param_offset[i] = pos;
        pos += numels[i];
        cur_bytes += b;
    }
    if (open) bucket_offsets[++nb] = pos;
    *n_buckets = nb;
    return ok();
}

int ddp_bucket_allreduce_avg(const uint16_t* const* rank_grads, int32_t nd,
                             const int64_t* bucket_offsets, int32_t first, int32_t count,
                             uint16_t* out, void* stream) {
    if (nd < 1) return fail(SHARDSTEP_ERR_INVALID, "nd must be >= 1 (got %d)", nd);
    if (nd > SHARDSTEP_MAX_ND)
        return fail(SHARDSTEP_ERR_CAPACITY, "nd %d > %d", nd, SHARDSTEP_MAX_ND);
    if (first < 0 || count < 0) return fail(SHARDSTEP_ERR_INVALID, "first / count negative");
    if (count == 0) return ok();
    if (bucket_offsets == nullptr || rank_grads == nullptr)
        return fail(SHARDSTEP_ERR_INVALID, "bucket_offsets / rank_grads is NULL");
    for (int32_t b = first; b < first + count; ++b)
        if (bucket_offsets[b] < 0 || bucket_offsets[b + 1] < bucket_offsets[b])
            return fail(SHARDSTEP_ERR_INVALID, "bucket offsets must be non-decreasing");
    const int64_t a0 = bucket_offsets[first], e0 = bucket_offsets[first + count];
    if (e0 == a0) return ok();                 // every bucket of the range is empty
    if (out == nullptr) return fail(SHARDSTEP_ERR_INVALID, "out is NULL");
    if (!aligned(out, 2)) return fail(SHARDSTEP_ERR_INVALID, "out is not 2-byte aligned");
    const Span os = span(out + a0, (e0 - a0) * 2);
    for (int32_t q = 0; q < nd; ++q) {
        if (rank_grads[q] == nullptr)
            return fail(SHARDSTEP_ERR_INVALID, "rank_grads[%d] is NULL", q);
        if (!aligned(rank_grads[q], 2))
            return fail(SHARDSTEP_ERR_INVALID, "rank_grads[%d] is not 2-byte aligned", q);
        if (overlap(span(rank_grads[q] + a0, (e0 - a0) * 2), os))
            return fail(SHARDSTEP_ERR_INVALID, "rank_grads[%d] overlaps out", q);
    }
    const MeanOp mo = mean_op(nd, nd);
    // the first launch of the call waits for everything before it in the
    // stream (the producers of the gradients); later buckets only follow
    // this call's own launches, on disjoint outputs, so they go out as
    // programmatic dependents and overlap the previous bucket's drain
    bool pdl = false;
    for (int32_t b = first; b < first + count; ++b) {
        const int64_t a = bucket_offsets[b], n = bucket_offsets[b + 1] - a;
        if (n == 0) continue;
        PtrTable tab;
        bool vec = aligned(out + a, 8),
             tma = vec && use_tma(TmaOp::kAllReduce, n, nd) && tma_reduce_fits(nd, 0);
        for (int32_t q = 0; q < SHARDSTEP_MAX_ND; ++q) {
            tab.p[q] = q < nd ? rank_grads[q] + a : nullptr;
            if (q < nd) {
                vec = vec && aligned(tab.p[q], 8);
                tma = tma && aligned(tab.p[q], 16);
            }
        }
        cudaError_t e = tma ? launch_allreduce_avg_tma(tab, nd, n, out + a, mo, pdl,
                                                       static_cast<cudaStream_t>(stream))
                            : launch_allreduce_avg(tab, nd, n, out + a, mo, vec, pdl,
                                                   static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "all-reduce kernel launch");
        if (tma)
            note_kernel("staged_stream<MeanOutOp> (TMA-staged)");
        else if (vec && nd >= 1 && nd <= 16)
            note_kernel("allreduce_avg_vec4<%d> (register-staged)", nd);
        else if (vec)
            note_kernel("allreduce_avg_vec4<any N_d = %d> (register-staged)", nd);
        else
            note_kernel("allreduce_avg_scalar");
        pdl = g_dependent_launch.load(std::memory_order_relaxed) != 0;
    }
    count_comm(allreduce_comm_bytes(nd, static_cast<double>(e0 - a0) * 2.0));
    return ok();
}

int ddp_bucket_allreduce_avg_adamw_cast(const uint16_t* const* rank_grads, int32_t nd,
                                        const int64_t* bucket_offsets, int32_t first,
                                        int32_t count, uint16_t* mean_out, float* master,
                                        float* m, float* v, uint16_t* params,
                                        const shardstep_adamw_t* hp, void* stream) {
    if (nd < 1) return fail(SHARDSTEP_ERR_INVALID, "nd must be >= 1 (got %d)", nd);
    if (nd > SHARDSTEP_MAX_ND)
        return fail(SHARDSTEP_ERR_CAPACITY, "nd %d > %d", nd, SHARDSTEP_MAX_ND);
    if (first < 0 || count < 0) return fail(SHARDSTEP_ERR_INVALID, "first / count negative");
    AdamScalars c{};
    if (int rc = adam_source(hp, nullptr, &c); rc != SHARDSTEP_OK) return rc;
    if (count == 0) return ok();
    if (bucket_offsets == nullptr || rank_grads == nullptr)
        return fail(SHARDSTEP_ERR_INVALID, "bucket_offsets / rank_grads is NULL");
    for (int32_t b = first; b < first + count; ++b)
        if (bucket_offsets[b] < 0 || bucket_offsets[b + 1] < bucket_offsets[b])
            return fail(SHARDSTEP_ERR_INVALID, "bucket offsets must be non-decreasing");
    const int64_t a0 = bucket_offsets[first], n = bucket_offsets[first + count] - a0;
    if (n == 0) return ok();
    // the buckets first..first+count-1 are contiguous: one launch over them
    Span outs[5];
    if (int rc = check_step_outputs(n, master ? master + a0 : nullptr, m ? m + a0 : nullptr,
                                    v ? v + a0 : nullptr, params ? params + a0 : nullptr, outs);
        rc != SHARDSTEP_OK)
        return rc;
    int n_outs = 4;
    if (mean_out != nullptr) {
        if (!aligned(mean_out, 2))
            return fail(SHARDSTEP_ERR_INVALID, "mean_out is not 2-byte aligned");
        outs[4] = span(mean_out + a0, n * 2);
        for (int a = 0; a < 4; ++a)
            if (overlap(outs[4], outs[a]))
                return fail(SHARDSTEP_ERR_INVALID, "mean_out overlaps output %d", a);
        n_outs = 5;
    }
    std::vector<const void*> slices(nd);
    for (int32_t q = 0; q < nd; ++q) {
        if (rank_grads[q] == nullptr)
            return fail(SHARDSTEP_ERR_INVALID, "rank_grads[%d] is NULL", q);
        slices[q] = rank_grads[q] + a0;
    }
    PtrTable tab;
    bool vec = false, tma = false;
    int rc = take_slices(slices.data(), SHARDSTEP_DTYPE_BF16, nd, n, outs, n_outs, &tab, &vec,
                         &tma);
    if (rc != SHARDSTEP_OK) return rc;
    vec = vec && aligned(master + a0, 16) && aligned(m + a0, 16) && aligned(v + a0, 16) &&
          aligned(params + a0, 8) && (mean_out == nullptr || aligned(mean_out + a0, 8));
    cudaError_t e = launch_ddp_allreduce_adamw_cast(
        tab, nd, n, mean_out ? mean_out + a0 : nullptr, master + a0, m + a0, v + a0,
        params + a0, c, mean_op(nd, nd), vec, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fused all-reduce + AdamW kernel launch");
    if (vec && (compiled_nd(nd, {1, 2, 3, 4, 6, 8}) || (nd >= 9 && nd <= 16)))
        note_kernel("ddp_allreduce_adamw_cast_vec4<%d> (register-staged)", nd);
    else if (vec && (nd == 5 || nd == 7))
        note_kernel("ddp_allreduce_adamw_cast_vec4<up to 8: %d> (register-staged)", nd);
    else if (vec)
        note_kernel("ddp_allreduce_adamw_cast_vec4<any N_d = %d> (register-staged)", nd);
    else
        note_kernel("ddp_allreduce_adamw_cast_scalar");
    count_comm(allreduce_comm_bytes(nd, static_cast<double>(n) * 2.0));
    return ok();
}

double shardstep_state_bytes(double psi, int32_t nd, int32_t stage, double k) {
    if (nd < 1) return -1.0;
    switch (stage) {
        case 0: return 2 * psi + 2 * psi + k * psi;
        case 1: return 2 * psi + 2 * psi + k * psi / nd;
        case 2: return 2 * psi + (2 * psi + k * psi) / nd;
        case 3: return (2 * psi + 2 * psi + k * psi) / nd;
        default: return -1.0;
    }
}

double shardstep_comm_bytes(double psi, int32_t nd, int32_t kind, int32_t exact) {
    if (nd < 1) return -1.0;
    const double f = exact ? static_cast<double>(nd - 1) / nd : 1.0;
    const double one = 2 * psi * f;  // one reduce-scatter or all-gather pass
    switch (kind) {
        case SHARDSTEP_COMM_REDUCE_SCATTER:
        case SHARDSTEP_COMM_ALL_GATHER: return one;
        case SHARDSTEP_COMM_ALL_REDUCE:
        case SHARDSTEP_COMM_ZERO1:
        case SHARDSTEP_COMM_ZERO2: return 2 * one;
        case SHARDSTEP_COMM_ZERO3: return 3 * one;
        default: return -1.0;
    }
}

}  // extern "C"
