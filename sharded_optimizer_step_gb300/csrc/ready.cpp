// Host-side readiness of the DDP gradient buckets across the N_d emulated
// ranks.  A bucket's all-reduce may start once every rank has produced every
// gradient in it ("4.1 数据并行详解", DDP section on buckets: a bucket is
// reduced as soon as all its gradients are ready).  A parameter whose
// gradient never arrives -- one the forward pass did not use -- leaves its
// bucket incomplete on that rank, and a collective that waited for it would
// hang; here the wait is on the host, bounded, and reports which (rank,
// parameter) is missing, so no kernel is ever launched for an incomplete
// bucket and nothing spins on the GPU.
//
// The table lives in memory the caller provides (ddp_ready_bytes tells how
// much); marks from several host threads (one per emulated rank) are atomic.
// Layout: a header, bucket_of_param[n_params], pending[n_buckets] (marks
// still missing: N_d x the bucket's parameters), marked[N_d * n_params].
#include <chrono>
#include <cstdint>
#include <cstring>
#include <thread>

#include "shardstep.h"

namespace shardstep {
int ready_fail(int code, const char* fmt, ...);  // api.cpp: sets the last error
int ready_ok();
}  // namespace shardstep

namespace {

constexpr uint32_t kMagic = 0x52445944u;  // "DYDR"

struct Header {
    uint32_t magic;
    int32_t n_params;
    int32_t n_buckets;
    int32_t nd;
};

size_t align8(size_t x) { return (x + 7) & ~size_t{7}; }

struct View {
    Header* h;
    int32_t* bucket_of;
    int32_t* pending;
    uint8_t* marked;
};

View view_of(void* table) {
    char* p = static_cast<char*>(table);
    View v;
    v.h = reinterpret_cast<Header*>(p);
    size_t off = align8(sizeof(Header));
    v.bucket_of = reinterpret_cast<int32_t*>(p + off);
    off = align8(off + sizeof(int32_t) * static_cast<size_t>(v.h->n_params));
    v.pending = reinterpret_cast<int32_t*>(p + off);
    off = align8(off + sizeof(int32_t) * static_cast<size_t>(v.h->n_buckets));
    v.marked = reinterpret_cast<uint8_t*>(p + off);
    return v;
}

int64_t bytes_for(int32_t n_params, int32_t n_buckets, int32_t nd) {
    size_t off = align8(sizeof(Header));
    off = align8(off + sizeof(int32_t) * static_cast<size_t>(n_params));
    off = align8(off + sizeof(int32_t) * static_cast<size_t>(n_buckets));
    off += static_cast<size_t>(nd) * static_cast<size_t>(n_params);
    return static_cast<int64_t>(align8(off));
}

bool valid(void* table) {
    if (table == nullptr || (reinterpret_cast<uintptr_t>(table) & 7u) != 0) return false;
    return static_cast<Header*>(table)->magic == kMagic;
}

void fill_pending(View v) {
    for (int32_t b = 0; b < v.h->n_buckets; ++b) v.pending[b] = 0;
    for (int32_t i = 0; i < v.h->n_params; ++i) v.pending[v.bucket_of[i]] += v.h->nd;
    std::memset(v.marked, 0, static_cast<size_t>(v.h->nd) * static_cast<size_t>(v.h->n_params));
}

}  // namespace

extern "C" {

int64_t ddp_ready_bytes(int32_t n_params, int32_t n_buckets, int32_t nd) {
    if (n_params < 0 || n_buckets < 1 || nd < 1 || nd > SHARDSTEP_MAX_ND) return -1;
    return bytes_for(n_params, n_buckets, nd);
}

int ddp_ready_init(void* table, int64_t table_bytes, const int32_t* bucket_of_param,
                   int32_t n_params, int32_t n_buckets, int32_t nd) {
    using namespace shardstep;
    const int64_t need = ddp_ready_bytes(n_params, n_buckets, nd);
    if (need < 0) return ready_fail(SHARDSTEP_ERR_INVALID, "bad n_params / n_buckets / nd");
    if (table == nullptr || (reinterpret_cast<uintptr_t>(table) & 7u) != 0)
        return ready_fail(SHARDSTEP_ERR_INVALID, "table must be 8-byte aligned host memory");
    if (table_bytes < need)
        return ready_fail(SHARDSTEP_ERR_CAPACITY, "table needs %lld bytes, got %lld",
                          static_cast<long long>(need), static_cast<long long>(table_bytes));
    if (n_params > 0 && bucket_of_param == nullptr)
        return ready_fail(SHARDSTEP_ERR_INVALID, "bucket_of_param is NULL");
    for (int32_t i = 0; i < n_params; ++i)
        if (bucket_of_param[i] < 0 || bucket_of_param[i] >= n_buckets)
            return ready_fail(SHARDSTEP_ERR_INVALID, "bucket_of_param[%d] = %d out of range", i,
                              bucket_of_param[i]);
    Header* h = static_cast<Header*>(table);
    h->n_params = n_params;
    h->n_buckets = n_buckets;
    h->nd = nd;
    View v = view_of(table);
    for (int32_t i = 0; i < n_params; ++i) v.bucket_of[i] = bucket_of_param[i];
    fill_pending(v);
    __atomic_store_n(&h->magic, kMagic, __ATOMIC_RELEASE);
    return ready_ok();
}

int ddp_ready_mark(void* table, int32_t rank, int32_t param, int32_t* bucket_done) {
    using namespace shardstep;
    if (!valid(table)) return ready_fail(SHARDSTEP_ERR_INVALID, "table not initialised");
    View v = view_of(table);
    if (rank < 0 || rank >= v.h->nd || param < 0 || param >= v.h->n_params)
        return ready_fail(SHARDSTEP_ERR_INVALID, "rank %d / param %d out of range", rank, param);
    uint8_t* flag = &v.marked[static_cast<size_t>(rank) * v.h->n_params + param];
    if (__atomic_exchange_n(flag, uint8_t{1}, __ATOMIC_ACQ_REL) != 0)
        return ready_fail(SHARDSTEP_ERR_INVALID, "rank %d marked param %d twice", rank, param);
    const int32_t b = v.bucket_of[param];
    const int32_t left = __atomic_sub_fetch(&v.pending[b], 1, __ATOMIC_ACQ_REL);
    if (bucket_done != nullptr) *bucket_done = left == 0 ? b : -1;
    return ready_ok();
}

int ddp_ready_wait(void* table, int32_t bucket, int64_t timeout_us, int32_t* missing_rank,
                   int32_t* missing_param) {
    using namespace shardstep;
    if (!valid(table)) return ready_fail(SHARDSTEP_ERR_INVALID, "table not initialised");
    View v = view_of(table);
    if (bucket < 0 || bucket >= v.h->n_buckets)
        return ready_fail(SHARDSTEP_ERR_INVALID, "bucket %d out of range", bucket);
    if (timeout_us < 0) return ready_fail(SHARDSTEP_ERR_INVALID, "timeout must be >= 0");
    const auto t0 = std::chrono::steady_clock::now();
    const auto limit = std::chrono::microseconds(timeout_us);
    for (;;) {
        if (__atomic_load_n(&v.pending[bucket], __ATOMIC_ACQUIRE) == 0) {
            if (missing_rank) *missing_rank = -1;
            if (missing_param) *missing_param = -1;
            return ready_ok();
        }
        if (std::chrono::steady_clock::now() - t0 >= limit) break;
        std::this_thread::sleep_for(std::chrono::microseconds(20));
    }
    // name one (rank, parameter) of the bucket that never arrived
    int32_t mr = -1, mp = -1;
    for (int32_t r = 0; r < v.h->nd && mr < 0; ++r)
        for (int32_t i = 0; i < v.h->n_params; ++i)
            if (v.bucket_of[i] == bucket &&
                __atomic_load_n(&v.marked[static_cast<size_t>(r) * v.h->n_params + i],
                                __ATOMIC_ACQUIRE) == 0) {
                mr = r;
                mp = i;
                break;
            }
    if (missing_rank) *missing_rank = mr;
    if (missing_param) *missing_param = mp;
    return ready_fail(SHARDSTEP_ERR_TIMEOUT,
                      "bucket %d not ready after %lld us: rank %d never marked param %d", bucket,
                      static_cast<long long>(timeout_us), mr, mp);
}

int ddp_ready_reset(void* table) {
    using namespace shardstep;
    if (!valid(table)) return ready_fail(SHARDSTEP_ERR_INVALID, "table not initialised");
    fill_pending(view_of(table));
    __atomic_thread_fence(__ATOMIC_SEQ_CST);
    return ready_ok();
}

}  // extern "C"
