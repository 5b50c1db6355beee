// Sharded checkpoint files (host only): every rank writes the shards it owns
// to a file of its own, with the metadata a load needs to restore them under
// another rank count; a load reads the pieces of the saved shards that make
// up its new shard (fsdp_reshard_plan + shardstep_ckpt_read).
//
// Rank file layout (little-endian):
//   header (64 B): magic "SHSTCKPT", u32 version, u32 header_bytes,
//                  i32 nd, i32 rank, i32 n_units, i32 n_sections, i64 step,
//                  u64 checksum of the unit and section tables, 16 B zero
//   unit totals:   n_units x i64 (elements of each unit's FlatParameter, T_u)
//   section table: n_sections x {i32 unit, i32 kind, i64 bytes, i64 offset,
//                  u64 checksum}
//   data:          each section at a 4096-byte aligned file offset
// Checksums: FNV-1a (64-bit offset basis and prime) over data taken as
// little-endian 64-bit words, a trailing partial word zero-padded.  The
// tables' checksum is one FNV-1a chain over the unit totals and then the
// section table.  A section's checksum (version 2) runs four FNV-1a chains
// from the offset basis, word j of the section going to chain j mod 4, and
// then folds the four chain values, in chain order, into one more FNV-1a
// chain from the basis: four independent multiply chains instead of one
// dependent one (a rank's 187 MB checksummed in 12 instead of 24 ms on the
// GB300 host's cores).  Version 1 files, whose sections have one chain like
// the tables, are still read and verified.
// The file is written to "<path>.tmp" and renamed into place, so a reader
// never sees a half-written checkpoint.
#include <cerrno>
#include <cstdio>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include "shardstep.h"

namespace shardstep {
int ckpt_fail(int code, const char* fmt, const char* a, long long b);
}

namespace {

constexpr char kMagic[8] = {'S', 'H', 'S', 'T', 'C', 'K', 'P', 'T'};
constexpr uint32_t kVersion = 2;       // written; versions 1 and 2 are read
constexpr int64_t kAlign = 4096;
constexpr uint64_t kFnvBasis = 14695981039346656037ull;
constexpr uint64_t kFnvPrime = 1099511628211ull;

struct Header {
    char magic[8];
    uint32_t version;
    uint32_t header_bytes;
    int32_t nd, rank, n_units, n_sections;
    int64_t step;
    uint64_t table_checksum;
    uint8_t zero[16];
};
static_assert(sizeof(Header) == 64, "header is 64 bytes");

struct SectionEntry {
    int32_t unit, kind;
    int64_t bytes, offset;
    uint64_t checksum;
};
static_assert(sizeof(SectionEntry) == 32, "section entry is 32 bytes");

uint64_t fnv_words(uint64_t h, const void* data, int64_t bytes) {
    const unsigned char* p = static_cast<const unsigned char*>(data);
    int64_t i = 0;
    for (; i + 8 <= bytes; i += 8) {
        uint64_t w;
        std::memcpy(&w, p + i, 8);
        h = (h ^ w) * kFnvPrime;
    }
    if (i < bytes) {
        uint64_t w = 0;
        std::memcpy(&w, p + i, static_cast<size_t>(bytes - i));
        h = (h ^ w) * kFnvPrime;
    }
    return h;
}

// A section's version-2 checksum, fed in pieces: every piece but the last
// holds whole 8-byte words.
struct LaneSum {
    uint64_t h[4] = {kFnvBasis, kFnvBasis, kFnvBasis, kFnvBasis};
    int64_t words = 0;  // words taken so far; the next goes to chain words % 4
    void word(uint64_t w) {
        uint64_t& x = h[words & 3];
        x = (x ^ w) * kFnvPrime;
        ++words;
    }
    void update(const void* data, int64_t bytes) {
        const unsigned char* p = static_cast<const unsigned char*>(data);
        int64_t i = 0;
        for (; i + 8 <= bytes && (words & 3) != 0; i += 8) {
            uint64_t w;
            std::memcpy(&w, p + i, 8);
            word(w);
        }
        uint64_t a = h[0], b = h[1], c = h[2], d = h[3];
        for (; i + 32 <= bytes; i += 32) {
            uint64_t w[4];
            std::memcpy(w, p + i, 32);
            a = (a ^ w[0]) * kFnvPrime;
            b = (b ^ w[1]) * kFnvPrime;
            c = (c ^ w[2]) * kFnvPrime;
            d = (d ^ w[3]) * kFnvPrime;
            words += 4;
        }
        h[0] = a;
        h[1] = b;
        h[2] = c;
        h[3] = d;
        for (; i + 8 <= bytes; i += 8) {
            uint64_t w;
            std::memcpy(&w, p + i, 8);
            word(w);
        }
        if (i < bytes) {
            uint64_t w = 0;
            std::memcpy(&w, p + i, static_cast<size_t>(bytes - i));
            word(w);
        }
    }
    uint64_t result() const {
        uint64_t c = kFnvBasis;
        for (uint64_t x : h) c = (c ^ x) * kFnvPrime;
        return c;
    }
};

uint64_t section_checksum(const void* data, int64_t bytes) {
    LaneSum s;
    s.update(data, bytes);
    return s.result();
}

int64_t align_up(int64_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct File {
    FILE* f = nullptr;
    ~File() {
        if (f) std::fclose(f);
    }
};

bool write_all(FILE* f, const void* p, int64_t n) {
    return n == 0 || std::fwrite(p, 1, static_cast<size_t>(n), f) == static_cast<size_t>(n);
}

bool read_at(FILE* f, int64_t off, void* p, int64_t n) {
    if (std::fseek(f, off, SEEK_SET) != 0) return false;
    return n == 0 || std::fread(p, 1, static_cast<size_t>(n), f) == static_cast<size_t>(n);
}

int load_tables(const char* path, File* file, Header* h, std::vector<int64_t>* totals,
                std::vector<SectionEntry>* sections) {
    if (path == nullptr) return shardstep::ckpt_fail(SHARDSTEP_ERR_INVALID, "path is NULL%s", "", 0);
    file->f = std::fopen(path, "rb");
    if (!file->f) return shardstep::ckpt_fail(SHARDSTEP_ERR_IO, "cannot open %s (errno %lld)", path, errno);
    if (!read_at(file->f, 0, h, sizeof(Header)) || std::memcmp(h->magic, kMagic, 8) != 0 ||
        (h->version != 1 && h->version != kVersion) || h->header_bytes != sizeof(Header) ||
        h->n_units < 0 ||
        h->n_sections < 0 || h->nd < 1 || h->rank < 0 || h->rank >= h->nd)
        return shardstep::ckpt_fail(SHARDSTEP_ERR_IO, "%s is not a rank checkpoint file", path, 0);
    totals->assign(h->n_units, 0);
    sections->assign(h->n_sections, SectionEntry{});
    if (!read_at(file->f, sizeof(Header), totals->data(), 8ll * h->n_units) ||
        !read_at(file->f, sizeof(Header) + 8ll * h->n_units, sections->data(),
                 static_cast<int64_t>(sizeof(SectionEntry)) * h->n_sections))
        return shardstep::ckpt_fail(SHARDSTEP_ERR_IO, "truncated tables in %s", path, 0);
    uint64_t c = fnv_words(kFnvBasis, totals->data(), 8ll * h->n_units);
    c = fnv_words(c, sections->data(), static_cast<int64_t>(sizeof(SectionEntry)) * h->n_sections);
    if (c != h->table_checksum)
        return shardstep::ckpt_fail(SHARDSTEP_ERR_IO, "table checksum mismatch in %s", path, 0);
    return SHARDSTEP_OK;
}

}  // namespace

extern "C" {

int shardstep_ckpt_save_rank(const char* path, int32_t nd, int32_t rank, int64_t step,
                             const int64_t* unit_totals, int32_t n_units,
                             const shardstep_ckpt_section_t* sections, int32_t n_sections) {
    if (path == nullptr) return shardstep::ckpt_fail(SHARDSTEP_ERR_INVALID, "path is NULL%s", "", 0);
    if (nd < 1 || rank < 0 || rank >= nd || n_units < 0 || n_sections < 0)
        return shardstep::ckpt_fail(SHARDSTEP_ERR_INVALID, "bad nd / rank / counts%s", "", 0);
    if ((n_units > 0 && unit_totals == nullptr) || (n_sections > 0 && sections == nullptr))
        return shardstep::ckpt_fail(SHARDSTEP_ERR_INVALID, "unit_totals / sections is NULL%s", "", 0);
    for (int32_t u = 0; u < n_units; ++u)
        if (unit_totals[u] < 0)
            return shardstep::ckpt_fail(SHARDSTEP_ERR_INVALID, "negative unit total%s", "", u);
    std::vector<SectionEntry> table(n_sections);
    const int64_t tables_end = static_cast<int64_t>(sizeof(Header)) + 8ll * n_units +
                               static_cast<int64_t>(sizeof(SectionEntry)) * n_sections;
    int64_t off = align_up(tables_end);
    for (int32_t s = 0; s < n_sections; ++s) {
        const shardstep_ckpt_section_t& sec = sections[s];
        if (sec.bytes < 0 || (sec.bytes > 0 && sec.data == nullptr) || sec.unit < 0 ||
            sec.unit >= n_units)
            return shardstep::ckpt_fail(SHARDSTEP_ERR_INVALID, "bad section%s", "", s);
        table[s] = SectionEntry{sec.unit, sec.kind, sec.bytes, off, 0};
        off = align_up(off + sec.bytes);
    }
    const std::string tmp = std::string(path) + ".tmp";
    {
        File f;
        f.f = std::fopen(tmp.c_str(), "wb");
        if (!f.f) return shardstep::ckpt_fail(SHARDSTEP_ERR_IO, "cannot create %s (errno %lld)", tmp.c_str(), errno);
        std::setvbuf(f.f, nullptr, _IOFBF, 1 << 22);
        // The sections' checksums are taken on a second thread while this one
        // writes the data behind a zeroed header and table, which are written
        // last (on the GB300 host: 12 ms of checksums under 30 ms of writing
        // per rank).  Without a thread, the checksums come first.
        auto checksum_all = [&table, sections, n_sections]() {
            for (int32_t s = 0; s < n_sections; ++s)
                table[s].checksum = section_checksum(sections[s].data, sections[s].bytes);
        };
        std::thread sums;
        try {
            sums = std::thread(checksum_all);
        } catch (...) {
            checksum_all();
        }
        static const char zeros[kAlign] = {0};
        bool ok = true;
        for (int64_t pos = 0; ok && pos < tables_end; pos += kAlign)
            ok = write_all(f.f, zeros, tables_end - pos < kAlign ? tables_end - pos : kAlign);
        int64_t pos = tables_end;
        for (int32_t s = 0; s < n_sections && ok; ++s) {
            ok = write_all(f.f, zeros, table[s].offset - pos) &&
                 write_all(f.f, sections[s].data, sections[s].bytes);
            pos = table[s].offset + sections[s].bytes;
        }
        if (sums.joinable()) sums.join();
        Header h{};
        std::memcpy(h.magic, kMagic, 8);
        h.version = kVersion;
        h.header_bytes = sizeof(Header);
        h.nd = nd;
        h.rank = rank;
        h.n_units = n_units;
        h.n_sections = n_sections;
        h.step = step;
        const uint64_t c = fnv_words(kFnvBasis, unit_totals, 8ll * n_units);
        h.table_checksum =
            fnv_words(c, table.data(), static_cast<int64_t>(sizeof(SectionEntry)) * n_sections);
        ok = ok && std::fseek(f.f, 0, SEEK_SET) == 0 && write_all(f.f, &h, sizeof h) &&
             write_all(f.f, unit_totals, 8ll * n_units) &&
             write_all(f.f, table.data(), static_cast<int64_t>(sizeof(SectionEntry)) * n_sections);
        ok = ok && std::fflush(f.f) == 0;
        if (!ok) {
            std::remove(tmp.c_str());
            return shardstep::ckpt_fail(SHARDSTEP_ERR_IO, "write to %s failed (errno %lld)", tmp.c_str(), errno);
        }
    }
    if (std::rename(tmp.c_str(), path) != 0)
        return shardstep::ckpt_fail(SHARDSTEP_ERR_IO, "cannot rename into %s (errno %lld)", path, errno);
    return SHARDSTEP_OK;
}

int shardstep_ckpt_info(const char* path, shardstep_ckpt_info_t* info, int64_t* unit_totals,
                        int32_t cap_units) {
    if (info == nullptr) return shardstep::ckpt_fail(SHARDSTEP_ERR_INVALID, "info is NULL%s", "", 0);
    File f;
    Header h;
    std::vector<int64_t> totals;
    std::vector<SectionEntry> secs;
    int rc = load_tables(path, &f, &h, &totals, &secs);
    if (rc != SHARDSTEP_OK) return rc;
    info->nd = h.nd;
    info->rank = h.rank;
    info->n_units = h.n_units;
    info->n_sections = h.n_sections;
    info->step = h.step;
    if (unit_totals != nullptr)
        for (int32_t u = 0; u < h.n_units && u < cap_units; ++u) unit_totals[u] = totals[u];
    return SHARDSTEP_OK;
}

int shardstep_ckpt_read(const char* path, int32_t unit, int32_t kind, int64_t byte_offset,
                        int64_t bytes, void* dst) {
    File f;
    Header h;
    std::vector<int64_t> totals;
    std::vector<SectionEntry> secs;
    int rc = load_tables(path, &f, &h, &totals, &secs);
    if (rc != SHARDSTEP_OK) return rc;
    for (const SectionEntry& s : secs) {
        if (s.unit != unit || s.kind != kind) continue;
        if (byte_offset < 0 || bytes < 0 || byte_offset + bytes > s.bytes || (bytes > 0 && !dst))
            return shardstep::ckpt_fail(SHARDSTEP_ERR_INVALID, "range outside section in %s", path, 0);
        if (!read_at(f.f, s.offset + byte_offset, dst, bytes))
            return shardstep::ckpt_fail(SHARDSTEP_ERR_IO, "short read from %s", path, 0);
        return SHARDSTEP_OK;
    }
    return shardstep::ckpt_fail(SHARDSTEP_ERR_INVALID, "no section of that unit and kind in %s", path, 0);
}

int shardstep_ckpt_verify(const char* path) {
    File f;
    Header h;
    std::vector<int64_t> totals;
    std::vector<SectionEntry> secs;
    int rc = load_tables(path, &f, &h, &totals, &secs);
    if (rc != SHARDSTEP_OK) return rc;
    std::vector<unsigned char> buf(1 << 22);
    for (const SectionEntry& s : secs) {
        uint64_t c = kFnvBasis;  // version 1: one chain
        LaneSum lanes;            // version 2
        if (std::fseek(f.f, s.offset, SEEK_SET) != 0)
            return shardstep::ckpt_fail(SHARDSTEP_ERR_IO, "seek failed in %s", path, 0);
        for (int64_t done = 0; done < s.bytes;) {
            const int64_t n = s.bytes - done < static_cast<int64_t>(buf.size())
                                  ? s.bytes - done
                                  : static_cast<int64_t>(buf.size());
            if (std::fread(buf.data(), 1, static_cast<size_t>(n), f.f) != static_cast<size_t>(n))
                return shardstep::ckpt_fail(SHARDSTEP_ERR_IO, "short read from %s", path, 0);
            // every chunk but the last is whole 8-byte words
            if (h.version == 1) c = fnv_words(c, buf.data(), n);
            else lanes.update(buf.data(), n);
            done += n;
        }
        if ((h.version == 1 ? c : lanes.result()) != s.checksum)
            return shardstep::ckpt_fail(SHARDSTEP_ERR_IO, "data checksum mismatch in %s", path, 0);
    }
    return SHARDSTEP_OK;
}

int fsdp_reshard_plan(int64_t total, int32_t old_nd, int32_t new_nd, int32_t new_rank,
                      shardstep_ckpt_piece_t* pieces, int32_t cap, int32_t* n_pieces) {
    if (total < 0 || old_nd < 1 || new_nd < 1 || new_rank < 0 || new_rank >= new_nd ||
        n_pieces == nullptr || (cap > 0 && pieces == nullptr))
        return shardstep::ckpt_fail(SHARDSTEP_ERR_INVALID, "bad reshard plan arguments%s", "", 0);
    const int64_t s_old = (total + old_nd - 1) / old_nd;
    const int64_t s_new = (total + new_nd - 1) / new_nd;
    int64_t g = static_cast<int64_t>(new_rank) * s_new;
    const int64_t end = g + s_new < total ? g + s_new : total;
    int32_t n = 0;
    while (g < end) {
        const int64_t q = g / s_old, off = g - q * s_old;
        const int64_t take = (s_old - off) < (end - g) ? (s_old - off) : (end - g);
        if (n < cap)
            pieces[n] = shardstep_ckpt_piece_t{static_cast<int32_t>(q), 0, off,
                                               g - static_cast<int64_t>(new_rank) * s_new, take};
        ++n;
        g += take;
    }
    *n_pieces = n;
    if (n > cap)
        return shardstep::ckpt_fail(SHARDSTEP_ERR_CAPACITY, "plan needs %s%lld pieces", "", n);
    return SHARDSTEP_OK;
}

}  // extern "C"
