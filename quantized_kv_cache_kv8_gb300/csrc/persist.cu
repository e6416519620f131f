// persist.cu -- versioned files of quantized row pools (host code only).
//
// The KV cache quantization pages keep the cache on disk across restarts and
// across mode changes ([P1] "KV persistence across mode changes"; [P2] "What's
// in it", .coli_kv bullet; [P1] Commits item 1, disk format v2):
//   - the file magic names the tier: COLIKV (v1, f32 rows), COLIKV2 (v2, KV8
//     codes), COLIKV3 (v3, TQ codes);
//   - header word h[7] carries the TQ codec and bit width as codec << 8 | bits;
//   - a file of another tier, codec or bit width is refused with an explicit
//     message and never misread; so is a container whose byte counts do not add
//     up;
//   - a v1 (f32) file can be read under a quantized mode (quantize on load) and
//     stays untouched until the first save rewrites it;
//   - appends heal a torn tail (bytes written after the last header update).
//
// Layout (little-endian, the byte order of every host this library builds on):
//   magic   8 bytes: "COLIKV\0\0" | "COLIKV2\0" | "COLIKV3\0"
//   h[0..7] 8 x int64: rows, row dimension D, number of scale blocks, block
//           dims (2), v_dim, TQ sign seed (0 for KV8 and f32), codec << 8 | bits
//           (TQ: codec 1 = rotated-int4 at 4 bits, codec 0 = PolarQuant at
//           2..6 bits; 0 for KV8 and f32)
//   payload one record per row -- v1: D f32; v2/v3: the row's codes then its
//           n_blocks f32 scales (584 bytes for a KV8 row of 512 + 64 dims, 296
//           for TQ4, 72 b + 8 for PolarQuant at b bits), so rows append in
//           place.  A v3 record's code bytes follow from h[7]: D b / 8 for
//           codec 1, the sum over blocks of ceil(n b / 8) for codec 0.
#include "kvq_internal.cuh"

#include <stdint.h>

#include <stdio.h>
#include <string.h>
#include <unistd.h>

#include <string>
#include <vector>

namespace {

constexpr int kHeaderWords = 8;
constexpr int64_t kHeaderBytes = 8 + kHeaderWords * 8;
constexpr int32_t kTq4Codec = 1, kTq4Bits = 4, kPolarCodec = 0;

// The tier (file version) and the TQ codec word of a format.
struct Mode {
    int version;
    int64_t codec_bits;   // h[7]
};

bool is_pq_format(kvq_format f) { return f >= KVQ_PQ2 && f <= KVQ_PQ6; }
bool format_ok(kvq_format f) { return f == KVQ_KV8 || f == KVQ_TQ4 || is_pq_format(f); }

Mode mode_of(kvq_format fmt) {
    if (fmt == KVQ_KV8) return {2, 0};
    if (fmt == KVQ_TQ4) return {3, (int64_t)kTq4Codec << 8 | kTq4Bits};
    return {3, (int64_t)kPolarCodec << 8 | ((int)fmt - 10)};
}

const char* magic_of(int version) {
    switch (version) {
        case 1: return "COLIKV\0\0";
        case 2: return "COLIKV2\0";
        default: return "COLIKV3\0";
    }
}

int version_of_magic(const char m[8]) {
    for (int v = 1; v <= 3; ++v)
        if (memcmp(m, magic_of(v), 8) == 0) return v;
    return 0;
}

const char* tier_name(int version) {
    return version == 1 ? "f32" : version == 2 ? "fp8 (KV8)" : "KV_TQ";
}

int64_t row_dim(const kvq_mla_layout& L) { return L.block_dim[0] + (L.n_blocks > 1 ? L.block_dim[1] : 0); }

// code bytes of one row of a TQ codec word (codec << 8 | bits)
int64_t tq_code_bytes(int64_t codec_bits, int64_t d0, int64_t d1) {
    const int64_t codec = codec_bits >> 8, bits = codec_bits & 255;
    if (codec == kPolarCodec) return (d0 * bits + 7) / 8 + (d1 * bits + 7) / 8;
    return (d0 + d1) * bits / 8;
}

int64_t row_bytes(kvq_format fmt, const kvq_mla_layout& L) {
    if (fmt == KVQ_KV8) return row_dim(L);
    return tq_code_bytes(mode_of(fmt).codec_bits, L.block_dim[0], L.n_blocks > 1 ? L.block_dim[1] : 0);
}

void put_msg(char* msg, size_t len, const std::string& s) {
    if (msg && len > 0) snprintf(msg, len, "%s", s.c_str());
}

bool layout_ok(const kvq_mla_layout* L) {
    if (!L || (L->n_blocks != 1 && L->n_blocks != 2)) return false;
    for (int b = 0; b < L->n_blocks; ++b)
        if (L->block_dim[b] <= 0) return false;
    return L->v_dim > 0 && L->v_dim <= row_dim(*L);
}

struct Header {
    int version;
    int64_t h[kHeaderWords];
};

void fill_header(Header* H, Mode m, const kvq_mla_layout& L, int64_t rows) {
    const int version = m.version;
    H->version = version;
    H->h[0] = rows;
    H->h[1] = row_dim(L);
    H->h[2] = L.n_blocks;
    H->h[3] = L.block_dim[0];
    H->h[4] = L.n_blocks > 1 ? L.block_dim[1] : 0;
    H->h[5] = L.v_dim;
    H->h[6] = version == 3 ? (int64_t)L.seed : 0;
    H->h[7] = version == 3 ? m.codec_bits : 0;
}

int64_t payload_row_bytes(const Header& H) {
    if (H.version == 1) return H.h[1] * 4;
    const int64_t codes = H.version == 2 ? H.h[1] : tq_code_bytes(H.h[7], H.h[3], H.h[4]);
    return codes + H.h[2] * 4;
}

bool write_header(FILE* f, const Header& H) {
    return fwrite(magic_of(H.version), 1, 8, f) == 8 && fwrite(H.h, 8, kHeaderWords, f) == (size_t)kHeaderWords;
}

// Reads and checks a header (known magic, consistent words) and returns the
// file's size; the callers compare it with the size h[0] rows need.
kvq_status read_header(FILE* f, Header* H, int64_t* file_bytes, char* msg, size_t msg_len) {
    char m[8];
    if (fread(m, 1, 8, f) != 8 || fread(H->h, 8, kHeaderWords, f) != (size_t)kHeaderWords) {
        put_msg(msg, msg_len, "not a quantized cache file (short header)");
        return KVQ_ERR_IO;
    }
    H->version = version_of_magic(m);
    if (H->version == 0) {
        put_msg(msg, msg_len, "not a quantized cache file (unknown magic)");
        return KVQ_ERR_IO;
    }
    const int64_t* h = H->h;
    if (h[0] < 0 || h[1] <= 0 || (h[2] != 1 && h[2] != 2) || h[3] <= 0 || h[4] < 0 || h[3] + h[4] != h[1] ||
        (h[2] == 2) != (h[4] > 0) || h[5] <= 0 || h[5] > h[1] ||
        (H->version == 3 && ((h[7] & 255) < 1 || (h[7] & 255) > 16 || (h[7] >> 8) < 0 || (h[7] >> 8) > 255))) {
        put_msg(msg, msg_len, "corrupt quantized cache header");
        return KVQ_ERR_IO;
    }
    // sizes computed from the header stay inside int64: a row dimension of at
    // most 2^20 and no more rows than the largest file could hold
    if (h[1] > (int64_t(1) << 20) || h[0] > (INT64_MAX - kHeaderBytes) / payload_row_bytes(*H)) {
        put_msg(msg, msg_len, "corrupt quantized cache header (sizes out of range)");
        return KVQ_ERR_IO;
    }
    if (fseek(f, 0, SEEK_END) != 0) return KVQ_ERR_IO;
    *file_bytes = ftell(f);
    return KVQ_OK;
}

kvq_status open_checked(const char* path, FILE** f, Header* H, int64_t* file_bytes, char* msg, size_t msg_len) {
    *f = fopen(path, "rb");
    if (!*f) {
        put_msg(msg, msg_len, std::string("cannot open ") + path);
        return KVQ_ERR_IO;
    }
    const kvq_status s = read_header(*f, H, file_bytes, msg, msg_len);
    if (s != KVQ_OK) {
        fclose(*f);
        *f = nullptr;
    }
    return s;
}

// The stored tier, codec and layout against the caller's; explains a refusal.
kvq_status check_mode(const Header& H, Mode want_mode, const kvq_mla_layout& L, char* msg, size_t msg_len) {
    const int want_version = want_mode.version;
    if (H.version != want_version) {
        put_msg(msg, msg_len, std::string("file is ") + tier_name(H.version) + ", current mode is " +
                                  tier_name(want_version) + ": refused");
        return KVQ_ERR_MISMATCH;
    }
    Header want;
    fill_header(&want, want_mode, L, 0);
    if (want_version == 3 && H.h[7] != want.h[7]) {
        char b[160];
        snprintf(b, sizeof b, "file is KV_TQ (codec %lld, %lld-bit), current is KV_TQ (codec %lld, %lld-bit): refused",
                 (long long)(H.h[7] >> 8), (long long)(H.h[7] & 255), (long long)(want.h[7] >> 8),
                 (long long)(want.h[7] & 255));
        put_msg(msg, msg_len, b);
        return KVQ_ERR_MISMATCH;
    }
    if (want_version == 3 && H.h[6] != want.h[6]) {
        put_msg(msg, msg_len, "file is KV_TQ with another rotation seed: refused");
        return KVQ_ERR_MISMATCH;
    }
    for (int i = 1; i <= 5; ++i)
        if (H.h[i] != want.h[i]) {
            put_msg(msg, msg_len, "file holds rows of another layout (block dims or v_dim): refused");
            return KVQ_ERR_MISMATCH;
        }
    return KVQ_OK;
}

// Writes header + records beside the target and renames it over the target,
// so a reader never sees a half-written file.
kvq_status write_file(const char* path, const Header& H, int64_t n, int64_t code_bytes, int64_t scale_bytes,
                      const void* codes, const void* scales) {
    const std::string tmp = std::string(path) + ".tmp";
    FILE* f = fopen(tmp.c_str(), "wb");
    if (!f) return KVQ_ERR_IO;
    bool ok = write_header(f, H);
    for (int64_t r = 0; ok && r < n; ++r) {
        if (code_bytes > 0)
            ok = fwrite(static_cast<const char*>(codes) + r * code_bytes, 1, (size_t)code_bytes, f) == (size_t)code_bytes;
        if (ok && scale_bytes > 0)
            ok = fwrite(static_cast<const char*>(scales) + r * scale_bytes, 1, (size_t)scale_bytes, f) ==
                 (size_t)scale_bytes;
    }
    ok = (fclose(f) == 0) && ok;
    if (!ok || rename(tmp.c_str(), path) != 0) {
        remove(tmp.c_str());
        return KVQ_ERR_IO;
    }
    return KVQ_OK;
}

// Reads n records into the two arrays (code_bytes and scale_bytes per row).
bool read_records(FILE* f, int64_t n, int64_t code_bytes, int64_t scale_bytes, void* codes, void* scales) {
    if (fseek(f, kHeaderBytes, SEEK_SET) != 0) return false;
    std::vector<char> rec((size_t)(code_bytes + scale_bytes));
    for (int64_t r = 0; r < n; ++r) {
        if (fread(rec.data(), 1, rec.size(), f) != rec.size()) return false;
        if (code_bytes > 0) memcpy(static_cast<char*>(codes) + r * code_bytes, rec.data(), (size_t)code_bytes);
        if (scale_bytes > 0)
            memcpy(static_cast<char*>(scales) + r * scale_bytes, rec.data() + code_bytes, (size_t)scale_bytes);
    }
    return true;
}

}  // namespace

extern "C" {

kvq_status kvq_cache_save(const char* path, kvq_format fmt, const kvq_mla_layout* layout, int64_t n_rows,
                          const uint8_t* codes, const float* scales) {
    if (!path || !layout_ok(layout) || !format_ok(fmt) || n_rows < 0) return KVQ_ERR_ARG;
    if (n_rows > 0 && (!codes || !scales)) return KVQ_ERR_ARG;
    Header H;
    fill_header(&H, mode_of(fmt), *layout, n_rows);
    return write_file(path, H, n_rows, row_bytes(fmt, *layout), layout->n_blocks * 4, codes, scales);
}

kvq_status kvq_cache_save_f32(const char* path, const kvq_mla_layout* layout, int64_t n_rows, const float* rows) {
    if (!path || !layout_ok(layout) || n_rows < 0 || (n_rows > 0 && !rows)) return KVQ_ERR_ARG;
    Header H;
    fill_header(&H, Mode{1, 0}, *layout, n_rows);
    return write_file(path, H, n_rows, row_dim(*layout) * 4, 0, rows, nullptr);
}

kvq_status kvq_cache_info(const char* path, int32_t* version, int64_t* n_rows, int64_t* header_words, char* msg,
                          size_t msg_len) {
    if (!path) return KVQ_ERR_ARG;
    FILE* f;
    Header H;
    int64_t bytes = 0;
    kvq_status s = open_checked(path, &f, &H, &bytes, msg, msg_len);
    if (s != KVQ_OK) return s;
    fclose(f);
    if (version) *version = H.version;
    if (n_rows) *n_rows = H.h[0];
    if (header_words) memcpy(header_words, H.h, sizeof H.h);
    return KVQ_OK;
}

// Shared by the two loaders: open, check the mode, check the byte count.
static kvq_status open_for_load(const char* path, Mode mode, const kvq_mla_layout& L, int64_t capacity, FILE** f,
                                Header* H, char* msg, size_t msg_len) {
    int64_t bytes = 0;
    kvq_status s = open_checked(path, f, H, &bytes, msg, msg_len);
    if (s != KVQ_OK) return s;
    if ((s = check_mode(*H, mode, L, msg, msg_len)) != KVQ_OK) {
        fclose(*f);
        return s;
    }
    if (bytes != kHeaderBytes + H->h[0] * payload_row_bytes(*H)) {
        fclose(*f);
        put_msg(msg, msg_len, "byte count does not match the header: refused");
        return KVQ_ERR_IO;
    }
    if (H->h[0] > capacity) {
        fclose(*f);
        put_msg(msg, msg_len, "file holds more rows than the buffers");
        return KVQ_ERR_WORKSPACE;
    }
    return KVQ_OK;
}

kvq_status kvq_cache_load(const char* path, kvq_format fmt, const kvq_mla_layout* layout, int64_t capacity,
                          uint8_t* codes, float* scales, int64_t* n_rows, char* msg, size_t msg_len) {
    if (!path || !layout_ok(layout) || !format_ok(fmt) || capacity < 0 || !n_rows)
        return KVQ_ERR_ARG;
    FILE* f;
    Header H;
    kvq_status s = open_for_load(path, mode_of(fmt), *layout, capacity, &f, &H, msg, msg_len);
    if (s != KVQ_OK) return s;
    const int64_t n = H.h[0];
    const bool ok = (n == 0 || (codes && scales)) &&
                    read_records(f, n, row_bytes(fmt, *layout), layout->n_blocks * 4, codes, scales);
    fclose(f);
    if (!ok) return KVQ_ERR_IO;
    *n_rows = n;
    return KVQ_OK;
}

kvq_status kvq_cache_load_f32(const char* path, const kvq_mla_layout* layout, int64_t capacity, float* rows,
                              int64_t* n_rows, char* msg, size_t msg_len) {
    if (!path || !layout_ok(layout) || capacity < 0 || !n_rows) return KVQ_ERR_ARG;
    FILE* f;
    Header H;
    kvq_status s = open_for_load(path, Mode{1, 0}, *layout, capacity, &f, &H, msg, msg_len);
    if (s != KVQ_OK) return s;
    const int64_t n = H.h[0];
    const bool ok = (n == 0 || rows) && read_records(f, n, row_dim(*layout) * 4, 0, rows, nullptr);
    fclose(f);
    if (!ok) return KVQ_ERR_IO;
    *n_rows = n;
    return KVQ_OK;
}

kvq_status kvq_cache_append(const char* path, kvq_format fmt, const kvq_mla_layout* layout, int64_t n_new,
                            const uint8_t* codes, const float* scales, int64_t* n_rows, char* msg, size_t msg_len) {
    if (!path || !layout_ok(layout) || !format_ok(fmt) || n_new < 0) return KVQ_ERR_ARG;
    if (n_new > 0 && (!codes || !scales)) return KVQ_ERR_ARG;
    FILE* f;
    Header H;
    int64_t bytes = 0;
    kvq_status s = open_checked(path, &f, &H, &bytes, msg, msg_len);
    if (s != KVQ_OK) return s;
    fclose(f);
    if ((s = check_mode(H, mode_of(fmt), *layout, msg, msg_len)) != KVQ_OK) return s;
    const int64_t rec = payload_row_bytes(H), committed = kHeaderBytes + H.h[0] * rec;
    if (bytes < committed) {
        put_msg(msg, msg_len, "file is shorter than its header says: refused");
        return KVQ_ERR_IO;
    }
    f = fopen(path, "r+b");
    if (!f) return KVQ_ERR_IO;
    bool ok = true;
    if (bytes > committed) {
        // self-heal: the bytes past the header's row count are an append that
        // was interrupted before its header update; they are dropped
        ok = fflush(f) == 0 && ftruncate(fileno(f), (off_t)committed) == 0;
        put_msg(msg, msg_len, "dropped the tail of an interrupted append");
    }
    ok = ok && fseek(f, committed, SEEK_SET) == 0;
    const int64_t cb = row_bytes(fmt, *layout), sb = layout->n_blocks * 4;
    for (int64_t r = 0; ok && r < n_new; ++r)
        ok = fwrite(codes + r * cb, 1, (size_t)cb, f) == (size_t)cb &&
             fwrite(reinterpret_cast<const char*>(scales) + r * sb, 1, (size_t)sb, f) == (size_t)sb;
    // the records reach the file before the header counts them
    ok = ok && fflush(f) == 0;
    const int64_t total = H.h[0] + n_new;
    ok = ok && fseek(f, 8, SEEK_SET) == 0 && fwrite(&total, 8, 1, f) == 1;
    ok = (fclose(f) == 0) && ok;
    if (!ok) return KVQ_ERR_IO;
    if (n_rows) *n_rows = total;
    return KVQ_OK;
}

}  // extern "C"
