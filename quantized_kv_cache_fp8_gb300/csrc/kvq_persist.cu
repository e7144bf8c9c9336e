// kvq_persist.cu — cache files: save, append (self-healing), probe, and load with
// refuse-on-mismatch and quantize-on-load of fp32 files.  colibri PR #399, Commit 1
// (".coli_kv v2 ... quantize-on-upgrade from v1, reject-on-mismatch, self-heal"),
// Commit 6 (the magic encodes the tier; a header word carries codec << 8 | bits) and
// the review thread (a cache written under one mode must be refused under another;
// containers whose byte counts do not add up are refused).  The byte layout is stated
// in kvq.h.  Host code only: planes move through host buffers with cudaMemcpy, in
// chunks of kChunkRows records.
#include <unistd.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <vector>

#include "kvq_internal.cuh"

namespace {

constexpr uint32_t kMagicF32 = 0x3151564Bu;   // "KVQ1"
constexpr uint32_t kMagicFp8 = 0x3251564Bu;   // "KVQ2"
constexpr uint32_t kMagicRot = 0x3351564Bu;   // "KVQ3"
constexpr uint32_t kVersion = 1;
constexpr int kHeaderWords = 16;
constexpr int64_t kChunkRows = 4096;
constexpr int kFmtF32 = 0;

bool quantized(int fmt) { return fmt == KVQ_FMT_FP8 || kvq::rotated_format(fmt); }

int64_t lat_bytes(int fmt)
{
    return fmt == kFmtF32 ? kvq::kDLat * 4 : fmt == KVQ_FMT_FP8 ? kvq::kDLat : kvq::kDLat * kvq::rotated_bits(fmt) / 8;
}

int64_t record_bytes(int fmt)
{
    return fmt == kFmtF32 ? (int64_t)(kvq::kDLat + kvq::kDRope) * 4 : lat_bytes(fmt) + 4 + kvq::kDRope + 4;
}

uint32_t magic_of(int fmt) { return fmt == kFmtF32 ? kMagicF32 : fmt == KVQ_FMT_FP8 ? kMagicFp8 : kMagicRot; }

uint32_t codec_bits(int fmt)
{
    return fmt == kFmtF32 ? 32u : fmt == KVQ_FMT_FP8 ? 8u : (1u << 8) | (uint32_t)kvq::rotated_bits(fmt);
}

int64_t data_offset(int fmt) { return 4 * kHeaderWords + (kvq::rotated_format(fmt) ? 64 : 0); }

struct File {
    FILE* f = nullptr;
    explicit File(const char* path, const char* mode) : f(std::fopen(path, mode)) {}
    ~File() { if (f) std::fclose(f); }
};

int io_fail(const char* entry, const char* path, const char* what)
{
    return kvq::set_last_error(KVQ_EIO, "%s: %s: %s", entry, path, what);
}

void fill_header(uint32_t (&w)[kHeaderWords], int fmt, int64_t n_rows)
{
    std::memset(w, 0, sizeof w);
    w[0] = magic_of(fmt);
    w[1] = kVersion;
    w[2] = kvq::kDLat;
    w[3] = kvq::kDRope;
    w[4] = (uint32_t)(uint64_t)n_rows;
    w[5] = (uint32_t)((uint64_t)n_rows >> 32);
    w[6] = (uint32_t)fmt;
    w[7] = codec_bits(fmt);
    w[8] = (uint32_t)record_bytes(fmt);
}

// read and check the header of an open file; fills info and the rotation signs
int read_header(FILE* f, const char* entry, const char* path, kvq_cache_info& info, uint32_t (&signs)[16])
{
    uint32_t w[kHeaderWords];
    if (std::fseek(f, 0, SEEK_END) != 0) return io_fail(entry, path, "cannot seek");
    const long long size = std::ftell(f);
    std::rewind(f);
    if (size < 4 * kHeaderWords || std::fread(w, 4, kHeaderWords, f) != (size_t)kHeaderWords)
        return io_fail(entry, path, "shorter than a header");
    const int fmt = (int)w[6];
    const bool known = fmt == kFmtF32 || quantized(fmt);
    if (!known || w[0] != magic_of(fmt) || w[1] != kVersion || w[2] != (uint32_t)kvq::kDLat ||
        w[3] != (uint32_t)kvq::kDRope || w[7] != codec_bits(fmt) || w[8] != (uint32_t)record_bytes(fmt))
        return io_fail(entry, path, "not a cache file of this layout");
    for (int i = 9; i < kHeaderWords; ++i)
        if (w[i] != 0) return io_fail(entry, path, "reserved header words are not zero");
    std::memset(signs, 0, sizeof signs);
    if (kvq::rotated_format(fmt) && std::fread(signs, 4, 16, f) != 16)
        return io_fail(entry, path, "rotation signs missing");
    info.format = fmt;
    info.codec = (int32_t)(w[7] >> 8);
    info.bits = (int32_t)(w[7] & 0xFF);
    info.d_lat = (int32_t)w[2];
    info.d_rope = (int32_t)w[3];
    info.n_rows = (int64_t)((uint64_t)w[4] | ((uint64_t)w[5] << 32));
    info.record_bytes = record_bytes(fmt);
    const long long need = data_offset(fmt) + info.n_rows * info.record_bytes;
    if (info.n_rows < 0 || size < need) return io_fail(entry, path, "fewer bytes than the header counts");
    info.trailing_bytes = size - need;
    return KVQ_OK;
}

bool planes_ok(const kvq_mla_cache* p)
{
    return p && p->lat && p->lat_scale && p->rope && p->rope_scale;
}

int cuda_fail(const char* entry, cudaError_t e)
{
    return kvq::set_last_error(KVQ_ECUDA, "%s: %s", entry, cudaGetErrorString(e));
}

// rows [r0, r0 + n) of the device planes as records in `rec`
cudaError_t planes_to_records(int fmt, const kvq_mla_cache& p, int64_t r0, int64_t n,
                              std::vector<uint8_t>& rec, std::vector<uint8_t>& tmp)
{
    const int64_t lb = lat_bytes(fmt), rb = record_bytes(fmt);
    tmp.resize((size_t)(n * (lb + 4 + kvq::kDRope + 4)));
    uint8_t* lat = tmp.data();
    uint8_t* ls = lat + n * lb;
    uint8_t* rope = ls + n * 4;
    uint8_t* rs = rope + n * kvq::kDRope;
    cudaError_t e = cudaMemcpy(lat, p.lat + r0 * lb, (size_t)(n * lb), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(ls, p.lat_scale + r0, (size_t)(n * 4), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(rope, p.rope + r0 * kvq::kDRope, (size_t)(n * kvq::kDRope), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(rs, p.rope_scale + r0, (size_t)(n * 4), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    rec.resize((size_t)(n * rb));
    for (int64_t i = 0; i < n; ++i) {
        uint8_t* d = rec.data() + i * rb;
        std::memcpy(d, lat + i * lb, (size_t)lb);
        std::memcpy(d + lb, ls + i * 4, 4);
        std::memcpy(d + lb + 4, rope + i * kvq::kDRope, kvq::kDRope);
        std::memcpy(d + lb + 4 + kvq::kDRope, rs + i * 4, 4);
    }
    return cudaSuccess;
}

int write_records(FILE* f, const char* entry, const char* path, int fmt, const kvq_mla_cache& p,
                  int64_t r0, int64_t rows)
{
    std::vector<uint8_t> rec, tmp;
    for (int64_t c = 0; c < rows; c += kChunkRows) {
        const int64_t n = std::min(kChunkRows, rows - c);
        const cudaError_t e = planes_to_records(fmt, p, r0 + c, n, rec, tmp);
        if (e != cudaSuccess) return cuda_fail(entry, e);
        if (std::fwrite(rec.data(), 1, rec.size(), f) != rec.size()) return io_fail(entry, path, "write failed");
    }
    return KVQ_OK;
}

}  // namespace

extern "C" {

int kvq_cache_probe(const char* path, kvq_cache_info* info)
{
    const char* E = "kvq_cache_probe";
    if (!path || !info) return kvq::set_last_error(KVQ_EINVAL, "%s: NULL argument", E);
    File f(path, "rb");
    if (!f.f) return io_fail(E, path, "cannot open");
    uint32_t signs[16];
    return read_header(f.f, E, path, *info, signs);
}

int kvq_cache_save(const char* path, int32_t format, const kvq_mla_cache* planes,
                   const uint32_t* signs, int64_t rows, kvq_stream_t stream)
{
    const char* E = "kvq_cache_save";
    if (!path || !planes_ok(planes)) return kvq::set_last_error(KVQ_EINVAL, "%s: NULL argument", E);
    if (!quantized(format)) return kvq::set_last_error(KVQ_EFORMAT, "%s: format %d is not a quantized tier", E, format);
    if (rows < 0 || rows > planes->n_rows) return kvq::set_last_error(KVQ_EINVAL, "%s: rows outside the planes", E);
    if (kvq::rotated_format(format) && !signs) return kvq::set_last_error(KVQ_EINVAL, "%s: rotation signs missing", E);
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(E, e);
    uint32_t hs[16] = {};
    if (kvq::rotated_format(format) && (e = cudaMemcpy(hs, signs, 64, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(E, e);
    File f(path, "wb");
    if (!f.f) return io_fail(E, path, "cannot open for writing");
    uint32_t w[kHeaderWords];
    fill_header(w, format, rows);
    if (std::fwrite(w, 4, kHeaderWords, f.f) != (size_t)kHeaderWords) return io_fail(E, path, "write failed");
    if (kvq::rotated_format(format) && std::fwrite(hs, 4, 16, f.f) != 16) return io_fail(E, path, "write failed");
    return write_records(f.f, E, path, format, *planes, 0, rows);
}

int kvq_cache_save_f32(const char* path, const float* lat, const float* rope, int64_t rows,
                       kvq_stream_t stream)
{
    const char* E = "kvq_cache_save_f32";
    if (!path || (rows > 0 && (!lat || !rope))) return kvq::set_last_error(KVQ_EINVAL, "%s: NULL argument", E);
    if (rows < 0) return kvq::set_last_error(KVQ_EINVAL, "%s: rows < 0", E);
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(E, e);
    File f(path, "wb");
    if (!f.f) return io_fail(E, path, "cannot open for writing");
    uint32_t w[kHeaderWords];
    fill_header(w, kFmtF32, rows);
    if (std::fwrite(w, 4, kHeaderWords, f.f) != (size_t)kHeaderWords) return io_fail(E, path, "write failed");
    std::vector<float> hl, hr, rec;
    for (int64_t c = 0; c < rows; c += kChunkRows) {
        const int64_t n = std::min(kChunkRows, rows - c);
        hl.resize((size_t)(n * kvq::kDLat));
        hr.resize((size_t)(n * kvq::kDRope));
        e = cudaMemcpy(hl.data(), lat + c * kvq::kDLat, hl.size() * 4, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(hr.data(), rope + c * kvq::kDRope, hr.size() * 4, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(E, e);
        rec.resize((size_t)(n * (kvq::kDLat + kvq::kDRope)));
        for (int64_t i = 0; i < n; ++i) {
            std::memcpy(&rec[i * (kvq::kDLat + kvq::kDRope)], &hl[i * kvq::kDLat], kvq::kDLat * 4);
            std::memcpy(&rec[i * (kvq::kDLat + kvq::kDRope) + kvq::kDLat], &hr[i * kvq::kDRope], kvq::kDRope * 4);
        }
        if (std::fwrite(rec.data(), 4, rec.size(), f.f) != rec.size()) return io_fail(E, path, "write failed");
    }
    return KVQ_OK;
}

int kvq_cache_append(const char* path, int32_t format, const kvq_mla_cache* planes, int64_t row0,
                     int64_t rows, kvq_stream_t stream)
{
    const char* E = "kvq_cache_append";
    if (!path || !planes_ok(planes)) return kvq::set_last_error(KVQ_EINVAL, "%s: NULL argument", E);
    if (row0 < 0 || rows < 0 || row0 + rows > planes->n_rows)
        return kvq::set_last_error(KVQ_EINVAL, "%s: rows outside the planes", E);
    kvq_cache_info info;
    uint32_t signs[16];
    long long keep = 0;
    {
        File f(path, "rb");
        if (!f.f) return io_fail(E, path, "cannot open");
        if (int st = read_header(f.f, E, path, info, signs)) return st;
        if (info.format != format)
            return kvq::set_last_error(KVQ_EMISMATCH, "%s: %s holds format %d, not %d", E, path, info.format, format);
        keep = data_offset(format) + info.n_rows * info.record_bytes;
    }
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(E, e);
    File f(path, "r+b");
    if (!f.f) return io_fail(E, path, "cannot open for writing");
    // self-heal: cut what an interrupted append left after the last complete record,
    // write the new records there, and only then the header's count
    if (info.trailing_bytes > 0 && ftruncate(fileno(f.f), (off_t)keep) != 0)
        return io_fail(E, path, "cannot cut the partial tail");
    if (std::fseek(f.f, (long)keep, SEEK_SET) != 0) return io_fail(E, path, "cannot seek");
    if (int st = write_records(f.f, E, path, format, *planes, row0, rows)) return st;
    if (std::fflush(f.f) != 0) return io_fail(E, path, "write failed");
    uint32_t w[kHeaderWords];
    fill_header(w, format, info.n_rows + rows);
    if (std::fseek(f.f, 0, SEEK_SET) != 0 || std::fwrite(w, 4, kHeaderWords, f.f) != (size_t)kHeaderWords)
        return io_fail(E, path, "header update failed");
    return KVQ_OK;
}

size_t kvq_cache_load_workspace(void)
{
    return (size_t)kChunkRows * (kvq::kDLat + kvq::kDRope) * sizeof(float);
}

int kvq_cache_load(const char* path, int32_t format, const uint32_t* signs,
                   const kvq_mla_cache* planes, int64_t capacity, int64_t* n_loaded,
                   void* workspace, size_t ws_bytes, kvq_stream_t stream)
{
    const char* E = "kvq_cache_load";
    if (!path || !planes_ok(planes)) return kvq::set_last_error(KVQ_EINVAL, "%s: NULL argument", E);
    if (!quantized(format)) return kvq::set_last_error(KVQ_EFORMAT, "%s: format %d is not a quantized tier", E, format);
    if (kvq::rotated_format(format) && !signs) return kvq::set_last_error(KVQ_EINVAL, "%s: rotation signs missing", E);
    File f(path, "rb");
    if (!f.f) return io_fail(E, path, "cannot open");
    kvq_cache_info info;
    uint32_t fsigns[16];
    if (int st = read_header(f.f, E, path, info, fsigns)) return st;
    const bool upgrade = info.format == kFmtF32;
    if (!upgrade && info.format != format)
        return kvq::set_last_error(KVQ_EMISMATCH, "%s: %s holds format %d (codec %d, %d bits), not %d", E, path,
                                   info.format, info.codec, info.bits, format);
    if (info.n_rows > capacity || info.n_rows > planes->n_rows)
        return kvq::set_last_error(KVQ_EINVAL, "%s: %lld rows do not fit", E, (long long)info.n_rows);
    if (upgrade && (!workspace || ws_bytes < kvq_cache_load_workspace()))
        return kvq::set_last_error(KVQ_EWORKSPACE, "%s: an upgrade needs %zu bytes of workspace", E,
                                   kvq_cache_load_workspace());
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(E, e);
    if (kvq::rotated_format(format)) {
        uint32_t hs[16];
        if ((e = cudaMemcpy(hs, signs, 64, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(E, e);
        if (!upgrade && std::memcmp(hs, fsigns, 64) != 0)
            return kvq::set_last_error(KVQ_EMISMATCH, "%s: %s was rotated with other signs", E, path);
    }
    uint8_t* lat = const_cast<uint8_t*>(planes->lat);
    float* ls = const_cast<float*>(planes->lat_scale);
    uint8_t* rope = const_cast<uint8_t*>(planes->rope);
    float* rs = const_cast<float*>(planes->rope_scale);
    const int64_t lb = lat_bytes(format), rb = info.record_bytes;
    std::vector<uint8_t> rec, pl;
    for (int64_t c = 0; c < info.n_rows; c += kChunkRows) {
        const int64_t n = std::min(kChunkRows, info.n_rows - c);
        rec.resize((size_t)(n * rb));
        if (std::fread(rec.data(), 1, rec.size(), f.f) != rec.size()) return io_fail(E, path, "read failed");
        if (upgrade) {
            // quantize on load: fp32 rows -> workspace -> the encoders write the planes
            std::vector<float> hl((size_t)(n * kvq::kDLat)), hr((size_t)(n * kvq::kDRope));
            for (int64_t i = 0; i < n; ++i) {
                std::memcpy(&hl[i * kvq::kDLat], rec.data() + i * rb, kvq::kDLat * 4);
                std::memcpy(&hr[i * kvq::kDRope], rec.data() + i * rb + kvq::kDLat * 4, kvq::kDRope * 4);
            }
            float* wl = static_cast<float*>(workspace);
            float* wr = wl + kChunkRows * kvq::kDLat;
            e = cudaMemcpyAsync(wl, hl.data(), hl.size() * 4, cudaMemcpyHostToDevice, s);
            if (e == cudaSuccess) e = cudaMemcpyAsync(wr, hr.data(), hr.size() * 4, cudaMemcpyHostToDevice, s);
            if (e == cudaSuccess)
                e = format == KVQ_FMT_FP8
                        ? kvq::launch_encode_fp8(wl, n, kvq::kDLat, kvq::kDLat, lat + c * lb, lb, ls + c, s)
                        : kvq::launch_encode_tq(wl, n, kvq::kDLat, kvq::kDLat, kvq::rotated_bits(format), signs,
                                                lat + c * lb, lb, ls + c, s);
            if (e == cudaSuccess)
                e = kvq::launch_encode_fp8(wr, n, kvq::kDRope, kvq::kDRope, rope + c * kvq::kDRope, kvq::kDRope,
                                           rs + c, s);
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);     // the staging is reused
            if (e != cudaSuccess) return cuda_fail(E, e);
            continue;
        }
        pl.resize((size_t)(n * (lb + 4 + kvq::kDRope + 4)));
        uint8_t* plat = pl.data();
        uint8_t* pls = plat + n * lb;
        uint8_t* prope = pls + n * 4;
        uint8_t* prs = prope + n * kvq::kDRope;
        for (int64_t i = 0; i < n; ++i) {
            const uint8_t* r = rec.data() + i * rb;
            std::memcpy(plat + i * lb, r, (size_t)lb);
            std::memcpy(pls + i * 4, r + lb, 4);
            std::memcpy(prope + i * kvq::kDRope, r + lb + 4, kvq::kDRope);
            std::memcpy(prs + i * 4, r + lb + 4 + kvq::kDRope, 4);
        }
        e = cudaMemcpy(lat + c * lb, plat, (size_t)(n * lb), cudaMemcpyHostToDevice);
        if (e == cudaSuccess) e = cudaMemcpy(ls + c, pls, (size_t)(n * 4), cudaMemcpyHostToDevice);
        if (e == cudaSuccess) e = cudaMemcpy(rope + c * kvq::kDRope, prope, (size_t)(n * kvq::kDRope), cudaMemcpyHostToDevice);
        if (e == cudaSuccess) e = cudaMemcpy(rs + c, prs, (size_t)(n * 4), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(E, e);
    }
    if (n_loaded) *n_loaded = info.n_rows;
    return KVQ_OK;
}

}  // extern "C"
