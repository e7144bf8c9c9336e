// kvq_api.cu — the C ABI of libkvq: host-side validation, then one or more launches.
//
// Every entry point validates its arguments completely before launching anything, so
// a non-OK return means nothing was enqueued and nothing written.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "kvq_internal.cuh"

namespace {

thread_local char g_last_error[512] = "";
std::atomic<uint64_t> g_wait_limit_ns{kvq::kDefaultWaitNs};

std::mutex g_fault_mu;
std::string g_fault_entry;
int g_fault_status = 0;
bool g_fault_env_read = false;

int fail(int status, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

int parse_fault(const char* spec)
{
    g_fault_entry.clear();
    g_fault_status = 0;
    if (!spec || !*spec) return KVQ_OK;
    const char* colon = strrchr(spec, ':');
    if (!colon || colon == spec) return KVQ_EINVAL;
    char* end = nullptr;
    long st = strtol(colon + 1, &end, 10);
    if (!end || *end != '\0' || st <= 0 || st > 1000) return KVQ_EINVAL;
    g_fault_entry.assign(spec, colon - spec);
    g_fault_status = (int)st;
    return KVQ_OK;
}

// returns a non-zero status when a fault is injected for `entry`
int injected(const char* entry)
{
    std::lock_guard<std::mutex> lk(g_fault_mu);
    if (!g_fault_env_read) {
        g_fault_env_read = true;
        if (const char* env = getenv("KVQ_FAULT")) parse_fault(env);
    }
    if (g_fault_status != 0 && g_fault_entry == entry) {
        fail(g_fault_status, "%s: fault injected (KVQ_FAULT / kvq_set_fault)", entry);
        return g_fault_status;
    }
    return 0;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }
bool is_pow2(int64_t n) { return n > 0 && (n & (n - 1)) == 0; }

int cuda_status(cudaError_t e, const char* entry)
{
    if (e == cudaSuccess) return KVQ_OK;
    return fail(KVQ_ECUDA, "%s: %s", entry, cudaGetErrorString(e));
}

}  // namespace

uint64_t kvq::wait_limit_ns() { return g_wait_limit_ns.load(); }

int kvq::set_last_error(int status, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

extern "C" {

int kvq_version(void) { return 100; }

const char* kvq_status_string(int status)
{
    switch (status) {
        case KVQ_OK: return "KVQ_OK";
        case KVQ_EINVAL: return "KVQ_EINVAL: invalid argument";
        case KVQ_ENOTPOW2: return "KVQ_ENOTPOW2: width is not a power of two";
        case KVQ_EFORMAT: return "KVQ_EFORMAT: unknown or mismatched format";
        case KVQ_EALIGN: return "KVQ_EALIGN: misaligned pointer or leading dimension";
        case KVQ_EWORKSPACE: return "KVQ_EWORKSPACE: workspace missing or too small";
        case KVQ_ECUDA: return "KVQ_ECUDA: CUDA error";
        case KVQ_EFAULT_INJECTED: return "KVQ_EFAULT_INJECTED: injected fault";
        default: return "unknown kvq status";
    }
}

const char* kvq_last_error(void) { return g_last_error; }

int kvq_set_fault(const char* spec)
{
    std::lock_guard<std::mutex> lk(g_fault_mu);
    g_fault_env_read = true;
    int st = parse_fault(spec);
    if (st != KVQ_OK) return fail(st, "kvq_set_fault: malformed spec (want \"entry:status\")");
    return KVQ_OK;
}

int kvq_set_wait_limit_ns(uint64_t ns)
{
    g_wait_limit_ns.store(ns == 0 ? kvq::kDefaultWaitNs : ns);
    return KVQ_OK;
}

int kvq_tq4_codebook(float centroids[16], float thresholds[15])
{
    if (!centroids || !thresholds) return fail(KVQ_EINVAL, "kvq_tq4_codebook: NULL output");
    for (int k = 0; k < 16; ++k) centroids[k] = kvq::kTq4Centroids[k];
    for (int k = 0; k < 15; ++k) thresholds[k] = kvq::kTq4Thresholds[k];
    return KVQ_OK;
}

int kvq_tq_codebook(int bits, float* centroids, float* thresholds)
{
    if (bits != 3 && bits != 4 && bits != 6) return fail(KVQ_EINVAL, "kvq_tq_codebook: bits %d not 3, 4 or 6", bits);
    if (!centroids || !thresholds) return fail(KVQ_EINVAL, "kvq_tq_codebook: NULL output");
    kvq::tq_codebook_values(bits, centroids, thresholds);
    return KVQ_OK;
}

int kvq_encode_fp8(const float* x, int64_t rows, int dim, int64_t ldx, uint8_t* codes,
                   int64_t ldc, float* scales, kvq_stream_t stream)
{
    const char* E = "kvq_encode_fp8";
    if (int st = injected(E)) return st;
    if (rows < 0) return fail(KVQ_EINVAL, "%s: rows < 0", E);
    if (dim < 1 || dim > 16384) return fail(KVQ_EINVAL, "%s: dim %d outside [1, 16384]", E, dim);
    if (ldx < dim || ldc < dim) return fail(KVQ_EINVAL, "%s: ldx/ldc smaller than dim", E);
    if (rows == 0) return KVQ_OK;
    if (!x || !codes || !scales) return fail(KVQ_EINVAL, "%s: NULL pointer", E);
    if (!aligned(x, 4) || !aligned(scales, 4)) return fail(KVQ_EALIGN, "%s: x/scales not 4-byte aligned", E);
    return cuda_status(kvq::launch_encode_fp8(x, rows, dim, ldx, codes, ldc, scales,
                                              (cudaStream_t)stream), E);
}

int kvq_encode_tq4(const float* x, int64_t rows, int dim, int64_t ldx,
                   const uint32_t* sign_bits, uint8_t* packed, int64_t ldp, float* radius,
                   kvq_stream_t stream)
{
    const char* E = "kvq_encode_tq4";
    if (int st = injected(E)) return st;
    if (!is_pow2(dim)) return fail(KVQ_ENOTPOW2, "%s: dim %d is not a power of two", E, dim);
    if (dim < 64 || dim > 1024) return fail(KVQ_EINVAL, "%s: dim %d outside [64, 1024]", E, dim);
    if (rows < 0) return fail(KVQ_EINVAL, "%s: rows < 0", E);
    if (ldx < dim || ldp < dim / 2) return fail(KVQ_EINVAL, "%s: ldx/ldp too small", E);
    if (rows == 0) return KVQ_OK;
    if (!x || !sign_bits || !packed || !radius) return fail(KVQ_EINVAL, "%s: NULL pointer", E);
    if (!aligned(x, 4) || !aligned(radius, 4) || !aligned(sign_bits, 4))
        return fail(KVQ_EALIGN, "%s: x/radius/sign_bits not 4-byte aligned", E);
    return cuda_status(kvq::launch_encode_tq4(x, rows, dim, ldx, sign_bits, packed, ldp, radius,
                                              (cudaStream_t)stream), E);
}

int kvq_encode_tq(const float* x, int64_t rows, int dim, int64_t ldx, int bits,
                  const uint32_t* sign_bits, uint8_t* packed, int64_t ldp, float* radius,
                  kvq_stream_t stream)
{
    const char* E = "kvq_encode_tq";
    if (int st = injected(E)) return st;
    if (bits != 3 && bits != 4 && bits != 6) return fail(KVQ_EINVAL, "%s: bits %d not 3, 4 or 6", E, bits);
    if (!is_pow2(dim)) return fail(KVQ_ENOTPOW2, "%s: dim %d is not a power of two", E, dim);
    if (dim < 64 || dim > 1024) return fail(KVQ_EINVAL, "%s: dim %d outside [64, 1024]", E, dim);
    if (rows < 0) return fail(KVQ_EINVAL, "%s: rows < 0", E);
    if (ldx < dim || ldp < (int64_t)dim * bits / 8) return fail(KVQ_EINVAL, "%s: ldx/ldp too small", E);
    if (rows == 0) return KVQ_OK;
    if (!x || !sign_bits || !packed || !radius) return fail(KVQ_EINVAL, "%s: NULL pointer", E);
    if (!aligned(x, 4) || !aligned(radius, 4) || !aligned(sign_bits, 4))
        return fail(KVQ_EALIGN, "%s: x/radius/sign_bits not 4-byte aligned", E);
    return cuda_status(kvq::launch_encode_tq(x, rows, dim, ldx, bits, sign_bits, packed, ldp, radius,
                                             (cudaStream_t)stream), E);
}

int kvq_encode_mla(const float* c_lat, int64_t ldx, const float* k_rope, int64_t ldr,
                   int64_t rows, int fmt, const uint32_t* sign_bits, uint8_t* lat,
                   int64_t ldl, float* lat_scale, uint8_t* rope, int64_t ldc,
                   float* rope_scale, kvq_stream_t stream)
{
    const char* E = "kvq_encode_mla";
    if (int st = injected(E)) return st;
    if (fmt != KVQ_FMT_FP8 && !kvq::rotated_format(fmt)) return fail(KVQ_EFORMAT, "%s: fmt %d", E, fmt);
    const int bits = fmt == KVQ_FMT_FP8 ? 8 : kvq::rotated_bits(fmt);
    if (rows < 0) return fail(KVQ_EINVAL, "%s: rows < 0", E);
    if (ldx < kvq::kDLat || ldr < kvq::kDRope || ldl < (int64_t)kvq::kDLat * bits / 8 || ldc < kvq::kDRope)
        return fail(KVQ_EINVAL, "%s: a row stride is smaller than its row", E);
    if (rows == 0) return KVQ_OK;
    if (!c_lat || !k_rope || !lat || !lat_scale || !rope || !rope_scale || (bits != 8 && !sign_bits))
        return fail(KVQ_EINVAL, "%s: NULL pointer", E);
    if (!aligned(c_lat, 4) || !aligned(k_rope, 4) || !aligned(lat_scale, 4) || !aligned(rope_scale, 4) ||
        (bits != 8 && !aligned(sign_bits, 4)))
        return fail(KVQ_EALIGN, "%s: a float or sign pointer is not 4-byte aligned", E);
    return cuda_status(kvq::launch_encode_mla(c_lat, ldx, k_rope, ldr, rows, fmt, sign_bits, lat, ldl,
                                              lat_scale, rope, ldc, rope_scale, (cudaStream_t)stream), E);
}

int kvq_append_q4(const float* k, const float* v, int n_seq, const int32_t* pos0, int n_tok,
                  int n_heads, int head_dim, const int32_t* page_table, int max_pages,
                  int page_size, int64_t n_cells, uint8_t* k_pool, uint8_t* v_pool,
                  uint32_t* dev_status, kvq_stream_t stream)
{
    const char* E = "kvq_append_q4";
    if (int st = injected(E)) return st;
    if (!is_pow2(head_dim)) return fail(KVQ_ENOTPOW2, "%s: head_dim %d is not a power of two", E, head_dim);
    if (head_dim != 256) return fail(KVQ_EINVAL, "%s: head_dim must be 256", E);
    if (n_seq < 0 || n_tok < 0 || n_heads < 1 || max_pages < 1 || page_size < 1 || n_cells < 0)
        return fail(KVQ_EINVAL, "%s: bad sizes", E);
    if ((int64_t)n_seq * n_tok == 0) return KVQ_OK;
    if (!k || !v || !pos0 || !page_table || !k_pool || !v_pool)
        return fail(KVQ_EINVAL, "%s: NULL pointer", E);
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16)) return fail(KVQ_EALIGN, "%s: pools not 16-byte aligned", E);
    if (!aligned(k, 4) || !aligned(v, 4)) return fail(KVQ_EALIGN, "%s: k/v not 4-byte aligned", E);
    return cuda_status(kvq::launch_append_q4(k, v, n_seq, pos0, n_tok, n_heads, page_table,
                                             max_pages, page_size, n_cells, k_pool, v_pool,
                                             dev_status, (cudaStream_t)stream), E);
}

int kvq_project_append_q4(const float* h, int n_seq, const int32_t* pos0, int n_tok, int d_model,
                          const void* w_k, const void* w_v, int w_type, int n_heads, int head_dim,
                          const int32_t* page_table, int max_pages, int page_size, int64_t n_cells,
                          uint8_t* k_pool, uint8_t* v_pool, uint32_t* dev_status, kvq_stream_t stream)
{
    const char* E = "kvq_project_append_q4";
    if (int st = injected(E)) return st;
    if (!is_pow2(head_dim)) return fail(KVQ_ENOTPOW2, "%s: head_dim %d is not a power of two", E, head_dim);
    if (head_dim != 256) return fail(KVQ_EINVAL, "%s: head_dim must be 256", E);
    if (n_seq < 0 || n_tok < 0 || n_heads < 1 || max_pages < 1 || page_size < 1 || n_cells < 0)
        return fail(KVQ_EINVAL, "%s: bad sizes", E);
    if (d_model < 4 || d_model % 4 != 0) return fail(KVQ_EINVAL, "%s: d_model %d is not a positive multiple of 4", E, d_model);
    if (w_type != KVQ_WEIGHT_F32 && w_type != KVQ_WEIGHT_BF16) return fail(KVQ_EINVAL, "%s: w_type %d", E, w_type);
    const int64_t n_tokens = (int64_t)n_seq * n_tok;
    if (n_tokens == 0) return KVQ_OK;
    if (n_tokens > (int64_t)65535 * 16) return fail(KVQ_EINVAL, "%s: more than 1048560 tokens", E);
    if ((int64_t)n_heads * 16 > INT32_MAX) return fail(KVQ_EINVAL, "%s: bad sizes", E);
    if (!h || !w_k || !w_v || !pos0 || !page_table || !k_pool || !v_pool)
        return fail(KVQ_EINVAL, "%s: NULL pointer", E);
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16)) return fail(KVQ_EALIGN, "%s: pools not 16-byte aligned", E);
    if (!aligned(h, 16)) return fail(KVQ_EALIGN, "%s: h not 16-byte aligned", E);
    if (!aligned(w_k, 16) || !aligned(w_v, 16)) return fail(KVQ_EALIGN, "%s: weights not 16-byte aligned", E);
    return cuda_status(kvq::launch_project_append_q4(h, n_seq, pos0, n_tok, d_model, w_k, w_v,
                                                     w_type == KVQ_WEIGHT_BF16, n_heads, page_table,
                                                     max_pages, page_size, n_cells, k_pool, v_pool,
                                                     dev_status, (cudaStream_t)stream), E);
}

int kvq_gather(const kvq_gather_desc* d, kvq_stream_t stream)
{
    const char* E = "kvq_gather";
    if (int st = injected(E)) return st;
    if (!d) return fail(KVQ_EINVAL, "%s: NULL descriptor", E);
    if (d->format == KVQ_FMT_Q4_0) {
        if (!is_pow2(d->head_dim)) return fail(KVQ_ENOTPOW2, "%s: head_dim not a power of two", E);
        if (d->head_dim != 256) return fail(KVQ_EINVAL, "%s: head_dim must be 256", E);
        if (d->n_seq < 0 || d->n_tok < 0 || d->n_heads < 1 || d->max_pages < 1 || d->page_size < 1)
            return fail(KVQ_EINVAL, "%s: bad sizes", E);
        if ((int64_t)d->n_seq * d->n_tok == 0) return KVQ_OK;
        if (!d->q4_pool || !d->pos0 || !d->page_table || !d->q4_out)
            return fail(KVQ_EINVAL, "%s: NULL pointer", E);
        if (!aligned(d->q4_pool, 16) || !aligned(d->q4_out, 16))
            return fail(KVQ_EALIGN, "%s: pool/out not 16-byte aligned", E);
        return cuda_status(kvq::launch_gather_q4(*d, (cudaStream_t)stream), E);
    }
    if (d->format == KVQ_FMT_FP8 || kvq::rotated_format(d->format)) {
        if (d->n_idx < 0 || d->mla_src_rows < 0) return fail(KVQ_EINVAL, "%s: bad sizes", E);
        if (d->n_idx == 0) return KVQ_OK;
        const kvq_mla_cache& c = d->mla_src;
        if (!c.lat || !c.lat_scale || !c.rope || !c.rope_scale || !d->idx || !d->dst_lat ||
            !d->dst_lat_scale || !d->dst_rope || !d->dst_rope_scale)
            return fail(KVQ_EINVAL, "%s: NULL pointer", E);
        if (d->page_table && (d->max_pages < 1 || d->page_size < 1))
            return fail(KVQ_EINVAL, "%s: bad paging sizes", E);
        if (!aligned(c.lat, 16) || !aligned(c.rope, 16) || !aligned(d->dst_lat, 16) ||
            !aligned(d->dst_rope, 16))
            return fail(KVQ_EALIGN, "%s: code planes not 16-byte aligned", E);
        return cuda_status(kvq::launch_gather_mla(*d, (cudaStream_t)stream), E);
    }
    return fail(KVQ_EFORMAT, "%s: unknown format %d", E, d->format);
}

static int validate_decode(const kvq_mla_problem* p, const char* E)
{
    if (!p) return fail(KVQ_EINVAL, "%s: NULL problem", E);
    if (p->d_lat != 512 || p->d_rope != 64) return fail(KVQ_EINVAL, "%s: d_lat/d_rope must be 512/64", E);
    if (p->n_seq < 0 || p->n_seq > 65535) return fail(KVQ_EINVAL, "%s: n_seq outside [0, 65535]", E);
    if (p->n_q < 1 || p->n_heads < 1 || p->max_seq_len < 0 || p->split_rows < 0)
        return fail(KVQ_EINVAL, "%s: bad sizes", E);
    if ((int64_t)p->n_q * ((p->n_heads + 7) / 8) > 65535) return fail(KVQ_EINVAL, "%s: n_q * n_heads too large", E);
    if (p->impl < 0 || p->impl > 5) return fail(KVQ_EINVAL, "%s: impl must be 0..5", E);
    if (p->overlap_prior != 0 && p->overlap_prior != 1) return fail(KVQ_EINVAL, "%s: overlap_prior must be 0 or 1", E);
    if (p->idx && p->top_k < 0) return fail(KVQ_EINVAL, "%s: top_k < 0", E);
    if (!p->seq_fmt && p->fmt != KVQ_FMT_FP8 && !kvq::rotated_format(p->fmt))
        return fail(KVQ_EFORMAT, "%s: fmt %d is not FP8, TQ3, TQ4 or TQ6", E, p->fmt);
    if ((p->impl == 2 || p->impl == 3) && !p->seq_fmt && (p->fmt == KVQ_FMT_TQ3 || p->fmt == KVQ_FMT_TQ6))
        return fail(KVQ_EFORMAT, "%s: impl 2 and 3 read FP8 and TQ4 rows only", E);
    if (p->impl == 5 && (p->seq_fmt || p->fmt != KVQ_FMT_FP8))
        return fail(KVQ_EFORMAT, "%s: impl 5 reads FP8 rows only (one format, no seq_fmt)", E);
    if (p->n_seq == 0) return KVQ_OK;
    if (!p->seq_len || !p->q_lat || !p->q_rope) return fail(KVQ_EINVAL, "%s: NULL pointer", E);
    const bool need_fp8 = p->seq_fmt || p->fmt == KVQ_FMT_FP8;
    const bool need_tq4 = p->seq_fmt || kvq::rotated_format(p->fmt);
    const kvq_mla_cache* tiers[2] = {need_fp8 ? &p->fp8 : nullptr, need_tq4 ? &p->tq4 : nullptr};
    for (const kvq_mla_cache* c : tiers) {
        if (!c) continue;
        if (!c->lat || !c->lat_scale || !c->rope || !c->rope_scale || c->n_rows < 0)
            return fail(KVQ_EINVAL, "%s: missing cache plane of a tier in use", E);
        if (!aligned(c->lat, 16) || !aligned(c->rope, 16) || !aligned(c->lat_scale, 4) ||
            !aligned(c->rope_scale, 4))
            return fail(KVQ_EALIGN, "%s: cache planes misaligned", E);
    }
    if (need_tq4 && !p->tq4_signs) return fail(KVQ_EINVAL, "%s: TQ4 rotation signs missing", E);
    if (p->block_table) {
        if (p->max_pages < 1 || p->page_size < 1) return fail(KVQ_EINVAL, "%s: bad paging sizes", E);
    } else if (p->seq_stride_rows < 0 || (p->n_seq > 1 && p->seq_stride_rows < p->max_seq_len)) {
        return fail(KVQ_EINVAL, "%s: seq_stride_rows smaller than max_seq_len", E);
    }
    if (!aligned(p->q_lat, 16) || !aligned(p->q_rope, 16))
        return fail(KVQ_EALIGN, "%s: queries not 16-byte aligned", E);
    return KVQ_OK;
}

size_t kvq_mla_decode_workspace(const kvq_mla_problem* p)
{
    if (validate_decode(p, "kvq_mla_decode_workspace") != KVQ_OK) return 0;
    kvq::DecodePlan plan;
    kvq::plan_decode(*p, plan);
    return plan.bytes;
}

int kvq_mla_decode_kernel(const kvq_mla_problem* p)
{
    if (int st = validate_decode(p, "kvq_mla_decode_kernel")) return -st;
    kvq::DecodePlan plan;
    kvq::plan_decode(*p, plan);
    return plan.by_fmt ? 6 : plan.tcf8 ? 5 : plan.tc16 ? 4 : plan.mma ? 3 : plan.tc ? 2 : 1;
}

}  // extern "C"

int kvq::fault_injected(const char* entry) { return injected(entry); }

int kvq::validate_mla_decode_call(const kvq_mla_problem* p, const float* out, const float* lse,
                                  const char* E)
{
    if (int st = validate_decode(p, E)) return st;
    if (p->n_seq == 0) return KVQ_OK;
    if (!out) return fail(KVQ_EINVAL, "%s: NULL out", E);
    if (!aligned(out, 16) || (lse && !aligned(lse, 4))) return fail(KVQ_EALIGN, "%s: out/lse misaligned", E);
    return KVQ_OK;
}

int kvq::mla_decode_checked(const kvq_mla_problem* p, float* out, float* lse, void* workspace,
                            size_t ws_bytes, uint32_t* dev_status, cudaStream_t stream, const char* E)
{
    if (int st = validate_mla_decode_call(p, out, lse, E)) return st;
    if (p->n_seq == 0) return KVQ_OK;
    kvq::DecodePlan plan;
    kvq::plan_decode(*p, plan);
    if (plan.bytes > 0 && (!workspace || ws_bytes < plan.bytes))
        return fail(KVQ_EWORKSPACE, "%s: workspace %zu bytes, need %zu", E, ws_bytes, plan.bytes);
    if (!aligned(workspace, 256)) return fail(KVQ_EALIGN, "%s: workspace not 256-byte aligned", E);
    return cuda_status(kvq::launch_mla_decode(*p, plan, out, lse, workspace, dev_status, stream), E);
}

extern "C" {

int kvq_mla_decode(const kvq_mla_problem* p, float* out, float* lse, void* workspace,
                   size_t ws_bytes, uint32_t* dev_status, kvq_stream_t stream)
{
    const char* E = "kvq_mla_decode";
    if (int st = injected(E)) return st;
    return kvq::mla_decode_checked(p, out, lse, workspace, ws_bytes, dev_status,
                                   (cudaStream_t)stream, E);
}

static int validate_q4_decode(const kvq_q4_problem* p, const char* E)
{
    if (!p) return fail(KVQ_EINVAL, "%s: NULL problem", E);
    if (p->head_dim != 256) return fail(KVQ_EINVAL, "%s: head_dim must be 256", E);
    if (p->n_seq < 0 || p->n_seq > 65535) return fail(KVQ_EINVAL, "%s: n_seq outside [0, 65535]", E);
    if (p->n_kv < 1 || p->n_kv > 65535 || p->n_qh < 1 || p->n_qh % p->n_kv != 0)
        return fail(KVQ_EINVAL, "%s: n_qh must be a positive multiple of n_kv", E);
    const int grp = p->n_qh / p->n_kv;
    if (grp != 1 && grp != 2 && grp != 4 && grp != 8)
        return fail(KVQ_EINVAL, "%s: n_qh / n_kv must be 1, 2, 4 or 8", E);
    if (p->max_seq_len < 0 || p->split_rows < 0) return fail(KVQ_EINVAL, "%s: bad sizes", E);
    if (p->max_pages < 1 || p->page_size < 1 || p->n_cells < 0)
        return fail(KVQ_EINVAL, "%s: bad paging sizes", E);
    if (!(p->sm_scale == p->sm_scale)) return fail(KVQ_EINVAL, "%s: sm_scale is NaN", E);
    if (p->n_seq == 0) return KVQ_OK;
    if (!p->seq_len || !p->page_table || !p->k_pool || !p->v_pool || !p->q)
        return fail(KVQ_EINVAL, "%s: NULL pointer", E);
    if (!aligned(p->k_pool, 16) || !aligned(p->v_pool, 16) || !aligned(p->q, 16) ||
        (p->gate && !aligned(p->gate, 16)))
        return fail(KVQ_EALIGN, "%s: pools, q and gate must be 16-byte aligned", E);
    return KVQ_OK;
}

size_t kvq_q4_decode_workspace(const kvq_q4_problem* p)
{
    if (validate_q4_decode(p, "kvq_q4_decode_workspace") != KVQ_OK) return 0;
    kvq::Q4Plan plan;
    kvq::plan_q4_decode(*p, plan);
    return plan.bytes;
}

int kvq_q4_decode(const kvq_q4_problem* p, float* out, float* lse, void* workspace,
                  size_t ws_bytes, uint32_t* dev_status, kvq_stream_t stream)
{
    const char* E = "kvq_q4_decode";
    if (int st = injected(E)) return st;
    if (int st = validate_q4_decode(p, E)) return st;
    if (p->n_seq == 0) return KVQ_OK;
    if (!out) return fail(KVQ_EINVAL, "%s: NULL out", E);
    if (!aligned(out, 16) || (lse && !aligned(lse, 4))) return fail(KVQ_EALIGN, "%s: out/lse misaligned", E);
    kvq::Q4Plan plan;
    kvq::plan_q4_decode(*p, plan);
    if (!workspace || ws_bytes < plan.bytes)
        return fail(KVQ_EWORKSPACE, "%s: workspace %zu bytes, need %zu", E, ws_bytes, plan.bytes);
    if (!aligned(workspace, 256)) return fail(KVQ_EALIGN, "%s: workspace not 256-byte aligned", E);
    return cuda_status(kvq::launch_q4_decode(*p, plan, out, lse, workspace, dev_status,
                                             (cudaStream_t)stream), E);
}

}  // extern "C"
