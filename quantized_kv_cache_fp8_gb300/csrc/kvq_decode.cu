// kvq_decode.cu — absorbed-MLA split-T decode over a quantized latent cache, the
// log-sum-exp combine, and the TQ4 query rotation / output unrotation.
//
// colibri PR #399: the MLA latent c_t is both key and value, so per query and head
//   s_t = tau (q_lat . c_t + q_rope . k_rope_t),  out = sum_t softmax(s)_t c_t;
// long contexts split T: each CTA reduces a chunk of rows to a partial softmax
// state (m, l, o) and a combine merges the chunks; the sparse (DSA-style) gather restricts the
// rows to a list of absolute indices; the native TQ4 consumer scores against
// rot(q) and accumulates in the rotated domain, unrotating the output once.
//
// This file holds the CUDA-core (SIMT) kernel, the reference-grade path for every
// shape.  Softmax runs in the log2 domain (scores pre-multiplied by log2 e).
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <atomic>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kRT = 32;              // rows per tile
constexpr int kGH = 8;               // heads per CTA
constexpr int kD = kDLat + kDRope;   // 576
constexpr int kLDT = kD + 4;         // padded shared row, floats (16-byte multiple)
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned kDevBadFormat = KVQ_DEV_BAD_FORMAT;

__constant__ float c_cb[16] = {
    kTq4Centroids[0], kTq4Centroids[1], kTq4Centroids[2], kTq4Centroids[3],
    kTq4Centroids[4], kTq4Centroids[5], kTq4Centroids[6], kTq4Centroids[7],
    kTq4Centroids[8], kTq4Centroids[9], kTq4Centroids[10], kTq4Centroids[11],
    kTq4Centroids[12], kTq4Centroids[13], kTq4Centroids[14], kTq4Centroids[15]};
__constant__ TqCodebook<8> c_cb3 = kTq3;
__constant__ TqCodebook<64> c_cb6 = kTq6;

struct DecodeArgs {
    kvq_mla_problem p;
    int split_rows, n_splits, n_hblk;
    float* q_rot;      // [n_seq][n_q][H][512]  (TQ4 sequences)
    float* part_ml;    // [n_seq][n_q][H][n_splits][2]
    float* part_o;     // [n_seq][n_q][H][n_splits][512]
    float* out;
    float* lse;
    uint32_t* status;
    int premix;        // rotated rows' partials carry the unrotation's stages h = 128, 256
};

__device__ __forceinline__ int seq_format(const kvq_mla_problem& p, int s)
{
    return p.seq_fmt ? p.seq_fmt[s] : p.fmt;
}

// pool row of logical row t of sequence s, or -1
__device__ __forceinline__ int64_t pool_row(const kvq_mla_problem& p, int s, int64_t t)
{
    if (!p.block_table) return (int64_t)s * p.seq_stride_rows + t;
    const int64_t page = t / p.page_size;
    if (page >= p.max_pages) return -1;
    const int64_t pid = p.block_table[(int64_t)s * p.max_pages + page];
    if (pid < 0) return -1;
    return pid * p.page_size + t % p.page_size;
}

// e4m3 code -> value; the pattern S.1111.111 (never written by the encoder) reads as 0
__device__ __forceinline__ float e4m3_to_float(uint32_t byte)
{
    if ((byte & 0x7Fu) == 0x7Fu) return 0.0f;
    const __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)byte, __NV_E4M3);
    return __half2float(__half(hr));
}

// ------------------------------------------------------------------------------------
// TQ4 query rotation: q_rot = (1/sqrt(512)) FWHT_512(s (.) q_lat), one warp per row.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) rotate_queries_kernel(DecodeArgs a)
{
    const kvq_mla_problem& p = a.p;
    const int lane = threadIdx.x & 31;
    const int64_t n_rows = (int64_t)p.n_seq * p.n_q * p.n_heads;
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    uint32_t neg = 0;
#pragma unroll
    for (int k = 0; k < 16; ++k) neg |= ((p.tq4_signs[k] >> lane) & 1u) << k;
    const float c = tq4_inv_sqrt(kDLat);
    for (int64_t r = warp; r < n_rows; r += n_warps) {
        const int s = (int)(r / ((int64_t)p.n_q * p.n_heads));
        if (!rotated_format(seq_format(p, s))) continue;
        const float* src = p.q_lat + r * kDLat;
        float y[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float v = src[k * 32 + lane];
            y[k] = ((neg >> k) & 1u) ? -v : v;
        }
        fwht_warp<16>(y, lane);
        float* dst = a.q_rot + r * kDLat;
#pragma unroll
        for (int k = 0; k < 16; ++k) dst[k * 32 + lane] = y[k] * c;
    }
}

// ------------------------------------------------------------------------------------
// Split-T decode, CUDA cores.  CTA = (split, sequence, query x head block of 8).
// Per tile of 32 rows: dequantise into shared fp32 (fp8: code * scale; TQ4: the
// rotated row cb[code] * radius / sqrt(512)); warp g scores head g against the 32 rows
// (lane = row); online softmax within the warp; every thread then accumulates two
// output columns for the 8 heads.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) mla_decode_simt_kernel(DecodeArgs a)
{
    extern __shared__ __align__(16) float smem[];
    float* s_q = smem;                      // [kGH][kLDT]
    float* s_kv = s_q + kGH * kLDT;         // [kRT][kLDT]
    float* s_p = s_kv + kRT * kLDT;         // [kRT][kGH]
    float* s_alpha = s_p + kRT * kGH;       // [kGH]
    int* s_valid = reinterpret_cast<int*>(s_alpha + kGH);   // [kRT]
    float* s_cb = reinterpret_cast<float*>(s_valid + kRT);  // [64] rotated-tier centroids

    const kvq_mla_problem& p = a.p;
    const int split = blockIdx.x, s = blockIdx.y;
    const int q = blockIdx.z / a.n_hblk;
    const int h0 = (blockIdx.z % a.n_hblk) * kGH;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nh = min(kGH, p.n_heads - h0);
    const int L = p.seq_len[s];
    const int fmt = seq_format(p, s);
    const int64_t n_cand = p.idx ? (int64_t)p.top_k : (int64_t)L;
    const int64_t r0 = (int64_t)split * a.split_rows;
    const int64_t r1 = min(r0 + (int64_t)a.split_rows, n_cand);
    const int64_t lim = p.causal ? (int64_t)L - p.n_q + q : (int64_t)L - 1;
    const int64_t qrow = ((int64_t)s * p.n_q + q) * p.n_heads;   // + h
    auto slot = [&](int h) { return (qrow + h) * a.n_splits + split; };

    const bool bad_fmt = (fmt != KVQ_FMT_FP8 && !rotated_format(fmt));
    if (r0 >= n_cand || bad_fmt) {
        if (bad_fmt && tid == 0 && split == 0 && a.status) atomicOr(a.status, kDevBadFormat);
        if (tid < nh) {
            a.part_ml[slot(h0 + tid) * 2] = -INFINITY;
            a.part_ml[slot(h0 + tid) * 2 + 1] = 0.0f;
        }
        return;
    }
    const bool tq4 = rotated_format(fmt);               // rows in the rotated domain
    const int bits = rotated_bits(fmt);
    const kvq_mla_cache& C = tq4 ? p.tq4 : p.fp8;
    if (tid < 64) s_cb[tid] = bits == 3 ? (tid < 8 ? c_cb3.cb[tid] : 0.0f)
                            : bits == 6 ? c_cb6.cb[tid] : (tid < 16 ? c_cb[tid] : 0.0f);

    for (int i = tid; i < kGH * kD; i += kThreads) {
        const int g = i / kD, k = i % kD;
        float v = 0.0f;
        if (g < nh) {
            const int64_t r = qrow + h0 + g;
            if (k < kDLat) v = tq4 ? a.q_rot[r * kDLat + k] : p.q_lat[r * kDLat + k];
            else v = p.q_rope[r * kDRope + (k - kDLat)];
        }
        s_q[g * kLDT + k] = v;
    }

    float m = -INFINITY, l = 0.0f;          // softmax state of head `warp` (log2 domain)
    float o[kGH][2];
#pragma unroll
    for (int g = 0; g < kGH; ++g) o[g][0] = o[g][1] = 0.0f;
    const float tau2 = p.sm_scale * kLog2e;
    const float c512 = tq4_inv_sqrt(kDLat);

    for (int64_t t0 = r0; t0 < r1; t0 += kRT) {
        __syncthreads();
        // ---- load + dequantise 32 rows (warp w: rows 4w .. 4w+3)
        for (int rr = 0; rr < kRT / 8; ++rr) {
            const int t = warp * (kRT / 8) + rr;
            const int64_t j = t0 + t;
            bool ok = false;
            int64_t row = -1;
            if (j < r1) {
                const int64_t tl = p.idx ? (int64_t)p.idx[((int64_t)s * p.n_q + q) * p.top_k + j] : j;
                if (tl < 0 || tl >= L) {
                    if (lane == 0 && a.status) atomicOr(a.status, (unsigned)KVQ_DEV_BAD_INDEX);
                } else if (tl <= lim) {
                    row = pool_row(p, s, tl);
                    if (row < 0 || row >= C.n_rows) {
                        if (lane == 0 && a.status) atomicOr(a.status, (unsigned)KVQ_DEV_BAD_PAGE);
                    } else {
                        ok = true;
                    }
                }
            }
            float* dst = s_kv + t * kLDT;
            if (lane == 0) s_valid[t] = ok ? 1 : 0;
            if (!ok) {
                for (int i = lane; i < kD; i += 32) dst[i] = 0.0f;
                continue;
            }
            const float sr = C.rope_scale[row];
            if (!tq4) {
                const float sc = C.lat_scale[row];
                const uint4 w = reinterpret_cast<const uint4*>(C.lat + row * kDLat)[lane];
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    dst[lane * 16 + e] = e4m3_to_float((ww[e >> 2] >> (8 * (e & 3))) & 0xFF) * sc;
            } else if (bits == 4) {
                const float sig = C.lat_scale[row] * c512;
                const uint2 w = reinterpret_cast<const uint2*>(C.lat + row * (kDLat / 2))[lane];
                const uint32_t ww[2] = {w.x, w.y};
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const uint32_t byte = (ww[e >> 3] >> (8 * ((e >> 1) & 3))) & 0xFF;
                    const uint32_t code = (e & 1) ? (byte >> 4) : (byte & 15);
                    dst[lane * 16 + e] = s_cb[code] * sig;
                }
            } else if (bits == 6) {
                // elements 16 lane .. 16 lane + 15: bits 96 lane .. +95 of the bit stream
                const float sig = C.lat_scale[row] * c512;
                const uint32_t* w = reinterpret_cast<const uint32_t*>(C.lat + row * (kDLat * 6 / 8) + lane * 12);
                const uint64_t lo = (uint64_t)w[0] | ((uint64_t)w[1] << 32);
                const uint32_t hi = w[2];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int b0 = 6 * e;          // 0 .. 90
                    uint32_t code;
                    if (b0 + 6 <= 64) code = (uint32_t)(lo >> b0) & 63u;
                    else if (b0 >= 64) code = (hi >> (b0 - 64)) & 63u;
                    else code = ((uint32_t)(lo >> b0) | (hi << (64 - b0))) & 63u;
                    dst[lane * 16 + e] = s_cb[code] * sig;
                }
            } else {
                // 3 bits: elements 16 lane .. +15 are bits 48 lane .. +47, six bytes
                const float sig = C.lat_scale[row] * c512;
                const uint16_t* w = reinterpret_cast<const uint16_t*>(C.lat + row * (kDLat * 3 / 8) + lane * 6);
                const uint64_t v = (uint64_t)w[0] | ((uint64_t)w[1] << 16) | ((uint64_t)w[2] << 32);
#pragma unroll
                for (int e = 0; e < 16; ++e) dst[lane * 16 + e] = s_cb[(uint32_t)(v >> (3 * e)) & 7u] * sig;
            }
            const unsigned short rw = reinterpret_cast<const unsigned short*>(C.rope + row * kDRope)[lane];
            dst[kDLat + 2 * lane] = e4m3_to_float(rw & 0xFF) * sr;
            dst[kDLat + 2 * lane + 1] = e4m3_to_float(rw >> 8) * sr;
        }
        __syncthreads();
        // ---- scores: warp = head g, lane = row t
        {
            const int g = warp, t = lane;
            float sc = -INFINITY;
            if (g < nh && t0 + t < r1 && s_valid[t]) {
                const float4* qa = reinterpret_cast<const float4*>(s_q + g * kLDT);
                const float4* ka = reinterpret_cast<const float4*>(s_kv + t * kLDT);
                float acc0 = 0.0f, acc1 = 0.0f;
#pragma unroll 8
                for (int k4 = 0; k4 < kD / 4; ++k4) {
                    const float4 x = qa[k4], y = ka[k4];
                    acc0 = fmaf(x.x, y.x, acc0);
                    acc1 = fmaf(x.y, y.y, acc1);
                    acc0 = fmaf(x.z, y.z, acc0);
                    acc1 = fmaf(x.w, y.w, acc1);
                }
                sc = (acc0 + acc1) * tau2;
            }
            float tmax = sc;
#pragma unroll
            for (int o2 = 16; o2 >= 1; o2 >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(kFull, tmax, o2));
            const float m_new = fmaxf(m, tmax);
            const float pv = (sc == -INFINITY) ? 0.0f : exp2f(sc - m_new);
            const float alpha = (m == -INFINITY) ? 0.0f : exp2f(m - m_new);
            float psum = pv;
#pragma unroll
            for (int o2 = 16; o2 >= 1; o2 >>= 1) psum += __shfl_xor_sync(kFull, psum, o2);
            l = l * alpha + psum;
            m = m_new;
            s_p[t * kGH + g] = pv;
            if (lane == 0) s_alpha[g] = alpha;
        }
        __syncthreads();
        // ---- context: columns tid and tid + 256, all heads
#pragma unroll
        for (int g = 0; g < kGH; ++g) {
            const float al = s_alpha[g];
            o[g][0] *= al;
            o[g][1] *= al;
        }
        const int nt = (int)min((int64_t)kRT, r1 - t0);
        for (int t = 0; t < nt; ++t) {
            const float v0 = s_kv[t * kLDT + tid];
            const float v1 = s_kv[t * kLDT + tid + 256];
            const float4 pa = reinterpret_cast<const float4*>(s_p + t * kGH)[0];
            const float4 pb = reinterpret_cast<const float4*>(s_p + t * kGH)[1];
            const float pp[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
            for (int g = 0; g < kGH; ++g) {
                o[g][0] = fmaf(pp[g], v0, o[g][0]);
                o[g][1] = fmaf(pp[g], v1, o[g][1]);
            }
        }
    }
    if (lane == 0 && warp < nh) {
        a.part_ml[slot(h0 + warp) * 2] = m;
        a.part_ml[slot(h0 + warp) * 2 + 1] = l;
    }
    for (int g = 0; g < nh; ++g) {
        float* dst = a.part_o + slot(h0 + g) * kDLat;
        dst[tid] = o[g][0];
        dst[tid + 256] = o[g][1];
    }
}

// ------------------------------------------------------------------------------------
// Log-sum-exp combine (+ TQ4 unrotation), grid (row, quarter) of 512-thread CTAs, row =
// (seq, query, head):
//   M = max_S m_S,  L = sum_S l_S 2^(m_S - M),  out = sum_S o_S 2^(m_S - M) / L,
//   lse = (M + log2 L) ln 2;  TQ4: out <- (1/sqrt 512) s (.) FWHT_512(out).
// With more than 80 splits a row (one CTA, 80 splits in flight) takes several dependent
// batches; then the grid has four quarters per row, and a row not in a rotated tier is
// split into four CTAs of 128 dims whose 16 split groups keep up to 192 splits' partials
// in flight at once.  A row of a rotated tier needs all 512 dims for the unrotation:
// quarter 0 does the whole row.  A split of a tensor-core kernel that gave up on a wait
// marks its partial m = +inf; a row with such a split is written as NaN (lse too).
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void combine_quarter(const DecodeArgs& a, int64_t r, int quarter, int ns, bool rot)
{
    constexpr int kGroups = 16, kPer = 12, kBatch = kGroups * kPer;
    __shared__ float s_w[kBatch];
    __shared__ __align__(16) float4 s_acc[kGroups][32];
    __shared__ float s_red[2][16];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = tid >> 5, j = tid & 31;       // split group, float4 column of the quarter
    const float* ml = a.part_ml + r * a.n_splits * 2;
    const float4* po = reinterpret_cast<const float4*>(a.part_o + r * a.n_splits * kDLat + quarter * 128) + j;
    // the partials come from the decode kernel launched just before this one
    grid_dependency_wait();
    // the first batch is requested before the maxima are known; splits with l = 0 (no
    // admissible row) may hold stale values and get weight 0 below
    float4 v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int S = grp + kGroups * i;
        v[i] = S < ns ? po[(int64_t)S * (kDLat / 4)] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    float M = -INFINITY;
    bool abort_mark = false;                      // a split that gave up (m = +inf)
    for (int S = tid; S < ns; S += 512) {
        const float2 x = reinterpret_cast<const float2*>(ml)[S];
        abort_mark |= x.x == INFINITY;
        if (x.y > 0.0f) M = fmaxf(M, x.x);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    if (lane == 0) s_red[0][warp] = M;
    const bool aborted = __syncthreads_or(abort_mark) != 0;
    M = s_red[0][0];
#pragma unroll
    for (int w = 1; w < 16; ++w) M = fmaxf(M, s_red[0][w]);
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float Lpart = 0.0f;
    for (int S0 = 0; S0 < ns; S0 += kBatch) {
        const int nb = min(kBatch, ns - S0);
        if (S0 > 0) {
            __syncthreads();                      // s_w of the previous batch is consumed
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                const int S = grp + kGroups * i;
                v[i] = S < nb ? po[(int64_t)(S0 + S) * (kDLat / 4)] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
        }
        if (tid < nb) {
            const float2 x = reinterpret_cast<const float2*>(ml)[S0 + tid];
            const float w = x.y > 0.0f ? exp2f(x.x - M) : 0.0f;
            s_w[tid] = w;
            Lpart += w > 0.0f ? x.y * w : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int S = grp + kGroups * i;
            const float w = S < nb ? s_w[S] : 0.0f;
            if (w != 0.0f) {
                acc.x = fmaf(v[i].x, w, acc.x);
                acc.y = fmaf(v[i].y, w, acc.y);
                acc.z = fmaf(v[i].z, w, acc.z);
                acc.w = fmaf(v[i].w, w, acc.w);
            }
        }
    }
    s_acc[grp][j] = acc;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) Lpart += __shfl_xor_sync(kFull, Lpart, o);
    if (lane == 0) s_red[1][warp] = Lpart;
    __syncthreads();
    if (tid >= 32) return;
    float Lt = 0.0f;
#pragma unroll
    for (int w = 0; w < 16; ++w) Lt += s_red[1][w];
    const bool empty = !(Lt > 0.0f);
    float4 res = s_acc[0][j];
#pragma unroll
    for (int g = 1; g < kGroups; ++g) {
        const float4 x = s_acc[g][j];
        res.x += x.x;
        res.y += x.y;
        res.z += x.z;
        res.w += x.w;
    }
    res = empty ? make_float4(0.0f, 0.0f, 0.0f, 0.0f)
                : make_float4(res.x / Lt, res.y / Lt, res.z / Lt, res.w / Lt);
    if (rot) {
        // the rest of the unrotation, (1/sqrt 512) s (.) FWHT_512(out): the decode kernel
        // applied the stages h = 128 and 256 (across the quarters) to each split's
        // partial; stages h = 1, 2 within the float4, h = 4 .. 64 across the lanes
        float e[4] = {res.x, res.y, res.z, res.w};
#pragma unroll
        for (int h = 1; h < 4; h <<= 1) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if ((c & h) == 0) {
                    const float x = e[c], y = e[c + h];
                    e[c] = x + y;
                    e[c + h] = x - y;
                }
            }
        }
#pragma unroll
        for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float o = __shfl_xor_sync(kFull, e[c], h);
                e[c] = (j & h) ? o - e[c] : e[c] + o;
            }
        }
        const int d0 = quarter * 128 + 4 * j;
        const uint32_t sw = a.p.tq4_signs[d0 >> 5] >> (d0 & 31);
        const float c = tq4_inv_sqrt(kDLat);
        res = make_float4(e[0] * c * ((sw & 1u) ? -1.0f : 1.0f), e[1] * c * ((sw & 2u) ? -1.0f : 1.0f),
                          e[2] * c * ((sw & 4u) ? -1.0f : 1.0f), e[3] * c * ((sw & 8u) ? -1.0f : 1.0f));
    }
    if (aborted) res = make_float4(NAN, NAN, NAN, NAN);
    reinterpret_cast<float4*>(a.out + r * kDLat + quarter * 128)[j] = res;
    if (quarter == 0 && tid == 0 && a.lse) a.lse[r] = aborted ? NAN : empty ? -INFINITY : (M + log2f(Lt)) * kLn2;
}

__global__ void __launch_bounds__(512) mla_combine_kernel(DecodeArgs a)
{
    constexpr int kBatch = 80;                    // splits whose partials load at once
    __shared__ float s_w[kBatch];
    __shared__ __align__(16) float s_part[4][kDLat];
    __shared__ float s_red[2][16];
    // a decode of the next call launched with overlap_prior may start now: it reads its
    // queries and writes the workspace only after this kernel has completed
    grid_dependents_launch();
    const kvq_mla_problem& p = a.p;
    const int64_t r = blockIdx.x;                 // (s * n_q + q) * H + h
    const int s = (int)(r / ((int64_t)p.n_q * p.n_heads));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = tid >> 7, j = tid & 127;      // split group, float4 column
    const int L = p.seq_len[s];
    const int fmt = seq_format(p, s);
    const int64_t n_cand = p.idx ? (int64_t)p.top_k : (int64_t)L;
    const int ns = (int)min((int64_t)a.n_splits, (n_cand + a.split_rows - 1) / a.split_rows);
    if (gridDim.y == 4 && (!rotated_format(fmt) || a.premix)) {
        combine_quarter(a, r, blockIdx.y, ns, rotated_format(fmt));
        return;
    }
    if (blockIdx.y != 0) return;                  // a rotated row: quarter 0 does it all
    const float* ml = a.part_ml + r * a.n_splits * 2;
    const float4* po = reinterpret_cast<const float4*>(a.part_o + r * a.n_splits * kDLat) + j;
    // the partials come from the decode kernel launched just before this one
    grid_dependency_wait();
    // the first batch of partials is requested before the maxima are known; splits
    // with l = 0 (no admissible row) may hold stale values and get weight 0 below
    float4 v[kBatch / 4];
#pragma unroll
    for (int i = 0; i < kBatch / 4; ++i) {
        const int S = grp + 4 * i;
        v[i] = S < ns ? po[(int64_t)S * (kDLat / 4)] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    float M = -INFINITY;
    float2 mine = make_float2(-INFINITY, 0.0f);   // (m, l) of split tid
    bool abort_mark = false;                      // a split that gave up (m = +inf)
    for (int S = tid; S < ns; S += 512) {
        const float2 x = reinterpret_cast<const float2*>(ml)[S];
        if (S == tid) mine = x;
        abort_mark |= x.x == INFINITY;
        if (x.y > 0.0f) M = fmaxf(M, x.x);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    if (lane == 0) s_red[0][warp] = M;
    const bool aborted = __syncthreads_or(abort_mark) != 0;
    M = s_red[0][0];
#pragma unroll
    for (int w = 1; w < 16; ++w) M = fmaxf(M, s_red[0][w]);
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float Lpart = 0.0f;
    for (int S0 = 0; S0 < ns; S0 += kBatch) {
        const int nb = min(kBatch, ns - S0);
        if (S0 > 0) {
            __syncthreads();                      // s_w of the previous batch is consumed
#pragma unroll
            for (int i = 0; i < kBatch / 4; ++i) {
                const int S = grp + 4 * i;
                v[i] = S < nb ? po[(int64_t)(S0 + S) * (kDLat / 4)] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
        }
        if (tid < nb) {
            const float2 x = (S0 + tid < 512) && S0 == 0 ? mine
                                                          : reinterpret_cast<const float2*>(ml)[S0 + tid];
            const float w = x.y > 0.0f ? exp2f(x.x - M) : 0.0f;
            s_w[tid] = w;
            Lpart += w > 0.0f ? x.y * w : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kBatch / 4; ++i) {
            const int S = grp + 4 * i;
            const float w = S < nb ? s_w[S] : 0.0f;
            if (w != 0.0f) {
                acc.x = fmaf(v[i].x, w, acc.x);
                acc.y = fmaf(v[i].y, w, acc.y);
                acc.z = fmaf(v[i].z, w, acc.z);
                acc.w = fmaf(v[i].w, w, acc.w);
            }
        }
    }
    reinterpret_cast<float4*>(s_part[grp])[j] = acc;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) Lpart += __shfl_xor_sync(kFull, Lpart, o);
    if (lane == 0) s_red[1][warp] = Lpart;
    __syncthreads();
    float Lt = 0.0f;
#pragma unroll
    for (int w = 0; w < 16; ++w) Lt += s_red[1][w];
    const bool empty = !(Lt > 0.0f);
    // thread tid owns output dim tid from here on
    float res = s_part[0][tid] + s_part[1][tid] + s_part[2][tid] + s_part[3][tid];
    res = empty ? 0.0f : res / Lt;
    if (rotated_format(fmt)) {
        // unrotate: (1/sqrt 512) s (.) FWHT_512(out); stages h < 32 within the warp,
        // h >= 32 through shared memory
#pragma unroll
        for (int h = 1; h < 32; h <<= 1) {
            const float o = __shfl_xor_sync(kFull, res, h);
            res = (tid & h) ? o - res : res + o;
        }
        float* s_o = s_part[0];
        for (int h = 32; h < kDLat; h <<= 1) {
            __syncthreads();
            s_o[tid] = res;
            __syncthreads();
            res = (tid & h) ? s_o[tid - h] - res : res + s_o[tid + h];
        }
        const bool ng = (p.tq4_signs[tid >> 5] >> (tid & 31)) & 1u;
        res = res * tq4_inv_sqrt(kDLat) * (ng ? -1.0f : 1.0f);
    }
    a.out[r * kDLat + tid] = aborted ? NAN : res;
    if (tid == 0 && a.lse) a.lse[r] = aborted ? NAN : empty ? -INFINITY : (M + log2f(Lt)) * kLn2;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// four quarters a row for many splits, or for rotated rows whose partials were premixed
dim3 combine_grid(int64_t rows, const DecodePlan& plan)
{
    return dim3((unsigned)rows, (plan.n_splits > 80 || plan.premix) ? 4 : 1);
}

}  // namespace

int sm_count()
{
    static std::atomic<int> cache[64];            // per device; 0 = not queried yet
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return kDefaultSMs;
    }
    int n = cache[dev].load();
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = kDefaultSMs;
        }
        cache[dev].store(n);
    }
    return n;
}

namespace {

// rows per split for the tensor-core kernels (whole 128-row tiles): one CTA per SM over
// all (sequence, query, head group) units, or about `waves` waves when the units alone
// fill the SMs
int64_t plan_tc_split_rows(int64_t units, int64_t n_cand, int64_t n_sm, int64_t waves)
{
    constexpr int kTile = 128;
    const int64_t tiles = std::max<int64_t>(1, (n_cand + kTile - 1) / kTile);
    int64_t split_tiles;
    if (units >= n_sm) {
        split_tiles = std::max<int64_t>(1, (units * tiles + waves * n_sm - 1) / (waves * n_sm));
    } else {
        const int64_t splits = std::max<int64_t>(1, std::min<int64_t>(tiles, n_sm / units));
        split_tiles = (tiles + splits - 1) / splits;
    }
    return split_tiles * kTile;
}

}  // namespace

bool plan_decode(const kvq_mla_problem& p, DecodePlan& plan)
{
    plan = DecodePlan();
    const int64_t n_sm = sm_count();
    const int64_t n_cand = p.idx ? (int64_t)p.top_k : (int64_t)p.max_seq_len;
    plan.n_cand_max = (int)n_cand;
    // The library's choice (impl 0), by measurement on GB300: fp8 problems of 8 or more heads
    // without a top-k list and with at least 64 tile-units of work run on the e4m3 tcgen05
    // kernel (codes read as they are); other
    // fp8 problems of at most 16 heads, or with a top-k index list, on the warp-level MMA
    // kernel (16 heads a CTA, each code converted once); TQ4 problems of 8 to 16 heads, and 3- and 6-bit problems
    // of 8 or more heads, on the 16-head tcgen05 kernel (each code converted once); other
    // problems of 8 or more heads on the 32-head tcgen05 kernel; below 8 heads the
    // CUDA-core kernel.
    const bool uniform_fp8 = !p.seq_fmt && p.fmt == KVQ_FMT_FP8;
    const bool uniform_tq4 = !p.seq_fmt && p.fmt == KVQ_FMT_TQ4;
    const bool uniform_tqb = !p.seq_fmt && (p.fmt == KVQ_FMT_TQ3 || p.fmt == KVQ_FMT_TQ6);
    // the e4m3 kernel's start-up (one CTA per SM, a 72 KB tile in flight before the first
    // score) pays off from 64 tile-units of work (T = 1024, 16 heads: 8 units, the
    // warp-level MMA kernel is faster; T = 32768: 256 units, the e4m3 kernel is)
    const int64_t tcf8_units = (int64_t)p.n_seq * p.n_q * ((p.n_heads + 15) / 16) * ((n_cand + 127) / 128);
    plan.tcf8 = p.impl == 5 || (p.impl == 0 && uniform_fp8 && p.n_heads >= 8 && !p.idx && tcf8_units >= 64);
    // a batch of per-sequence formats (fp8 and TQ4) of as much work: its fp8 sequences on
    // the e4m3 kernel and its TQ4 sequences on the 32-head kernel, into one set of partials
    plan.by_fmt = p.impl == 0 && p.seq_fmt != nullptr && p.n_heads >= 8 && !p.idx && tcf8_units >= 64;
    plan.tc16 = !plan.tcf8 && (p.impl == 4 || (p.impl == 0 && p.n_heads >= 8 &&
                                ((uniform_tq4 && p.n_heads <= 16) || uniform_tqb)));
    plan.mma = p.impl == 3 || (p.impl == 0 && !plan.tcf8 && uniform_fp8 && (p.n_heads <= 16 || p.idx != nullptr));
    plan.tc = p.impl == 2 || plan.by_fmt ||
              (p.impl == 0 && !plan.tcf8 && !plan.mma && !plan.tc16 && p.n_heads >= 8 &&
               !(p.fmt == KVQ_FMT_TQ3 || p.fmt == KVQ_FMT_TQ6));
    int64_t split_rows = p.split_rows;
    // A batch of several sequences is split into about 16 waves of CTAs rather than 4: its
    // sequences may have many lengths (the plan sees only the longest), so shorter splits
    // even out the last wave (ragged batch of 32 sequences on the 32-head kernel: 4855 us
    // in 4 waves, 4107 us in 16).
    const int64_t waves = p.n_seq > 1 ? 16 : 4;
    if (plan.tc16 || plan.tcf8) {
        constexpr int kHeads = 16;
        plan.head_block = kHeads;
        const int64_t units = std::max<int64_t>(1, (int64_t)p.n_seq * p.n_q * ((p.n_heads + kHeads - 1) / kHeads));
        if (split_rows <= 0) split_rows = plan_tc_split_rows(units, n_cand, n_sm, waves);
    } else if (plan.mma) {
        plan.head_block = mma_head_block();
        if (split_rows <= 0) plan_mma_splits(p, n_cand, split_rows);
    } else if (plan.tc) {
        // (a batch split by tier takes these splits for both of its kernels)
        constexpr int kHeads = 32;
        plan.head_block = kHeads;
        const int64_t units = std::max<int64_t>(1, (int64_t)p.n_seq * p.n_q * ((p.n_heads + kHeads - 1) / kHeads));
        if (split_rows <= 0) split_rows = plan_tc_split_rows(units, n_cand, n_sm, waves);
    } else {
        plan.head_block = kGH;
        const int64_t n_hblk = (p.n_heads + kGH - 1) / kGH;
        if (split_rows <= 0) {
            const int64_t units = std::max<int64_t>(1, (int64_t)p.n_seq * p.n_q * n_hblk);
            int64_t splits = (2 * n_sm + units - 1) / units;
            const int64_t max_splits = std::max<int64_t>(1, (n_cand + 63) / 64);
            splits = std::min(std::max<int64_t>(splits, 1), max_splits);
            split_rows = (n_cand + splits - 1) / splits;
            split_rows = std::max<int64_t>(kRT, (split_rows + kRT - 1) / kRT * kRT);
        }
    }
    plan.split_rows = (int)split_rows;
    // Few rows (say 16 heads of one query): the combine of a rotated row, which needs all
    // 512 dims for the unrotation, would run on as many CTAs as there are rows.  Then tc /
    // tc16 apply the unrotation's stages that mix the 128-dim quarters to each partial and
    // the combine takes four quarters a row (TQ4, T = 131072, 16 heads: 46.6 -> 44.4 us).
    // With more rows the one-CTA-a-row combine is already spread over the SMs, and the
    // extra epilogue work costs more than it saves (64 heads: 43.8 against 45.1 us).
    plan.premix = (plan.tc || plan.tc16) && (p.seq_fmt != nullptr || rotated_format(p.fmt)) &&
                  (int64_t)p.n_seq * p.n_q * p.n_heads <= 32;
    plan.n_splits = (int)std::max<int64_t>(1, (n_cand + split_rows - 1) / split_rows);
    const size_t rows = (size_t)p.n_seq * p.n_q * p.n_heads;
    const bool any_tq4 = p.seq_fmt != nullptr || rotated_format(p.fmt);
    size_t off = 0;
    plan.off_qrot = off;
    off += any_tq4 ? align256(rows * kDLat * sizeof(float)) : 0;
    plan.off_qimg = off;
    off += plan.tc ? tc_q_image_bytes(p) : plan.tc16 ? tc16_q_image_bytes(p) : 0;
    plan.off_ml = off;
    off += align256(rows * plan.n_splits * 2 * sizeof(float));
    plan.off_o = off;
    off += align256(rows * plan.n_splits * kDLat * sizeof(float));
    plan.bytes = off;
    return true;
}

cudaError_t launch_mla_decode(const kvq_mla_problem& p, const DecodePlan& plan, float* out,
                              float* lse, void* ws, uint32_t* dev_status, cudaStream_t s)
{
    if (p.n_seq == 0) return cudaSuccess;
    DecodeArgs a;
    a.p = p;
    a.split_rows = plan.split_rows;
    a.n_splits = plan.n_splits;
    a.n_hblk = (p.n_heads + kGH - 1) / kGH;
    char* base = static_cast<char*>(ws);
    a.q_rot = reinterpret_cast<float*>(base + plan.off_qrot);
    a.part_ml = reinterpret_cast<float*>(base + plan.off_ml);
    a.part_o = reinterpret_cast<float*>(base + plan.off_o);
    a.out = out;
    a.lse = lse;
    a.status = dev_status;
    a.premix = plan.premix ? 1 : 0;
    const int64_t rows = (int64_t)p.n_seq * p.n_q * p.n_heads;
    const bool any_tq4 = p.seq_fmt != nullptr || rotated_format(p.fmt);
    if (any_tq4 && !plan.tc && !plan.mma && !plan.tcf8 && !plan.tc16) {   // read by the CUDA-core kernel only
        int64_t g = std::min<int64_t>((rows + 7) / 8, (int64_t)sm_count() * 8);
        rotate_queries_kernel<<<(int)std::max<int64_t>(g, 1), kThreads, 0, s>>>(a);
    }
    if (plan.by_fmt) {
        // the fp8 sequences on the e4m3 kernel, then the TQ4 ones on the 32-head kernel
        // (an ordinary launch of its query image after the e4m3 kernel, so the combine,
        // dependent on the 32-head kernel, reads the partials of both)
        cudaError_t e = launch_mla_decode_tcf8(p, plan, a.part_ml, a.part_o, dev_status, s, true);
        if (e != cudaSuccess) return e;
        e = launch_mla_decode_tc(p, plan, a.q_rot, base + plan.off_qimg, a.part_ml, a.part_o,
                                 dev_status, s, true);
        if (e != cudaSuccess) return e;
        return launch_dependent(mla_combine_kernel, combine_grid(rows, plan), dim3(512), 0, s, a);
    }
    if (plan.tcf8) {
        cudaError_t e = launch_mla_decode_tcf8(p, plan, a.part_ml, a.part_o, dev_status, s, false);
        if (e != cudaSuccess) return e;
        return launch_dependent(mla_combine_kernel, combine_grid(rows, plan), dim3(512), 0, s, a);
    }
    if (plan.tc16) {
        cudaError_t e = launch_mla_decode_tc16(p, plan, base + plan.off_qimg, a.part_ml, a.part_o,
                                               dev_status, s);
        if (e != cudaSuccess) return e;
        return launch_dependent(mla_combine_kernel, combine_grid(rows, plan), dim3(512), 0, s, a);
    }
    if (plan.mma) {
        cudaError_t e = launch_mla_decode_mma(p, plan, a.part_ml, a.part_o, dev_status, s);
        if (e != cudaSuccess) return e;
        return launch_dependent(mla_combine_kernel, combine_grid(rows, plan), dim3(512), 0, s, a);
    }
    if (plan.tc) {
        cudaError_t e = launch_mla_decode_tc(p, plan, a.q_rot, base + plan.off_qimg, a.part_ml,
                                             a.part_o, dev_status, s, false);
        if (e != cudaSuccess) return e;
        return launch_dependent(mla_combine_kernel, combine_grid(rows, plan), dim3(512), 0, s, a);
    }
    const size_t smem = (size_t)(kGH * kLDT + kRT * kLDT + kRT * kGH + kGH) * sizeof(float)
                        + kRT * sizeof(int) + 64 * sizeof(float);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    static std::atomic<uint64_t> attr_set{0};       // one bit per device
    const uint64_t bit = 1ull << (device & 63);
    if (!(attr_set.load() & bit)) {
        e = cudaFuncSetAttribute(mla_decode_simt_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(bit);
    }
    dim3 grid(plan.n_splits, p.n_seq, p.n_q * a.n_hblk);
    mla_decode_simt_kernel<<<grid, kThreads, smem, s>>>(a);
    return launch_dependent(mla_combine_kernel, combine_grid(rows, plan), dim3(512), 0, s, a);
}

}  // namespace kvq
