/*
 * kvq.h — C ABI of libkvq: a quantized KV cache for an MLA-style latent on one
 * NVIDIA GB300 (sm_103a).
 *
 * The operations follow two pages:
 *   colibri PR #399 "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant (KV_TQ) on
 *     CPU, CUDA, and Metal" — the fp8 tier (Summary; Commit 1), the rotated-int4 tier
 *     ("Why rotated-int4 for the 4-bit tier"), split-T decode and the DSA-aware gather
 *     (Commit 2), the native TQ4 consumer identities and the non-power-of-two refusal
 *     (review-thread rebase notes);
 *   Strata PR #2533 "metal: q4_0 KV cache on the Mac engine" — the q4_0 block codec
 *     with the FWHT256 rotation, the paged append and the gather (kv_q4.metal port
 *     commit; parity-fixture commit), and the decode attention over the q4_0 pools
 *     (qsa decode commit).
 *
 * Conventions for every entry point
 *   - Pointers to tensors are DEVICE pointers owned by the caller.  libkvq allocates no
 *     device memory, keeps no per-call state, and writes only the declared outputs,
 *     the caller's workspace and *dev_status.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default stream) and
 *     returns a host-side status.  Argument errors are detected on the host before any
 *     launch: the call then launches nothing, writes nothing and returns the status;
 *     kvq_last_error() holds a one-line reason (per calling thread).
 *   - Data-dependent faults (a row index or page id out of range) never trap: the
 *     offending row is skipped (or written as zeros where stated) and a bit is OR-ed
 *     into *dev_status (if non-NULL), which the caller reads after synchronizing.
 *   - Row-major layouts; leading dimensions are in elements; 16-byte-aligned bases and
 *     leading dimensions are required where stated (KVQ_EALIGN otherwise).
 *   - Non-finite inputs are outside the contract of every codec.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kvq_stream_t;   /* a cudaStream_t */

typedef enum kvq_status {
    KVQ_OK = 0,
    KVQ_EINVAL = 1,          /* a size, count or pointer argument is invalid           */
    KVQ_ENOTPOW2 = 2,        /* a rotated codec was given a non-power-of-two width      */
    KVQ_EFORMAT = 3,         /* unknown or mismatched format enum                      */
    KVQ_EALIGN = 4,          /* a base pointer or leading dimension is misaligned      */
    KVQ_EWORKSPACE = 5,      /* the workspace is NULL or smaller than required         */
    KVQ_ECUDA = 6,           /* a CUDA launch or attribute call failed                 */
    KVQ_EFAULT_INJECTED = 7, /* host-side fault injection (kvq_set_fault) fired        */
    KVQ_EMISMATCH = 8,       /* a cache file written under another mode: refused       */
    KVQ_EIO = 9              /* a cache file cannot be opened, read or written, or its
                                byte counts do not add up                              */
} kvq_status;

/* bits of *dev_status */
enum {
    KVQ_DEV_BAD_INDEX = 1u,  /* a sparse / gather row index outside [0, rows)          */
    KVQ_DEV_BAD_PAGE = 2u,   /* a position past the page table, or a page id outside
                                the pool                                               */
    KVQ_DEV_TIMEOUT = 4u,    /* a bounded device wait expired                          */
    KVQ_DEV_BAD_FORMAT = 8u  /* a per-sequence format the kernel in use cannot read    */
};

typedef enum kvq_format {
    KVQ_FMT_FP8 = 1,         /* e4m3 codes + one fp32 scale per row                    */
    KVQ_FMT_TQ4 = 2,         /* rotated-int4: 4-bit Lloyd-Max codes + one fp32 radius  */
    KVQ_FMT_Q4_0 = 3,        /* FWHT256-rotated 18-byte q4_0 blocks                    */
    KVQ_FMT_TQ6 = 4,         /* rotated tier, 6-bit codes (64 levels) + fp32 radius     */
    KVQ_FMT_TQ3 = 5          /* rotated tier, 3-bit codes (8 levels) + fp32 radius      */
} kvq_format;

/* element type of a projection weight matrix */
typedef enum kvq_weight_type {
    KVQ_WEIGHT_F32 = 0,      /* fp32                                                   */
    KVQ_WEIGHT_BF16 = 1      /* bfloat16 (the upper half of an fp32 pattern; widened
                                exactly)                                               */
} kvq_weight_type;

/* Library version (major*10000 + minor*100 + patch). */
int kvq_version(void);

/* Static text of a kvq_status value. */
const char* kvq_status_string(int status);

/* One-line reason for the last non-OK status returned to the calling thread. */
const char* kvq_last_error(void);

/*
 * Host-side fault injection for tests of the error paths.  spec = "<entry>:<status>"
 * makes the named entry point (e.g. "kvq_encode_fp8:6") return that status before any
 * launch; NULL or "" clears it.  The environment variable KVQ_FAULT, read at the first
 * call, sets the initial spec.  Returns KVQ_EINVAL for a malformed spec.
 */
int kvq_set_fault(const char* spec);

/*
 * Test hook for the failure path of the tensor-core decode kernels (impl 2, 4 and 5).  Every
 * wait in their pipelines (for a copy, an MMA or another warp's hand-over) gives up after
 * `ns` nanoseconds of %globaltimer time; ns = 0 restores the default of 2 s.  The limit
 * is process-wide and read at each launch.  A CTA that gives up sets KVQ_DEV_TIMEOUT in
 * *dev_status, stops its pipeline, waits (with the default limit) for every copy and MMA
 * it already issued, frees its tensor memory and returns; its partial result is written
 * as (m, l) = (+inf, +inf), which the combine turns into NaN for every output row it
 * feeds, so an aborted row never reads as a result.  Returns KVQ_OK.
 */
int kvq_set_wait_limit_ns(uint64_t ns);

/*
 * The TQ4 codebook in use: the 16 centroids (the Lloyd-Max fixed point of N(0,1) with
 * 16 levels, each rounded to the nearest binary16 value, ascending) and the 15
 * thresholds (midpoints of adjacent centroids).  Host arrays, written by the call.
 * colibri PR #399, "Why rotated-int4 for the 4-bit tier".
 */
int kvq_tq4_codebook(float centroids[16], float thresholds[15]);

/*
 * The codebook of the rotated tier of width bits = 3, 4 or 6 (colibri PR #399: the
 * TurboQuant tier's bit widths, KV_TQ=6 and a 3-bit setting besides the 4-bit one): the
 * 2^bits centroids (Lloyd-Max outputs of N(0,1), each rounded to the nearest binary16
 * value, ascending) and the 2^bits - 1 thresholds (midpoints).  Host arrays of at least
 * 2^bits and 2^bits - 1 floats.  KVQ_EINVAL for another width or a NULL output.
 */
int kvq_tq_codebook(int bits, float* centroids, float* thresholds);

/*
 * fp8 (KV8) per-row encode — colibri PR #399, Summary and Commit 1 (e4m3 codes with one
 * scale per row, the row's largest magnitude over 448, rounding to nearest even).  For each
 * row r:
 *     amax = max_i |x[r][i]|,  scales[r] = amax / 448 (IEEE fp32 division),
 *     codes[r][i] = e4m3 nearest-even of (x[r][i] / scales[r]), saturating at +-448;
 * a row with amax = 0 stores scale 0 and all-zero codes.
 *   x       device fp32 [rows][ldx]   (dim <= ldx)
 *   codes   device u8   [rows][ldc]   (dim <= ldc)
 *   scales  device fp32 [rows]
 * 1 <= dim <= 16384.  The MLA cache encodes the 512-wide latent and the 64-wide rope
 * key as separate calls (separate scales).  rows = 0 is a no-op.
 */
int kvq_encode_fp8(const float* x, int64_t rows, int dim, int64_t ldx,
                   uint8_t* codes, int64_t ldc, float* scales, kvq_stream_t stream);

/*
 * Rotated-int4 (TQ4) encode — colibri PR #399, "Why rotated-int4 for the 4-bit tier":
 * a randomized-Hadamard rotation, then a 16-level N(0,1) Lloyd-Max codebook scaled by
 * radius/sqrt(n).  For each row, with n = dim and c = fp32(1/sqrt(n)):
 *   1. w_i = s_i x_i, s_i = -1 where bit i of sign_bits is 1 (bit i%32 of word i/32);
 *   2. w = FWHT_n(w), radix-2 stages h = 1, 2, ..., n/2 in that order, fp32; y = w * c;
 *   3. ss = sum y_i^2 as 32 partial sums (partial l: i = l, l+32, ... ascending, one
 *      fused multiply-add each) folded by p_l += p_(l xor o), o = 16, 8, 4, 2, 1;
 *   4. radius = sqrt(ss) (IEEE); sigma = radius * c; radius 0 -> all-zero bytes;
 *   5. code_i = #{k : y_i / sigma >= thresholds[k]} (IEEE division);
 *   6. packed[r][j] = code_(2j) | code_(2j+1) << 4.
 *   x        device fp32 [rows][ldx]
 *   sign_bits device u32 [dim/32]
 *   packed   device u8   [rows][ldp]  (dim/2 <= ldp)
 *   radius   device fp32 [rows]
 * dim must be a power of two (KVQ_ENOTPOW2 otherwise, per the page's refusal of
 * non-power-of-two widths) in [64, 1024].  The 64-wide rope key of a TQ4 row is
 * stored with kvq_encode_fp8.
 */
int kvq_encode_tq4(const float* x, int64_t rows, int dim, int64_t ldx,
                   const uint32_t* sign_bits, uint8_t* packed, int64_t ldp,
                   float* radius, kvq_stream_t stream);

/*
 * Rotated-tier encode at bits = 3, 4 or 6: steps 1-5 of kvq_encode_tq4 with the codebook
 * of that width (kvq_tq_codebook), then
 *   6'. the codes form a little-endian bit stream: code i occupies bits
 *       bits*i .. bits*i + bits - 1 of the row's dim*bits/8 bytes (bit 0 = low bit of
 *       byte 0).  For bits = 4 this is step 6 of kvq_encode_tq4, which it calls.
 *   packed   device u8 [rows][ldp], ldp >= dim*bits/8
 * Same dims, alignment and errors as kvq_encode_tq4, plus KVQ_EINVAL for another width.
 */
int kvq_encode_tq(const float* x, int64_t rows, int dim, int64_t ldx, int bits,
                  const uint32_t* sign_bits, uint8_t* packed, int64_t ldp, float* radius,
                  kvq_stream_t stream);

/*
 * Quantize-on-append of MLA rows, both planes in one call — colibri PR #399, Commit 1
 * (the fp8 tier) and Commit 2 (the rotated tier): the latent of a row goes to the
 * cache's tier, its rope key to fp8.  Row r's latent c_lat[r] (512 dims) is encoded as
 * kvq_encode_fp8 (fmt KVQ_FMT_FP8) or kvq_encode_tq (KVQ_FMT_TQ3 / TQ4 / TQ6, rotation
 * signs `sign_bits`) would encode it, into lat + r * ldl and lat_scale[r]; its rope key
 * k_rope[r] (64 dims) as kvq_encode_fp8 would, into rope + r * ldc and rope_scale[r].
 * The bytes equal those of the separate calls.  With 16-byte aligned input rows and
 * 4-byte aligned fp8 code rows the two encoders run as one kernel launch (the latent and
 * rope CTAs side by side), so a per-token append costs one launch; otherwise they run as
 * the two separate kernels.
 *   c_lat      device fp32 [rows] x ldx  (ldx >= 512)
 *   k_rope     device fp32 [rows] x ldr  (ldr >= 64)
 *   lat        device u8   [rows] x ldl  (ldl >= 512 * bits / 8; 8 bits for fp8)
 *   lat_scale  device fp32 [rows]         (fp8: amax/448; rotated: the row radius)
 *   rope       device u8   [rows] x ldc  (ldc >= 64)
 *   rope_scale device fp32 [rows]
 * Errors: KVQ_EFORMAT for another fmt; KVQ_EINVAL for rows < 0, a stride too small or
 * a NULL pointer (sign_bits only for the rotated tiers); KVQ_EALIGN for a float pointer
 * that is not 4-byte aligned.  rows == 0 is a no-op.
 */
int kvq_encode_mla(const float* c_lat, int64_t ldx, const float* k_rope, int64_t ldr,
                   int64_t rows, int fmt, const uint32_t* sign_bits, uint8_t* lat,
                   int64_t ldl, float* lat_scale, uint8_t* rope, int64_t ldc,
                   float* rope_scale, kvq_stream_t stream);

/*
 * q4_0 paged append — Strata PR #2533, kv_q4.metal port commit (fwht256, q4_group /
 * q4_store, the tie rule, the fp16 scale) and the page-table commit.  Token t of
 * sequence s sits at position pos = pos0[s] + t and cell
 *     page_table[s][pos / page_size] * page_size + pos % page_size;
 * its row of head h (K and V alike) is rotated, z = FWHT_256(x) / 16 (stages
 * h = 1..128 ascending, fp32), and stored as 8 blocks of 18 bytes at byte offset
 * (cell * n_heads + h) * 144 of the pool.  Per 32-element block: mval = the element of
 * largest |z| (a tie goes to the larger value, +0 over -0), d = mval / -8,
 * id = (d != 0) ? 1/d : 0, q_j = clamp(trunc(fma(z_j, id, 8.5)), 0, 15); bytes 0-1 =
 * binary16(d) nearest-even, little endian; byte 2+j = q_j | q_(j+16) << 4.
 *   k, v       device fp32 [n_seq][n_tok][n_heads][256]
 *   pos0       device i32  [n_seq]
 *   page_table device i32  [n_seq][max_pages]
 *   k_pool, v_pool device u8 [n_cells][n_heads][144]  (16-byte aligned)
 * head_dim must be 256.  A position past the table or a page id outside the pool sets
 * KVQ_DEV_BAD_PAGE and that token is skipped.
 */
int kvq_append_q4(const float* k, const float* v, int n_seq, const int32_t* pos0,
                  int n_tok, int n_heads, int head_dim, const int32_t* page_table,
                  int max_pages, int page_size, int64_t n_cells,
                  uint8_t* k_pool, uint8_t* v_pool, uint32_t* dev_status,
                  kvq_stream_t stream);

/*
 * q4_0 append with the K/V projection fused into its producer — Strata PR #2533, the qsa
 * decode commit (fwht_row256 applied inside qsa_prep, the kernel that produces the rows,
 * so no unrotated fp32 row makes a round trip through memory) with the q4_0 layout of
 * the kv_q4.metal port commit.  Token t of sequence s has the hidden row
 * h[s][t][0 .. d_model - 1]; its K row of head g is
 *     k[c] = sum_k h[k] * w_k[k][256 g + c],   c < 256   (V alike with w_v),
 * summed in this fixed fp32 order: the k range is cut into 64 chunks of
 * L = 4 * ceil(d_model / 256) consecutive terms (the last chunks short or empty); each
 * chunk is the chain acc = fmaf(h[k], w[k][col], acc) from acc = 0 in ascending k; the
 * 64 chunk sums are added pairwise ((0 + 1), (2 + 3), ..., then the 32, 16, 8, 4 and 2
 * results the same way).
 * The rows are then rotated, quantized and stored exactly as kvq_append_q4 stores its k
 * and v rows (same pool layout, page rule and status), in the same launch: the bytes
 * equal kvq_append_q4 applied to those fp32 rows.
 *   h          device fp32 [n_seq][n_tok][d_model], 16-byte aligned; d_model % 4 == 0
 *   w_k, w_v   device [d_model][n_heads * 256], row-major, of `w_type`, 16-byte aligned
 *   pos0, page_table, pools, dev_status: as kvq_append_q4 (head_dim 256)
 * The projection reads every weight once per group of 16 tokens: it is built for the
 * few new tokens of a decode step, not for a prefill.  Errors: KVQ_EINVAL for bad sizes
 * (d_model < 4 or not a multiple of 4, more than 1048560 tokens), a NULL pointer or another
 * w_type; KVQ_EALIGN as above.  n_seq * n_tok == 0 is a no-op.
 */
int kvq_project_append_q4(const float* h, int n_seq, const int32_t* pos0, int n_tok,
                          int d_model, const void* w_k, const void* w_v, int w_type,
                          int n_heads, int head_dim, const int32_t* page_table,
                          int max_pages, int page_size, int64_t n_cells, uint8_t* k_pool,
                          uint8_t* v_pool, uint32_t* dev_status, kvq_stream_t stream);

/* Planes of one MLA cache tier (device pointers, pool-row indexed). */
typedef struct kvq_mla_cache {
    const uint8_t* lat;        /* FP8: [n_rows][512] e4m3; TQ4: [n_rows][256] nibbles   */
    const float*   lat_scale;  /* FP8: [n_rows] scale;    TQ4: [n_rows] radius          */
    const uint8_t* rope;       /* [n_rows][64] e4m3 codes of the rope key               */
    const float*   rope_scale; /* [n_rows]                                              */
    int64_t        n_rows;     /* rows in the pool                                      */
} kvq_mla_cache;

/*
 * Gather — two modes selected by `format`.
 *
 * KVQ_FMT_Q4_0 (Strata PR #2533, kv_gather_q4 and the qsa decode commit, where a block
 * value is its nibble minus 8 times the fp32 value of the binary16 scale): for s < n_seq,
 * t < n_tok, h < n_heads,
 *     q4_out[s][t][h][32b + j] = binary16_rne((q_j - 8) * float(d_b))
 * from the pool row of position pos0[s] + t (as in kvq_append_q4), i.e. in the ROTATED
 * domain.  q4_out: device u16 (binary16 bits) [n_seq][n_tok][n_heads][256].  A bad
 * position or page sets KVQ_DEV_BAD_PAGE and that token's rows are left untouched.
 *
 * KVQ_FMT_FP8 / KVQ_FMT_TQ4 / KVQ_FMT_TQ6 / KVQ_FMT_TQ3 (colibri PR #399, Commit 2: the
 * gather by absolute row index for DSA-style sparse attention; rows of 512, 256, 384 or
 * 192 code bytes): copies the
 * n_idx rows idx[j] of the cache `mla_src` (through page_table / page_size when
 * page_table is non-NULL, one sequence) byte for byte into the compact cache dst_*
 * (row j).  An index outside [0, mla_src_rows) sets KVQ_DEV_BAD_INDEX and row j is
 * written as zeros.
 */
typedef struct kvq_gather_desc {
    int32_t format;
    /* q4_0 */
    const uint8_t* q4_pool;
    int32_t n_seq, n_tok, n_heads, head_dim;
    const int32_t* pos0;
    int64_t n_cells;
    uint16_t* q4_out;
    /* paging (both modes) */
    const int32_t* page_table;
    int32_t max_pages, page_size;
    /* fp8 / TQ4 rows */
    kvq_mla_cache mla_src;
    int64_t mla_src_rows;           /* logical rows addressable by idx                 */
    const int32_t* idx;             /* device [n_idx]                                  */
    int64_t n_idx;
    uint8_t* dst_lat; float* dst_lat_scale; uint8_t* dst_rope; float* dst_rope_scale;
    uint32_t* dev_status;
} kvq_gather_desc;

int kvq_gather(const kvq_gather_desc* d, kvq_stream_t stream);

/*
 * Absorbed-MLA decode attention over a quantized cache — colibri PR #399: the MLA
 * latent c_t is both key and value; per query and head
 *     s_t = sm_scale * (q_lat . c_t + q_rope . k_rope_t),  out = sum_t softmax(s)_t c_t,
 *     lse = log sum_t exp(s_t)
 * over the admissible rows, computed as split-T partials (m, l, o) merged by a
 * log-sum-exp combine (Commit 2: the kernels that split T).  Rows are dequantised inside the
 * kernel: fp8 c_t = code * scale; the rotated tiers (TQ4, and TQ3 / TQ6 from
 * kvq_encode_tq) in the rotated domain (the page's identity q . xhat = rot(q) . yhat;
 * the combine unrotates the output).  The tensor-core kernels read FP8 and TQ4 rows, and
 * impl 4 also a problem of one 3- or 6-bit format (impl 2 or 3 with such a `fmt` is
 * refused with KVQ_EFORMAT); impl 5 reads problems of FP8 rows only (any other `fmt`, or
 * a seq_fmt batch, is refused with KVQ_EFORMAT) and keeps the codes in e4m3 inside the
 * tensor core, carrying q and the softmax weights as sums of 5 and 4 e4m3 values of
 * decreasing power-of-two weight; in a seq_fmt batch on a tensor-core kernel the 3- and 6-bit
 * sequences set KVQ_DEV_BAD_FORMAT (use impl 1 for such batches).  Admissible rows of
 * query j of sequence i (holding L = seq_len[i] rows): t < L; with `causal`,
 * t <= L - n_q + j (draft + verify); with idx, only t in idx[i][j][:] (an index
 * outside [0, L) sets KVQ_DEV_BAD_INDEX and is skipped).  A query with no admissible
 * row gets out = 0 and lse = -inf.
 */
typedef struct kvq_mla_problem {
    int32_t n_seq, n_q, n_heads;
    int32_t d_lat, d_rope;          /* must be 512 and 64                               */
    int32_t causal;
    int32_t max_seq_len;            /* host: >= every seq_len[i] (sizes the grid)        */
    const int32_t* seq_len;         /* device [n_seq]                                   */
    const int32_t* seq_fmt;         /* device [n_seq] FP8 / TQ3 / TQ4 / TQ6, or NULL:
                                       all `fmt`                                          */
    int32_t fmt;
    const int32_t* block_table;     /* device [n_seq][max_pages] pool page ids, or NULL */
    int32_t max_pages, page_size;
    int64_t seq_stride_rows;        /* no block table: seq i row t = pool row i*stride+t */
    kvq_mla_cache fp8, tq4;         /* the pools of each tier (unused tier: zeros); `tq4`
                                       holds the rotated tier's rows, 512 * b / 8 bytes
                                       of codes each for the b-bit format in use          */
    const uint32_t* tq4_signs;      /* device [16]: the rotation signs of the rotated tier */
    const float* q_lat;             /* device [n_seq][n_q][n_heads][512]                */
    const float* q_rope;            /* device [n_seq][n_q][n_heads][64]                 */
    const int32_t* idx;             /* device [n_seq][n_q][top_k] or NULL               */
    int32_t top_k;
    float sm_scale;
    int32_t split_rows;             /* rows per split; 0: the library chooses            */
    int32_t impl;                   /* 0: library chooses; 1: CUDA-core kernel;
                                       2: tensor-core (tcgen05) kernel, 32 heads a CTA;
                                       3: warp-level MMA kernel, 16 heads a CTA;
                                       4: tcgen05 kernel, 16 heads a CTA, each code
                                          converted to binary16 once;
                                       5: tcgen05 kernel of the fp8 tier, 16 heads a
                                          CTA, e4m3 codes read by the tensor core as
                                          they are (kind::f8f6f4)                        */
    int32_t overlap_prior;          /* 0: the call starts after everything before it on
                                       the stream.  1 (used by kernel 5 alone; the others
                                       ignore it): the decode may start while the kernel
                                       just before it still runs, once that kernel lets
                                       dependents launch (this library's combine does, so
                                       back-to-back calls overlap a decode's start with the
                                       previous call's combine).  It reads the queries and
                                       writes the workspace and outputs only after that
                                       kernel has completed, but reads the cache rows and
                                       scales, seq_len, seq_fmt and block_table, and may set
                                       dev_status bits, before: set 1 only when the kernel
                                       just before the call writes none of those.  0 or 1. */
} kvq_mla_problem;

/* Bytes of workspace kvq_mla_decode needs for this problem (0 if invalid). */
size_t kvq_mla_decode_workspace(const kvq_mla_problem* p);

/*
 * The decode kernel kvq_mla_decode runs for this problem: 1 the CUDA-core kernel, 2 the
 * tcgen05 kernel with 32 heads a CTA, 3 the warp-level MMA kernel, 4 the tcgen05 kernel
 * with 16 heads a CTA and each code converted once, 5 the e4m3 tcgen05 kernel of the fp8
 * tier, 6 both 5 (for the batch's fp8 sequences) and 2 (for its TQ4 sequences) in one
 * call; `impl` when it is non-zero, else the library's choice.  With W =
 * n_seq * n_q * ceil(H / 16) * ceil(rows / 128) tile-units of work: fp8 problems of 8 or
 * more heads without a top-k list and W >= 64: 5; batches of per-sequence formats
 * (seq_fmt) of 8 or more heads without a top-k list and W >= 64: 6; other fp8 problems of
 * at most 16 heads or with a top-k list: 3; TQ4 problems of 8 to 16 heads and 3- or 6-bit
 * problems of 8 or more heads: 4; other problems of 8 or more heads: 2; the rest: 1.  Host
 * only, nothing enqueued.  An invalid problem returns the negated status
 * kvq_mla_decode would return (-KVQ_EINVAL, -KVQ_EFORMAT, -KVQ_EALIGN).
 */
int kvq_mla_decode_kernel(const kvq_mla_problem* p);

/*
 *   out        device fp32 [n_seq][n_q][n_heads][512]
 *   lse        device fp32 [n_seq][n_q][n_heads] or NULL (natural log)
 *   workspace  device, >= kvq_mla_decode_workspace(p) bytes, 256-byte aligned
 *   dev_status device u32 or NULL
 */
int kvq_mla_decode(const kvq_mla_problem* p, float* out, float* lse, void* workspace,
                   size_t ws_bytes, uint32_t* dev_status, kvq_stream_t stream);

/*
 * kvq_mla_decode without a workspace argument.  The pages have no counterpart: this is a
 * convenience of the library for callers that cannot allocate device memory when they
 * decode, such as code running inside a memory pool or custom allocator that owns the
 * whole device, a latency-critical loop that must not enter the allocator, or an
 * embedding that only receives pre-placed input and output buffers.
 *
 * Same problem, outputs, status word and errors as kvq_mla_decode; the scratch comes
 * from one fixed 64 MiB device array inside the library, which every GPU that loads the
 * library holds until the process exits.  A problem whose kvq_mla_decode_workspace()
 * exceeds 64 MiB is rejected with KVQ_EWORKSPACE (nothing launched).  The call allocates
 * nothing.  Its first call on a device looks up that array's device address (with the
 * device current); make that first call before any stream capture.  All calls share the
 * array: calls that overlap on the GPU (several streams or host threads) race, so
 * serialise them.  No scratch byte needs to be zero beforehand.
 */
int kvq_mla_decode_noalloc(const kvq_mla_problem* p, float* out, float* lse,
                           uint32_t* dev_status, kvq_stream_t stream);

/*
 * q4_0 paged decode attention, grouped-query, head_dim 256 — Strata PR #2533, the qsa
 * decode commit: the query rows pass through the orthonormal 256-point FWHT (the
 * rotation the K and V rows received when kvq_append_q4 stored them), attention reads
 * the q4_0 pools, each 4-bit code of a block standing for its value less 8 times the
 * block's binary16 scale, and the merged output row is rotated back (the orthonormal
 * FWHT is its own inverse) before the optional multiply by sigmoid(gate).  For sequence s and query head h, with KV head
 * g = h / (n_qh / n_kv) and the tokens at positions 0 .. seq_len[s] - 1:
 *   q_rot = FWHT256(q[s][h]) / 16,  score_t = sm_scale * q_rot . k_t,
 *   out[s][h] = FWHT256(sum_t softmax(score)_t v_t) / 16  [* sigmoid(gate[s][h])],
 *   lse[s][h] = log sum_t exp(score_t).
 * Positions map to pool cells as in kvq_append_q4: page_table[s][t / page_size] *
 * page_size + t % page_size.  A page index past max_pages, a missing page id (< 0) or a
 * cell outside the pool skips that position and sets KVQ_DEV_BAD_PAGE; a sequence with no
 * position gives out = 0, lse = -inf.  seq_len[s] is clamped to [0, max_seq_len].
 * Computed as split-T partials (one warp per split, sequence and KV head) merged by a
 * log-sum-exp combine.  Errors: KVQ_EINVAL (sizes, group ratio, NULL pointers),
 * KVQ_EALIGN, KVQ_EWORKSPACE (workspace below kvq_q4_decode_workspace(p)), KVQ_ECUDA.
 */
typedef struct kvq_q4_problem {
    int32_t n_seq;
    int32_t n_qh;                   /* query heads                                      */
    int32_t n_kv;                   /* KV heads; n_qh / n_kv is 1, 2, 4 or 8            */
    int32_t head_dim;               /* 256                                              */
    const int32_t* seq_len;         /* device [n_seq] tokens held                       */
    int32_t max_seq_len;            /* host bound on every seq_len (sizes the splits)   */
    const int32_t* page_table;      /* device [n_seq][max_pages]                        */
    int32_t max_pages, page_size;
    int64_t n_cells;                /* cells in each pool                               */
    const uint8_t* k_pool;          /* device [n_cells][n_kv][144], 16-byte aligned      */
    const uint8_t* v_pool;          /* device [n_cells][n_kv][144], 16-byte aligned      */
    const float* q;                 /* device [n_seq][n_qh][256], not rotated, 16 B al. */
    const float* gate;              /* device [n_seq][n_qh][256] or NULL                */
    float sm_scale;
    int32_t split_rows;             /* positions per split; 0: the library chooses      */
} kvq_q4_problem;

/* Bytes of workspace kvq_q4_decode needs for this problem (0 if invalid). */
size_t kvq_q4_decode_workspace(const kvq_q4_problem* p);

/*
 *   out        device fp32 [n_seq][n_qh][256]
 *   lse        device fp32 [n_seq][n_qh] or NULL (natural log)
 *   workspace  device, >= kvq_q4_decode_workspace(p) bytes, 256-byte aligned
 *   dev_status device u32 or NULL
 */
int kvq_q4_decode(const kvq_q4_problem* p, float* out, float* lse, void* workspace,
                  size_t ws_bytes, uint32_t* dev_status, kvq_stream_t stream);

/*
 * Cache persistence — colibri PR #399, Commit 1 (".coli_kv v2: quantize-on-upgrade from
 * v1, reject-on-mismatch, self-heal"), Commit 6 (v3: the magic encodes the tier and a
 * header word carries codec << 8 | bits) and the review thread (a cache written under
 * one mode and read under another must be refused, never misread; containers whose
 * byte counts do not add up are refused).  The layout is this library's own:
 *
 *   header  16 little-endian u32 words
 *     w0  magic: 0x3151564B "KVQ1" fp32 rows, 0x3251564B "KVQ2" fp8 tier,
 *                0x3351564B "KVQ3" rotated tier
 *     w1  layout version = 1
 *     w2  d_lat = 512      w3  d_rope = 64
 *     w4  n_rows (low)     w5  n_rows (high)      complete records
 *     w6  format: 0 (fp32 rows), KVQ_FMT_FP8, KVQ_FMT_TQ3, KVQ_FMT_TQ4, KVQ_FMT_TQ6
 *     w7  codec << 8 | bits: (0, 32) fp32, (0, 8) fp8, (1, b) rotated b-bit
 *     w8  record bytes      w9 .. w15  zero
 *   rotated tier: the 16 u32 rotation-sign words
 *   n_rows records, row after row:
 *     fp32     lat f32[512], rope f32[64]                                  (2304 B)
 *     fp8      lat u8[512], lat_scale f32, rope u8[64], rope_scale f32     (584 B)
 *     rotated  lat u8[512 b / 8], radius f32, rope u8[64], rope_scale f32  (264/328/456 B)
 *
 * These calls are synchronous: they synchronize `stream`, move the planes through host
 * memory (they allocate host buffers, never device memory) and return when done.
 */
typedef struct kvq_cache_info {
    int32_t format;           /* w6                                                      */
    int32_t codec, bits;      /* w7                                                      */
    int32_t d_lat, d_rope;
    int64_t n_rows;           /* complete records the header counts                      */
    int64_t record_bytes;
    int64_t trailing_bytes;   /* bytes after those records (an interrupted append)      */
} kvq_cache_info;

/* Read and check a cache file's header (host only).  KVQ_EIO if it cannot be read, is
 * not a cache file, or holds fewer bytes than its header counts. */
int kvq_cache_probe(const char* path, kvq_cache_info* info);

/*
 * Write rows [0, rows) of a quantized cache (format KVQ_FMT_FP8 / TQ3 / TQ4 / TQ6) to
 * `path`, replacing it.  planes: device planes of that format (lat rows of 512 or
 * 512 b / 8 bytes); signs: device u32[16] rotation signs (rotated tiers; else NULL).
 */
int kvq_cache_save(const char* path, int32_t format, const kvq_mla_cache* planes,
                   const uint32_t* signs, int64_t rows, kvq_stream_t stream);

/* Write an fp32 (layout "KVQ1") file of rows: lat device f32 [rows][512], rope device f32
 * [rows][64] — the unquantized cache an upgrade starts from. */
int kvq_cache_save_f32(const char* path, const float* lat, const float* rope, int64_t rows,
                       kvq_stream_t stream);

/*
 * Append rows [row0, row0 + rows) of the planes to a quantized cache file in place.
 * Self-heal: bytes after the header's n_rows records (a record an interrupted append
 * left behind) are cut first; the records are written, then n_rows.  KVQ_EMISMATCH if
 * the file holds another format; KVQ_EIO as for kvq_cache_probe.
 */
int kvq_cache_append(const char* path, int32_t format, const kvq_mla_cache* planes,
                     int64_t row0, int64_t rows, kvq_stream_t stream);

/* Device workspace bytes kvq_cache_load needs to upgrade an fp32 file (0 otherwise
 * suffices for same-format loads). */
size_t kvq_cache_load_workspace(void);

/*
 * Load a cache file under `format` into device planes with room for `capacity` rows
 * (*n_loaded = the file's n_rows):
 *   - the file holds `format` (rotated: the same width and the same signs as `signs`):
 *     its records are copied into the planes;
 *   - the file holds fp32 rows ("KVQ1") and `format` is quantized: quantize on load —
 *     the rows are encoded by kvq_encode_fp8 / kvq_encode_tq (and the rope by
 *     kvq_encode_fp8) through `workspace`; the file is left as it is;
 *   - any other pairing: KVQ_EMISMATCH, nothing written.
 * KVQ_EINVAL if n_rows > capacity; KVQ_EWORKSPACE for an upgrade without
 * kvq_cache_load_workspace() bytes.  Trailing bytes after the n_rows records are
 * ignored (kvq_cache_append cuts them).
 */
int kvq_cache_load(const char* path, int32_t format, const uint32_t* signs,
                   const kvq_mla_cache* planes, int64_t capacity, int64_t* n_loaded,
                   void* workspace, size_t ws_bytes, kvq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif
