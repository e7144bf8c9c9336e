/*
 * kvq_oracle.h — declarations of the CPU oracle (TEST INFRASTRUCTURE ONLY).
 *
 * The oracle is a plain, slow, obviously-correct restatement of what the quantized
 * MLA KV-cache path computes.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load it.  It shares no code, header, table or constant
 * with the CUDA library: every rounding rule here is written from the definition of
 * the number format, and every step of a codec from the method's description.
 *
 * Sources (pages, by title and section):
 *   [KV8/TQ]  colibri PR #399 "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant
 *             (KV_TQ) on CPU, CUDA, and Metal" — Summary, Commits 1-2 and 6,
 *             "Why rotated-int4 for the 4-bit tier", Validation, and the review
 *             thread's rebase notes (fp8 bit-math fallback; non-power-of-two refusal;
 *             native TQ4 identities).
 *   [Q4_0]    Strata PR #2533 "metal: q4_0 KV cache on the Mac engine" — the
 *             kv_q4.metal port commit (fwht256, q4_group/q4_store, tie rule, fp16 RNE),
 *             the parity-fixture commit (all-zero group bits) and the qsa decode commit
 *             (dequantization as (nibble - 8) * f32_from_f16(d)).
 *
 * Conventions shared with the library are INTERFACE conventions (byte layouts, the
 * argument meaning) and are restated independently on each side.
 */
#ifndef KVQ_ORACLE_H
#define KVQ_ORACLE_H
#include <stdint.h>

#define ORC_FMT_FP8 1
#define ORC_FMT_TQ4 2
#define ORC_FMT_TQ6 4
#define ORC_FMT_TQ3 5

/* ---- number formats ---------------------------------------------------------- */
double   orc_e4m3_value(uint8_t code);     /* value of an e4m3 code (S.1111.111 reads 0) */
uint8_t  orc_e4m3_rne(float v);            /* round-to-nearest-even, saturate to +-448   */
uint16_t orc_f16_rne(double v);            /* IEEE binary16 round-to-nearest-even        */
double   orc_f16_value(uint16_t h);        /* value of a binary16 pattern                */

/* ---- fp8 (KV8) per-row encode ------------------------------------------------- */
void orc_encode_fp8(const float* x, int64_t rows, int dim, int64_t ldx,
                    uint8_t* codes, int64_t ldc, float* scales);
void orc_decode_fp8(const uint8_t* codes, int64_t rows, int dim, int64_t ldc,
                    const float* scales, double* out);

/* ---- rotated tiers: TQ-b, b = 3, 4, 6 (TQ4 = rotated-int4) --------------------- */
int  orc_tq_codebook(int bits, double* lloyd, float* cb, float* thr, int* iters);
int  orc_encode_tq(int bits, const float* x, int64_t rows, int dim, int64_t ldx,
                   const uint32_t* sign_bits, uint8_t* packed, int64_t ldp, float* radius);
int  orc_decode_tq(int bits, const uint8_t* packed, int64_t rows, int dim, int64_t ldp,
                   const float* radius, const uint32_t* sign_bits, double* xhat, double* yhat);
int  orc_tq4_codebook(double lloyd[16], float cb[16], float thr[15], int* iters);
void orc_fwht_f32(float* w, int n);
void orc_fwht_f64(double* w, int n);
int  orc_encode_tq4(const float* x, int64_t rows, int dim, int64_t ldx,
                    const uint32_t* sign_bits, uint8_t* packed, int64_t ldp,
                    float* radius);
int  orc_decode_tq4(const uint8_t* packed, int64_t rows, int dim, int64_t ldp,
                    const float* radius, const uint32_t* sign_bits,
                    double* xhat, double* yhat);

/* ---- q4_0 paged cache ---------------------------------------------------------- */
void orc_fwht256_q4(const float* x, float* z);
void orc_q4_block(const float* z, uint8_t out[18]);
int  orc_append_q4(const float* k, const float* v, int n_seq, const int32_t* pos0,
                   int n_tok, int n_heads, int head_dim, const int32_t* page_table,
                   int max_pages, int page_size, int64_t n_cells,
                   uint8_t* k_pool, uint8_t* v_pool);
int  orc_gather_q4(const uint8_t* pool, int n_seq, const int32_t* pos0, int n_tok,
                   int n_heads, int head_dim, const int32_t* page_table,
                   int max_pages, int page_size, int64_t n_cells, uint16_t* out);
/* projection producer of the q4_0 append: y = h . w in the library's fixed fp32 order */
void orc_project_rows(const float* h, int64_t rows, int d_model, const void* w, int w_bf16,
                      int64_t n_out, float* y);
int  orc_project_append_q4(const float* h, int n_seq, const int32_t* pos0, int n_tok,
                           int d_model, const void* w_k, const void* w_v, int w_bf16,
                           int n_heads, const int32_t* page_table, int max_pages,
                           int page_size, int64_t n_cells, uint8_t* k_pool, uint8_t* v_pool);

/* ---- absorbed-MLA decode attention, fp64 ---------------------------------------- */
typedef struct orc_mla {
    int32_t n_seq, n_q, n_heads, d_lat, d_rope, causal;
    const int32_t* seq_len;       /* [n_seq] rows held by each sequence                  */
    const int32_t* seq_fmt;       /* [n_seq] ORC_FMT_FP8, _TQ4, _TQ6 or _TQ3 (the rotated
                                     tiers share the tq4_* planes, n*b/8 bytes a row)     */
    const int32_t* block_table;   /* [n_seq][max_pages] pool page ids, or NULL            */
    int32_t max_pages, page_size;
    int64_t seq_stride_rows;      /* without a block table: seq i row t = i*stride + t    */
    const uint8_t* fp8_lat;   const float* fp8_lat_scale;
    const uint8_t* fp8_rope;  const float* fp8_rope_scale;
    const uint8_t* tq4_lat;   const float* tq4_radius;
    const uint8_t* tq4_rope;  const float* tq4_rope_scale;
    const uint32_t* tq4_signs;
    const float* q_lat;           /* [n_seq][n_q][H][d_lat]                               */
    const float* q_rope;          /* [n_seq][n_q][H][d_rope]                              */
    const int32_t* idx;           /* [n_seq][n_q][top_k] absolute row ids, or NULL        */
    int32_t top_k;
    float sm_scale;
    int32_t n_split;              /* 0: direct softmax; >0: split-T partials + combine    */
    int32_t head_lo, head_hi;     /* heads to compute (others untouched)                  */
    const int32_t* seq_sel;       /* optional subset of sequences to compute              */
    int32_t n_sel;
} orc_mla;

int orc_mla_decode(const orc_mla* p, double* out, double* lse, uint32_t* bad_index);

/* ---- q4_0 paged decode attention (GQA, head_dim 256), fp64 ------------------------ */
int orc_q4_decode(int n_seq, int n_qh, int n_kv, const int32_t* seq_len,
                  const int32_t* page_table, int max_pages, int page_size, int64_t n_cells,
                  const uint8_t* k_pool, const uint8_t* v_pool, const float* q,
                  const float* gate, double sm_scale, const int32_t* seq_sel, int n_sel,
                  double* out, double* lse, uint32_t* bad_page);

#endif
