// kvq_decode_mma.cu — absorbed-MLA split-T decode for blocks of up to 16 query-heads on
// the warp-level tensor-core instruction (mma.sync m16n8k16, fp16 operands, fp32
// accumulation).
//
// colibri PR #399: per query and head s_t = tau (q_lat . c_t + q_rope . k_rope_t) and
// out = sum_t softmax(s)_t c_t over the latent rows (Commit 2, the kernels that split T: each
// CTA reduces a chunk of rows to (m, l, o), the log-sum-exp combine merges the chunks;
// the sparse (DSA-style) gather restricts the rows to a list of indices; TQ4 rows are scored
// against rot(q) and accumulated in the rotated domain).  Same contract and the same
// partials (m and l in the log2 domain, o unnormalised) as the other decode kernels;
// mla_combine_kernel merges them.
//
// Why a third kernel: with at most 16 heads the contraction per row is small and the
// codes stream at the HBM rate, so converting a code to fp16 must cost a few
// instructions.  Here each code is converted once, straight into the score's B
// fragment register, which is also stored for the context.
//
// Per CTA (256 threads, 8 warps; one sequence, one query, 16 heads, one split), two
// independent groups of four warps take alternate 32-row tiles of the split, each with
// its own staging ring, softmax state and named barriers, so that one group's softmax
// and barriers overlap the other's matrix work; the two states merge at the end.  Per
// group and tile:
//  * rows arrive by cp.async (a contiguous cache: the tile's run of codes piece by
//    piece; paged and sparse caches: 8 threads per row), 2 (fp8) or 4 (TQ4) tiles in flight
//    beside the one being computed; inadmissible rows are zero-filled and flagged;
//  * score  S[16 heads x 32 rows] = Q[16 x 576] C^T: warp q covers all 32 rows and a
//    quarter of the 36 k-steps (latent dims 128 q .. 128 q + 127 and rope dims 16 t +
//    4 q ..); A = the query image (fp16 hi and lo parts, both accumulated into one fp32
//    accumulator), B = the codes of column g's row, converted in registers;
//  * the score also stores the codes it converted into an fp16 copy of the tile's
//    latent rows, so each code is converted once;
//  * the four quarters sum their partial scores through shared memory, each keeping one
//    8-row n-tile; the per-head maximum over the tile is reduced across the group;
//    w = p * scale(row) goes to shared memory as fp16 hi | lo;
//  * context O[16 x 512] += W[16 x 32] C: warp q owns output dims 128 q .. 128 q + 127;
//    B comes from the fp16 tile by transposing matrix loads, A = W hi, then W lo.
// The CTA requests its query before its first tiles and builds the query image (fp16 hi
// | lo, rotated in fp32 for TQ4) while they land; it lets the combine launch early
// (programmatic dependent launch; the combine waits for this grid).
// The split-fp16 operands keep the products exact to ~2^-22 relative, which the 1e-4
// tolerance needs; the codes themselves are exact in fp16.
//
// Shared-memory layouts are chosen so that every fragment load is free of bank
// conflicts: rows inside an 8-row n-tile are permuted (rho below), and the 16-byte
// pieces of a staged row are XOR-swizzled by a function of the row.
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cmath>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int kH = 16;                                   // heads per CTA: M of every MMA
constexpr int kT = 32;                                   // rows per tile
constexpr int kWarps = 8;                                // two groups of four
constexpr int kThreads = kWarps * 32;
constexpr int kGroupThreads = 128;
constexpr int kKSteps = (kDLat + kDRope) / 16;           // 36
constexpr int kQImgBytes = kKSteps * 2 * kH * 16 * 2;    // [k-step][hi, lo][16 heads][16] fp16
constexpr int kPHalfBytes = kH * kT * 2;                 // [16 heads][32 positions] fp16
constexpr int kXBytes = 4 * 3 * 4 * 32 * 4;              // [n-tile][other quarter][4][lane]
constexpr int kRedBytes = 4 * kH * 4;                    // [quarter][head]
constexpr int kF16RowBytes = kDLat * 2;                  // one converted latent row
// per group: fp16 tile | swap area (W shares it, see the loop) | maxima | staging ring
constexpr int kGOffX = kT * kF16RowBytes;
constexpr int kGOffRed = kGOffX + kXBytes;
constexpr int kGOffStage = kGOffRed + kRedBytes;
constexpr int kOffGroups = kQImgBytes;
static_assert(2 * kPHalfBytes <= kXBytes, "W fits in the swap area");
constexpr float kLog2e = 1.4426950408889634f;

// Staged row layout of each tier: the latent codes, then the 64 rope codes, in 16-byte
// pieces; after the rows, one float2 (latent scale, rope scale) and one flag per row.
struct Fp8Rows {
    static constexpr int kRowBytes = 576, kLatChunks = 32, kLatBytes = 512, kStages = 3;   // per group
    static constexpr bool kFp8 = true;
};
struct Tq4Rows {
    static constexpr int kRowBytes = 320, kLatChunks = 16, kLatBytes = 256, kStages = 5;   // per group
    static constexpr bool kFp8 = false;
};
template <class R>
constexpr int stage_bytes() { return kT * R::kRowBytes + kT * 8 + kT * 4; }
constexpr int kStageArea = std::max(Fp8Rows::kStages * stage_bytes<Fp8Rows>(),
                                    Tq4Rows::kStages * stage_bytes<Tq4Rows>());
constexpr int kGroupBytes = kGOffStage + kStageArea;
constexpr int kSmemBytes = kOffGroups + 2 * kGroupBytes;
static_assert(kGOffStage % 16 == 0 && kGroupBytes % 16 == 0 && stage_bytes<Fp8Rows>() % 16 == 0 &&
              stage_bytes<Tq4Rows>() % 16 == 0, "16-byte alignment of the staged rows");
static_assert(kH * kDLat * 4 <= kStageArea, "a group's output fits in its staging ring");
static_assert(kH * (kDLat + kDRope + 4) * 4 <= kGOffStage, "the staged query fits before group 0's ring");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

// Row of column n inside an 8-row n-tile.  With this order the four rows that one
// shared-memory wavefront of the context loads (columns 2t, or 2t + 1, for t = 0..3)
// fall into four different bank groups, as do the row pairs of a score load.
__device__ __forceinline__ int rho(int n) { return (n & 1) ? 4 + ((n >> 1) ^ 1) : (n >> 1); }

// 16-byte piece c of staged row r is stored at piece swz(c, r).
template <class R>
__device__ __forceinline__ int swz(int c, int r)
{
    if (R::kFp8) return c ^ (r & 2);
    return c < R::kLatChunks ? c ^ ((r & 6) ^ ((r >> 1) & 2)) : c;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src, uint32_t bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// the four warps of a group (named barriers 1..4 for group 0, 5..8 for group 1; 0 is
// __syncthreads)
__device__ __forceinline__ void group_barrier(int id)
{
    asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Clear every byte of the form S.1111.111 (an e4m3 NaN, never written by the encoder,
// read as 0): (b & 0x7F) + 1 has bit 7 set exactly for those bytes, and prmt's sign
// mode (selector 8 + i) spreads that bit over byte i.
__device__ __forceinline__ uint32_t e4m3_clear_nan(uint32_t w)
{
    const uint32_t m = prmt((w & 0x7F7F7F7Fu) + 0x01010101u, 0u, 0xBA98u);
    return w & ~m;
}

// two e4m3 codes (the two bytes of the low, or high, 16 bits of w) -> half2 (exact)
__device__ __forceinline__ uint32_t e4m3x2_lo(uint32_t w)
{
    uint32_t r;
    asm("{.reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e4m3x2 %0, l;}" : "=r"(r) : "r"(w));
    return r;
}
__device__ __forceinline__ uint32_t e4m3x2_hi(uint32_t w)
{
    uint32_t r;
    asm("{.reg .b16 l, h; mov.b32 {l, h}, %1; cvt.rn.f16x2.e4m3x2 %0, h;}" : "=r"(r) : "r"(w));
    return r;
}

// TQ4 centroids without a table in memory: the codebook is symmetric (code 15 - k is
// code k negated) with a positive upper half, so code k is +m[k - 8] or -m[7 - k], and
// the bytes of the eight binary16 magnitudes m[j] sit in four constants that byte
// permutes index by j.
constexpr bool tq4_symmetric()
{
    for (int k = 0; k < 8; ++k) {
        if (kTq4CentroidBits[15 - k] != (kTq4CentroidBits[k] ^ 0x8000u)) return false;
        if (kTq4CentroidBits[8 + k] & 0x8000u) return false;
    }
    return true;
}
static_assert(tq4_symmetric(), "the TQ4 codebook must be symmetric");

constexpr uint32_t tq4_mag_bytes(int hi, int part)
{
    uint32_t r = 0;
    for (int b = 0; b < 4; ++b) {
        const uint32_t h = kTq4CentroidBits[8 + 4 * part + b];
        r |= (hi ? (h >> 8) : (h & 0xFFu)) << (8 * b);
    }
    return r;
}

// eight TQ4 codes (code i in nibble i of w) -> h[q] = half2(centroid 2q, centroid 2q + 1)
__device__ __forceinline__ void tq4x8_to_half2(uint32_t w, uint32_t (&h)[4])
{
    constexpr uint32_t kL0 = tq4_mag_bytes(0, 0), kL1 = tq4_mag_bytes(0, 1);
    constexpr uint32_t kH0 = tq4_mag_bytes(1, 0), kH1 = tq4_mag_bytes(1, 1);
    const uint32_t pos = (w >> 3) & 0x11111111u;                        // 1: code >= 8
    const uint32_t j = (w & 0x77777777u) ^ ((pos ^ 0x11111111u) * 7u);  // magnitude index
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint32_t js = j >> (16 * q), ps = pos >> (16 * q);
        const uint32_t lo = prmt(kL0, kL1, js);
        const uint32_t hi = prmt(kH0, kH1, js) | prmt(0x80u, 0u, ps);   // sign bit 0x80
        h[2 * q] = prmt(lo, hi, 0x5140u);
        h[2 * q + 1] = prmt(lo, hi, 0x7362u);
    }
}

struct MmaArgs {
    kvq_mla_problem p;
    int split_rows, n_splits, n_hblk;
    float* part_ml;          // [n_seq][n_q][H][n_splits][2]
    float* part_o;           // [n_seq][n_q][H][n_splits][512]
    uint32_t* status;
};

struct Split {
    int s, q, h0, nh, L, split;
    int64_t r0, r1, lim, qrow;
};

// pool row of candidate j, or -1 when it is not admissible (flags bad indices and pages)
__device__ __forceinline__ int64_t candidate_row(const kvq_mla_problem& p, const kvq_mla_cache& C,
                                                 const Split& sp, int64_t j, bool flag, uint32_t* status)
{
    if (j >= sp.r1) return -1;
    const int64_t tl = p.idx ? (int64_t)p.idx[((int64_t)sp.s * p.n_q + sp.q) * p.top_k + j] : j;
    if (tl < 0 || tl >= sp.L) {
        if (flag && status) atomicOr(status, (unsigned)KVQ_DEV_BAD_INDEX);
        return -1;
    }
    if (tl > sp.lim) return -1;
    int64_t row;
    if (!p.block_table) {
        row = (int64_t)sp.s * p.seq_stride_rows + tl;
    } else {
        const int64_t page = tl / p.page_size;
        const int64_t pid = page < p.max_pages ? (int64_t)p.block_table[(int64_t)sp.s * p.max_pages + page] : -1;
        row = pid < 0 ? -1 : pid * p.page_size + tl % p.page_size;
    }
    if (row < 0 || row >= C.n_rows) {
        if (flag && status) atomicOr(status, (unsigned)KVQ_DEV_BAD_PAGE);
        return -1;
    }
    return row;
}

// ---- query image: block ks = 4 kk + e (kk < 8 latent dims 64 kk.., kk = 8 rope),
// column kap of block ks holds dim 64 kk + 16 (kap % 8 / 2) + 4 e + kap % 2 + 2 (kap / 8),
// the order in which a thread's 4-byte code word feeds its B fragment.  Head h's 32-byte
// row stores its two 16-byte halves swapped when bit 2 of h is set.
//
// The query image of (sequence, query) row sq, heads h0 .. h0 + nh - 1, built into
// shared memory by the CTA in two steps.  (1) Warp w stages heads w and w + 8 (rotated
// sequences: rot(q) = (1/sqrt 512) FWHT_512(s (.) q), in fp32 registers) into an fp32
// copy [16 heads][kQStageLd].  (2) Thread i of item list (k-step, head, column
// pair) writes one 4-byte hi pair and one lo pair of the image: a warp covers 128
// contiguous bytes of one k-step block, free of bank conflicts.
constexpr int kQStageLd = kDLat + kDRope + 4;            // floats per staged head

// This warp's two heads of the query (w and w + 8; zeros past nh) and the rotation signs
// of its lanes, requested at the start of the kernel so that their latency overlaps the
// first tile loads.
struct QRegs {
    float y[2][16];
    float2 r2[2];
    uint32_t signs[16];
};

__device__ __forceinline__ void load_q(QRegs& q, const kvq_mla_problem& p, int64_t sq, int h0, int nh,
                                       bool rotated)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < 16; ++j) q.signs[j] = rotated ? p.tq4_signs[j] : 0u;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int h = warp + 8 * hh;
        const bool ok = h < nh;
        const int64_t r = sq * p.n_heads + h0 + (ok ? h : 0);
#pragma unroll
        for (int j = 0; j < 16; ++j) q.y[hh][j] = ok ? p.q_lat[r * kDLat + j * 32 + lane] : 0.0f;
        q.r2[hh] = ok ? reinterpret_cast<const float2*>(p.q_rope + r * kDRope)[lane] : make_float2(0.0f, 0.0f);
    }
}

__device__ __forceinline__ void build_q_image(uint8_t* s_q, float* s_stage_q, QRegs& q, bool rotated)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t neg = 0;                                // rotation signs of elements j * 32 + lane
#pragma unroll
    for (int j = 0; j < 16; ++j) neg |= ((q.signs[j] >> lane) & 1u) << j;
    const float c512 = tq4_inv_sqrt(kDLat);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int h = warp + 8 * hh;
        float (&y)[16] = q.y[hh];
        if (rotated) {                               // CTA-uniform
#pragma unroll
            for (int j = 0; j < 16; ++j) y[j] = ((neg >> j) & 1u) ? -y[j] : y[j];
            fwht_warp<16>(y, lane);
#pragma unroll
            for (int j = 0; j < 16; ++j) y[j] *= c512;
        }
        float* row = s_stage_q + h * kQStageLd;
#pragma unroll
        for (int j = 0; j < 16; ++j) row[j * 32 + lane] = y[j];
        reinterpret_cast<float2*>(row + kDLat)[lane] = q.r2[hh];
    }
    __syncthreads();
    // item i: column pair m = i % 8 (columns 2m, 2m + 1), head (i / 8) % 16, k-step i / 128
    constexpr int kItems = kKSteps * kH * 8;
    static_assert(kItems % kThreads == 0, "image items per thread");
#pragma unroll 2
    for (int i = tid; i < kItems; i += kThreads) {
        const int m = i & 7, h = (i >> 3) & 15, ks = i >> 7;
        // column 2m of k-step ks = 4 kk + e is dim 64 kk + 16 (m % 4) + 4 e + 2 (m / 4)
        const int d0 = 64 * (ks >> 2) + 16 * (m & 3) + 4 * (ks & 3) + 2 * (m >> 2);
        const float2 v = *reinterpret_cast<const float2*>(s_stage_q + h * kQStageLd + d0);
        const __half2 hi = __floats2half2_rn(v.x, v.y);
        const float2 hf = __half22float2(hi);
        const __half2 lo = __floats2half2_rn(v.x - hf.x, v.y - hf.y);
        const int off = ks * 1024 + h * 32 + (((m >> 2) ^ ((h >> 2) & 1)) << 4) + 4 * (m & 3);
        *reinterpret_cast<__half2*>(s_q + off) = hi;
        *reinterpret_cast<__half2*>(s_q + off + 512) = lo;
    }
}

template <class R>
__device__ __forceinline__ void decode_split(const MmaArgs& a, uint8_t* smem, const Split& sp)
{
    constexpr int kSB = stage_bytes<R>();
    constexpr int kS = R::kStages;
    const kvq_mla_problem& p = a.p;
    const kvq_mla_cache& C = R::kFp8 ? p.fp8 : p.tq4;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = warp >> 2, qq = warp & 3, gt = tid & (kGroupThreads - 1);
    const int g = lane >> 2, t = lane & 3;
    const int bar0 = 1 + 4 * grp;                  // this group's named barriers bar0 .. bar0 + 3
    uint8_t* s_q = smem;
    uint8_t* gbase = smem + kOffGroups + grp * kGroupBytes;
    uint8_t* s_f16 = gbase;
    float* s_x = reinterpret_cast<float*>(gbase + kGOffX);
    uint8_t* s_p = gbase + kGOffX;
    float* s_red = reinterpret_cast<float*>(gbase + kGOffRed);
    uint8_t* s_stage = gbase + kGOffStage;
    const int n_tiles = (int)((sp.r1 - sp.r0 + kT - 1) / kT);
    const int my_tiles = (n_tiles - grp + 1) / 2;  // tiles grp, grp + 2, ...
    const float lat_mul = R::kFp8 ? 1.0f : tq4_inv_sqrt(kDLat);   // TQ4: radius / sqrt(512)

    // ---- loads of this group's k-th tile.  A contiguous cache holds the tile's rows as
    // one run: thread gt copies 16-byte pieces gt, gt + 128, .. of the run's latent and
    // rope codes (a warp request = 512 contiguous bytes), and a row's admissibility is
    // arithmetic.  Paged and sparse caches: thread = (row gt / 8 + 16 pass, pieces
    // gt % 8 + 8 m), a warp request covering 128 contiguous bytes of each of four rows.
    const bool contiguous = !p.block_table && !p.idx;
    const int64_t seq_base = (int64_t)sp.s * p.seq_stride_rows;
    auto issue = [&](int k) {
        uint8_t* st = s_stage + (k % kS) * kSB;
        float* sc = reinterpret_cast<float*>(st + kT * R::kRowBytes);
        int* valid = reinterpret_cast<int*>(st + kT * R::kRowBytes + kT * 8);
        const int64_t j0 = sp.r0 + (int64_t)(grp + 2 * k) * kT;      // first candidate of the tile
        if (contiguous) {
            // row tr is admissible when j0 + tr < r1, <= lim and inside the pool; a row the
            // split asks for past the end of the pool flags a bad page, as per row
            const int64_t want = min(min(sp.r1 - 1, sp.lim), j0 + kT - 1);
            const int64_t last = min(want, C.n_rows - 1 - seq_base);
            const int n_ok = (int)max((int64_t)0, min((int64_t)kT, last - j0 + 1));
            if (gt == 0 && want >= j0 && last < want && a.status) atomicOr(a.status, (unsigned)KVQ_DEV_BAD_PAGE);
            const int64_t row0 = seq_base + j0;
            constexpr int kLatPieces = kT * R::kLatChunks;             // latent pieces of the tile
#pragma unroll
            for (int i = gt; i < kLatPieces; i += kGroupThreads) {
                const int tr = i / R::kLatChunks, c = i % R::kLatChunks;
                const bool ok = tr < n_ok;
                const uint8_t* src = C.lat + (ok ? (row0 + tr) * R::kLatBytes + 16 * c : 0);
                cp_async16(st + tr * R::kRowBytes + 16 * swz<R>(c, tr), src, ok ? 16u : 0u);
            }
            {
                const int tr = gt >> 2, c = gt & 3;                       // rope: 4 pieces a row
                const bool ok = tr < n_ok;
                const uint8_t* src = C.rope + (ok ? (row0 + tr) * kDRope + 16 * c : 0);
                cp_async16(st + tr * R::kRowBytes + 16 * swz<R>(R::kLatChunks + c, tr), src, ok ? 16u : 0u);
            }
            if (gt < 2 * kT) {
                const int tr = gt >> 1;
                const bool ok = tr < n_ok;
                const float* src = (gt & 1) ? C.rope_scale : C.lat_scale;
                cp_async4(sc + gt, src + (ok ? row0 + tr : 0), ok ? 4u : 0u);
                if ((gt & 1) == 0) valid[tr] = ok ? 1 : 0;
            }
            return;
        }
        const int l8 = gt & 7;
#pragma unroll
        for (int pass = 0; pass < kT / 16; ++pass) {
            const int tr = (gt >> 3) + 16 * pass;
            const int64_t row = candidate_row(p, C, sp, j0 + tr, l8 == 0, a.status);
            const bool ok = row >= 0;
            const uint32_t nb = ok ? 16u : 0u;
            const int64_t rr = ok ? row : 0;
            const uint8_t* lat = C.lat + rr * R::kLatBytes;
            const uint8_t* rope = C.rope + rr * kDRope;
            uint8_t* dst = st + tr * R::kRowBytes;
#pragma unroll
            for (int c = l8; c < R::kLatChunks + 4; c += 8) {
                const uint8_t* src = c < R::kLatChunks ? lat + 16 * c : rope + 16 * (c - R::kLatChunks);
                cp_async16(dst + 16 * swz<R>(c, tr), src, nb);
            }
            if (l8 == 0) valid[tr] = ok ? 1 : 0;
            if (l8 == 1) cp_async4(sc + 2 * tr, C.lat_scale + rr, ok ? 4u : 0u);
            if (l8 == 2) cp_async4(sc + 2 * tr + 1, C.rope_scale + rr, ok ? 4u : 0u);
        }
    };

    // ---- the query's loads, the first tiles, then (while they land) the query image
    QRegs qr;
    load_q(qr, p, (int64_t)sp.s * p.n_q + sp.q, sp.h0, sp.nh, !R::kFp8);
#pragma unroll
    for (int k = 0; k < kS - 1; ++k) {
        if (k < my_tiles) issue(k);
        cp_async_commit();
    }
    grid_dependents_launch();                      // the combine may launch; it waits for us
    // staging: group 0's fp16 tile and swap area, unused until its first score
    build_q_image(s_q, reinterpret_cast<float*>(smem + kOffGroups), qr, !R::kFp8);
    __syncthreads();                               // the query image is complete

    // this lane's ldmatrix row: matrix lane / 8 = (heads 0-7 | 8-15) x (columns 0-7 | 8-15)
    const int lm = lane >> 3, lr = lane & 7;
    const int a_head = lr + 8 * (lm & 1);
    const uint32_t q_lane = smem_u32(s_q) + a_head * 32 + (((lm >> 1) ^ ((a_head >> 2) & 1)) << 4);
    // W: [hi, lo][16 heads][32 positions] fp16, 16-byte piece c of head h at c ^ (h / 2 % 4)
    const uint32_t p_lane = smem_u32(s_p) + a_head * (kT * 2);
    const int p_x = (a_head >> 1) & 3;
    // the context's transposed loads: k-slot 8 (lm % 2) + lr of k-step j is tile row
    // 16 j + 8 (lm % 2) + rho(lr)
    const uint32_t f_lane = smem_u32(s_f16) + (8 * (lm & 1) + rho(lr)) * kF16RowBytes;

    const float tau2 = p.sm_scale * kLog2e;
    float m0 = -INFINITY, m1 = -INFINITY;          // running maxima of heads g and g + 8
    float l0 = 0.0f, l1 = 0.0f;                    // this thread's share of the row sums
    float o[16][4];
#pragma unroll
    for (int b = 0; b < 16; ++b) o[b][0] = o[b][1] = o[b][2] = o[b][3] = 0.0f;
    // column g of n-tile n is tile row 8 n + rho(g); the swizzles depend on the row's low
    // three bits only, which rho(g) fixes
    const int rg = rho(g);
    const int cb_rope = R::kLatChunks + (R::kFp8 ? (t ^ (rg & 2)) : t);
    const int lat_x = R::kFp8 ? (rg & 2) : ((rg & 6) ^ ((rg >> 1) & 2));

#pragma unroll 1
    for (int k = 0; k < my_tiles; ++k) {
        cp_async_wait<kS - 2>();
        group_barrier(bar0);                       // tile k visible; tile k - 1 fully used
        if (k + kS - 1 < my_tiles) issue(k + kS - 1);
        cp_async_commit();
        const uint8_t* st = s_stage + (k % kS) * kSB;
        const float2* sc = reinterpret_cast<const float2*>(st + kT * R::kRowBytes);
        const int* valid = reinterpret_cast<const int*>(st + kT * R::kRowBytes + kT * 8);

        // ---------------- score ----------------
        float acc[4][4], accr[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[n][c] = accr[n][c] = 0.0f;
        const uint8_t* brow = st + rg * R::kRowBytes;   // n-tile n: + 8 n rows
        // the rope k-step of this quarter: dims 512 + 16 t + 4 qq .. + 3 of every row
        {
            uint32_t ahi[4], alo[4];
            ldsm_x4(ahi, q_lane + (32 + qq) * 1024);
            ldsm_x4(alo, q_lane + (32 + qq) * 1024 + 512);
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const uint32_t x = e4m3_clear_nan(
                    *reinterpret_cast<const uint32_t*>(brow + 8 * n * R::kRowBytes + 16 * cb_rope + 4 * qq));
                const uint32_t b0 = e4m3x2_lo(x), b1 = e4m3x2_hi(x);
                mma16816(accr[n], ahi, b0, b1);
                mma16816(accr[n], alo, b0, b1);
            }
        }
        // two latent groups of 4 k-steps (64 dims each): groups 2 qq and 2 qq + 1
#pragma unroll
        for (int kk = 2 * qq; kk < 2 * qq + 2; ++kk) {
            uint32_t b[4][4][2];
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const uint8_t* rowp = brow + 8 * n * R::kRowBytes;
                if (R::kFp8) {
                    const uint4 u = *reinterpret_cast<const uint4*>(rowp + 16 * ((4 * kk + t) ^ lat_x));
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t x = e4m3_clear_nan(w[e]);
                        b[n][e][0] = e4m3x2_lo(x);
                        b[n][e][1] = e4m3x2_hi(x);
                    }
                } else {
                    const uint2 u = *reinterpret_cast<const uint2*>(rowp + 16 * ((2 * kk + (t >> 1)) ^ lat_x) + 8 * (t & 1));
                    uint32_t h[4];
                    tq4x8_to_half2(u.x, h);
                    b[n][0][0] = h[0]; b[n][0][1] = h[1]; b[n][1][0] = h[2]; b[n][1][1] = h[3];
                    tq4x8_to_half2(u.y, h);
                    b[n][2][0] = h[0]; b[n][2][1] = h[1]; b[n][3][0] = h[2]; b[n][3][1] = h[3];
                }
            }
            // the converted codes (dims 64 kk + 16 t .. + 15 of each row) go to the fp16
            // tile the context reads: 16-byte piece c of row r at piece c ^ (r % 8)
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                uint8_t* f = s_f16 + (8 * n + rg) * kF16RowBytes;
                *reinterpret_cast<uint4*>(f + (((8 * kk + 2 * t) ^ rg) << 4)) =
                    make_uint4(b[n][0][0], b[n][0][1], b[n][1][0], b[n][1][1]);
                *reinterpret_cast<uint4*>(f + (((8 * kk + 2 * t + 1) ^ rg) << 4)) =
                    make_uint4(b[n][2][0], b[n][2][1], b[n][3][0], b[n][3][1]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int ks = 4 * kk + e;
                uint32_t ahi[4], alo[4];
                ldsm_x4(ahi, q_lane + ks * 1024);
                ldsm_x4(alo, q_lane + ks * 1024 + 512);
#pragma unroll
                for (int n = 0; n < 4; ++n) mma16816(acc[n], ahi, b[n][e][0], b[n][e][1]);
#pragma unroll
                for (int n = 0; n < 4; ++n) mma16816(acc[n], alo, b[n][e][0], b[n][e][1]);
            }
        }

        // scaled partial scores; columns 2t, 2t + 1 of n-tile n are rows ra, rb
        float part[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int ra = 8 * n + rho(2 * t), rb = 8 * n + rho(2 * t + 1);
            const float2 sa = sc[ra], sb = sc[rb];
            const float la = sa.x * lat_mul, lb = sb.x * lat_mul;
            part[n][0] = fmaf(accr[n][0], sa.y, acc[n][0] * la);
            part[n][1] = fmaf(accr[n][1], sb.y, acc[n][1] * lb);
            part[n][2] = fmaf(accr[n][2], sa.y, acc[n][2] * la);
            part[n][3] = fmaf(accr[n][3], sb.y, acc[n][3] * lb);
        }
        // quarter qq keeps n-tile qq; the other three are summed in by their owners.
        // Layout [n-tile][sender among the other three][value][lane].
        float kept[4];
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            if (n == qq) continue;
            const int slot = qq < n ? qq : qq - 1;
#pragma unroll
            for (int c = 0; c < 4; ++c) s_x[((n * 3 + slot) * 4 + c) * 32 + lane] = part[n][c];
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
            kept[c] = qq == 0 ? part[0][c] : qq == 1 ? part[1][c] : qq == 2 ? part[2][c] : part[3][c];
        group_barrier(bar0 + 1);
#pragma unroll
        for (int slot = 0; slot < 3; ++slot) {
#pragma unroll
            for (int c = 0; c < 4; ++c) kept[c] += s_x[((qq * 3 + slot) * 4 + c) * 32 + lane];
        }
        // final scores (log2 domain) of the kept n-tile, -inf for inadmissible rows
        const int ra = 8 * qq + rho(2 * t), rb = 8 * qq + rho(2 * t + 1);
        const bool va = valid[ra] != 0, vb = valid[rb] != 0;
        float sv[4];
        sv[0] = va ? kept[0] * tau2 : -INFINITY;
        sv[1] = vb ? kept[1] * tau2 : -INFINITY;
        sv[2] = va ? kept[2] * tau2 : -INFINITY;
        sv[3] = vb ? kept[3] * tau2 : -INFINITY;
        float x0 = fmaxf(sv[0], sv[1]), x1 = fmaxf(sv[2], sv[3]);
#pragma unroll
        for (int o2 = 1; o2 <= 2; o2 <<= 1) {
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, o2));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, o2));
        }
        if (t == 0) {
            s_red[qq * kH + g] = x0;
            s_red[qq * kH + g + 8] = x1;
        }
        group_barrier(bar0 + 2);
        float t0 = -INFINITY, t1 = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            t0 = fmaxf(t0, s_red[w * kH + g]);
            t1 = fmaxf(t1, s_red[w * kH + g + 8]);
        }
        const float mn0 = fmaxf(m0, t0), mn1 = fmaxf(m1, t1);
        const float al0 = mn0 == -INFINITY ? 1.0f : exp2f(m0 - mn0);
        const float al1 = mn1 == -INFINITY ? 1.0f : exp2f(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        {
            const float wa = sc[ra].x * lat_mul, wb = sc[rb].x * lat_mul;
            float pv[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float m = c < 2 ? mn0 : mn1;
                pv[c] = sv[c] == -INFINITY ? 0.0f : exp2f(sv[c] - m);
            }
            l0 = fmaf(l0, al0, pv[0] + pv[1]);
            l1 = fmaf(l1, al1, pv[2] + pv[3]);
            // w = p * latent scale, as fp16 hi | lo, positions 8 qq + 2t, + 1 (W shares the
            // swap area: every read of the swap values precedes the barrier above)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int head = g + 8 * hh;
                const float w0 = pv[2 * hh] * wa, w1 = pv[2 * hh + 1] * wb;
                const __half2 hi = __floats2half2_rn(w0, w1);
                const float2 hf = __half22float2(hi);
                const __half2 lo = __floats2half2_rn(w0 - hf.x, w1 - hf.y);
                const int off = head * (kT * 2) + ((qq ^ ((head >> 1) & 3)) << 4) + 4 * t;
                *reinterpret_cast<__half2*>(s_p + off) = hi;
                *reinterpret_cast<__half2*>(s_p + kPHalfBytes + off) = lo;
            }
        }
        group_barrier(bar0 + 3);                   // W and the fp16 tile of tile k complete

        // ---------------- context ----------------
#pragma unroll
        for (int b = 0; b < 16; ++b) {
            o[b][0] *= al0;
            o[b][1] *= al0;
            o[b][2] *= al1;
            o[b][3] *= al1;
        }
#pragma unroll
        for (int j = 0; j < kT / 16; ++j) {
            uint32_t whi[4], wlo[4];
            const uint32_t pa = p_lane + (((2 * j + (lm >> 1)) ^ p_x) << 4);
            ldsm_x4(whi, pa);
            ldsm_x4(wlo, pa + kPHalfBytes);
            // B of n-tiles b, b + 1 (dims 128 qq + 8 b ..) from the fp16 tile, transposed:
            // lane = (matrix lm: k-half lm % 2, n-tile b + lm / 2; line lr)
            const uint32_t f_row = f_lane + (16 * j) * kF16RowBytes;
#pragma unroll
            for (int b = 0; b < 16; b += 2) {
                uint32_t bb[4];
                ldsm_x4_trans(bb, f_row + (((16 * qq + b + (lm >> 1)) ^ rho(lr)) << 4));
                mma16816(o[b], whi, bb[0], bb[1]);
                mma16816(o[b + 1], whi, bb[2], bb[3]);
                mma16816(o[b], wlo, bb[0], bb[1]);
                mma16816(o[b + 1], wlo, bb[2], bb[3]);
            }
        }
    }
    cp_async_wait<0>();

    // ---- the group's state: (m, l) per head and o; group 1 hands its state to group 0 ----
#pragma unroll
    for (int o2 = 1; o2 <= 2; o2 <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
    }
    group_barrier(bar0);                           // the group is past its last read of s_red
    if (t == 0) {
        s_red[qq * kH + g] = l0;
        s_red[qq * kH + g + 8] = l1;
    }
    group_barrier(bar0 + 1);
    float lg0 = 0.0f, lg1 = 0.0f;                  // the group's row sums of heads g, g + 8
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        lg0 += s_red[w * kH + g];
        lg1 += s_red[w * kH + g + 8];
    }
    // group 1's o goes to its (now idle) staging ring as [warp][value][lane]
    float* hand = reinterpret_cast<float*>(smem + kOffGroups + kGroupBytes + kGOffStage);
    float* hand_ml = reinterpret_cast<float*>(smem + kOffGroups + kGroupBytes + kGOffRed);
    __syncthreads();                               // group 1's s_red reads are done
    if (grp == 1) {
#pragma unroll
        for (int b = 0; b < 16; ++b)
#pragma unroll
            for (int c = 0; c < 4; ++c) hand[((qq * 16 + b) * 4 + c) * 32 + lane] = o[b][c];
        if (qq == 0 && t == 0) {
            hand_ml[g] = m0;
            hand_ml[g + 8] = m1;
            hand_ml[16 + g] = lg0;
            hand_ml[24 + g] = lg1;
        }
    }
    __syncthreads();
    if (grp == 1) return;
    const float mo0 = hand_ml[g], mo1 = hand_ml[g + 8];
    const float lo0 = hand_ml[16 + g], lo1 = hand_ml[24 + g];
    const float M0 = fmaxf(m0, mo0), M1 = fmaxf(m1, mo1);
    const float a0 = m0 == -INFINITY ? 0.0f : exp2f(m0 - M0), b0 = mo0 == -INFINITY ? 0.0f : exp2f(mo0 - M0);
    const float a1 = m1 == -INFINITY ? 0.0f : exp2f(m1 - M1), b1 = mo1 == -INFINITY ? 0.0f : exp2f(mo1 - M1);
    auto slot = [&](int h) { return (sp.qrow + sp.h0 + h) * a.n_splits + sp.split; };
    if (qq == 0 && t == 0) {
        if (g < sp.nh) {
            a.part_ml[slot(g) * 2] = M0;
            a.part_ml[slot(g) * 2 + 1] = lg0 * a0 + lo0 * b0;
        }
        if (g + 8 < sp.nh) {
            a.part_ml[slot(g + 8) * 2] = M1;
            a.part_ml[slot(g + 8) * 2 + 1] = lg1 * a1 + lo1 * b1;
        }
    }
    // n-tile b, columns 2t, 2t + 1 are dims 128 qq + 8 b + 2t, + 1
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int h = g + 8 * hh;
        if (h >= sp.nh) continue;
        const float wa = hh ? a1 : a0, wb = hh ? b1 : b0;
        float* dst = a.part_o + slot(h) * kDLat + 128 * qq + 2 * t;
#pragma unroll
        for (int b = 0; b < 16; ++b) {
            const float x = o[b][2 * hh] * wa + hand[((qq * 16 + b) * 4 + 2 * hh) * 32 + lane] * wb;
            const float y = o[b][2 * hh + 1] * wa + hand[((qq * 16 + b) * 4 + 2 * hh + 1) * 32 + lane] * wb;
            *reinterpret_cast<float2*>(dst + 8 * b) = make_float2(x, y);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) mla_decode_mma_kernel(MmaArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const kvq_mla_problem& p = a.p;
    Split sp;
    sp.split = blockIdx.x;
    sp.s = blockIdx.y;
    sp.q = blockIdx.z / a.n_hblk;
    sp.h0 = (blockIdx.z % a.n_hblk) * kH;
    sp.nh = min(kH, p.n_heads - sp.h0);
    sp.L = p.seq_len[sp.s];
    const int fmt = p.seq_fmt ? p.seq_fmt[sp.s] : p.fmt;
    const int64_t n_cand = p.idx ? (int64_t)p.top_k : (int64_t)sp.L;
    sp.r0 = (int64_t)sp.split * a.split_rows;
    sp.r1 = min(sp.r0 + (int64_t)a.split_rows, n_cand);
    sp.lim = p.causal ? (int64_t)sp.L - p.n_q + sp.q : (int64_t)sp.L - 1;
    sp.qrow = ((int64_t)sp.s * p.n_q + sp.q) * p.n_heads;
    const bool bad_fmt = fmt != KVQ_FMT_FP8 && fmt != KVQ_FMT_TQ4;
    if (sp.r0 >= n_cand || bad_fmt) {
        if (bad_fmt && threadIdx.x == 0 && sp.split == 0 && a.status)
            atomicOr(a.status, (unsigned)KVQ_DEV_BAD_FORMAT);
        if ((int)threadIdx.x < sp.nh) {
            const int64_t slot = (sp.qrow + sp.h0 + threadIdx.x) * a.n_splits + sp.split;
            a.part_ml[slot * 2] = -INFINITY;
            a.part_ml[slot * 2 + 1] = 0.0f;
        }
        return;
    }
    if (fmt == KVQ_FMT_FP8) decode_split<Fp8Rows>(a, smem, sp);
    else decode_split<Tq4Rows>(a, smem, sp);
}

}  // namespace

int mma_head_block() { return kH; }

void plan_mma_splits(const kvq_mla_problem& p, int64_t n_cand, int64_t& split_rows)
{
    const int64_t units = std::max<int64_t>(1, (int64_t)p.n_seq * p.n_q * ((p.n_heads + kH - 1) / kH));
    // the two warp groups of a CTA take alternate tiles: splits are whole pairs of tiles
    constexpr int kPair = 2 * kT;
    const int64_t tiles = std::max<int64_t>(1, (n_cand + kPair - 1) / kPair);
    int64_t split_tiles;
    const int64_t n_sm = sm_count();
    if (units >= n_sm) {
        split_tiles = std::max<int64_t>(1, (units * tiles + 4 * n_sm - 1) / (4 * n_sm));
    } else {
        const int64_t splits = std::min<int64_t>(tiles, n_sm / units);
        split_tiles = (tiles + splits - 1) / splits;
    }
    split_rows = split_tiles * kPair;
}

cudaError_t launch_mla_decode_mma(const kvq_mla_problem& p, const DecodePlan& plan, float* part_ml, float* part_o, uint32_t* dev_status,
                                  cudaStream_t s)
{
    MmaArgs a;
    a.p = p;
    a.split_rows = plan.split_rows;
    a.n_splits = plan.n_splits;
    a.n_hblk = (p.n_heads + kH - 1) / kH;
    a.part_ml = part_ml;
    a.part_o = part_o;
    a.status = dev_status;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    static std::atomic<uint64_t> attr_set{0};       // one bit per device
    const uint64_t bit = 1ull << (device & 63);
    if (!(attr_set.load() & bit)) {
        e = cudaFuncSetAttribute(mla_decode_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(bit);
    }
    dim3 grid(plan.n_splits, p.n_seq, p.n_q * a.n_hblk);
    mla_decode_mma_kernel<<<grid, kThreads, kSmemBytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kvq
