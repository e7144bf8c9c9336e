// kvq_decode_tc.cu — the tensor-core (tcgen05) split-T absorbed-MLA decode.
//
// Same operation as the CUDA-core kernel in kvq_decode.cu (colibri PR #399: score
// s_t = tau (q_lat . c_t + q_rope . k_rope_t), context sum_t softmax(s)_t c_t, split-T
// partials), restated as two dense contractions per tile of 128 rows:
//
//   S^T[rows x heads] = C_tile[rows x 576] . Q^T        (rows on M = 128, heads on N)
//   O^T[dims x heads] += V_tile^T[dims x rows] . W^T     (dims on M, 4 M-tiles of 128)
//
// The codes are exact in fp16 (every e4m3 value; every TQ4 centroid is a binary16
// value), and per-row scales are factored out: the latent and rope scores accumulate
// separately and are scaled per row afterwards; the context weight of row t is
// w = p_t * scale_t.  The fp32 operands q and w are split into fp16 hi + lo halves
// that are stacked along N (N = 64 for 32 heads), so each A tile read serves both
// halves; D accumulates in fp32 in tensor memory.
//
// Every wait is bounded (%globaltimer); a timeout sets KVQ_DEV_TIMEOUT, raises a
// CTA-wide abort flag, drains the MMAs in flight and frees tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <climits>
#include <cstring>
#include <atomic>

#include "kvq_internal.cuh"
#include "kvq_sm100.cuh"
#include "kvq_tc_common.cuh"

namespace kvq {

using namespace sm100;

namespace {

using namespace tc;

constexpr int kRT = 128;                 // rows per tile (MMA M)
constexpr int kGQ = 32;                  // query-heads per CTA
constexpr int kN = 2 * kGQ;              // MMA N: hi | lo stacked
constexpr int kChunkBytes = kRT * 128;   // [128 rows x 64 fp16], 128B-swizzled
constexpr int kQSlabBytes = kN * 128;    // [64 rows x 64 fp16]
constexpr int kQBytes = 9 * kQSlabBytes; // 72 KB
constexpr int kPBytes = kRT * 128;       // [128 rows x 64 fp16] MN-major
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.0f;            // rescale only when the max grows by > 2^8
constexpr uint64_t kTimeoutNs = kDefaultWaitNs;   // drains

// TMEM columns
constexpr uint32_t kColO = 256;      // O^T M-tile m at 256 + 64m

struct TcArgs {
    // tensor maps of the code planes ([0] fp8 tier, [1] TQ4 tier), used when use_tma
    CUtensorMap tm_lat[2], tm_rope[2];
    int use_tma;                         // contiguous rows: chunks arrive by TMA
    kvq_mla_problem p;
    int split_rows, n_splits, n_hg;      // n_hg: head groups of 32
    int fmt_split;                       // skip fp8 sequences (the e4m3 kernel reads them)
    const float* q_rot;                  // [n_seq][n_q][H][512] (TQ4 sequences)
    uint8_t* q_img;                      // [n_seq][n_q][n_hg][kQBytes]
    float* part_ml;
    float* part_o;
    uint32_t* status;
    uint64_t wait_ns;                    // limit of the pipeline waits
    int premix;                          // TQ4 rows: partials carry stages h = 128, 256
};

// Q image of 32-head groups (see build_q_image): [9 slabs][64 rows][128 B], 72 KB.
__global__ void __launch_bounds__(256) q_image_kernel(TcArgs a)
{
    grid_dependents_launch();                    // the decode may start loading codes
    build_q_image<kGQ>(a.p, a.n_hg, a.q_img);
}

// ====================================================================================
// The decode kernel.
//  * Roles (512 threads): warps 0-7 are two producer sets of four warps (thread = row)
//    that convert alternate chunks of codes to fp16, so two chains of ring waits,
//    stores and arrivals run at once and every warp scheduler holds one warp of each
//    set; warps 8-11 run the softmax (thread = row) and the epilogue (thread = output
//    dim); warp 12 allocates tensor memory and issues the score MMAs, warp 15 the
//    context MMAs, each from one elected lane (two issuing warps on two schedulers, so
//    neither chain of waits and issues queues behind the other); warps 13 and 14 load
//    code chunks by TMA for producer sets 0 and 1 (contiguous caches).
//  * Order of work, common to producers, loaders and MMA issuers: per step i, the 9
//    score chunks of tile i (8 latent, 1 rope) if i < NT, then the 8 latent context
//    chunks of tile i-1.  Score chunks go to tensor memory (thread = row = TMEM lane)
//    and are read from there by the MMA; context chunks go to a shared-memory ring,
//    the two chunks of an M-tile in adjacent slots.
//  * Raw codes: contiguous caches stream [128 rows x 32 or 64 bytes] boxes by TMA
//    into the owning set's stages; paged and sparse caches copy each row's 16-byte
//    pieces with cp.async.  Either way a set's next kStages chunks are in flight.
//  * TQ4 codes decode without a table in memory: the codebook is symmetric, so code k
//    is +m[k - 8] (k >= 8) or -m[7 - k], and the bytes of the 8 binary16 magnitudes
//    m[j] sit in four registers that byte permutes (prmt) index by j.
//  * The per-head maximum over a tile's rows is a transposing butterfly (31 shuffles
//    per warp); the running maxima live in shared memory, and the row sums of p are
//    reduced the same way into one register per lane.
//  * W (the context operand) is single-buffered: the softmax writes W(i) only after
//    the context MMAs of tile i-1, which read W(i-1), have completed.
//  * The Q image arrives by one bulk asynchronous copy while the first codes load.
// TMEM: S lat 0..63, S rope 64..127, score-A ring 4 x 32 columns at 128.., O^T 256..511.
// ====================================================================================
constexpr int kRingA = 4;                // TMEM score-A slots (32 columns each)
constexpr int kRingC = 4;                // shared-memory context slots (pairs adjacent)
constexpr int kStages = 4;               // raw-code stages in flight per producer set
constexpr int kStageBytes = kRT * 64;    // one chunk of raw codes, [4 pieces][128 rows][16 B]
constexpr uint32_t kColA = 128;
constexpr int kThreads = 512;           // 8 producer, 4 softmax, 2 MMA and 2 loader warps
constexpr int kOffQ = 0;
constexpr int kOffRing = kOffQ + kQBytes;
constexpr int kOffP = kOffRing + kRingC * kChunkBytes;
constexpr int kOffStage = kOffP + kPBytes;
constexpr int kOffRed = kOffStage + 2 * kStages * kStageBytes;   // [4][32] f32
constexpr int kOffM = kOffRed + 4 * 32 * 4;             // [32] running maxima
constexpr int kOffAlpha = kOffM + 32 * 4;               // [32] rescale factors
constexpr int kOffFlag = kOffAlpha + 32 * 4;            // some head rescales O
constexpr int kOffBar = kOffFlag + 16;
// full_a[4], empty_a[4], full_c[4], empty_c[4], s_full, s_empty, p_full, o_done, drain,
// q_full, raw_full[2][kStages], raw_empty[2][kStages], drain_c
constexpr int kNumBars = 2 * kRingA + 2 * kRingC + 6 + 4 * kStages + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

struct Shared {
    uint8_t* base;
    __device__ uint8_t* q() const { return base + kOffQ; }
    __device__ uint8_t* slot(int i) const { return base + kOffRing + i * kChunkBytes; }
    __device__ uint8_t* pbuf() const { return base + kOffP; }
    __device__ uint8_t* stage(int set, int d) const { return base + kOffStage + (set * kStages + d) * kStageBytes; }
    __device__ float* red() const { return reinterpret_cast<float*>(base + kOffRed); }
    __device__ float* m_run() const { return reinterpret_cast<float*>(base + kOffM); }
    __device__ float* alpha() const { return reinterpret_cast<float*>(base + kOffAlpha); }
    __device__ volatile int* flag() const { return reinterpret_cast<volatile int*>(base + kOffFlag); }
    __device__ uint64_t* bar(int i) const { return reinterpret_cast<uint64_t*>(base + kOffBar) + i; }
    __device__ uint64_t* full_a(int i) const { return bar(i); }
    __device__ uint64_t* empty_a(int i) const { return bar(kRingA + i); }
    __device__ uint64_t* full_c(int i) const { return bar(2 * kRingA + i); }
    __device__ uint64_t* empty_c(int i) const { return bar(2 * kRingA + kRingC + i); }
    __device__ uint64_t* s_full() const { return bar(2 * kRingA + 2 * kRingC); }
    __device__ uint64_t* s_empty() const { return bar(2 * kRingA + 2 * kRingC + 1); }
    __device__ uint64_t* p_full() const { return bar(2 * kRingA + 2 * kRingC + 2); }
    __device__ uint64_t* o_done() const { return bar(2 * kRingA + 2 * kRingC + 3); }
    __device__ uint64_t* drain() const { return bar(2 * kRingA + 2 * kRingC + 4); }
    __device__ uint64_t* q_full() const { return bar(2 * kRingA + 2 * kRingC + 5); }
    __device__ uint64_t* raw_full(int set, int d) const { return bar(2 * kRingA + 2 * kRingC + 6 + set * kStages + d); }
    __device__ uint64_t* raw_empty(int set, int d) const { return bar(2 * kRingA + 2 * kRingC + 6 + 2 * kStages + set * kStages + d); }
    __device__ uint64_t* drain_c() const { return bar(2 * kRingA + 2 * kRingC + 6 + 4 * kStages); }
    __device__ uint32_t* tmem_base() const { return reinterpret_cast<uint32_t*>(base + kOffMisc); }
    __device__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(base + kOffMisc + 4); }
};

__device__ __forceinline__ bool wait_bar(const Shared& sh, uint64_t* bar, uint32_t parity,
                                          uint32_t* status, uint64_t limit_ns)
{
    // try_wait may sleep inside the instruction until the phase completes, which hides a
    // deadline shorter than its sleep; a short limit (set only to exercise this path)
    // therefore polls with the non-blocking test and reads the timer on every pass
    const bool poll = limit_ns < 100000;
    if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!(poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity))) {
        if (*sh.abort_flag()) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *sh.abort_flag() = 1;
            if (status) atomicOr(status, (unsigned)KVQ_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void named_bar_softmax() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Item j of a producer set that converts the chunks of parity `par` (NS = its score
// chunks per tile: 5 for parity 0 of ch = 0..8, 4 for parity 1).  The common order is,
// per step i: S(i) chunks 0..8 if i < NT, then C(i-1) latent chunks 0..7 if i >= 1.
struct OwnItem {
    int tile, ch;
    bool score;
};

template <int NS>
__device__ __forceinline__ int own_count(int NT) { return NS + (NT - 1) * (NS + 4) + 4; }

// position n of the common order
__device__ __forceinline__ OwnItem common_item(int n, int NT)
{
    OwnItem o;
    if (n < 9) {
        o.tile = 0; o.ch = n; o.score = true;
        return o;
    }
    const int m = n - 9, i = 1 + m / 17, j = m - (m / 17) * 17;
    if (i < NT && j < 9) {
        o.tile = i; o.ch = j; o.score = true;
    } else {
        o.tile = i - 1; o.ch = i < NT ? j - 9 : j; o.score = false;
    }
    return o;
}

template <int NS>
__device__ __forceinline__ OwnItem own_item(int j, int par, int NT)
{
    OwnItem o;
    if (j < NS) {
        o.tile = 0; o.ch = 2 * j + par; o.score = true;
        return o;
    }
    constexpr int B = NS + 4;
    const int jj = j - NS, i = 1 + jj / B, r = jj - (jj / B) * B;
    if (i < NT && r < NS) {
        o.tile = i; o.ch = 2 * r + par; o.score = true;
    } else {
        o.tile = i - 1; o.ch = 2 * (i < NT ? r - NS : r) + par; o.score = false;
    }
    return o;
}

// 15 warps: warp w runs on sub-partition w % 4, so sub-partitions 0-2 hold four warps
// each and their 16K registers cap every thread at 128
__global__ void __maxnreg__(128) mla_decode_tc_kernel(const __grid_constant__ TcArgs a)
{
    extern __shared__ uint8_t dsm[];
    Shared sh{reinterpret_cast<uint8_t*>(((uintptr_t)dsm + 1023) & ~(uintptr_t)1023)};
    const kvq_mla_problem& p = a.p;
    const int split = blockIdx.x, s = blockIdx.y;
    const int q = blockIdx.z / a.n_hg, hg = blockIdx.z % a.n_hg;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h0 = hg * kGQ;
    const int nh = min(kGQ, p.n_heads - h0);
    const int L = p.seq_len[s];
    const int fmt = seq_fmt_of(p, s);
    const int64_t n_cand = p.idx ? (int64_t)p.top_k : (int64_t)L;
    const int64_t r0 = (int64_t)split * a.split_rows;
    const int64_t r1 = min(r0 + (int64_t)a.split_rows, n_cand);
    const int64_t qrow = ((int64_t)s * p.n_q + q) * p.n_heads;
    const bool bad_fmt = fmt != KVQ_FMT_FP8 && fmt != KVQ_FMT_TQ4;
    grid_dependents_launch();                    // the combine may start launching
    if (fmt == KVQ_FMT_FP8 && a.fmt_split) return;   // the e4m3 kernel writes these partials

    if (r0 >= n_cand || bad_fmt) {
        if (bad_fmt && tid == 0 && split == 0 && a.status) atomicOr(a.status, (unsigned)KVQ_DEV_BAD_FORMAT);
        if (tid < nh) {
            const int64_t sl = (qrow + h0 + tid) * a.n_splits + split;
            a.part_ml[sl * 2] = -INFINITY;
            a.part_ml[sl * 2 + 1] = 0.0f;
        }
        return;
    }
    const bool tq4 = fmt == KVQ_FMT_TQ4;
    const kvq_mla_cache& C = tq4 ? p.tq4 : p.fp8;
    const int NT = (int)((r1 - r0 + kRT - 1) / kRT);
    const RowCtx rc{&p, s, q, L, r1, p.causal ? (int64_t)L - p.n_q + q : (int64_t)L - 1, &C, a.status};
    // Contiguous rows: each loader sets up its set's stage barriers and requests the set's
    // first kStages chunks before the CTA-wide setup below (tensor memory, the other
    // barriers), which would otherwise delay the first loads.
    const bool pre = a.use_tma != 0;
    if ((warp == 13 || warp == 14) && pre && lane == 0) {
        const int set = warp - 13;
        for (int d = 0; d < kStages; ++d) {
            mbar_init(sh.raw_full(set, d), 1);
            mbar_init(sh.raw_empty(set, d), 4);       // one per warp of the set
        }
        fence_mbar_init();
        const int64_t row0 = (int64_t)s * p.seq_stride_rows + r0;
        int j = 0;
        for (int n = 0; n < 17 * NT && j < kStages; ++n) {
            const OwnItem it = common_item(n, NT);
            if ((it.ch & 1) != set) continue;
            const bool rope = it.ch == 8;
            const int inner = (rope || !tq4) ? 64 : 32;
            mbar_arrive_expect_tx(sh.raw_full(set, j), (uint32_t)(inner * kRT));
            tma_load_2d(sh.stage(set, j), rope ? &a.tm_rope[tq4 ? 1 : 0] : &a.tm_lat[tq4 ? 1 : 0],
                        rope ? 0 : it.ch * inner, (int)(row0 + (int64_t)it.tile * kRT), sh.raw_full(set, j));
            ++j;
        }
    }

    if (warp == 12) {
        if (lane == 0) {
            for (int i = 0; i < kRingA; ++i) {
                mbar_init(sh.full_a(i), 4);          // one arrival per warp of the owning set
                mbar_init(sh.empty_a(i), 1);
            }
            for (int i = 0; i < kRingC; ++i) {
                mbar_init(sh.full_c(i), 4);
                mbar_init(sh.empty_c(i), 1);
            }
            mbar_init(sh.s_full(), 1);
            mbar_init(sh.s_empty(), 4);              // one arrival per softmax warp
            mbar_init(sh.p_full(), 4);
            mbar_init(sh.o_done(), 1);
            mbar_init(sh.drain(), 1);
            mbar_init(sh.drain_c(), 1);
            mbar_init(sh.q_full(), 1);
            for (int i = 0; i < 2 * kStages && !pre; ++i) {
                mbar_init(sh.raw_full(i / kStages, i % kStages), 1);
                mbar_init(sh.raw_empty(i / kStages, i % kStages), 4);   // one per warp of the set
            }
            *sh.abort_flag() = 0;
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(sh.tmem_base(), 512);
        tmem_relinquish();
    }
    if (tid < kGQ) sh.m_run()[tid] = -INFINITY;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sh.tmem_base();
    const int n_items = 17 * NT;

    if (warp < 8) {
        // ================================ producers ======================================
        // Two sets of four warps (thread = row).  Set k converts the chunks of parity k
        // (score chunks ch = k, k + 2, ..; context chunks c = k, k + 2, ..) in the common
        // order into ring slots that only it writes: score-A slots k and k + 2, context
        // slots k, k + 2, k + 4, so the two chunks of a context M-tile sit in adjacent
        // slots.  The two sets' chains of waits, stores and arrivals overlap.
        const int set = warp >> 2;
        const int t = (warp & 3) * 32 + lane;             // row within the tile
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int n_own = set == 0 ? own_count<5>(NT) : own_count<4>(NT);
        int64_t row_c0 = -1, row_c1 = -1;                 // rows of the last two tiles
        int tile_c0 = -1, tile_c1 = -1;
        // stage d holds piece p of row t at (p * 128 + t) * 16: conflict-free reads
        auto issue = [&](int j) {
            if (j < n_own) {
                const OwnItem it = set == 0 ? own_item<5>(j, 0, NT) : own_item<4>(j, 1, NT);
                int64_t row;
                if (it.tile == tile_c0) row = row_c0;
                else if (it.tile == tile_c1) row = row_c1;
                else {
                    row = rc.row(r0 + (int64_t)it.tile * kRT + t, false);
                    if (it.tile & 1) { tile_c1 = it.tile; row_c1 = row; }
                    else { tile_c0 = it.tile; row_c0 = row; }
                }
                const bool fp8 = it.ch == 8 || !tq4;
                const uint8_t* src = row < 0 ? C.rope
                                   : it.ch == 8 ? C.rope + row * kDRope
                                   : tq4 ? C.lat + row * (kDLat / 2) + it.ch * 32
                                         : C.lat + row * kDLat + it.ch * 64;
                const uint32_t nb = row < 0 ? 0u : 16u;      // invalid rows read as zeros
                uint8_t* st = sh.stage(set, j % kStages) + t * 16;
                cp_async16(st, src, nb);
                cp_async16(st + kRT * 16, src + 16, nb);
                if (fp8) {
                    cp_async16(st + 2 * kRT * 16, src + 32, nb);
                    cp_async16(st + 3 * kRT * 16, src + 48, nb);
                }
            }
            cp_async_commit();                            // one group per item, maybe empty
        };
        const bool tma = a.use_tma != 0;
        if (!tma) {
#pragma unroll
            for (int d = 0; d < kStages; ++d) issue(d);
        }
        int a_ord = 0, c_ord = 0;
        bool ok = true;
        for (int j = 0; j < n_own && ok; ++j) {
            const OwnItem it = set == 0 ? own_item<5>(j, 0, NT) : own_item<4>(j, 1, NT);
            const bool fp8 = it.ch == 8 || !tq4;
            uint4 raw[4];
            if (tma) {
                // the loader's box: row t at t * (bytes per row of the chunk), its 16-byte
                // pieces swizzled (64-byte rows: piece i at i ^ ((t >> 1) & 3); 32-byte rows:
                // i ^ ((t >> 2) & 1)) so that the rows a quarter-warp reads share no bank
                const int d = j % kStages;
                ok = __all_sync(kFull, wait_bar(sh, sh.raw_full(set, d), (uint32_t)(j / kStages) & 1u, a.status, a.wait_ns));
                if (!ok) break;
                const uint8_t* st = sh.stage(set, d) + t * (fp8 ? 64 : 32);
                if (fp8) {
                    const int x = (t >> 1) & 3;
#pragma unroll
                    for (int i = 0; i < 4; ++i) raw[i] = *reinterpret_cast<const uint4*>(st + 16 * (i ^ x));
                } else {
                    const int x = (t >> 2) & 1;
                    raw[0] = *reinterpret_cast<const uint4*>(st + 16 * x);
                    raw[1] = *reinterpret_cast<const uint4*>(st + 16 * (1 ^ x));
                    raw[2] = make_uint4(0u, 0u, 0u, 0u);
                    raw[3] = make_uint4(0u, 0u, 0u, 0u);
                }
            } else {
                cp_async_wait<kStages - 1>();             // item j's group has landed
                const uint8_t* st = sh.stage(set, j % kStages) + t * 16;
                raw[0] = *reinterpret_cast<const uint4*>(st);
                raw[1] = *reinterpret_cast<const uint4*>(st + kRT * 16);
                raw[2] = fp8 ? *reinterpret_cast<const uint4*>(st + 2 * kRT * 16) : make_uint4(0u, 0u, 0u, 0u);
                raw[3] = fp8 ? *reinterpret_cast<const uint4*>(st + 3 * kRT * 16) : make_uint4(0u, 0u, 0u, 0u);
                issue(j + kStages);                       // refills the stage just read
            }
            uint32_t h[32];
            codes_to_half(raw, 0, fp8, *reinterpret_cast<uint32_t(*)[16]>(h));
            codes_to_half(raw, 1, fp8, *reinterpret_cast<uint32_t(*)[16]>(h + 16));
            if (tma) {
                // the stage is released once every lane's reads of it have been consumed
                __syncwarp();
                if (lane == 0) mbar_arrive(sh.raw_empty(set, j % kStages));
            }
            if (it.score) {
                const int slot = set + 2 * (a_ord & 1);
                ok = wait_bar(sh, sh.empty_a(slot), ((uint32_t)(a_ord >> 1) & 1u) ^ 1u, a.status, a.wait_ns);
                ok = __all_sync(kFull, ok);
                if (!ok) break;
                tc_fence_after();
                tmem_st_x32(tmem + lane_base + kColA + 32 * slot, h);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sh.full_a(slot));
                ++a_ord;
            } else {
                const int slot = 2 * (c_ord & 1) + set;
                ok = wait_bar(sh, sh.empty_c(slot), ((uint32_t)(c_ord >> 1) & 1u) ^ 1u, a.status, a.wait_ns);
                ok = __all_sync(kFull, ok);
                if (!ok) break;
                uint8_t* dst = sh.slot(slot);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(dst + sw128(t, c)) =
                        make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(sh.full_c(slot));
                ++c_ord;
            }
        }
        cp_async_wait_all();                              // nothing lands after the CTA ends
    } else if (warp < 12) {
        // ================================ softmax ========================================
        // Control flow is identical in all 128 threads (the named barriers need every one
        // of them); `ok` only guards work and is kept warp-uniform.
        const int t = tid - 256;                      // row within the tile
        const int wq = warp - 8;                      // TMEM lane quarter
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        const float tau2 = p.sm_scale * kLog2e;
        const float c512 = tq4_inv_sqrt(kDLat);
        float* red = sh.red();
        float* m_s = sh.m_run();
        float* alpha_s = sh.alpha();
        float l_lane = 0.0f;                          // sum of p over this warp's rows, head `lane`
        bool ok = true;
        for (int i = 0; i < NT; ++i) {
            const int64_t row = rc.row(r0 + (int64_t)i * kRT + t, true);
            float sc_lat = 0.0f, sc_rope = 0.0f;
            if (row >= 0) {
                sc_lat = tq4 ? C.lat_scale[row] * c512 : C.lat_scale[row];
                sc_rope = C.rope_scale[row];
            }
            if (ok) ok = wait_bar(sh, sh.s_full(), (uint32_t)i & 1u, a.status, a.wait_ns);
            ok = __all_sync(kFull, ok);
            float sv[kGQ];
#pragma unroll
            for (int g = 0; g < kGQ; ++g) sv[g] = 0.0f;
            if (ok) {
                tc_fence_after();
                uint32_t x[16], y[16];
#pragma unroll
                for (int c = 0; c < kN; c += 16) {
                    tmem_ld_x16(tmem + lane_base + c, x);
                    tmem_ld_x16(tmem + lane_base + 64 + c, y);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        sv[(c + e) & (kGQ - 1)] += fmaf(sc_lat, __uint_as_float(x[e]),
                                                        sc_rope * __uint_as_float(y[e]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sh.s_empty());
            }
#pragma unroll
            for (int g = 0; g < kGQ; ++g) sv[g] = (row >= 0 && ok) ? sv[g] * tau2 : -INFINITY;
            {
                float mx[kGQ];
#pragma unroll
                for (int g = 0; g < kGQ; ++g) mx[g] = sv[g];
                warp_reduce_transpose<true>(mx, lane);
                red[wq * 32 + lane] = mx[0];
            }
            named_bar_softmax();
            if (wq == 0) {
                const float tm = fmaxf(fmaxf(red[lane], red[32 + lane]), fmaxf(red[64 + lane], red[96 + lane]));
                const float mo = m_s[lane];
                float al = 1.0f;
                bool resc = false;
                if (tm > mo + kLazy || (mo == -INFINITY && tm > -INFINITY)) {
                    al = (mo == -INFINITY) ? 0.0f : exp2f(mo - tm);
                    m_s[lane] = tm;
                    resc = i > 0;
                }
                alpha_s[lane] = al;
                const bool any = __any_sync(kFull, resc);
                if (lane == 0) *sh.flag() = any ? 1 : 0;
            }
            named_bar_softmax();
            const bool need_rescale = *sh.flag() != 0;
            // Consume o_done's phase i-1 (the context MMAs of tile i-1) at every tile,
            // so that this wait and the epilogue's never trail the barrier by more than
            // one phase (a parity wait cannot tell phase k from phase k+2); it also
            // makes O safe to rescale.
            if (i > 0 && ok) ok = wait_bar(sh, sh.o_done(), (uint32_t)(i - 1) & 1u, a.status, a.wait_ns);
            ok = __all_sync(kFull, ok);
            if (need_rescale) {
                l_lane *= alpha_s[lane];
                if (ok) {
                    tc_fence_after();
#pragma unroll 1
                    for (int m = 0; m < 4; ++m) {
#pragma unroll 1
                        for (int c = 0; c < kN; c += 16) {
                            uint32_t x[16];
                            tmem_ld_x16(tmem + lane_base + kColO + 64 * m + c, x);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 16; e += 4) {
                                const float4 al = *reinterpret_cast<const float4*>(alpha_s + ((c + e) & (kGQ - 1)));
                                x[e] = __float_as_uint(__uint_as_float(x[e]) * al.x);
                                x[e + 1] = __float_as_uint(__uint_as_float(x[e + 1]) * al.y);
                                x[e + 2] = __float_as_uint(__uint_as_float(x[e + 2]) * al.z);
                                x[e + 3] = __float_as_uint(__uint_as_float(x[e + 3]) * al.w);
                            }
                            tmem_st_x16(tmem + lane_base + kColO + 64 * m + c, x);
                        }
                    }
                    tmem_st_wait();
                }
            }
            // weights: p = 2^(s - m), w = p * latent scale, split hi | lo
            uint32_t wh[kGQ / 2], wl[kGQ / 2];
#pragma unroll
            for (int g = 0; g < kGQ; g += 4) {
                const float4 mv = *reinterpret_cast<const float4*>(m_s + g);
                const float mm[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const float p0 = sv[g + e] == -INFINITY ? 0.0f : exp2f(sv[g + e] - mm[e]);
                    const float p1 = sv[g + e + 1] == -INFINITY ? 0.0f : exp2f(sv[g + e + 1] - mm[e + 1]);
                    sv[g + e] = p0;
                    sv[g + e + 1] = p1;
                    const float w0 = p0 * sc_lat, w1 = p1 * sc_lat;
                    const __half2 hi = __floats2half2_rn(w0, w1);
                    const float2 hf = __half22float2(hi);
                    const __half2 lo = __floats2half2_rn(w0 - hf.x, w1 - hf.y);
                    wh[(g + e) / 2] = *reinterpret_cast<const uint32_t*>(&hi);
                    wl[(g + e) / 2] = *reinterpret_cast<const uint32_t*>(&lo);
                }
            }
            // W of tile i-1 was consumed by the context MMAs that o_done(i-1) covers
            if (ok) {
                uint8_t* pb = sh.pbuf();
                // row t of W^T: 64 fp16, chunks 0..3 the hi halves, 4..7 the lo halves
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    *reinterpret_cast<uint4*>(pb + sw128(t, c)) =
                        make_uint4(wh[4 * c], wh[4 * c + 1], wh[4 * c + 2], wh[4 * c + 3]);
                    *reinterpret_cast<uint4*>(pb + sw128(t, c + 4)) =
                        make_uint4(wl[4 * c], wl[4 * c + 1], wl[4 * c + 2], wl[4 * c + 3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(sh.p_full());
            }
            warp_reduce_transpose<false>(sv, lane);
            l_lane += sv[0];
        }
        // ---- epilogue: l over the 128 rows, O^T -> partials ------------------------------
        if (ok) ok = wait_bar(sh, sh.o_done(), (uint32_t)(NT - 1) & 1u, a.status, a.wait_ns);
        ok = __all_sync(kFull, ok);
        red[wq * 32 + lane] = l_lane;
        named_bar_softmax();
        // every wait that can give up lies before o_done(NT - 1): a CTA whose pipeline
        // completed has no abort flag, and one that gave up (anywhere) poisons its partial
        if (*sh.abort_flag()) {
            if (t < nh) {
                const int64_t sl = (qrow + h0 + t) * a.n_splits + split;
                a.part_ml[sl * 2] = INFINITY;
                a.part_ml[sl * 2 + 1] = INFINITY;
            }
        } else if (ok) {
            tc_fence_after();
            if (t < nh) {
                const float lt = red[t] + red[32 + t] + red[64 + t] + red[96 + t];
                const int64_t sl = (qrow + h0 + t) * a.n_splits + split;
                a.part_ml[sl * 2] = m_s[t];
                a.part_ml[sl * 2 + 1] = lt;
            }
            // Premixed TQ4 rows: eight heads at a time, all four M-tiles (dims 128 m + 32 wq
            // + lane) of each, with the unrotation's stages h = 128 and 256, which mix the
            // M-tiles; the combine does the rest.  Otherwise M-tile by M-tile.
#pragma unroll 1
            for (int hb = 0; hb < kGQ && a.premix && tq4; hb += 8) {
                uint32_t x[4][8], y[4][8];           // every load issued, then one wait
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    tmem_ld_x8(tmem + lane_base + kColO + 64 * m + hb, x[m]);
                    tmem_ld_x8(tmem + lane_base + kColO + 64 * m + kGQ + hb, y[m]);
                }
                tmem_ld_wait();
                float v[4][8];
#pragma unroll
                for (int m = 0; m < 4; ++m)
#pragma unroll
                    for (int g = 0; g < 8; ++g) v[m][g] = __uint_as_float(x[m][g]) + __uint_as_float(y[m][g]);
                {
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        const float a0 = v[0][g] + v[1][g], a1 = v[0][g] - v[1][g];    // h = 128
                        const float a2 = v[2][g] + v[3][g], a3 = v[2][g] - v[3][g];
                        v[0][g] = a0 + a2;                                             // h = 256
                        v[2][g] = a0 - a2;
                        v[1][g] = a1 + a3;
                        v[3][g] = a1 - a3;
                    }
                }
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int d = 128 * m + 32 * wq + lane;
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        if (hb + g < nh)
                            a.part_o[((qrow + h0 + hb + g) * a.n_splits + split) * kDLat + d] = v[m][g];
                }
            }
#pragma unroll 1
            for (int m = 0; m < 4 && !(a.premix && tq4); ++m) {
                const int d = 128 * m + 32 * wq + lane;
                uint32_t x[16], y[16];
#pragma unroll
                for (int c = 0; c < kGQ; c += 16) {
                    tmem_ld_x16(tmem + lane_base + kColO + 64 * m + c, x);
                    tmem_ld_x16(tmem + lane_base + kColO + 64 * m + kGQ + c, y);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int g = c + e;
                        if (g < nh)
                            a.part_o[((qrow + h0 + g) * a.n_splits + split) * kDLat + d] =
                                __uint_as_float(x[e]) + __uint_as_float(y[e]);
                    }
                }
            }
        }
    } else if (warp == 13 || warp == 14) {
        // ================================ loaders ========================================
        // Contiguous rows: one TMA box per chunk ([128 rows x 32 or 64 bytes]) into the
        // owning producer set's next stage, in the common order.  Warp 13 loads set 0's
        // chunks and warp 14 set 1's, so a set that falls behind does not hold back the
        // other set's refills.
        const int my_set = warp - 13;
        if (a.use_tma) {
            const bool leader = elect_one();
            const CUtensorMap* m_lat = &a.tm_lat[tq4 ? 1 : 0];
            const CUtensorMap* m_rope = &a.tm_rope[tq4 ? 1 : 0];
            const int64_t row0 = (int64_t)s * p.seq_stride_rows + r0;   // pool row of candidate r0
            int o0 = 0, o1 = 0;
            bool ok = true;
            for (int n = 0; n < n_items && ok; ++n) {
                const OwnItem it = common_item(n, NT);
                const int set = it.ch & 1;
                if (set != my_set) continue;
                const int j = set ? o1++ : o0++;
                if (j < kStages) continue;            // requested at the start
                const int d = j % kStages;
                ok = __all_sync(kFull, wait_bar(sh, sh.raw_empty(set, d), ((uint32_t)(j / kStages) & 1u) ^ 1u, a.status, a.wait_ns));
                if (!ok) break;
                if (leader) {
                    const bool rope = it.ch == 8;
                    const int inner = (rope || !tq4) ? 64 : 32;
                    mbar_arrive_expect_tx(sh.raw_full(set, d), (uint32_t)(inner * kRT));
                    tma_load_2d(sh.stage(set, d), rope ? m_rope : m_lat, rope ? 0 : it.ch * inner,
                                (int)(row0 + (int64_t)it.tile * kRT), sh.raw_full(set, d));
                }
                __syncwarp();
            }
            // every box issued has landed before the CTA's shared memory is released
            if (leader) {
                for (int set = my_set; set == my_set; ++set) {
                    const int o = set ? o1 : o0;
                    for (int d = 0; d < kStages && d < o; ++d) {
                        const int jl = d + kStages * ((o - 1 - d) / kStages);
                        if (!mbar_wait(sh.raw_full(set, d), (uint32_t)(jl / kStages) & 1u, kTimeoutNs) && a.status)
                            atomicOr(a.status, (unsigned)KVQ_DEV_TIMEOUT);
                    }
                }
            }
            __syncwarp();
        }
    } else if (warp == 15) {
        // ============================ context MMA issuer =================================
        // The context of tile i after its softmax, chunk pair by chunk pair as the
        // producers fill the ring.  A second issuing warp, on another scheduler, so that
        // the score of the next tile is not queued behind this chain of waits and issues.
        const bool leader = elect_one();
        const uint32_t idesc_c = idesc_f16_f32(kRT, kN, true, true);     // V^T . W^T
        const uint64_t p_desc = desc_sw128(smem_u32(sh.pbuf()), 1024);
        const uint64_t v_desc = desc_sw128_lbo(smem_u32(sh.slot(0)), kChunkBytes, 1024);
        bool ok = true;
        for (int tile = 0; tile < NT && ok; ++tile) {
            ok = __all_sync(kFull, wait_bar(sh, sh.p_full(), (uint32_t)tile & 1u, a.status, a.wait_ns));
            if (!ok) break;
            tc_fence_after();
            for (int c = 0; c < 8; ++c) {
                // chunk c comes from set c & 1: its ord-th context chunk, in slot
                // 2 (ord % 2) + (c & 1), next to its M-tile partner
                const int ord = 4 * tile + (c >> 1);
                const int slot = 2 * (ord & 1) + (c & 1);
                ok = __all_sync(kFull, wait_bar(sh, sh.full_c(slot), (uint32_t)(ord >> 1) & 1u, a.status, a.wait_ns));
                if (!ok) break;
                tc_fence_after();
                if (c & 1) {
                    // M-tile m = c/2 spans the slots of chunks c-1 (this - 1) and c
                    const int m = c >> 1;
                    const uint64_t a_desc = v_desc + (uint64_t)(((slot - 1) * kChunkBytes) >> 4);
                    const uint32_t d = tmem + kColO + 64 * m;
                    if (leader) {
#pragma unroll
                        for (int ks = 0; ks < kRT / 16; ++ks)
                            mma_f16_ss(d, a_desc + (uint64_t)((2048 * ks) >> 4), p_desc + (uint64_t)((2048 * ks) >> 4),
                                       idesc_c, (tile == 0 && ks == 0) ? 0u : 1u);
                        mma_commit(sh.empty_c(slot - 1));
                        mma_commit(sh.empty_c(slot));
                    }
                    __syncwarp();
                }
            }
            if (!ok) break;
            if (leader) mma_commit(sh.o_done());
            __syncwarp();
        }
        // drain: this warp's MMAs complete before tensor memory is freed
        if (leader) {
            mma_commit(sh.drain_c());
            if (!mbar_wait(sh.drain_c(), 0, kTimeoutNs) && a.status)
                atomicOr(a.status, (unsigned)KVQ_DEV_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ============================= score MMA issuer ==================================
        // The whole warp runs the loop (operands are computed warp-uniformly); one elected
        // lane issues the MMAs and commits.
        const bool leader = elect_one();
        const uint32_t idesc_s = idesc_f16_f32(kRT, kN, false, false);   // C . Q^T
        const uint64_t q_desc = desc_sw128(smem_u32(sh.q()), 1024);
        // the Q image is written by the kernel launched just before this one
        grid_dependency_wait();
        if (leader) {
            mbar_arrive_expect_tx(sh.q_full(), kQBytes);
            bulk_copy_g2s(sh.q(), a.q_img + (((int64_t)s * p.n_q + q) * a.n_hg + hg) * (int64_t)kQBytes,
                          kQBytes, sh.q_full());
        }
        __syncwarp();
        bool ok = __all_sync(kFull, wait_bar(sh, sh.q_full(), 0u, a.status, a.wait_ns));
        tc_fence_after();
        for (int i = 0; i < NT && ok; ++i) {
            if (i >= 1) ok = __all_sync(kFull, wait_bar(sh, sh.s_empty(), (uint32_t)(i - 1) & 1u, a.status, a.wait_ns));
            if (!ok) break;
            tc_fence_after();
            for (int ch = 0; ch < 9; ++ch) {
                // chunk ch comes from producer set ch & 1: its ord-th score chunk
                const int ord = i * ((ch & 1) ? 4 : 5) + (ch >> 1);
                const int slot = (ch & 1) + 2 * (ord & 1);
                ok = __all_sync(kFull, wait_bar(sh, sh.full_a(slot), (uint32_t)(ord >> 1) & 1u, a.status, a.wait_ns));
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem + (ch == 8 ? 64u : 0u);
                const uint32_t a_tm = tmem + kColA + 32 * slot;
                const uint64_t b_desc = q_desc + (uint64_t)((ch * kQSlabBytes) >> 4);
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16_ts(d, a_tm + 8 * ks, b_desc + 2 * ks, idesc_s,
                                   (ch == 0 || ch == 8) ? (ks > 0) : 1u);
                    mma_commit(sh.empty_a(slot));
                }
                __syncwarp();
            }
            if (!ok) break;
            if (leader) mma_commit(sh.s_full());
            __syncwarp();
        }
        // drain: this warp's MMAs complete before tensor memory is freed, and the Q copy
        // has landed before the CTA's shared memory is released
        if (leader) {
            mma_commit(sh.drain());
            if (!mbar_wait(sh.drain(), 0, kTimeoutNs) && a.status)
                atomicOr(a.status, (unsigned)KVQ_DEV_TIMEOUT);
            if (!mbar_wait(sh.q_full(), 0, kTimeoutNs) && a.status)
                atomicOr(a.status, (unsigned)KVQ_DEV_TIMEOUT);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 12) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t tc_q_image_bytes(const kvq_mla_problem& p)
{
    const size_t n_hg = (size_t)(p.n_heads + kGQ - 1) / kGQ;
    return align256((size_t)p.n_seq * p.n_q * n_hg * kQBytes);
}

namespace {

}  // namespace

cudaError_t launch_mla_decode_tc(const kvq_mla_problem& p, const DecodePlan& plan,
                                 const float* q_rot, void* q_img, float* part_ml, float* part_o,
                                 uint32_t* dev_status, cudaStream_t s, bool fmt_split)
{
    TcArgs a;
    memset(&a, 0, sizeof(a));
    if (!p.block_table && !p.idx) {
        bool ok = true;
        for (int k = 0; k < 2 && ok; ++k) {
            const bool used = p.seq_fmt || p.fmt == (k ? KVQ_FMT_TQ4 : KVQ_FMT_FP8);
            if (!used) continue;
            const kvq_mla_cache& c = k ? p.tq4 : p.fp8;
            ok = make_code_map(&a.tm_lat[k], c.lat, c.n_rows, k ? kDLat / 2 : kDLat, k ? 32 : 64) &&
                 make_code_map(&a.tm_rope[k], c.rope, c.n_rows, kDRope, 64);
        }
        a.use_tma = ok ? 1 : 0;
    }
    a.p = p;
    a.split_rows = plan.split_rows;
    a.n_splits = plan.n_splits;
    a.n_hg = (p.n_heads + kGQ - 1) / kGQ;
    a.fmt_split = fmt_split ? 1 : 0;
    a.q_rot = q_rot;
    a.q_img = static_cast<uint8_t*>(q_img);
    a.part_ml = part_ml;
    a.part_o = part_o;
    a.status = dev_status;
    a.wait_ns = wait_limit_ns();
    a.premix = plan.premix ? 1 : 0;
    const int64_t items = (int64_t)p.n_seq * p.n_q * a.n_hg * kGQ;
    q_image_kernel<<<(int)std::max<int64_t>(1, std::min<int64_t>((items + 7) / 8, (int64_t)sm_count() * 8)), 256, 0, s>>>(a);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    static std::atomic<uint64_t> attr_set{0};
    const uint64_t bit = 1ull << (device & 63);
    if (!(attr_set.load() & bit)) {
        e = cudaFuncSetAttribute(mla_decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(bit);
    }
    dim3 grid(plan.n_splits, p.n_seq, p.n_q * a.n_hg);
    return launch_dependent(mla_decode_tc_kernel, grid, dim3(kThreads), kSmemBytes, s, a);
}

}  // namespace kvq
