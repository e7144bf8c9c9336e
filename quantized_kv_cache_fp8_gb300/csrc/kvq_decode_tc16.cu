// kvq_decode_tc16.cu — the tensor-core (tcgen05) split-T absorbed-MLA decode for groups
// of 16 query-heads, with every code converted to binary16 once.
//
// Same operation as the other decode kernels (colibri PR #399: score
// s_t = tau (q_lat . c_t + q_rope . k_rope_t), context sum_t softmax(s)_t c_t, split-T
// partials merged by the log-sum-exp combine; Commit 2), as two dense contractions per
// tile of 128 rows:
//
//   S^T[rows x 32] = C_tile[rows x 576] . Q^T        rows on M = 128, N = 16 heads hi | lo
//   O^T[dims x 32] += V_tile^T[dims x rows] . W^T    dims on M (4 M-tiles), same N
//
// A producer thread (one row) converts a 64-code chunk once into a tensor-memory slot
// that the score MMA reads as A (lane = row); latent chunks are later copied from there
// into a 128B-swizzled shared-memory slot that the context MMA reads as the MN-major A
// operand V^T once the softmax of the tile has produced W.  Three producer sets take
// every third chunk, so three chains of conversion and hand-over latency overlap.  The codes are exact in fp16
// (every e4m3 value; every TQ4 centroid is a binary16 value); the fp32 operands q and
// w = p * scale are split into fp16 hi + lo halves stacked along N, and D accumulates in
// fp32 in tensor memory.
//
// Why 16 heads: a tcgen05.mma of M = 128, K = 16 costs the same ~46 cycles for every
// N <= 64 (measured on GB300), so 16 heads cost as much tensor time per row as 32; the
// win is shared memory.  The V tile of 128 rows (128 KB of fp16) must live from its
// conversion until the context MMAs after the softmax; next to a 36 KB query image it
// fits, next to the 72 KB image of 32 heads it does not.
//
// Every wait is bounded (%globaltimer); a timeout sets KVQ_DEV_TIMEOUT, raises a
// CTA-wide abort flag, drains the MMAs and copies in flight and frees tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstring>

#include "kvq_internal.cuh"
#include "kvq_sm100.cuh"
#include "kvq_tc_common.cuh"

namespace kvq {

using namespace sm100;

namespace {

using namespace tc;

constexpr int kRT = 128;                  // rows per tile (score M)
constexpr int kGQ = 16;                   // query-heads per CTA
constexpr int kN = 2 * kGQ;               // MMA N: 16 hi | 16 lo
constexpr int kQSlab = kN * 128;          // [32 rows x 64 k] fp16, 128B-swizzled
constexpr int kQBytes = 9 * kQSlab;       // 36 KB
constexpr int kWSlab = kN * 128;          // W image: [32 n x 64 rows] per slab
constexpr int kWBytes = 2 * kWSlab;       // rows 0..63 and 64..127
constexpr int kVSlot = kRT * 128;         // [128 rows x 64 dims] fp16, 128B-swizzled
constexpr int kSets = 3;                  // producer sets; set s converts chunks ch = s mod 3
constexpr int kPer = 3;                   // chunks per set and tile (9 = rope + 8 latent)
constexpr int kStages = 2;                // raw-code stages per producer set
constexpr int kStageBytes = kRT * 64;     // one chunk of raw codes
constexpr int kWarpSmx = 4 * kSets;       // first softmax warp
constexpr int kWarpMma = kWarpSmx + 4;   // score MMA issuer; allocates tensor memory
constexpr int kWarpCtx = kWarpMma + 1;   // context MMA issuer
constexpr int kWarpLoad = kWarpCtx + 1;  // TMA loader of the three sets
constexpr int kThreads = 32 * (kWarpLoad + 1);   // 12 producer, 4 softmax, 2 MMA, 1 loader warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.0f;             // rescale only when the max grows by > 2^8
constexpr uint64_t kTimeoutNs = kDefaultWaitNs;   // drains

// tensor memory columns: S (latent scores at 0, rope scores at 32), O^T, and one score-A
// slot per chunk of a tile (slot k of set s holds the set's k-th chunk)
constexpr uint32_t kColO = 64;            // O^T M-tile m at 64 + 32 m
constexpr uint32_t kColA = 192;           // score-A slot k of set s at 192 + 32 (3 s + k)
static_assert(kColA + 32 * kSets * kPer <= 512, "tensor memory columns");

// shared memory
constexpr int kOffQ = 0;
constexpr int kOffW = kOffQ + kQBytes;
constexpr int kOffV = kOffW + kWBytes;                    // slot j: latent chunk j
constexpr int kOffStage = kOffV + 8 * kVSlot;
constexpr int kOffRed = kOffStage + kSets * kStages * kStageBytes;   // [4][16] f32
constexpr int kOffM = kOffRed + 4 * 16 * 4;               // [16] running maxima
constexpr int kOffAlpha = kOffM + 16 * 4;                 // [16] rescale factors
constexpr int kOffFlag = kOffAlpha + 16 * 4;              // some head rescales O
constexpr int kOffVote = kOffFlag + 16;                   // [2][4] "a row exceeds the max"
constexpr int kOffTab = kOffVote + 32;                    // [64] binary16 centroids (3/6 bits)
constexpr int kOffBar = kOffTab + 128;
// full_a[3][3], empty_a[3][3], full_v[8], empty_v[8], s_full, s_empty, p_full, o_done,
// drain[2] (one per MMA issuer), q_full, raw_full[3][kStages], raw_empty[3][kStages]
constexpr int kNumA = kSets * kPer;
constexpr int kNumBars = 2 * kNumA + 16 + 7 + 2 * kSets * kStages;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert(kOffV % 1024 == 0 && kOffW % 1024 == 0 && kOffStage % 1024 == 0, "swizzle atoms");

struct Tc16Args {
    CUtensorMap tm_lat[2], tm_rope[2];   // code planes ([0] fp8 tier, [1] TQ4 tier)
    int use_tma;                         // contiguous rows: chunks arrive by TMA
    kvq_mla_problem p;
    int split_rows, n_splits, n_hg;      // n_hg: head groups of 16
    uint8_t* q_img;                      // [n_seq][n_q][n_hg][kQBytes]
    float* part_ml;
    float* part_o;
    uint32_t* status;
    uint64_t wait_ns;                    // limit of the pipeline waits
    int premix;                          // rotated rows: partials carry stages h = 128, 256
    uint16_t cb_tab[64];                 // binary16 centroids of a 3- or 6-bit problem
};

__global__ void __launch_bounds__(256) q_image16_kernel(Tc16Args a)
{
    grid_dependents_launch();                    // the decode may start loading codes
    build_q_image<kGQ>(a.p, a.n_hg, a.q_img);
}

struct Shared {
    uint8_t* base;
    __device__ uint8_t* q() const { return base + kOffQ; }
    __device__ uint8_t* w() const { return base + kOffW; }
    // V slot of latent chunk j (dims 64j..64j+63); M-tile m is slots 2m and 2m+1
    __device__ uint8_t* v(int j) const { return base + kOffV + j * kVSlot; }
    __device__ uint8_t* stage(int set, int d) const { return base + kOffStage + (set * kStages + d) * kStageBytes; }
    __device__ float* red() const { return reinterpret_cast<float*>(base + kOffRed); }
    __device__ float* m_run() const { return reinterpret_cast<float*>(base + kOffM); }
    __device__ float* alpha() const { return reinterpret_cast<float*>(base + kOffAlpha); }
    __device__ volatile int* flag() const { return reinterpret_cast<volatile int*>(base + kOffFlag); }
    __device__ volatile int* vote(int par) const { return reinterpret_cast<volatile int*>(base + kOffVote) + 4 * par; }
    __device__ uint16_t* tab() const { return reinterpret_cast<uint16_t*>(base + kOffTab); }
    __device__ uint64_t* bar(int i) const { return reinterpret_cast<uint64_t*>(base + kOffBar) + i; }
    __device__ uint64_t* full_a(int s, int k) const { return bar(s * kPer + k); }
    __device__ uint64_t* empty_a(int s, int k) const { return bar(kNumA + s * kPer + k); }
    __device__ uint64_t* full_v(int j) const { return bar(2 * kNumA + j); }
    __device__ uint64_t* empty_v(int j) const { return bar(2 * kNumA + 8 + j); }
    __device__ uint64_t* s_full() const { return bar(2 * kNumA + 16); }
    __device__ uint64_t* s_empty() const { return bar(2 * kNumA + 17); }
    __device__ uint64_t* p_full() const { return bar(2 * kNumA + 18); }
    __device__ uint64_t* o_done() const { return bar(2 * kNumA + 19); }
    __device__ uint64_t* drain(int w) const { return bar(2 * kNumA + 20 + w); }
    __device__ uint64_t* q_full() const { return bar(2 * kNumA + 22); }
    __device__ uint64_t* raw_full(int s, int d) const { return bar(2 * kNumA + 23 + s * kStages + d); }
    __device__ uint64_t* raw_empty(int s, int d) const { return bar(2 * kNumA + 23 + kSets * kStages + s * kStages + d); }
    __device__ uint32_t* tmem_base() const { return reinterpret_cast<uint32_t*>(base + kOffMisc); }
    __device__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(base + kOffMisc + 4); }
};

__device__ __forceinline__ bool wait_bar(const Shared& sh, uint64_t* bar, uint32_t parity, uint32_t* status,
                                         uint64_t limit_ns)
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

// Per-tile chunk order: ch = 0 the rope key, ch = 1 + j latent chunk j (dims 64j..64j+63).
// Producer set s converts the chunks with ch % 3 == s, three a tile: the k-th chunk of set
// s in tile i has the set ordinal o = 3 i + k and ch = 3 k + s.
static_assert(kSets * kPer == 9, "nine chunks a tile");

// ====================================================================================
// The decode kernel.
//  * Warps 0-11: three producer sets of four warps (thread = row of the tile).  Per chunk:
//    raw codes from the set's stage ring -> binary16 -> the set's score-A slot of the
//    chunk in tensor memory (tcgen05.st; one slot per chunk of a tile, so converting a
//    tile waits only on the score MMAs of the tile before).  Once the set's three chunks
//    of tile i are converted, it copies its latent chunks from their A slots (tcgen05.ld)
//    into the V slots in shared memory, each as the context of tile i-1 frees it.  So
//    the conversion of tile i+1 runs during the softmax and context of tile i.
//  * Warps 12-15: softmax (thread = row): S from tensor memory, per-head tile maxima,
//    lazy O rescale, W = p * scale as fp16 hi | lo into the K-major W image; epilogue
//    (thread = output dim) writes the split's (m, l, o) partials.
//  * Warp 16: allocates tensor memory; issues the score MMAs chunk by chunk as the A
//    slots fill (the first chunk of tile i after the softmax has read S of tile i-1).
//  * Warp 17: issues the context MMAs of tile i after its softmax, M-tile by M-tile as
//    the V copies land.  Two issuing warps, on two schedulers, keep the chain of waits
//    and MMA issues off the critical path; each waits only on other roles.
//  * Warp 18: the TMA loader of the three sets (contiguous caches), polling their stages;
//    paged and sparse caches are copied by the producers themselves with cp.async.
// ====================================================================================
// kB = 0: fp8 and TQ4 rows (per sequence, mixed batches included); kB = 6 or 3: the
// rotated tier at 6 or 3 bits in a problem of that one format.
template <int kB>
__global__ void __maxnreg__(96) mla_decode_tc16_kernel(const __grid_constant__ Tc16Args a)
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
    // the 3- and 6-bit rotated tiers are read in problems of one format (the rotated
    // planes of a seq_fmt batch hold 4-bit rows)
    const bool bad_fmt = kB == 0 ? !(fmt == KVQ_FMT_FP8 || fmt == KVQ_FMT_TQ4)
                                 : (p.seq_fmt != nullptr || fmt != (kB == 6 ? KVQ_FMT_TQ6 : KVQ_FMT_TQ3));
    grid_dependents_launch();                    // the combine may start launching

    if (r0 >= n_cand || bad_fmt) {
        if (bad_fmt && tid == 0 && split == 0 && a.status) atomicOr(a.status, (unsigned)KVQ_DEV_BAD_FORMAT);
        if (tid < nh) {
            const int64_t sl = (qrow + h0 + tid) * a.n_splits + split;
            a.part_ml[sl * 2] = -INFINITY;
            a.part_ml[sl * 2 + 1] = 0.0f;
        }
        return;
    }
    const bool rot = fmt != KVQ_FMT_FP8;               // a rotated tier: 3, 4 or 6 bits
    const int bits = kB != 0 ? kB : rot ? 4 : 8;
    const int lat_cb = 8 * bits;                        // bytes of a latent chunk of a row
    const kvq_mla_cache& C = rot ? p.tq4 : p.fp8;
    const int NT = (int)((r1 - r0 + kRT - 1) / kRT);
    const RowCtx rc{&p, s, q, L, r1, p.causal ? (int64_t)L - p.n_q + q : (int64_t)L - 1, &C, a.status};
    // Contiguous rows: the loader sets up the stage barriers itself and requests each set's
    // first kStages chunks at once, before the CTA-wide setup below (tensor memory, the
    // other barriers), which would otherwise delay the first loads by ~1 us.
    const bool pre = a.use_tma != 0;
    if (warp == kWarpLoad && pre && lane == 0) {
        for (int st = 0; st < kSets; ++st) {
            for (int d = 0; d < kStages; ++d) {
                mbar_init(sh.raw_full(st, d), 1);
                mbar_init(sh.raw_empty(st, d), 4);       // one per warp of the set
            }
        }
        fence_mbar_init();
        const int64_t row0 = (int64_t)s * p.seq_stride_rows + r0;
        static_assert(kStages <= kPer, "the first kStages chunks of a set are in tile 0");
        for (int st = 0; st < kSets; ++st) {
            for (int d = 0; d < kStages; ++d) {
                const int ch = kSets * d + st;
                const bool rope = ch == 0;
                const int inner = rope ? 64 : lat_cb;
                mbar_arrive_expect_tx(sh.raw_full(st, d), (uint32_t)(inner * kRT));
                tma_load_2d(sh.stage(st, d), rope ? &a.tm_rope[rot ? 1 : 0] : &a.tm_lat[rot ? 1 : 0],
                            rope ? 0 : (ch - 1) * inner, (int)row0, sh.raw_full(st, d));
            }
        }
    }

    if (warp == kWarpMma) {
        if (lane == 0) {
            for (int st = 0; st < kSets; ++st) {
                for (int k = 0; k < kPer; ++k) {
                    mbar_init(sh.full_a(st, k), 4);      // one arrival per warp of the set
                    mbar_init(sh.empty_a(st, k), 1);     // MMA commit
                }
                for (int d = 0; d < kStages && !pre; ++d) {
                    mbar_init(sh.raw_full(st, d), 1);
                    mbar_init(sh.raw_empty(st, d), 4);   // one per warp of the set
                }
            }
            for (int j = 0; j < 8; ++j) {
                mbar_init(sh.full_v(j), 4);
                mbar_init(sh.empty_v(j), 1);
            }
            mbar_init(sh.s_full(), 1);
            mbar_init(sh.s_empty(), 4);                  // one arrival per softmax warp
            mbar_init(sh.p_full(), 4);
            mbar_init(sh.o_done(), 1);
            mbar_init(sh.drain(0), 1);
            mbar_init(sh.drain(1), 1);
            mbar_init(sh.q_full(), 1);
            *sh.abort_flag() = 0;
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(sh.tmem_base(), 512);
        tmem_relinquish();
    }
    if (tid < kGQ) sh.m_run()[tid] = -INFINITY;
    if (tid < 64) sh.tab()[tid] = a.cb_tab[tid];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sh.tmem_base();

    if (warp < kWarpSmx) {
        // ================================ producers ======================================
        const int set = warp >> 2;
        const int t = (warp & 3) * 32 + lane;             // row within the tile
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int n_own = kPer * NT;
        int64_t row_c = -1;                               // pool row of this thread, tile tile_c
        int tile_c = -1;
        // non-TMA staging: piece p of row t at (p * 128 + t) * 16 of the stage (conflict-free)
        auto issue = [&](int o) {
            if (o < n_own) {
                const int tile = o / kPer, ch = kSets * (o - tile * kPer) + set;
                if (tile != tile_c) {
                    tile_c = tile;
                    row_c = rc.row(r0 + (int64_t)tile * kRT + t, false);
                }
                const int64_t row = row_c;
                const bool rope = ch == 0;
                const int cb = rope ? 64 : lat_cb;
                const uint8_t* src = row < 0 ? C.rope
                                   : rope ? C.rope + row * kDRope
                                          : C.lat + row * (kDLat * bits / 8) + (ch - 1) * lat_cb;
                uint8_t* st = sh.stage(set, o % kStages);
                const uint32_t nb = row < 0 ? 0u : 16u;       // invalid rows read as zeros
                if (cb == 24) {
                    // a 3-bit chunk starts 0 or 8 bytes past a 16-byte boundary (24 j):
                    // copy the two aligned 16-byte pieces that hold its 24 bytes
                    const uint8_t* s16 = row < 0 ? src : src - ((ch - 1) & 1) * 8;
                    cp_async16(st + t * 16, s16, nb);
                    cp_async16(st + (kRT + t) * 16, s16 + 16, nb);
                } else {
                    for (int pc = 0; pc < cb / 16; ++pc) cp_async16(st + (pc * kRT + t) * 16, src + 16 * pc, nb);
                }
            }
            cp_async_commit();                            // one group per item, maybe empty
        };
        const bool tma = a.use_tma != 0;
        // the raw codes of chunk o into registers (TMA: after its box landed)
        auto fetch = [&](int o, uint4 (&raw)[4]) -> bool {
            const int tile = o / kPer, ch = kSets * (o - tile * kPer) + set;
            const int cb = ch == 0 ? 64 : lat_cb;
            raw[1] = raw[2] = raw[3] = make_uint4(0u, 0u, 0u, 0u);
            if (tma) {
                // the loader's box: row t at t * cb; its 16-byte pieces swizzled by the TMA
                // (64-byte rows: piece i at i ^ ((t >> 1) & 3); 32-byte rows: i ^ ((t >> 2)
                // & 1); 48-byte rows unswizzled, conflict-free as they are)
                const int d = o % kStages;
                if (!__all_sync(kFull, wait_bar(sh, sh.raw_full(set, d), (uint32_t)(o / kStages) & 1u, a.status, a.wait_ns)))
                    return false;
                const uint8_t* st = sh.stage(set, d) + t * cb;
                if (cb == 64) {
                    const int x = (t >> 1) & 3;
#pragma unroll
                    for (int i = 0; i < 4; ++i) raw[i] = *reinterpret_cast<const uint4*>(st + 16 * (i ^ x));
                } else if (cb == 32) {
                    const int x = (t >> 2) & 1;
                    raw[0] = *reinterpret_cast<const uint4*>(st + 16 * x);
                    raw[1] = *reinterpret_cast<const uint4*>(st + 16 * (1 ^ x));
                } else {
#pragma unroll
                    for (int i = 0; i < 3; ++i) raw[i] = *reinterpret_cast<const uint4*>(st + 16 * i);
                }
            } else {
                cp_async_wait<kStages - 1>();             // item o's group has landed
                const uint8_t* st = sh.stage(set, o % kStages);
                if (cb == 24) {
                    const uint4 a0 = *reinterpret_cast<const uint4*>(st + t * 16);
                    const uint4 a1 = *reinterpret_cast<const uint4*>(st + (kRT + t) * 16);
                    if (((ch - 1) & 1) == 0) {            // the chunk's 24 bytes start at byte 0
                        raw[0] = a0;
                        raw[1] = make_uint4(a1.x, a1.y, 0u, 0u);
                    } else {                              // ... at byte 8
                        raw[0] = make_uint4(a0.z, a0.w, a1.x, a1.y);
                        raw[1] = make_uint4(a1.z, a1.w, 0u, 0u);
                    }
                } else {
                    for (int i = 0; i < cb / 16; ++i) raw[i] = *reinterpret_cast<const uint4*>(st + (i * kRT + t) * 16);
                }
            }
            return true;
        };
        if (!tma) {
#pragma unroll
            for (int d = 0; d < kStages; ++d) issue(d);
        }
        uint4 raw[4];
        bool ok = n_own > 0 && fetch(0, raw);
        for (int o = 0; o < n_own && ok; ++o) {
            const int tile = o / kPer, k = o - tile * kPer;
            const bool rope = kSets * k + set == 0;
            {
                uint32_t h[32];
                if (kB == 0 || rope) {
                    const bool fp8 = rope || bits == 8;
                    codes_to_half(raw, 0, fp8, *reinterpret_cast<uint32_t(*)[16]>(h));
                    codes_to_half(raw, 1, fp8, *reinterpret_cast<uint32_t(*)[16]>(h + 16));
                } else {
                    tqb_codes_to_half<kB == 0 ? 6 : kB>(raw, sh.tab(), h);
                }
                // the stage is free once every lane's reads of it are consumed
                if (tma) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sh.raw_empty(set, o % kStages));
                } else {
                    issue(o + kStages);                   // refills the stage just read
                }
                // score operand: the chunk's 64 binary16 values as TMEM lane t, 32 columns,
                // in slot k of the set (free once the score of the tile before read it)
                ok = __all_sync(kFull, wait_bar(sh, sh.empty_a(set, k), ((uint32_t)tile & 1u) ^ 1u, a.status, a.wait_ns));
                if (!ok) break;
                tc_fence_after();
                tmem_st_x32(tmem + lane_base + kColA + 32 * (kPer * set + k), h);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sh.full_a(set, k));
            }
            // the next chunk's raw codes (for the last chunk of the tile, read before the
            // copies below)
            if (o + 1 < n_own) {
                ok = fetch(o + 1, raw);
                if (!ok) break;
            }
            if (k + 1 < kPer) continue;
            // The set's chunks of this tile are converted: copy its latent chunks from their
            // A slots into the V slots as the context of the tile before frees them.
            const uint32_t vpar = ((uint32_t)tile & 1u) ^ 1u;
            for (int kk = 0; kk < kPer && ok; ++kk) {
                const int ch = kSets * kk + set;
                if (ch == 0) continue;                    // the rope key has no V
                ok = __all_sync(kFull, wait_bar(sh, sh.empty_v(ch - 1), vpar, a.status, a.wait_ns));
                if (!ok) break;
                uint32_t h[32];
                const uint32_t src = tmem + lane_base + kColA + 32 * (kPer * set + kk);
                tmem_ld_x16(src, *reinterpret_cast<uint32_t(*)[16]>(h));
                tmem_ld_x16(src + 16, *reinterpret_cast<uint32_t(*)[16]>(h + 16));
                tmem_ld_wait();
                uint8_t* dst = sh.v(ch - 1);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(dst + sw128(t, c)) =
                        make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sh.full_v(ch - 1));
            }
        }
        cp_async_wait_all();                              // nothing lands after the CTA ends
    } else if (warp < kWarpMma) {
        // ================================ softmax ========================================
        // Control flow is identical in all 128 threads (the named barriers need every one
        // of them); `ok` only guards work and is kept warp-uniform.
        const int t = tid - 32 * kWarpSmx;            // row within the tile
        const int wq = warp - kWarpSmx;               // TMEM lane quarter
        const int g16 = lane & 15;                    // head of this lane after a reduction
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        const float tau2 = p.sm_scale * kLog2e;
        const float c512 = tq4_inv_sqrt(kDLat);
        float* red = sh.red();
        float* m_s = sh.m_run();
        float* alpha_s = sh.alpha();
        uint8_t* wimg = sh.w() + (t >> 6) * kWSlab;   // this row's W slab
        const int kk = t & 63;                        // k (row) within the slab
        float l_lane = 0.0f;                          // sum of p over this warp's rows, head g16
        bool ok = true;
        for (int i = 0; i < NT; ++i) {
            const int64_t row = rc.row(r0 + (int64_t)i * kRT + t, true);
            float sc_lat = 0.0f, sc_rope = 0.0f;
            if (row >= 0) {
                sc_lat = rot ? C.lat_scale[row] * c512 : C.lat_scale[row];
                sc_rope = C.rope_scale[row];
            }
            if (ok) ok = wait_bar(sh, sh.s_full(), (uint32_t)i & 1u, a.status, a.wait_ns);
            ok = __all_sync(kFull, ok);
            float sv[kGQ];
#pragma unroll
            for (int g = 0; g < kGQ; ++g) sv[g] = 0.0f;
            if (ok) {
                tc_fence_after();
                uint32_t xh[16], xl[16], yh[16], yl[16];
                const uint32_t cs = tmem + lane_base;
                tmem_ld_x16(cs, xh);
                tmem_ld_x16(cs + 16, xl);
                tmem_ld_x16(cs + 32, yh);
                tmem_ld_x16(cs + 48, yl);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sh.s_empty());   // S may take the next tile's scores
#pragma unroll
                for (int g = 0; g < kGQ; ++g)
                    sv[g] = fmaf(sc_lat, __uint_as_float(xh[g]) + __uint_as_float(xl[g]),
                                 sc_rope * (__uint_as_float(yh[g]) + __uint_as_float(yl[g])));
            }
#pragma unroll
            for (int g = 0; g < kGQ; ++g) sv[g] = (row >= 0 && ok) ? sv[g] * tau2 : -INFINITY;
            // The running maxima move only when a head's tile maximum exceeds them by more
            // than 2^kLazy.  Each warp votes whether one of its rows does; the votes of tile
            // i sit in buffer i % 2 (a warp can run at most one tile ahead of a reader, since
            // the vote barrier of the next tile needs all four warps), so every warp reads
            // the same four votes and takes the same path through the barriers below.
            bool exceed = false;
#pragma unroll
            for (int g = 0; g < kGQ; g += 4) {
                const float4 mv = *reinterpret_cast<const float4*>(m_s + g);
                exceed |= sv[g] > mv.x + kLazy || sv[g + 1] > mv.y + kLazy ||
                          sv[g + 2] > mv.z + kLazy || sv[g + 3] > mv.w + kLazy;
            }
            exceed = __any_sync(kFull, exceed);
            if (lane == 0) sh.vote(i & 1)[wq] = exceed ? 1 : 0;
            named_bar_softmax();
            bool need_rescale = false;
            {
                volatile int* v = sh.vote(i & 1);
                if (v[0] | v[1] | v[2] | v[3]) {
                    float mx[kGQ];
#pragma unroll
                    for (int g = 0; g < kGQ; ++g) mx[g] = sv[g];
                    warp_reduce_transpose<true>(mx, lane);
                    if (lane < kGQ) red[wq * kGQ + lane] = mx[0];
                    named_bar_softmax();
                    if (wq == 0) {
                        const float tm = fmaxf(fmaxf(red[g16], red[16 + g16]), fmaxf(red[32 + g16], red[48 + g16]));
                        const float mo = m_s[g16];
                        // lanes l and l + 16 compute the same head; lanes 0..15 store it
                        const bool upd = tm > mo + kLazy || (mo == -INFINITY && tm > -INFINITY);
                        const float al = !upd ? 1.0f : (mo == -INFINITY) ? 0.0f : exp2f(mo - tm);
                        const bool any = __any_sync(kFull, upd && i > 0);   // also orders the reads of m_s
                        if (lane < kGQ) {
                            if (upd) m_s[lane] = tm;
                            alpha_s[lane] = al;
                        }
                        if (lane == 0) *sh.flag() = any ? 1 : 0;
                    }
                    named_bar_softmax();
                    need_rescale = *sh.flag() != 0;
                }
            }
            // Consume o_done's phase i-1 (the context MMAs of tile i-1) at every tile, so
            // that this wait and the epilogue's never trail the barrier by more than one
            // phase; it also makes O safe to rescale and the W image safe to rewrite.
            if (i > 0 && ok) ok = wait_bar(sh, sh.o_done(), (uint32_t)(i - 1) & 1u, a.status, a.wait_ns);
            ok = __all_sync(kFull, ok);
            if (need_rescale) {
                l_lane *= alpha_s[g16];
                if (ok) {
                    tc_fence_after();
                    float al[kGQ];
#pragma unroll
                    for (int g = 0; g < kGQ; ++g) al[g] = alpha_s[g];
#pragma unroll 1
                    for (int m = 0; m < 4; ++m) {
#pragma unroll
                        for (int c = 0; c < kN; c += 16) {
                            uint32_t x[16];
                            tmem_ld_x16(tmem + lane_base + kColO + 32 * m + c, x);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 16; ++e) x[e] = __float_as_uint(__uint_as_float(x[e]) * al[e]);
                            tmem_st_x16(tmem + lane_base + kColO + 32 * m + c, x);
                        }
                    }
                    tmem_st_wait();
                }
            }
            // weights: p = 2^(s - m), w = p * latent scale, split hi | lo into the W image
            // (K-major: row n = head (hi) or 16 + head (lo), k = this row)
            if (ok) {
#pragma unroll
                for (int g = 0; g < kGQ; g += 2) {
                    const float2 mm = *reinterpret_cast<const float2*>(m_s + g);
                    const float p0 = sv[g] == -INFINITY ? 0.0f : exp2f(sv[g] - mm.x);
                    const float p1 = sv[g + 1] == -INFINITY ? 0.0f : exp2f(sv[g + 1] - mm.y);
                    sv[g] = p0;
                    sv[g + 1] = p1;
                    const float w0 = p0 * sc_lat, w1 = p1 * sc_lat;
                    const __half2 hi = __floats2half2_rn(w0, w1);
                    const float2 hf = __half22float2(hi);
                    const __half2 lo = __floats2half2_rn(w0 - hf.x, w1 - hf.y);
                    const uint32_t off = (kk & 7) * 2;
                    *reinterpret_cast<__half*>(wimg + sw128(g, kk >> 3) + off) = __low2half(hi);
                    *reinterpret_cast<__half*>(wimg + sw128(g + 1, kk >> 3) + off) = __high2half(hi);
                    *reinterpret_cast<__half*>(wimg + sw128(kGQ + g, kk >> 3) + off) = __low2half(lo);
                    *reinterpret_cast<__half*>(wimg + sw128(kGQ + g + 1, kk >> 3) + off) = __high2half(lo);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(sh.p_full());
            } else {
#pragma unroll
                for (int g = 0; g < kGQ; ++g) sv[g] = 0.0f;
            }
            warp_reduce_transpose<false>(sv, lane);
            l_lane += sv[0];
        }
        // ---- epilogue: l over the 128 rows, O^T -> partials ------------------------------
        if (ok) ok = wait_bar(sh, sh.o_done(), (uint32_t)(NT - 1) & 1u, a.status, a.wait_ns);
        ok = __all_sync(kFull, ok);
        if (lane < kGQ) red[wq * kGQ + lane] = l_lane;
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
                const float lt = red[t] + red[16 + t] + red[32 + t] + red[48 + t];
                const int64_t sl = (qrow + h0 + t) * a.n_splits + split;
                a.part_ml[sl * 2] = m_s[t];
                a.part_ml[sl * 2 + 1] = lt;
            }
            // Premixed rotated rows: eight heads at a time, all four M-tiles (dims 128 m +
            // 32 wq + lane) of each, with the unrotation's stages h = 128 and 256, which mix
            // the M-tiles; the combine does the rest.  Otherwise M-tile by M-tile.
#pragma unroll 1
            for (int hb = 0; hb < kGQ && a.premix && rot; hb += 8) {
                uint32_t x[4][8], y[4][8];           // every load issued, then one wait
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    tmem_ld_x8(tmem + lane_base + kColO + 32 * m + hb, x[m]);
                    tmem_ld_x8(tmem + lane_base + kColO + 32 * m + 16 + hb, y[m]);
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
            for (int m = 0; m < 4 && !(a.premix && rot); ++m) {
                const int d = 128 * m + 32 * wq + lane;
                uint32_t x[16], y[16];
                tmem_ld_x16(tmem + lane_base + kColO + 32 * m, x);
                tmem_ld_x16(tmem + lane_base + kColO + 32 * m + 16, y);
                tmem_ld_wait();
#pragma unroll
                for (int g = 0; g < kGQ; ++g)
                    if (g < nh)
                        a.part_o[((qrow + h0 + g) * a.n_splits + split) * kDLat + d] =
                            __uint_as_float(x[g]) + __uint_as_float(y[g]);
            }
        }
    } else if (warp == kWarpLoad) {
        // ================================ loader =========================================
        // Contiguous rows: one TMA box per chunk ([128 rows x 32, 48 or 64 bytes]) into the
        // next stage of the chunk's producer set.  One warp serves the three sets, polling
        // their stages, so a lagging set does not hold back the refills of the others.
        if (a.use_tma) {
            const bool leader = elect_one();
            const CUtensorMap* m_lat = &a.tm_lat[rot ? 1 : 0];
            const CUtensorMap* m_rope = &a.tm_rope[rot ? 1 : 0];
            const int64_t row0 = (int64_t)s * p.seq_stride_rows + r0;   // pool row of candidate r0
            const int n_own = kPer * NT;
            int nxt[kSets];                               // next item of each set
#pragma unroll
            for (int set = 0; set < kSets; ++set) nxt[set] = kStages;   // the first went out at the start
            bool ok = true;
            uint64_t idle_since = 0;
            while (ok && (nxt[0] < n_own || nxt[1] < n_own || nxt[2] < n_own)) {
                bool progress = false;
#pragma unroll
                for (int set = 0; set < kSets; ++set) {
                    const int o = nxt[set];
                    if (o >= n_own) continue;
                    const int d = o % kStages;
                    int r = 0;
                    if (lane == 0) r = mbar_test_wait(sh.raw_empty(set, d), ((uint32_t)(o / kStages) & 1u) ^ 1u) ? 1 : 0;
                    if (!__shfl_sync(kFull, r, 0)) continue;
                    if (leader) {
                        const int tile = o / kPer, ch = kSets * (o - tile * kPer) + set;
                        const bool rope = ch == 0;
                        const int inner = rope ? 64 : lat_cb;
                        mbar_arrive_expect_tx(sh.raw_full(set, d), (uint32_t)(inner * kRT));
                        tma_load_2d(sh.stage(set, d), rope ? m_rope : m_lat, rope ? 0 : (ch - 1) * inner,
                                    (int)(row0 + (int64_t)tile * kRT), sh.raw_full(set, d));
                    }
                    __syncwarp();
                    nxt[set] = o + 1;
                    progress = true;
                }
                if (progress) {
                    idle_since = 0;
                } else if (*sh.abort_flag()) {
                    ok = false;
                } else {
                    const uint64_t now = globaltimer_ns();
                    if (idle_since == 0) {
                        idle_since = now;
                    } else if (now - idle_since > a.wait_ns) {
                        if (lane == 0) {
                            *sh.abort_flag() = 1;
                            if (a.status) atomicOr(a.status, (unsigned)KVQ_DEV_TIMEOUT);
                        }
                        ok = false;
                    }
                }
                ok = __all_sync(kFull, ok);
            }
            // every box issued has landed before the CTA's shared memory is released
            if (leader) {
#pragma unroll
                for (int set = 0; set < kSets; ++set) {
                    for (int d = 0; d < kStages && d < nxt[set]; ++d) {
                        const int jl = d + kStages * ((nxt[set] - 1 - d) / kStages);
                        if (!mbar_wait(sh.raw_full(set, d), (uint32_t)(jl / kStages) & 1u, kTimeoutNs) && a.status)
                            atomicOr(a.status, (unsigned)KVQ_DEV_TIMEOUT);
                    }
                }
            }
            __syncwarp();
        }
    } else if (warp == kWarpCtx) {
        // ============================ context MMA issuer =================================
        // O^T += V^T . W^T per tile, after the tile's softmax, M-tile by M-tile as the V
        // copies land
        const bool leader = elect_one();
        const uint32_t idesc_c = idesc_f16_f32(kRT, kN, true, false);    // V^T (MN-major) . W^T
        const uint32_t w_addr = smem_u32(sh.w());
        bool ok = true;
        for (int i = 0; i < NT && ok; ++i) {
            ok = __all_sync(kFull, wait_bar(sh, sh.p_full(), (uint32_t)i & 1u, a.status, a.wait_ns));
            for (int m = 0; m < 4 && ok; ++m) {
                ok = __all_sync(kFull, wait_bar(sh, sh.full_v(2 * m), (uint32_t)i & 1u, a.status, a.wait_ns));
                if (ok) ok = __all_sync(kFull, wait_bar(sh, sh.full_v(2 * m + 1), (uint32_t)i & 1u, a.status, a.wait_ns));
                if (!ok) break;
                tc_fence_after();
                // A = V^T of M-tile m: its two 64-dim halves in adjacent slots; K = rows,
                // 16 rows (2048 B) per step
                const uint64_t a_desc = desc_sw128_lbo(smem_u32(sh.v(2 * m)), kVSlot, 1024);
                const uint32_t d = tmem + kColO + 32 * m;
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < kRT / 16; ++ks) {
                        const uint64_t b_desc = desc_sw128(w_addr + (ks >> 2) * kWSlab + 32 * (ks & 3), 1024);
                        mma_f16_ss(d, a_desc + (uint64_t)((2048 * ks) >> 4), b_desc, idesc_c,
                                   (i == 0 && ks == 0) ? 0u : 1u);
                    }
                    mma_commit(sh.empty_v(2 * m));
                    mma_commit(sh.empty_v(2 * m + 1));
                    if (m == 3) mma_commit(sh.o_done());
                }
                __syncwarp();
            }
        }
        // drain: this warp's MMAs complete before tensor memory is freed
        if (leader) {
            mma_commit(sh.drain(1));
            if (!mbar_wait(sh.drain(1), 0, kTimeoutNs) && a.status)
                atomicOr(a.status, (unsigned)KVQ_DEV_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ============================= score MMA issuer ==================================
        // S^T = C . Q^T per tile, chunk by chunk as the producers fill the A slots; the
        // first chunk waits until the softmax has read S of the tile before
        const bool leader = elect_one();
        const uint32_t idesc_s = idesc_f16_f32(kRT, kN, false, false);   // C . Q^T
        const uint64_t q_desc = desc_sw128(smem_u32(sh.q()), 1024);
        grid_dependency_wait();                 // the Q image comes from the kernel before
        if (leader) {
            mbar_arrive_expect_tx(sh.q_full(), kQBytes);
            bulk_copy_g2s(sh.q(), a.q_img + (((int64_t)s * p.n_q + q) * a.n_hg + hg) * (int64_t)kQBytes,
                          kQBytes, sh.q_full());
        }
        __syncwarp();
        bool ok = __all_sync(kFull, wait_bar(sh, sh.q_full(), 0u, a.status, a.wait_ns));
        tc_fence_after();
        for (int i = 0; i < NT && ok; ++i) {
            if (i > 0) ok = __all_sync(kFull, wait_bar(sh, sh.s_empty(), (uint32_t)(i - 1) & 1u, a.status, a.wait_ns));
            for (int ch = 0; ch < 9 && ok; ++ch) {
                const int set = ch % kSets, k = ch / kSets;
                ok = __all_sync(kFull, wait_bar(sh, sh.full_a(set, k), (uint32_t)i & 1u, a.status, a.wait_ns));
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem + (ch == 0 ? 32u : 0u);
                const uint32_t a_tm = tmem + kColA + 32 * (kPer * set + k);
                const uint64_t b_desc = q_desc + (uint64_t)(((ch == 0 ? 8 : ch - 1) * kQSlab) >> 4);
                const bool first = ch <= 1;             // first chunk of its accumulator
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16_ts(d, a_tm + 8 * ks, b_desc + 2 * ks, idesc_s, first ? (ks > 0) : 1u);
                    mma_commit(sh.empty_a(set, k));
                    if (ch == 8) mma_commit(sh.s_full());
                }
                __syncwarp();
            }
        }
        // drain: this warp's MMAs complete before tensor memory is freed, and the Q copy
        // has landed before the CTA's shared memory is released
        if (leader) {
            mma_commit(sh.drain(0));
            if (!mbar_wait(sh.drain(0), 0, kTimeoutNs) && a.status)
                atomicOr(a.status, (unsigned)KVQ_DEV_TIMEOUT);
            if (!mbar_wait(sh.q_full(), 0, kTimeoutNs) && a.status)
                atomicOr(a.status, (unsigned)KVQ_DEV_TIMEOUT);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

size_t tc16_q_image_bytes(const kvq_mla_problem& p)
{
    const size_t n_hg = (size_t)(p.n_heads + kGQ - 1) / kGQ;
    return align256((size_t)p.n_seq * p.n_q * n_hg * kQBytes);
}

cudaError_t launch_mla_decode_tc16(const kvq_mla_problem& p, const DecodePlan& plan, void* q_img,
                                   float* part_ml, float* part_o, uint32_t* dev_status, cudaStream_t s)
{
    Tc16Args a;
    memset(&a, 0, sizeof(a));
    // TMA boxes of one 64-dim chunk: 64 B (fp8), 32 B (4 bits), 48 B (6 bits); 3-bit
    // chunks (24 B) are no multiple of 16 bytes and go by cp.async
    const int rot_bits = p.seq_fmt ? 4 : rotated_bits(p.fmt);
    if (!p.block_table && !p.idx && !(!p.seq_fmt && p.fmt == KVQ_FMT_TQ3)) {
        bool ok = true;
        for (int k = 0; k < 2 && ok; ++k) {
            const bool used = p.seq_fmt || (k ? rotated_format(p.fmt) : p.fmt == KVQ_FMT_FP8);
            if (!used) continue;
            const kvq_mla_cache& c = k ? p.tq4 : p.fp8;
            ok = make_code_map(&a.tm_lat[k], c.lat, c.n_rows, k ? kDLat * rot_bits / 8 : kDLat,
                               k ? 8 * rot_bits : 64) &&
                 make_code_map(&a.tm_rope[k], c.rope, c.n_rows, kDRope, 64);
        }
        a.use_tma = ok ? 1 : 0;
    }
    a.p = p;
    a.split_rows = plan.split_rows;
    a.n_splits = plan.n_splits;
    a.n_hg = (p.n_heads + kGQ - 1) / kGQ;
    a.q_img = static_cast<uint8_t*>(q_img);
    a.part_ml = part_ml;
    a.part_o = part_o;
    a.status = dev_status;
    a.wait_ns = wait_limit_ns();
    a.premix = plan.premix ? 1 : 0;
    for (int k = 0; k < 64; ++k)
        a.cb_tab[k] = p.fmt == KVQ_FMT_TQ6 ? kTq6CentroidBits[k] : p.fmt == KVQ_FMT_TQ3 ? kTq3CentroidBits[k & 7] : 0;
    const int64_t items = (int64_t)p.n_seq * p.n_q * a.n_hg * kGQ;
    const int n_sm = sm_count();
    q_image16_kernel<<<(int)std::max<int64_t>(1, std::min<int64_t>((items + 7) / 8, (int64_t)n_sm * 8)), 256, 0, s>>>(a);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    static std::atomic<uint64_t> attr_set{0};
    const uint64_t bit = 1ull << (device & 63);
    if (!(attr_set.load() & bit)) {
        for (auto* k : {mla_decode_tc16_kernel<0>, mla_decode_tc16_kernel<6>, mla_decode_tc16_kernel<3>}) {
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e != cudaSuccess) return e;
        }
        attr_set.fetch_or(bit);
    }
    dim3 grid(plan.n_splits, p.n_seq, p.n_q * a.n_hg);
    auto* kern = (!p.seq_fmt && p.fmt == KVQ_FMT_TQ6) ? mla_decode_tc16_kernel<6>
               : (!p.seq_fmt && p.fmt == KVQ_FMT_TQ3) ? mla_decode_tc16_kernel<3> : mla_decode_tc16_kernel<0>;
    return launch_dependent(kern, grid, dim3(kThreads), kSmemBytes, s, a);
}

}  // namespace kvq
