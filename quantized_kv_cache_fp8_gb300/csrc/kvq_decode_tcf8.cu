// kvq_decode_tcf8.cu — the tensor-core split-T absorbed-MLA decode of the fp8 tier
// (tcgen05 kind::f8f6f4), 16 query-heads a CTA, with the tensor core reading the e4m3
// codes straight from the tiles that the TMA lands: no code is converted.
//
// Same operation as the other decode kernels (colibri PR #399: score
// s_t = tau (q_lat . c_t + q_rope . k_rope_t), context sum_t softmax(s)_t c_t, split-T
// partials merged by the log-sum-exp combine; Commit 2), as two contractions per tile of
// 128 rows whose operands are all e4m3:
//
//   S^T[rows x 80]  = C_tile[rows x 576] . Qd^T     rows on M = 128; N = 5 digits x 16 heads
//   O^T[dims x 64] += V_tile^T[dims x rows] . Wd^T  dims on M (4 M-tiles); N = 4 digits x 16
//
// Each 128-dim block of a tile's latent codes is one [128 rows x 128 B] box, 128B-swizzled:
// the score MMA reads it K-major (rows on M) and the context MMA reads the same bytes
// MN-major (dims on M), so one copy of the codes serves both.  The rope key is a
// [128 x 64 B] box, 64B-swizzled.  The per-row scales stay outside the MMAs: the softmax
// applies them to the scores in fp32 and folds the latent scale into the weights.
//
// The fp32 operands are sums of e4m3 "digits" with power-of-two weights, each digit in
// its own block of N columns so that the fp32 accumulators keep them apart:
//   q_h ~ 2^-sigma_h sum_{j<5} 2^-4j Qd_j     Qd_j = RN_e4m3(r_j 2^(sigma_h + 4j)), r_j the residual
//   w_t ~ sum_{j<4} 2^-4j Wd_j                 (0 <= w_t <= 2^8, see below)
// An e4m3 rounding keeps 4 significant bits, so 5 digits carry q to ~2^-20 and 4 digits
// carry w to ~2^-16 of its value; the product of two e4m3 values is exact and the tensor
// core sums them in fp32 (measured on GB300: error below 3e-7 of the sum of |terms|).
//
// Softmax with two running maxima per head: m_s over the scores (normalizer l = sum_t
// 2^(s_t - m_s)) and m_u over u_t = s_t + log2(latent scale_t) (weights w_t = 2^(u_t - m_u),
// i.e. p_t * scale_t * 2^(m_s - m_u)); each moves only when a tile exceeds it by more than
// 2^8, so every w_t <= 2^8 fits e4m3 and the split's partial output is 2^(m_u - m_s) O.
//
// The e4m3 pattern S.1111.111, which the encoder never writes, reads as 0 in every decode
// kernel; the tensor core would read it as NaN.  A row whose score comes out NaN is
// rescored on the CUDA cores with those bytes cleared in shared memory (so that the
// context MMA reads them as 0 too), and rows outside the split are cleared the same way.
//
// Every wait is bounded (%globaltimer); a timeout sets KVQ_DEV_TIMEOUT, raises a
// CTA-wide abort flag, drains the MMAs and copies in flight and frees tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

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


constexpr int kRT = 128;                  // rows per tile
constexpr int kGQ = 16;                   // query-heads per CTA
constexpr int kGH = 4;                    // heads per softmax warp
constexpr int kHP = 16 / kGH;             // softmax warps per row (lane quarter)
constexpr int kDQ = 5;                    // e4m3 digits of q
constexpr int kDW = 4;                    // e4m3 digits of the weights
constexpr int kNS = kGQ * kDQ;            // score MMA N (column n = 16 digit + head)
constexpr int kNC = kGQ * kDW;            // context MMA N (same order)
constexpr int kBox = kRT * 128;           // [128 rows x 128 dims] e4m3, 128B-swizzled
constexpr int kRopeBox = kRT * 64;        // [128 rows x 64 dims], 64B-swizzled
constexpr int kStageBytes = 4 * kBox + kRopeBox;
constexpr int kStages = 2;
constexpr int kPrefetch = 2;              // tiles are prefetched into L2 this far ahead of their load
                                          // (measured on GB300: 3, 6 and 10 were no faster)
constexpr int kQBlk = kNS * 128;          // Q digits of one 128-dim block: [80 x 128 B]
constexpr int kQRope = 4 * kQBlk;         // offset of the rope digits [80 x 64 B]
constexpr int kQScale = kQRope + kNS * 64;   // 16 floats: 2^-sigma_h
constexpr int kQBytes = kQScale + 64;
constexpr int kWBuf = kRT * kNC;          // W digits: [128 rows (K) x 64 B], MN-major
constexpr int kSmx = 4 * kHP;             // softmax warps: lane quarter w % 4, heads kGH (w / 4) ..
constexpr int kWarpLoad = kSmx;           // TMA loader
constexpr int kWarpS = kSmx + 1;          // score MMA issuer (allocates tensor memory)
constexpr int kWarpC = kSmx + 2;          // context MMA issuer
constexpr int kWarpGather = kSmx + 3;     // two warps: cp.async gather of paged / sparse rows
constexpr int kGatherThreads = 64;        // two rows a thread
constexpr int kThreads = 32 * kWarpGather + kGatherThreads;
constexpr int kPieces = 36 / kHP;         // 16-byte pieces of a row that each head part clears
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLazy = 8.0f;             // a maximum moves only when exceeded by > 2^8
constexpr uint64_t kTimeoutNs = kDefaultWaitNs;   // drains
// tensor memory columns
constexpr uint32_t kColSL = 0;            // latent score digits [0, 80)
constexpr uint32_t kColSR = kNS;          // rope score digits [80, 160)
constexpr uint32_t kColO = 256;           // O^T M-tile m at 256 + 64 m

// shared memory
constexpr int kOffStage = 0;
constexpr int kOffQ = kOffStage + kStages * kStageBytes;
constexpr int kOffW = (kOffQ + kQBytes + 1023) / 1024 * 1024;
constexpr int kOffRed = kOffW + 2 * kWBuf;               // [2][4][16] f32: s and u maxima
constexpr int kOffM = kOffRed + 2 * 4 * 16 * 4;          // m_s[16], m_u[16], al_s[16], al_u[16]
constexpr int kOffFlag = kOffM + 4 * 16 * 4;
constexpr int kOffVote = kOffFlag + 16;                  // [2][kSmx]
constexpr int kOffScratch = kOffVote + 2 * kSmx * 4;     // [kHP][128][kGH] f32: rescored rows
constexpr int kOffBar = kOffScratch + kHP * kRT * kGH * 4;
// full[2][5], empty[2][5] (per box: four latent blocks and the rope key), s_full,
// s_empty, p_full, o_done, drain_s, drain_c, q_full
constexpr int kBoxes = 5;
constexpr int kNumBars = 2 * kStages * kBoxes + 7;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory");
static_assert(kStageBytes % 1024 == 0 && kOffQ % 1024 == 0 && kQRope % 512 == 0 && kQBytes % 16 == 0,
              "swizzle atoms and bulk copies");

struct F8Args {
    CUtensorMap tm_lat, tm_rope;         // fp8 code planes ([128 x 128 B] and [128 x 64 B] boxes)
    int use_tma;                         // tiles arrive by TMA (contiguous rows, or pages)
    int paged;                           // by TMA from pages: two boxes of 64 rows a tile
    kvq_mla_problem p;
    int split_rows, n_splits, n_hg;      // n_hg: head groups of 16
    int fmt_split;                       // skip non-fp8 sequences (another kernel reads them)
    float* part_ml;
    float* part_o;
    uint32_t* status;
    uint64_t wait_ns;                    // limit of the pipeline waits
};


// ------------------------------------------------------------------------------------
// Q digit image of the CTA's 16 heads in shared memory: the B operand of the score MMA,
// K-major, rows n = 16 j + head (digit j).  Latent k in four 128B-swizzled blocks
// [80 x 128 B], rope k in one 64B-swizzled block [80 x 64 B], then 2^-sigma_h per head.
// sigma_h puts max|q_h| in [128, 256): Qd_0 = RN(q 2^sigma), Qd_{j+1} = RN(16 (x_j - Qd_j))
// with x_j the scaled residual (all exact in fp32).  One softmax warp per head: its 18
// values a lane are loaded first thing in the CTA (ahead of the tile loads, which would
// otherwise queue in front of them), the digits written once the tiles are on their way.
// ------------------------------------------------------------------------------------
__device__ __forceinline__ void load_q_head(const kvq_mla_problem& p, int64_t qrow, int h, int lane, float (&y)[18])
{
    if (h < p.n_heads) {
        const int64_t r = qrow + h;
#pragma unroll
        for (int j = 0; j < 16; ++j) y[j] = p.q_lat[r * kDLat + j * 32 + lane];
        y[16] = p.q_rope[r * kDRope + lane];
        y[17] = p.q_rope[r * kDRope + 32 + lane];
    } else {
#pragma unroll
        for (int j = 0; j < 18; ++j) y[j] = 0.0f;
    }
}

__device__ __forceinline__ void write_q_digits(const float (&y)[18], int n, int lane, uint8_t* img)
{
    float mx = 0.0f;
#pragma unroll
    for (int j = 0; j < 18; ++j) mx = fmaxf(mx, fabsf(y[j]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    int e = 0;
    (void)frexpf(mx, &e);                        // mx < 2^e
    const int sigma = mx > 0.0f ? std::min(100, std::max(-100, 8 - e)) : 0;
    const float scale = ldexpf(1.0f, sigma);
#pragma unroll
    for (int j = 0; j < 18; ++j) {
        float x = y[j] * scale;
        const int k = (j & 15) * 32 + lane;      // latent dim (j < 16) or rope dim (j >= 16)
#pragma unroll
        for (int d = 0; d < kDQ; ++d) {
            const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
            const int row = 16 * d + n;
            uint8_t* dst;
            if (j < 16) {
                const int kk = k & 127;
                dst = img + (k >> 7) * kQBlk + row * 128 + (((kk >> 4) ^ (row & 7)) << 4) + (kk & 15);
            } else {
                dst = img + kQRope + row * 64 + (((k >> 4) ^ ((row >> 1) & 3)) << 4) + (k & 15);
            }
            *dst = c;
            x = (x - __half2float(__half(__nv_cvt_fp8_to_halfraw(c, __NV_E4M3)))) * 16.0f;
        }
    }
    if (lane == 0) reinterpret_cast<float*>(img + kQScale)[n] = ldexpf(1.0f, -sigma);
}

struct Shared {
    uint8_t* base;
    __device__ uint8_t* stage(int st) const { return base + kOffStage + st * kStageBytes; }
    __device__ uint8_t* q() const { return base + kOffQ; }
    __device__ uint8_t* w(int b) const { return base + kOffW + b * kWBuf; }
    __device__ float* red(int which) const { return reinterpret_cast<float*>(base + kOffRed) + which * 64; }
    __device__ float* m_s() const { return reinterpret_cast<float*>(base + kOffM); }
    __device__ float* m_u() const { return reinterpret_cast<float*>(base + kOffM) + 16; }
    __device__ float* al_s() const { return reinterpret_cast<float*>(base + kOffM) + 32; }
    __device__ float* al_u() const { return reinterpret_cast<float*>(base + kOffM) + 48; }
    __device__ volatile int* flag() const { return reinterpret_cast<volatile int*>(base + kOffFlag); }
    __device__ volatile int* vote(int par) const { return reinterpret_cast<volatile int*>(base + kOffVote) + kSmx * par; }
    __device__ float* scratch(int hp, int t) const { return reinterpret_cast<float*>(base + kOffScratch) + (hp * kRT + t) * kGH; }
    __device__ uint64_t* bar(int i) const { return reinterpret_cast<uint64_t*>(base + kOffBar) + i; }
    __device__ uint64_t* full(int st, int b) const { return bar(st * kBoxes + b); }
    __device__ uint64_t* empty(int st, int b) const { return bar((kStages + st) * kBoxes + b); }
    __device__ uint64_t* s_full() const { return bar(2 * kStages * kBoxes); }
    __device__ uint64_t* s_empty() const { return bar(2 * kStages * kBoxes + 1); }
    __device__ uint64_t* p_full() const { return bar(2 * kStages * kBoxes + 2); }
    __device__ uint64_t* o_done() const { return bar(2 * kStages * kBoxes + 3); }
    __device__ uint64_t* drain_s() const { return bar(2 * kStages * kBoxes + 4); }
    __device__ uint64_t* drain_c() const { return bar(2 * kStages * kBoxes + 5); }
    __device__ uint64_t* q_full() const { return bar(2 * kStages * kBoxes + 6); }
    __device__ uint32_t* tmem_base() const { return reinterpret_cast<uint32_t*>(base + kOffMisc); }
    __device__ volatile int* abort_flag() const { return reinterpret_cast<volatile int*>(base + kOffMisc + 4); }
};

__device__ __forceinline__ bool give_up(const Shared& sh, uint32_t* status)
{
    *sh.abort_flag() = 1;
    if (status) atomicOr(status, (unsigned)KVQ_DEV_TIMEOUT);
    return false;
}

// Wait for a phase, bounded by %globaltimer.  kSpin: poll the non-blocking test (no
// suspension; for the softmax warps, whose hand-overs are the critical path); otherwise
// try_wait, which may suspend the thread and so leaves the issue slots of its scheduler
// to the softmax warps.  A limit below 100 us (set only to exercise the failure path)
// always polls, since a suspended try_wait can outlast it.
constexpr bool kSmxSpin = true;           // softmax warps poll
constexpr bool kRoleSpin = false;         // loader and MMA issuers sleep in try_wait
template <bool kSpin>
__device__ __forceinline__ bool wait_bar(const Shared& sh, uint64_t* bar, uint32_t parity, uint32_t* status,
                                         uint64_t limit_ns)
{
    const bool spin = kSpin || limit_ns < 100000;
    if (spin ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int k = 0; k < 4; ++k)
            if (spin ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (*sh.abort_flag()) return false;
        if (globaltimer_ns() - t0 > limit_ns) return give_up(sh, status);
    }
}

__device__ __forceinline__ void named_bar_softmax() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kSmx) : "memory"); }

// kGH consecutive columns of the warp's lane quarter
template <int G>
__device__ __forceinline__ void tmem_ld_heads(uint32_t taddr, uint32_t (&r)[G])
{
    static_assert(G == 4 || G == 8, "4 or 8 heads a warp");
    if constexpr (G == 4) tmem_ld_x4(taddr, r);
    else tmem_ld_x8(taddr, r);
}
template <int G>
__device__ __forceinline__ void tmem_st_heads(uint32_t taddr, const uint32_t (&r)[G])
{
    static_assert(G == 4 || G == 8, "4 or 8 heads a warp");
    if constexpr (G == 4) tmem_st_x4(taddr, r);
    else tmem_st_x8(taddr, r);
}

// byte offsets of row t's 16-byte pieces in a stage: piece pc < 32 is latent block pc / 8,
// piece pc % 8; pieces 32..35 are the rope key's
__device__ __forceinline__ uint32_t row_piece(int t, int pc)
{
    return pc < 32 ? (pc >> 3) * kBox + t * 128 + (((pc & 7) ^ (t & 7)) << 4)
                   : 4 * kBox + t * 64 + (((pc - 32) ^ ((t >> 1) & 3)) << 4);
}

// clear every byte of the form S.1111.111 in a 32-bit word
__device__ __forceinline__ uint32_t clear_unwritten(uint32_t w)
{
    const uint32_t m = prmt((w & 0x7F7F7F7Fu) + 0x01010101u, 0u, 0xBA98u);
    return w & ~m;
}

// A row with an unwritten code, for the kGH heads hb .. : score it on the CUDA cores from
// the codes with those bytes cleared and q (fp32), sv[g] = tau2 (ls q_lat . c + rs q_rope . k),
// into `out` in shared memory (so that the caller's scores stay in registers); the warp
// of head part hp also writes the cleared bytes of its kPieces pieces back, so that the
// context MMA reads them as 0.  Rare by construction: the encoder never writes the pattern.
__device__ __noinline__ void rescore_row(uint8_t* stage, int t, int hp, const float* ql, const float* qr,
                                         int nh, float ls, float rs, float tau2, float* out)
{
    float al[kGH], ar[kGH];
#pragma unroll
    for (int g = 0; g < kGH; ++g) al[g] = ar[g] = 0.0f;
    const int hb = kGH * hp;
    for (int pc = 0; pc < 36; ++pc) {
        uint4* ptr = reinterpret_cast<uint4*>(stage + row_piece(t, pc));
        uint4 v = *ptr;
        v.x = clear_unwritten(v.x);
        v.y = clear_unwritten(v.y);
        v.z = clear_unwritten(v.z);
        v.w = clear_unwritten(v.w);
        if (pc / kPieces == hp) *ptr = v;
        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
        const bool rope = pc >= 32;
        const int k0 = rope ? (pc - 32) * 16 : pc * 16;
        for (int e = 0; e < 16; ++e) {
            const float c = __half2float(__half(__nv_cvt_fp8_to_halfraw(
                (__nv_fp8_storage_t)((wd[e >> 2] >> (8 * (e & 3))) & 0xFFu), __NV_E4M3)));
            if (c == 0.0f) continue;
            for (int g = 0; g < kGH; ++g) {
                if (hb + g >= nh) break;
                if (rope) ar[g] = fmaf(qr[(int64_t)(hb + g) * kDRope + k0 + e], c, ar[g]);
                else al[g] = fmaf(ql[(int64_t)(hb + g) * kDLat + k0 + e], c, al[g]);
            }
        }
    }
#pragma unroll
    for (int g = 0; g < kGH; ++g) out[g] = hb + g < nh ? tau2 * fmaf(ls, al[g], rs * ar[g]) : 0.0f;
}

// ====================================================================================
// The decode kernel.
//  * Warps 0-7: softmax.  Thread = row of the tile (lane quarter warp % 4) for the 8 heads
//    8 (warp / 4) .. +7: S digits from tensor memory -> scores, two running maxima per head
//    with lazy updates, O rescale when m_u moves, the weight digits into the MN-major W
//    image; epilogue (thread = output dim) writes the split's (m, l, o) partials.
//  * Warp 8: TMA loader (contiguous rows): five boxes a tile into a two-stage ring.
//  * Warp 9: allocates tensor memory and issues the score MMAs; warp 10 issues the context
//    MMAs.  Each waits only for its own inputs, so neither order holds the other up.
//  * Warps 11-14: paged or sparse rows, gathered with cp.async into the same layout.
// ====================================================================================
__global__ void __launch_bounds__(kThreads, 1) mla_decode_tcf8_kernel(const __grid_constant__ F8Args a)
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
    const int64_t n_cand = p.idx ? (int64_t)p.top_k : (int64_t)L;
    const int64_t r0 = (int64_t)split * a.split_rows;
    const int64_t r1 = min(r0 + (int64_t)a.split_rows, n_cand);
    const int64_t qrow = ((int64_t)s * p.n_q + q) * p.n_heads;
    const bool bad_fmt = seq_fmt_of(p, s) != KVQ_FMT_FP8;
    grid_dependents_launch();                    // the combine may start launching
    if (bad_fmt && a.fmt_split) return;          // the other tier's kernel writes these partials

    if (r0 >= n_cand || bad_fmt) {
        grid_dependency_wait();                  // the workspace may still be read before us
        if (bad_fmt && tid == 0 && split == 0 && a.status) atomicOr(a.status, (unsigned)KVQ_DEV_BAD_FORMAT);
        if (tid < nh) {
            const int64_t sl = (qrow + h0 + tid) * a.n_splits + split;
            a.part_ml[sl * 2] = -INFINITY;
            a.part_ml[sl * 2 + 1] = 0.0f;
        }
        return;
    }
    const kvq_mla_cache& C = p.fp8;
    const int NT = (int)((r1 - r0 + kRT - 1) / kRT);
    const RowCtx rc{&p, s, q, L, r1, p.causal ? (int64_t)L - p.n_q + q : (int64_t)L - 1, &C, a.status};
    const bool tma = a.use_tma != 0;
    // Contiguous rows: the loader sets up the stage barriers itself and requests the first
    // kStages tiles at once, before the CTA-wide setup below (tensor memory, the other
    // barriers, the query loads), which would otherwise delay the first loads by ~1 us.
    const int pre = (tma && !a.paged) ? min(NT, kStages) : 0;
    if (warp == kWarpLoad && pre > 0 && lane == 0) {
        for (int st = 0; st < kStages; ++st) {
            for (int b = 0; b < kBoxes; ++b) {
                mbar_init(sh.full(st, b), 1);
                mbar_init(sh.empty(st, b), 1);
            }
        }
        fence_mbar_init();
        const int64_t row0 = (int64_t)s * p.seq_stride_rows + r0;
        for (int i = 0; i < pre; ++i) {
            const int y = (int)(row0 + (int64_t)i * kRT);
            for (int b = 0; b < kBoxes; ++b) {
                mbar_arrive_expect_tx(sh.full(i, b), b < 4 ? kBox : kRopeBox);
                tma_load_2d(sh.stage(i) + b * kBox, b < 4 ? &a.tm_lat : &a.tm_rope, b < 4 ? 128 * b : 0, y,
                            sh.full(i, b));
            }
        }
    }

    if (warp == kWarpS) {
        if (lane == 0) {
            for (int st = 0; st < kStages && pre == 0; ++st) {
                for (int b = 0; b < kBoxes; ++b) {
                    mbar_init(sh.full(st, b), tma ? 1 : kGatherThreads);   // TMA: the loader; else every gather thread
                    mbar_init(sh.empty(st, b), 1);
                }
            }
            mbar_init(sh.s_full(), 1);
            mbar_init(sh.s_empty(), kSmx);
            mbar_init(sh.p_full(), kSmx);
            mbar_init(sh.o_done(), 1);
            mbar_init(sh.drain_s(), 1);
            mbar_init(sh.drain_c(), 1);
            mbar_init(sh.q_full(), kSmx);            // one arrival per softmax warp (= head)
            *sh.abort_flag() = 0;
            fence_mbar_init();
        }
        __syncwarp();
        tmem_alloc(sh.tmem_base(), 512);
        tmem_relinquish();
    }
    if (tid < kGQ) {
        sh.m_s()[tid] = -INFINITY;
        sh.m_u()[tid] = -INFINITY;
    }
    static_assert(kSmx == kGQ, "one softmax warp per head builds the query digits");
    float qv[18];
    if (warp < kSmx) {
        // with overlap_prior the kernel before this call may still run: the queries, and
        // every write these warps make to the workspace, come after it has completed (an
        // immediate return for an ordinary launch)
        grid_dependency_wait();
        load_q_head(p, qrow, h0 + warp, lane, qv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sh.tmem_base();

    if (warp < kSmx) {
        // ================================ softmax ========================================
        // Control flow is identical in all 256 threads (the named barriers need every one
        // of them); `ok` only guards work and is kept warp-uniform.
        const int wq = warp & 3;                      // TMEM lane quarter
        const int hp = warp >> 2;                     // head part: heads hb .. hb + kGH - 1
        const int hb = kGH * hp;
        const int t = wq * 32 + lane;                 // row within the tile
        const int g16 = lane & 15;                    // head of this lane (warp 0's update)
        const int gl = lane & (kGH - 1);              // head hb + gl after a reduction
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        const float tau2 = p.sm_scale * kLog2e;
        const float* ql = p.q_lat + (qrow + h0) * kDLat;
        const float* qr = p.q_rope + (qrow + h0) * kDRope;
        float* m_s = sh.m_s();
        float* m_u = sh.m_u();
        // row t of the W image: 64 bytes at (t / 8) 512 + (t % 8) 64, 16-byte chunk d (the
        // weight digit d of the 16 heads) at d ^ ((t / 2) % 4); this warp's heads are the
        // chunk's bytes hb .. hb + kGH - 1
        const uint32_t w_row = (t >> 3) * 512 + (t & 7) * 64 + hb;
        const int wx = (t >> 1) & 3;
        float l_lane = 0.0f;                          // sum of p over this warp's rows, head hb + gl
        float G[kGH];                                 // tau2 2^-sigma_h
        write_q_digits(qv, warp, lane, sh.q());
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(sh.q_full());
        bool ok = wait_bar<kSmxSpin>(sh, sh.q_full(), 0u, a.status, a.wait_ns);
        ok = __all_sync(kFull, ok);
        {
            const float* f0 = reinterpret_cast<const float*>(sh.q() + kQScale) + hb;
#pragma unroll
            for (int g = 0; g < kGH; ++g) G[g] = tau2 * f0[g];
        }
        // the pool row and scales of this thread's row, read one tile ahead
        int64_t row_n = rc.row(r0 + t, hp == 0);
        float ls_n = row_n >= 0 ? C.lat_scale[row_n] : 0.0f;
        float rs_n = row_n >= 0 ? C.rope_scale[row_n] : 0.0f;
        for (int i = 0; i < NT; ++i) {
            const int st = i % kStages;
            const int64_t row = row_n;
            const float ls = ls_n, rs = rs_n;
            if (i + 1 < NT) {
                row_n = rc.row(r0 + (int64_t)(i + 1) * kRT + t, hp == 0);
                ls_n = row_n >= 0 ? C.lat_scale[row_n] : 0.0f;
                rs_n = row_n >= 0 ? C.rope_scale[row_n] : 0.0f;
            }
            if (ok) ok = wait_bar<kSmxSpin>(sh, sh.s_full(), (uint32_t)i & 1u, a.status, a.wait_ns);
            ok = __all_sync(kFull, ok);
            float sv[kGH];
#pragma unroll
            for (int g = 0; g < kGH; ++g) sv[g] = 0.0f;
            if (ok) {
                tc_fence_after();
                uint32_t xl[kDQ][kGH], xr[kDQ][kGH];
#pragma unroll
                for (int d = 0; d < kDQ; ++d) {
                    tmem_ld_heads(tmem + lane_base + kColSL + 16 * d + hb, xl[d]);
                    tmem_ld_heads(tmem + lane_base + kColSR + 16 * d + hb, xr[d]);
                }
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sh.s_empty());
#pragma unroll
                for (int g = 0; g < kGH; ++g) {
                    float al = __uint_as_float(xl[kDQ - 1][g]), ar = __uint_as_float(xr[kDQ - 1][g]);
#pragma unroll
                    for (int d = kDQ - 2; d >= 0; --d) {
                        al = fmaf(al, 0.0625f, __uint_as_float(xl[d][g]));
                        ar = fmaf(ar, 0.0625f, __uint_as_float(xr[d][g]));
                    }
                    sv[g] = G[g] * fmaf(ls, al, rs * ar);
                }
            }
            float u[kGH];
            if (row < 0) {
                // outside the split: clear the row in the stage so that the context MMA reads
                // zeros (whatever bytes the box brought in); each head part clears kPieces
                if (ok) {
                    uint8_t* stg = sh.stage(st);
                    for (int pc = kPieces * hp; pc < kPieces * hp + kPieces; ++pc)
                        *reinterpret_cast<uint4*>(stg + row_piece(t, pc)) = make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int g = 0; g < kGH; ++g) sv[g] = u[g] = -INFINITY;
            } else {
                bool bad = false;
#pragma unroll
                for (int g = 0; g < kGH; ++g) bad |= isnan(sv[g]);
                if (bad && ok) {
                    rescore_row(sh.stage(st), t, hp, ql, qr, nh, ls, rs, tau2, sh.scratch(hp, t));
#pragma unroll
                    for (int g = 0; g < kGH; ++g) sv[g] = sh.scratch(hp, t)[g];
                }
                const float lg = ls > 0.0f ? log2f(ls) : -INFINITY;
#pragma unroll
                for (int g = 0; g < kGH; ++g) {
                    if (!ok) sv[g] = -INFINITY;
                    u[g] = sv[g] + lg;
                }
            }
            // The running maxima move only when a tile exceeds them by more than 2^kLazy.
            // Each warp votes whether one of its rows does; the votes of tile i sit in buffer
            // i % 2, so every warp reads the same eight votes and takes the same path
            // through the barriers below.
            bool exceed = false;
#pragma unroll
            for (int g4 = 0; g4 < kGH; g4 += 4) {
                const float4 ms = *reinterpret_cast<const float4*>(m_s + hb + g4);
                const float4 mu = *reinterpret_cast<const float4*>(m_u + hb + g4);
                exceed |= sv[g4] > ms.x + kLazy || sv[g4 + 1] > ms.y + kLazy || sv[g4 + 2] > ms.z + kLazy ||
                          sv[g4 + 3] > ms.w + kLazy || u[g4] > mu.x + kLazy || u[g4 + 1] > mu.y + kLazy ||
                          u[g4 + 2] > mu.z + kLazy || u[g4 + 3] > mu.w + kLazy;
            }
            exceed = __any_sync(kFull, exceed);
            if (lane == 0) sh.vote(i & 1)[warp] = exceed ? 1 : 0;
            named_bar_softmax();
            bool rescale_o = false;
            {
                volatile int* v = sh.vote(i & 1);
                int any_vote = 0;
#pragma unroll
                for (int w = 0; w < kSmx; ++w) any_vote |= v[w];
                if (any_vote) {
                    float mx[kGH], mv[kGH];
#pragma unroll
                    for (int g = 0; g < kGH; ++g) {
                        mx[g] = sv[g];
                        mv[g] = u[g];
                    }
                    warp_reduce_transpose<true>(mx, lane);
                    warp_reduce_transpose<true>(mv, lane);
                    if (lane < kGH) {
                        sh.red(0)[wq * kGQ + hb + lane] = mx[0];
                        sh.red(1)[wq * kGQ + hb + lane] = mv[0];
                    }
                    named_bar_softmax();
                    if (warp == 0) {
                        // lanes l and l + 16 compute the same head; lanes 0..15 store it
                        const float* rsd = sh.red(0);
                        const float* rud = sh.red(1);
                        const float ts = fmaxf(fmaxf(rsd[g16], rsd[16 + g16]), fmaxf(rsd[32 + g16], rsd[48 + g16]));
                        const float tu = fmaxf(fmaxf(rud[g16], rud[16 + g16]), fmaxf(rud[32 + g16], rud[48 + g16]));
                        const float ms = m_s[g16], mu = m_u[g16];
                        const bool ups = ts > ms + kLazy || (ms == -INFINITY && ts > -INFINITY);
                        const bool upu = tu > mu + kLazy || (mu == -INFINITY && tu > -INFINITY);
                        const float as = !ups ? 1.0f : (ms == -INFINITY) ? 0.0f : exp2f(ms - ts);
                        const float au = !upu ? 1.0f : (mu == -INFINITY) ? 0.0f : exp2f(mu - tu);
                        const bool any = __any_sync(kFull, upu && i > 0);   // also orders the reads
                        if (lane < kGQ) {
                            if (ups) m_s[lane] = ts;
                            if (upu) m_u[lane] = tu;
                            sh.al_s()[lane] = as;
                            sh.al_u()[lane] = au;
                        }
                        if (lane == 0) *sh.flag() = any ? 1 : 0;
                    }
                    named_bar_softmax();
                    rescale_o = *sh.flag() != 0;
                    l_lane *= sh.al_s()[hb + gl];
                }
            }
            // p for the normalizer, w for the context, split into e4m3 digits: digit d of
            // heads hb .. hb + kGH - 1 in wd[d] (byte g = head hb + g)
            float pv[kGH];
            uint32_t wd[kDW][kGH / 4];
#pragma unroll
            for (int g = 0; g < kGH; g += 2) {
                const float2 ms = *reinterpret_cast<const float2*>(m_s + hb + g);
                const float2 mu = *reinterpret_cast<const float2*>(m_u + hb + g);
                pv[g] = sv[g] == -INFINITY ? 0.0f : exp2f(sv[g] - ms.x);
                pv[g + 1] = sv[g + 1] == -INFINITY ? 0.0f : exp2f(sv[g + 1] - ms.y);
                float2 x = make_float2(u[g] == -INFINITY ? 0.0f : exp2f(u[g] - mu.x),
                                       u[g + 1] == -INFINITY ? 0.0f : exp2f(u[g + 1] - mu.y));
#pragma unroll
                for (int d = 0; d < kDW; ++d) {
                    const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
                    if ((g & 2) == 0) wd[d][g >> 2] = (uint32_t)c;
                    else wd[d][g >> 2] |= (uint32_t)c << 16;
                    if (d + 1 < kDW) {
                        const float2 back = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(c, __NV_E4M3)));
                        x.x = (x.x - back.x) * 16.0f;
                        x.y = (x.y - back.y) * 16.0f;
                    }
                }
            }
            // the W buffer of tile i was last read by the context of tile i-2, which the
            // o_done wait of the previous tile covered
            if (ok) {
                uint8_t* wimg = sh.w(i & 1) + w_row;
#pragma unroll
                for (int d = 0; d < kDW; ++d) {
                    if constexpr (kGH == 4) *reinterpret_cast<uint32_t*>(wimg + ((d ^ wx) << 4)) = wd[d][0];
                    else *reinterpret_cast<uint2*>(wimg + ((d ^ wx) << 4)) = make_uint2(wd[d][0], wd[d][1]);
                }
            }
            // Consume o_done's phase i-1 (the context of tile i-1) at every tile, so that this
            // wait and the epilogue's never trail the barrier by more than one phase; it also
            // makes O safe to rescale and keeps p_full from running a phase ahead.
            if (i > 0 && ok) ok = wait_bar<kSmxSpin>(sh, sh.o_done(), (uint32_t)(i - 1) & 1u, a.status, a.wait_ns);
            ok = __all_sync(kFull, ok);
            if (rescale_o && ok) {
                tc_fence_after();
                float au[kGH];
#pragma unroll
                for (int g = 0; g < kGH; ++g) au[g] = sh.al_u()[hb + g];
#pragma unroll 1
                for (int m = 0; m < 4; ++m) {
#pragma unroll
                    for (int d = 0; d < kDW; ++d) {
                        uint32_t x[kGH];
                        const uint32_t col = tmem + lane_base + kColO + kNC * m + 16 * d + hb;
                        tmem_ld_heads(col, x);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < kGH; ++e) x[e] = __float_as_uint(__uint_as_float(x[e]) * au[e]);
                        tmem_st_heads(col, x);
                    }
                }
                tmem_st_wait();
            }
            if (ok) {
                tc_fence_before();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(sh.p_full());
            } else {
#pragma unroll
                for (int g = 0; g < kGH; ++g) pv[g] = 0.0f;
            }
            warp_reduce_transpose<false>(pv, lane);
            l_lane += pv[0];
        }
        // ---- epilogue: l over the 128 rows, O^T -> partials ------------------------------
        if (ok) ok = wait_bar<kSmxSpin>(sh, sh.o_done(), (uint32_t)(NT - 1) & 1u, a.status, a.wait_ns);
        ok = __all_sync(kFull, ok);
        float* red = sh.red(0);
        if (lane < kGH) red[wq * kGQ + hb + lane] = l_lane;
        named_bar_softmax();
        if (*sh.abort_flag()) {
            if (warp == 0 && lane < nh) {
                const int64_t sl = (qrow + h0 + lane) * a.n_splits + split;
                a.part_ml[sl * 2] = INFINITY;
                a.part_ml[sl * 2 + 1] = INFINITY;
            }
        } else if (ok) {
            tc_fence_after();
            if (warp == 0 && lane < nh) {
                const float lt = red[lane] + red[16 + lane] + red[32 + lane] + red[48 + lane];
                const int64_t sl = (qrow + h0 + lane) * a.n_splits + split;
                a.part_ml[sl * 2] = m_s[lane];
                a.part_ml[sl * 2 + 1] = lt;
            }
            float fac[kGH];
#pragma unroll
            for (int g = 0; g < kGH; ++g) {
                const float ms = m_s[hb + g], mu = m_u[hb + g];
                fac[g] = (ms == -INFINITY || mu == -INFINITY) ? 0.0f : exp2f(mu - ms);
            }
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
                const int dim = 128 * m + 32 * wq + lane;
                uint32_t x[kDW][kGH];
#pragma unroll
                for (int d = 0; d < kDW; ++d) tmem_ld_heads(tmem + lane_base + kColO + kNC * m + 16 * d + hb, x[d]);
                tmem_ld_wait();
#pragma unroll
                for (int g = 0; g < kGH; ++g) {
                    float o = __uint_as_float(x[kDW - 1][g]);
#pragma unroll
                    for (int d = kDW - 2; d >= 0; --d) o = fmaf(o, 0.0625f, __uint_as_float(x[d][g]));
                    if (hb + g < nh) a.part_o[((qrow + h0 + hb + g) * a.n_splits + split) * kDLat + dim] = o * fac[g];
                }
            }
        }
    } else if (warp == kWarpLoad) {
        // ================================ TMA loader =====================================
        if (tma) {
            const bool leader = elect_one();
            const int64_t row0 = (int64_t)s * p.seq_stride_rows + r0;   // pool row of candidate r0
            // Tile i+2 can land only once the context of tile i has freed its stage, so a
            // stage refill from DRAM would sit on the critical path; tiles are prefetched
            // into L2 kPrefetch tiles ahead of their load instead.
            constexpr uint32_t kBoxBytes[kBoxes] = {kBox, kBox, kBox, kBox, kRopeBox};
            // paged: the pool row of the 64-row half h of tile j, or -1 when the half holds
            // no admissible row or its page is not in the table (the softmax clears the
            // rows of the stage that are not admissible, whatever they hold)
            auto half_row = [&](int j, int h) -> int {
                const int64_t sr = r0 + (int64_t)j * kRT + 64 * h;
                if (sr >= r1 || sr >= L) return -1;
                const int64_t pr = pool_row_of(p, s, sr);
                return (pr < 0 || pr > (int64_t)INT32_MAX - 64) ? -1 : (int)pr;
            };
            auto prefetch = [&](int j) {
                if (leader && j < NT && !a.paged) {
                    const int y = (int)(row0 + (int64_t)j * kRT);
#pragma unroll
                    for (int b = 0; b < 4; ++b) tma_prefetch_2d(&a.tm_lat, 128 * b, y);
                    tma_prefetch_2d(&a.tm_rope, 0, y);
                }
            };
            for (int j = kStages; j < kPrefetch; ++j) prefetch(j);
            for (int j = 0; j < pre; ++j) prefetch(j + kPrefetch);
            bool ok = true;
            int i = pre;                              // the first `pre` tiles went out at the start
            int nb = pre * kBoxes;                    // boxes issued
            int hy0 = 0, hy1 = 0;                     // paged: pool rows of tile i's halves
            if (a.paged) {
                hy0 = half_row(0, 0);
                hy1 = half_row(0, 1);
            }
            for (; i < NT && ok; ++i) {
                const int st = i % kStages;
                const int y = (int)(row0 + (int64_t)i * kRT);
                const int y0 = hy0, y1 = hy1;
                if (a.paged && i + 1 < NT) {          // the next tile's page lookups, in flight
                    hy0 = half_row(i + 1, 0);         // while this tile's boxes wait
                    hy1 = half_row(i + 1, 1);
                }
                // box b of tile i, as soon as the MMAs of tile i-2 are done with box b
                for (int b = 0; b < kBoxes && ok; ++b) {
                    ok = __all_sync(kFull, wait_bar<kRoleSpin>(sh, sh.empty(st, b), ((uint32_t)(i / kStages) & 1u) ^ 1u, a.status, a.wait_ns));
                    if (!ok) break;
                    if (leader) {
                        const CUtensorMap* map = b < 4 ? &a.tm_lat : &a.tm_rope;
                        uint8_t* dst = sh.stage(st) + b * kBox;
                        const int x = b < 4 ? 128 * b : 0;
                        if (!a.paged) {
                            mbar_arrive_expect_tx(sh.full(st, b), kBoxBytes[b]);
                            tma_load_2d(dst, map, x, y, sh.full(st, b));
                        } else {
                            // two boxes of 64 rows; their swizzle is that of one 128-row box
                            const uint32_t half = kBoxBytes[b] / 2;
                            mbar_arrive_expect_tx(sh.full(st, b), (y0 >= 0 ? half : 0u) + (y1 >= 0 ? half : 0u));
                            if (y0 >= 0) tma_load_2d(dst, map, x, y0, sh.full(st, b));
                            if (y1 >= 0) tma_load_2d(dst + half, map, x, y1, sh.full(st, b));
                        }
                    }
                    ++nb;
                }
                if (!ok) break;
                prefetch(i + kPrefetch);
                __syncwarp();
            }
            // every box issued has landed before the CTA's shared memory is released
            if (leader) {
                for (int k = 0; k < nb; ++k) {
                    const int ti = k / kBoxes, b = k % kBoxes;
                    // the issue of box b of tile ti + 2 implies that tile ti's box b landed
                    if ((ti + kStages) * kBoxes + b < nb) continue;
                    if (!mbar_wait(sh.full(ti % kStages, b), (uint32_t)(ti / kStages) & 1u, kTimeoutNs) && a.status)
                        atomicOr(a.status, (unsigned)KVQ_DEV_TIMEOUT);
                }
            }
            __syncwarp();
        }
    } else if (warp >= kWarpGather) {
        // ================================ cp.async gather ================================
        // Paged or sparse rows: thread = row of the tile, 36 pieces of 16 bytes into the
        // swizzled positions that the boxes would have; rows that are not admissible read
        // as zeros.  Tile i is issued, then tile i-1 waited for and handed over.
        if (!tma) {
            const int tg = tid - 32 * kWarpGather;    // rows tg and tg + 64 of each tile
            bool ok = true;
            int i = 0;
            for (; i < NT && ok; ++i) {
                const int st = i % kStages;
                for (int b = 0; b < kBoxes && ok; ++b)
                    ok = __all_sync(kFull, wait_bar<kRoleSpin>(sh, sh.empty(st, b), ((uint32_t)(i / kStages) & 1u) ^ 1u, a.status, a.wait_ns));
                if (!ok) break;
                uint8_t* stg = sh.stage(st);
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int t = tg + kGatherThreads * hr;
                    const int64_t row = rc.row(r0 + (int64_t)i * kRT + t, false);
                    const uint8_t* lat = row < 0 ? C.lat : C.lat + row * kDLat;
                    const uint8_t* rope = row < 0 ? C.rope : C.rope + row * kDRope;
                    const uint32_t nb = row < 0 ? 0u : 16u;
#pragma unroll
                    for (int pc = 0; pc < 32; ++pc) cp_async16(stg + row_piece(t, pc), lat + 16 * pc, nb);
#pragma unroll
                    for (int pc = 0; pc < 4; ++pc) cp_async16(stg + row_piece(t, 32 + pc), rope + 16 * pc, nb);
                }
                cp_async_commit();
                if (i > 0) {
                    cp_async_wait<1>();
                    fence_proxy_async_smem();
                    for (int b = 0; b < kBoxes; ++b) mbar_arrive(sh.full((i - 1) % kStages, b));
                }
            }
            cp_async_wait_all();
            if (ok && i == NT) {
                fence_proxy_async_smem();
                for (int b = 0; b < kBoxes; ++b) mbar_arrive(sh.full((NT - 1) % kStages, b));
            }
        }
    } else if (warp == kWarpS) {
        // ================================ score MMAs ======================================
        const bool leader = elect_one();
        constexpr uint32_t idesc_s = idesc_e4m3_f32(kRT, kNS, false, false);   // C . Qd^T
        const uint32_t q_addr = smem_u32(sh.q());
        bool ok = __all_sync(kFull, wait_bar<kRoleSpin>(sh, sh.q_full(), 0u, a.status, a.wait_ns));
        for (int i = 0; i < NT && ok; ++i) {
            const int st = i % kStages;
            const uint32_t par = (uint32_t)(i / kStages) & 1u;
            // S(i) overwrites S(i-1): the softmax has read it
            if (i > 0) ok = __all_sync(kFull, wait_bar<kRoleSpin>(sh, sh.s_empty(), (uint32_t)(i - 1) & 1u, a.status, a.wait_ns));
            const uint32_t stg = smem_u32(sh.stage(st));
            // each box's K steps as soon as it has landed
            for (int b = 0; b < kBoxes && ok; ++b) {
                ok = __all_sync(kFull, wait_bar<kRoleSpin>(sh, sh.full(st, b), par, a.status, a.wait_ns));
                if (!ok) break;
                tc_fence_after();
                if (leader) {
                    if (b < 4) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t ad = desc_smem(stg + b * kBox + k * 32, 16, 1024, kSwizzle128);
                            const uint64_t bd = desc_smem(q_addr + b * kQBlk + k * 32, 16, 1024, kSwizzle128);
                            mma_e4m3_ss(tmem + kColSL, ad, bd, idesc_s, (b | k) ? 1u : 0u);
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const uint64_t ad = desc_smem(stg + 4 * kBox + k * 32, 16, 512, kSwizzle64);
                            const uint64_t bd = desc_smem(q_addr + kQRope + k * 32, 16, 512, kSwizzle64);
                            mma_e4m3_ss(tmem + kColSR, ad, bd, idesc_s, k > 0 ? 1u : 0u);
                        }
                        mma_commit(sh.s_full());
                        mma_commit(sh.empty(st, 4));      // the context does not read the rope key
                    }
                }
                __syncwarp();
            }
        }
        // drain: every MMA issued here completes before tensor memory is freed
        if (leader) {
            mma_commit(sh.drain_s());
            if (!mbar_wait(sh.drain_s(), 0, kTimeoutNs) && a.status)
                atomicOr(a.status, (unsigned)KVQ_DEV_TIMEOUT);
        }
        __syncwarp();
    } else if (warp == kWarpC) {
        // ================================ context MMAs ====================================
        const bool leader = elect_one();
        constexpr uint32_t idesc_c = idesc_e4m3_f32(kRT, kNC, true, true);     // V^T . Wd^T, both MN-major
        bool ok = true;
        for (int i = 0; i < NT && ok; ++i) {
            ok = __all_sync(kFull, wait_bar<kRoleSpin>(sh, sh.p_full(), (uint32_t)i & 1u, a.status, a.wait_ns));
            if (!ok) break;
            tc_fence_after();
            const uint32_t stg = smem_u32(sh.stage(i % kStages));
            const uint32_t wb = smem_u32(sh.w(i & 1));
            if (leader) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
#pragma unroll
                    for (int ks = 0; ks < kRT / 32; ++ks) {
                        // A = V^T of M-tile m: 32 rows (4 groups of 8 x 128 B) a step; B = W
                        // digits: 32 rows (4 groups of 8 x 64 B) a step
                        const uint64_t ad = desc_smem(stg + m * kBox + ks * 4096, 16, 1024, kSwizzle128);
                        const uint64_t bd = desc_smem(wb + ks * 2048, 16, 512, kSwizzle64);
                        mma_e4m3_ss(tmem + kColO + kNC * m, ad, bd, idesc_c, (i == 0 && ks == 0) ? 0u : 1u);
                    }
                    mma_commit(sh.empty(i % kStages, m));   // box m is free for tile i+2
                }
                mma_commit(sh.o_done());
            }
            __syncwarp();
        }
        if (leader) {
            mma_commit(sh.drain_c());
            if (!mbar_wait(sh.drain_c(), 0, kTimeoutNs) && a.status)
                atomicOr(a.status, (unsigned)KVQ_DEV_TIMEOUT);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kWarpS) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_mla_decode_tcf8(const kvq_mla_problem& p, const DecodePlan& plan, float* part_ml,
                                   float* part_o, uint32_t* dev_status, cudaStream_t s, bool fmt_split)
{
    F8Args a;
    memset(&a, 0, sizeof(a));
    if (!p.block_table && !p.idx) {
        a.use_tma = make_code_map(&a.tm_lat, p.fp8.lat, p.fp8.n_rows, kDLat, 128) &&
                    make_code_map(&a.tm_rope, p.fp8.rope, p.fp8.n_rows, kDRope, 64) ? 1 : 0;
    } else if (p.block_table && !p.idx && p.page_size % 64 == 0 && plan.split_rows % 64 == 0) {
        // pages of a multiple of 64 rows and splits on 64-row boundaries: each 64-row half
        // of a tile lies in one page
        a.use_tma = make_code_map(&a.tm_lat, p.fp8.lat, p.fp8.n_rows, kDLat, 128, 64) &&
                    make_code_map(&a.tm_rope, p.fp8.rope, p.fp8.n_rows, kDRope, 64, 64) ? 1 : 0;
        a.paged = a.use_tma;
    }
    a.p = p;
    a.split_rows = plan.split_rows;
    a.n_splits = plan.n_splits;
    a.n_hg = (p.n_heads + kGQ - 1) / kGQ;
    a.fmt_split = fmt_split ? 1 : 0;
    a.part_ml = part_ml;
    a.part_o = part_o;
    a.status = dev_status;
    a.wait_ns = wait_limit_ns();
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    static std::atomic<uint64_t> attr_set{0};
    const uint64_t bit = 1ull << (device & 63);
    if (!(attr_set.load() & bit)) {
        e = cudaFuncSetAttribute(mla_decode_tcf8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set.fetch_or(bit);
    }
    // an ordinary launch: the first kernel of the call reads the cache and the queries
    // only after every kernel before it in the stream (an append, say) has completed;
    // with overlap_prior (not in a batch split by tier) a programmatic one, which may start
    // once the kernel before it lets dependents launch
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.n_splits, p.n_seq, p.n_q * a.n_hg);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (p.overlap_prior && !fmt_split) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, mla_decode_tcf8_kernel, a);
}

}  // namespace kvq
