// kvq_q4_decode.cu — decode attention over the paged q4_0 pools (grouped-query,
// head_dim 256): Strata PR #2533, the qsa decode commit.  The query is rotated by the
// orthonormal FWHT256 (the rotation the stored K and V rows carry), each block is
// dequantised as (nibble - 8) * f32(d), and the merged output is rotated back before
// the optional sigmoid gate.
//
// One warp per (split, sequence, KV head) [and half of the 8 query heads when a KV head
// serves 8]; four such warps per CTA, each with its own 3-stage cp.async ring of 16-row
// tiles (the K and V rows of 16 positions, 4.5 KB); three CTAs per SM.  A warp computes
// tile i + 1's scores and tile i's context in one straight-line body.  Each landed row is
// rewritten in place as its 8 blocks' code bytes (16-byte aligned) and then its 8 scales,
// so the operands come from ldmatrix and 16-byte loads instead of 2-byte ones.
// Both contractions of a tile run on the tensor cores with register operands
// (mma.sync m16n8k16, fp16 in, fp32 out; the operands are built in registers, so
// there is no shared-memory or tensor-memory operand image to stage):
//   score    S[row][n]  = sum_k (code - 8)[row][k] * Q[k][n]      per 32-element block,
//                         then sum over blocks of d_K[row][block] * S_block
//   context  O[dim][n] += sum_row (code - 8)[row][dim] * P[row][n][block(dim)]
// The codes are exact in fp16: one lop3 puts two nibbles into the mantissas of 1024 + c
// and one packed subtract (or fma, for high nibbles) leaves c - 8.  The fp32 operands
// (the rotated query; P = p * d_V) are split into fp16 value + fp16 residual columns
// (n = 2 * head + part), so the products keep ~22 bits; a power-of-two scale keeps
// them inside the fp16 range (fixed per split for Q, per tile for P with the running
// output rescaled when it changes).  Split-T partials (m, l, o in the rotated domain,
// log2 units) are merged by a combine kernel that also rotates back and gates.
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cmath>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kRowBytes = 144;           // 8 blocks of 18 bytes
constexpr int kMaxDevices = 64;

struct Q4Args {
    kvq_q4_problem p;
    int split_rows, n_splits;
    int n_hg;                            // warps per (split, sequence, KV head): 2 when 8 heads share it
    int64_t n_units;                     // n_splits * n_seq * n_kv * n_hg
    float* part_ml;                      // [n_seq][n_qh][n_splits][2]
    float* part_o;                       // [n_seq][n_qh][n_splits][256]
    float* out;
    float* lse;
    uint32_t* status;
};

// FWHT256 of a row held as 8 consecutive elements per lane (element 8 * lane + k):
// stages h = 1, 2, 4 inside the lane, h = 8 .. 128 across lanes, in that order.
__device__ __forceinline__ void fwht256_lane8(float (&z)[8], int lane)
{
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if ((k & h) == 0) {
                const float a = z[k], b = z[k + h];
                z[k] = a + b;
                z[k + h] = a - b;
            }
        }
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const float sgn = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float o = __shfl_xor_sync(kFull, z[k], m);
            z[k] = fmaf(sgn, z[k], o);
        }
    }
}

__device__ __forceinline__ float exp2i(int k)             // 2^k, k in [-126, 127]
{
    return __int_as_float((k + 127) << 23);
}

__device__ __forceinline__ float h2f(uint16_t bits) { return __half2float(__ushort_as_half(bits)); }

// {lo, hi} -> f16x2 (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void unpack_h2(uint32_t h, float& lo, float& hi)
{
    asm("{.reg .b16 l, h; mov.b32 {l, h}, %2; cvt.f32.f16 %0, l; cvt.f32.f16 %1, h;}"
        : "=f"(lo), "=f"(hi) : "r"(h));
}

// The fp16 values (part 0) or the fp16 residuals x - f16(x) (part 1) of a pair.
__device__ __forceinline__ uint32_t split_pair(float x, float y, float part)
{
    float hx, hy;
    unpack_h2(pack_h2(x, y), hx, hy);
    return pack_h2(fmaf(-part, hx, x), fmaf(-part, hy, y));
}

// Nibbles at bits 0-3 and 16-19 of x as f16x2 {c - 8, c' - 8}: 0x6400 | c is 1024 + c.
__device__ __forceinline__ uint32_t nib_lo(uint32_t x)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "r"(0x000F000Fu), "r"(0x64006400u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(r), "r"(0x64086408u));        // - 1032
    return r;
}

// Nibbles at bits 4-7 and 20-23: 0x6400 | 16c is 1024 + 16c; (1024 + 16c) / 16 - 72 = c - 8.
__device__ __forceinline__ uint32_t nib_hi(uint32_t x)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "r"(0x00F000F0u), "r"(0x64006400u));
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(r), "r"(0x2C002C00u), "r"(0xD480D480u));
    return r;
}

// D += A (16 x 16, row-major) * B (16 x 8, column-major), fp16 in, fp32 accumulate
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Four 8 x 8 matrices of 16-bit elements (a code byte pair each) from shared memory; lanes
// 8m .. 8m + 7 give the 16-byte rows of matrix m.  Lane (g, t) receives elements 2t, 2t + 1
// of row g (plain) or elements g of rows 2t, 2t + 1 (transposed): the A fragments of
// m16n8k16 for rows on M (score) and for V^T (context).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}

// A staged row of 8 blocks [scale (2 B) | 16 code bytes] rewritten in place as the 8
// blocks' code bytes (block b at 16 b, 16-byte aligned for ldmatrix) followed by the 8
// binary16 scales (block b at 128 + 2 b).  Block 2e starts at word 9e, so its scale is
// the low half of that word and its codes straddle words; block 2e + 1's scale is the
// high half of word 9e + 4 and its codes are words 9e + 5 .. 9e + 8.  Returns the row's
// largest |scale| as binary16 bits.
__device__ __forceinline__ uint32_t repack_row(uint8_t* row)
{
    uint4* r4 = reinterpret_cast<uint4*>(row);
    uint32_t w[36];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        const uint4 v = r4[i];
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
    uint32_t c[32], s[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            c[8 * e + k] = __byte_perm(w[9 * e + k], w[9 * e + k + 1], 0x5432);
            c[8 * e + 4 + k] = w[9 * e + 5 + k];
        }
        s[e] = __byte_perm(w[9 * e], w[9 * e + 4], 0x7610);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) r4[i] = make_uint4(c[4 * i], c[4 * i + 1], c[4 * i + 2], c[4 * i + 3]);
    r4[8] = make_uint4(s[0], s[1], s[2], s[3]);
    const uint32_t m2 = __vmaxu2(__vmaxu2(s[0] & 0x7FFF7FFFu, s[1] & 0x7FFF7FFFu),
                                 __vmaxu2(s[2] & 0x7FFF7FFFu, s[3] & 0x7FFF7FFFu));
    return max(m2 & 0xFFFFu, m2 >> 16);
}

// binary16 scale of block b from a row's four scale words
__device__ __forceinline__ float scale_of(const uint4& s, int b)
{
    const uint32_t w = (b >> 1) == 0 ? s.x : (b >> 1) == 1 ? s.y : (b >> 1) == 2 ? s.z : s.w;
    return h2f((uint16_t)((b & 1) ? (w >> 16) : (w & 0xFFFFu)));
}

constexpr int kTileRows = 16;
constexpr int kStages = 3;
constexpr int kWarps = 4;
constexpr int kStageBytes = 2 * kTileRows * kRowBytes;    // K rows 0..15, then V rows 0..15

// dynamic shared memory: per warp kStages tiles, then per warp the score's B fragments
// (8 blocks x 32 lanes x 16 B), then per warp kStages row-validity masks.  The rotated
// query rows (fp32, at most 4 KB) are built in the last stage, which the prologue leaves
// free.
constexpr int kFragBytes = 8 * 32 * 16;
constexpr size_t kQ4SmemBytes = (size_t)kWarps * (kStages * kStageBytes + kFragBytes + kStages * 4);
static_assert(4 * 256 * 4 <= kStageBytes, "query scratch must fit in one stage");

template <int GH>   // query heads per warp: 1, 2 or 4
__global__ void __launch_bounds__(32 * kWarps, 3) q4_decode_kernel(const __grid_constant__ Q4Args a)
{
    extern __shared__ __align__(16) uint8_t q4_smem[];
    grid_dependents_launch();                        // the combine may start launching
    const kvq_q4_problem& p = a.p;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t u = (int64_t)blockIdx.x * kWarps + warp;
    if (u >= a.n_units) return;
    const int hh = (int)(u % a.n_hg);
    int64_t rest = u / a.n_hg;
    const int kvh = (int)(rest % p.n_kv);
    rest /= p.n_kv;
    const int s = (int)(rest % p.n_seq);
    const int split = (int)(rest / p.n_seq);
    const int64_t head0 = (int64_t)s * p.n_qh + (int64_t)kvh * (p.n_qh / p.n_kv) + hh * GH;
    const int L = min(max(p.seq_len[s], 0), p.max_seq_len);
    const int64_t r0 = (int64_t)split * a.split_rows;
    const int64_t r1 = min(r0 + (int64_t)a.split_rows, (int64_t)L);
    if (r0 >= r1) {
        if (lane < GH) {
            const int64_t sl = (head0 + lane) * a.n_splits + split;
            a.part_ml[sl * 2] = -INFINITY;
            a.part_ml[sl * 2 + 1] = 0.0f;
        }
        return;
    }
    const int g = lane >> 2, t = lane & 3;
    uint8_t (*tiles)[kStageBytes] = reinterpret_cast<uint8_t (*)[kStageBytes]>(q4_smem + warp * kStages * kStageBytes);
    uint4* frag = reinterpret_cast<uint4*>(q4_smem + kWarps * kStages * kStageBytes + warp * kFragBytes);
    unsigned* valid_of = reinterpret_cast<unsigned*>(q4_smem + kWarps * (kStages * kStageBytes + kFragBytes)) + warp * kStages;
    float* qs = reinterpret_cast<float*>(tiles[kStages - 1]);

    // ---- tile loads: lane l copies row l & 15 of K (l < 16) or V (l >= 16), 9 x 16 B
    const int n_tiles = (int)((r1 - r0 + kTileRows - 1) / kTileRows);
    const int64_t cell_stride = (int64_t)p.n_kv * kRowBytes;
    const uint8_t* pool = (lane < 16 ? p.k_pool : p.v_pool) + (int64_t)kvh * kRowBytes;
    const int32_t* table = p.page_table + (int64_t)s * p.max_pages;
    // positions are below 2^31 (seq_len is int32): 32-bit page arithmetic
    auto page_id = [&](int tile) -> int {
        const int pos = (int)r0 + tile * kTileRows + (lane & 15);
        if (pos >= (int)r1) return -1;
        const int page = pos / p.page_size;
        return page < p.max_pages ? __ldg(table + page) : -1;
    };
    auto issue = [&](int tile, int pid) {
        const int pos = (int)r0 + tile * kTileRows + (lane & 15);
        int64_t cell = -1;
        if (pos < (int)r1) {
            cell = (int64_t)pid * p.page_size + (pos - (pos / p.page_size) * p.page_size);
            if (pid < 0 || cell >= p.n_cells) {
                if (a.status) atomicOr(a.status, (unsigned)KVQ_DEV_BAD_PAGE);
                cell = -1;
            }
        }
        const int st = tile % kStages;
        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(tiles[st] + lane * kRowBytes);
        const uint8_t* src = pool + (cell < 0 ? 0 : cell) * cell_stride;
        const uint32_t nb = cell < 0 ? 0u : 16u;     // 0: zero-fill, read nothing
#pragma unroll
        for (int i = 0; i < kRowBytes / 16; ++i) cp_async16(dst + 16 * i, src + 16 * i, nb);
        const unsigned m = __ballot_sync(kFull, cell >= 0) & 0xFFFFu;
        if (lane == 0) valid_of[st] = m;
    };
#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) {
        if (i < n_tiles) issue(i, page_id(i));
        cp_async_commit();
    }
    int pid_next = (kStages - 1 < n_tiles) ? page_id(kStages - 1) : -1;

    // ---- query: rotate, scale into log2 units, choose a power of two for the fp16 split
    const float qmul = p.sm_scale * kLog2e * (1.0f / 16.0f);
    float qmax = 0.0f;
#pragma unroll
    for (int j = 0; j < GH; ++j) {
        const float4* qp = reinterpret_cast<const float4*>(p.q + (head0 + j) * 256 + 8 * lane);
        const float4 x0 = qp[0], x1 = qp[1];
        float z[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        fwht256_lane8(z, lane);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            z[k] *= qmul;
            qmax = fmaxf(qmax, fabsf(z[k]));
        }
        float4* qd = reinterpret_cast<float4*>(qs + j * 256 + 8 * lane);
        qd[0] = make_float4(z[0], z[1], z[2], z[3]);
        qd[1] = make_float4(z[4], z[5], z[6], z[7]);
    }
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(kFull, qmax, w));
    const int qexp = qmax > 0.0f ? (int)((__float_as_uint(qmax) >> 23) & 0xFF) - 127 : 0;
    const int sigma = min(max(13 - qexp, -100), 100);   // max |Q| * 2^sigma in [2^13, 2^14)
    const float qscale = exp2i(sigma), sinv = exp2i(-sigma);
    __syncwarp();
    // B operand of the score: column n = g is head g >> 1, part g & 1; rows k = 2t, 2t+1
    // are code bytes 4t, 4t+2 and rows 2t+8, 2t+9 bytes 4t+1, 4t+3 of the block
    const int jq = g >> 1;
    const float part = (g & 1) ? 1.0f : 0.0f;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        uint32_t w[4];
#pragma unroll
        for (int hn = 0; hn < 2; ++hn) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (jq < GH) v = *reinterpret_cast<const float4*>(qs + jq * 256 + 32 * b + 16 * hn + 4 * t);
            w[2 * hn] = split_pair(v.x * qscale, v.z * qscale, part);
            w[2 * hn + 1] = split_pair(v.y * qscale, v.w * qscale, part);
        }
        frag[b * 32 + lane] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncwarp();                                    // the query scratch becomes a stage again

    float o[8][2][4];
#pragma unroll
    for (int b = 0; b < 8; ++b)
#pragma unroll
        for (int k = 0; k < 4; ++k) o[b][0][k] = o[b][1][k] = 0.0f;
    float m_run = -INFINITY, l_run = 0.0f;           // head t (t < GH)
    int tau = 40;                                    // P carries 2^tau
    const bool head_ok = t < GH;

    // scores of rows g and g + 8 of a repacked tile for head t (unscaled); aK is the
    // tile's shared-memory address
    auto scores = [&](uint32_t aK, const uint8_t* sK, float& sg, float& sg8) {
        sg = 0.0f;
        sg8 = 0.0f;
        const uint4 dg = *reinterpret_cast<const uint4*>(sK + g * kRowBytes + 128);
        const uint4 dg8 = *reinterpret_cast<const uint4*>(sK + (g + 8) * kRowBytes + 128);
        // lanes 0..15 give rows 0..15 of block 2bp, lanes 16..31 those of block 2bp + 1
        const uint32_t arow = aK + (lane & 15) * kRowBytes + 16 * (lane >> 4);
#pragma unroll
        for (int bp = 0; bp < 4; ++bp) {
            uint32_t x[4];                           // code bytes 4t..4t+3 of rows g, g + 8
            ldsm_x4(arow + 32 * bp, x);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int b = 2 * bp + h;
                const uint32_t xg = x[2 * h], xg8 = x[2 * h + 1];
                const uint4 bq = frag[b * 32 + lane];
                float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                mma16816(c, nib_lo(xg), nib_lo(xg8), nib_lo(xg >> 8), nib_lo(xg8 >> 8), bq.x, bq.y);
                mma16816(c, nib_hi(xg), nib_hi(xg8), nib_hi(xg >> 8), nib_hi(xg8 >> 8), bq.z, bq.w);
                sg = fmaf(scale_of(dg, b), c[0] + c[1], sg);
                sg8 = fmaf(scale_of(dg8, b), c[2] + c[3], sg8);
            }
        }
    };
    // online softmax of head t over a tile's 16 rows (lanes of equal t); returns the
    // factor the running output takes before this tile's context, and this tile's
    // weights of head g >> 1 for rows 2t, 2t+1, 2t+8, 2t+9 times 2^tau
    float f = 1.0f, pa = 0.0f, pb = 0.0f, pc = 0.0f, pd = 0.0f;
    auto softmax = [&](float sg, float sg8, unsigned valid, uint32_t dm) {
        const bool vg = head_ok && ((valid >> g) & 1u), vg8 = head_ok && ((valid >> (g + 8)) & 1u);
        const float s0 = vg ? sg * sinv : -INFINITY;
        const float s1 = vg8 ? sg8 * sinv : -INFINITY;
        float mx = fmaxf(s0, s1);
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
        const float m_new = fmaxf(m_run, mx);
        const float alpha = (m_new == m_run) ? 1.0f : exp2f(m_run - m_new);
        const float p0 = vg ? exp2f(s0 - m_new) : 0.0f;
        const float p1 = vg8 ? exp2f(s1 - m_new) : 0.0f;
        float ps = p0 + p1;
        ps += __shfl_xor_sync(kFull, ps, 4);
        ps += __shfl_xor_sync(kFull, ps, 8);
        ps += __shfl_xor_sync(kFull, ps, 16);
        l_run = l_run * alpha + ps;
        m_run = m_new;
        // the tile's largest V block scale bounds P = p * d (p <= 1): P * 2^tau < 2^15;
        // dm is a V row's largest |scale| (lanes 16..31) or 0 (lanes 0..15)
#pragma unroll
        for (int w = 16; w >= 1; w >>= 1) dm = max(dm, __shfl_xor_sync(kFull, dm, w));
        int tau_new = tau;
        if (dm != 0) tau_new = min(tau, 14 - (dm >= 0x400u ? (int)(dm >> 10) - 15 : -15));
        f = alpha * exp2i(tau_new - tau);
        tau = tau_new;
        // B operand of the context: column n = g (head g >> 1, part g & 1), rows
        // k = 2t, 2t+1, 2t+8, 2t+9 of the tile, taken from the score lanes
        const int src = 8 * t + (g >> 1);
        const float pscale = ((g >> 1) < GH) ? exp2i(tau) : 0.0f;
        pa = __shfl_sync(kFull, p0, src) * pscale;
        pb = __shfl_sync(kFull, p0, src + 4) * pscale;
        pc = __shfl_sync(kFull, p1, src) * pscale;
        pd = __shfl_sync(kFull, p1, src + 4) * pscale;
    };
    // context of a repacked tile's V rows (shared-memory address aV) with the current weights
    auto context = [&](uint32_t aV, const uint8_t* sV) {
        if (__any_sync(kFull, f != 1.0f)) {
#pragma unroll
            for (int b = 0; b < 8; ++b)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    o[b][0][k] *= f;
                    o[b][1][k] *= f;
                }
        }
        const uint8_t* v0 = sV + 2 * t * kRowBytes + 128;     // scales of rows 2t, 2t+1, 2t+8, 2t+9
        const uint4 d0 = *reinterpret_cast<const uint4*>(v0);
        const uint4 d1 = *reinterpret_cast<const uint4*>(v0 + kRowBytes);
        const uint4 d2 = *reinterpret_cast<const uint4*>(v0 + 8 * kRowBytes);
        const uint4 d3 = *reinterpret_cast<const uint4*>(v0 + 9 * kRowBytes);
        const uint32_t arow = aV + (lane & 15) * kRowBytes + 16 * (lane >> 4);
#pragma unroll
        for (int bp = 0; bp < 4; ++bp) {
            // A = V^T: m = g is code byte 2g, m = g + 8 byte 2g + 1; k = rows.  X holds the
            // byte pair g of rows 2t, 2t+1, Y that of rows 2t+8, 2t+9.
            uint32_t x[4];
            ldsm_x4_trans(arow + 32 * bp, x);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int b = 2 * bp + h;
                const uint32_t X = x[2 * h], Y = x[2 * h + 1];
                const uint32_t b0 = split_pair(pa * scale_of(d0, b), pb * scale_of(d1, b), part);
                const uint32_t b1 = split_pair(pc * scale_of(d2, b), pd * scale_of(d3, b), part);
                mma16816(o[b][0], nib_lo(X), nib_lo(X >> 8), nib_lo(Y), nib_lo(Y >> 8), b0, b1);
                mma16816(o[b][1], nib_hi(X), nib_hi(X >> 8), nib_hi(Y), nib_hi(Y >> 8), b0, b1);
            }
        }
    };

    // Software pipeline: iteration i computes the scores of tile i + 1 and the context of
    // tile i in one straight-line body (two independent chains for the scheduler), then
    // the softmax of tile i + 1.  Each lane repacks the row it copied once its copies
    // have landed; the warp then reads the tile through ldmatrix.  The last iteration's
    // scores read a stale stage and are discarded.
    const uint32_t tiles_sa = (uint32_t)__cvta_generic_to_shared(tiles[0]);
    cp_async_wait<kStages - 2>();                    // tile 0 has landed
    {
        const uint32_t dm0 = repack_row(tiles[0] + lane * kRowBytes);
        __syncwarp();
        float sg, sg8;
        scores(tiles_sa, tiles[0], sg, sg8);
        softmax(sg, sg8, valid_of[0], lane >= 16 ? dm0 : 0u);
    }
    for (int i = 0; i < n_tiles; ++i) {
        const int ti = i + kStages - 1;
        if (ti < n_tiles) {
            issue(ti, pid_next);
            if (ti + 1 < n_tiles) pid_next = page_id(ti + 1);
        }
        cp_async_commit();
        cp_async_wait<kStages - 2>();                // tile i + 1 has landed
        const int sn = (i + 1) % kStages, sc = i % kStages;
        uint32_t dmn = 0;
        if (i + 1 < n_tiles) dmn = repack_row(tiles[sn] + lane * kRowBytes);
        __syncwarp();
        float sg, sg8;
        scores(tiles_sa + sn * kStageBytes, tiles[sn], sg, sg8);
        context(tiles_sa + sc * kStageBytes + kTileRows * kRowBytes, tiles[sc] + kTileRows * kRowBytes);
        __syncwarp();                                // tile i's stage is refilled next iteration
        if (i + 1 < n_tiles) softmax(sg, sg8, valid_of[sn], lane >= 16 ? dmn : 0u);
    }
    // ---- partials: (m, l) of head t from lane t, o of head t: dims 32b + 16mt + 2g (+1)
    if (t < GH) {
        const int64_t sl = (head0 + t) * a.n_splits + split;
        if (g == 0) {
            a.part_ml[sl * 2] = m_run;
            a.part_ml[sl * 2 + 1] = l_run;
        }
        const float inv = exp2i(-tau);
        float* dst = a.part_o + sl * 256 + 2 * g;
#pragma unroll
        for (int b = 0; b < 8; ++b)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
                *reinterpret_cast<float2*>(dst + 32 * b + 16 * mt) =
                    make_float2((o[b][mt][0] + o[b][mt][1]) * inv, (o[b][mt][2] + o[b][mt][3]) * inv);
    }
}

// One CTA of 8 warps per (sequence, query head): warp w folds splits w, w + 8, ... into
// its partial row (independent loads, lane = 8 dims); the 8 partial rows are summed in
// shared memory, and warp 0 rotates back and gates.
constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(32 * kCombineWarps) q4_combine_kernel(const __grid_constant__ Q4Args a)
{
    __shared__ __align__(16) float s_z[kCombineWarps][256];
    __shared__ float s_l[kCombineWarps];
    const kvq_q4_problem& p = a.p;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row = blockIdx.x;
    const int s = (int)(row / p.n_qh);
    const int L = min(max(p.seq_len[s], 0), p.max_seq_len);
    const int ns = (int)min((int64_t)a.n_splits, ((int64_t)L + a.split_rows - 1) / a.split_rows);
    grid_dependency_wait();                          // the partials of the decode kernel
    const float* ml = a.part_ml + row * a.n_splits * 2;
    float M = -INFINITY;
    for (int S = lane; S < ns; S += 32)
        if (ml[2 * S + 1] > 0.0f) M = fmaxf(M, ml[2 * S]);
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, w));
    float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float Lt = 0.0f;
    const float* po = a.part_o + row * a.n_splits * 256 + 8 * lane;
#pragma unroll 4
    for (int S = warp; S < ns; S += kCombineWarps) {  // every split below ns wrote its row
        const float lS = ml[2 * S + 1];
        const float w = lS > 0.0f ? exp2f(ml[2 * S] - M) : 0.0f;
        Lt = fmaf(w, lS, Lt);
        const float4* src = reinterpret_cast<const float4*>(po + (int64_t)S * 256);
        const float4 x0 = src[0], x1 = src[1];
        z[0] = fmaf(w, x0.x, z[0]); z[1] = fmaf(w, x0.y, z[1]);
        z[2] = fmaf(w, x0.z, z[2]); z[3] = fmaf(w, x0.w, z[3]);
        z[4] = fmaf(w, x1.x, z[4]); z[5] = fmaf(w, x1.y, z[5]);
        z[6] = fmaf(w, x1.z, z[6]); z[7] = fmaf(w, x1.w, z[7]);
    }
    float4* zs = reinterpret_cast<float4*>(&s_z[warp][8 * lane]);
    zs[0] = make_float4(z[0], z[1], z[2], z[3]);
    zs[1] = make_float4(z[4], z[5], z[6], z[7]);
    if (lane == 0) s_l[warp] = Lt;
    __syncthreads();
    if (warp != 0) return;
    Lt = 0.0f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) Lt += s_l[w];
#pragma unroll
    for (int w = 1; w < kCombineWarps; ++w) {
        const float4* zw = reinterpret_cast<const float4*>(&s_z[w][8 * lane]);
        const float4 y0 = zw[0], y1 = zw[1];
        z[0] += y0.x; z[1] += y0.y; z[2] += y0.z; z[3] += y0.w;
        z[4] += y1.x; z[5] += y1.y; z[6] += y1.z; z[7] += y1.w;
    }
    const bool empty = !(Lt > 0.0f);
    const float inv = empty ? 0.0f : 1.0f / (16.0f * Lt);
    fwht256_lane8(z, lane);                          // rotate back, then gate
    float r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) r[k] = z[k] * inv;
    if (p.gate) {
        const float4* gp = reinterpret_cast<const float4*>(p.gate + row * 256 + 8 * lane);
        const float4 g0 = gp[0], g1 = gp[1];
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) r[k] *= 1.0f / (1.0f + expf(-g[k]));
    }
    float4* dst = reinterpret_cast<float4*>(a.out + row * 256 + 8 * lane);
    dst[0] = make_float4(r[0], r[1], r[2], r[3]);
    dst[1] = make_float4(r[4], r[5], r[6], r[7]);
    if (lane == 0 && a.lse) a.lse[row] = empty ? -INFINITY : (M + log2f(Lt)) * kLn2;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

bool plan_q4_decode(const kvq_q4_problem& p, Q4Plan& plan)
{
    plan = Q4Plan();
    int64_t split_rows = p.split_rows;
    if (split_rows <= 0) {
        // about 24 warps per SM over all (sequence, KV head) units: 1.5 waves of the 16
        // resident warps, enough splits to hide the ragged end of each
        const int64_t hg = (p.n_kv > 0 && p.n_qh / p.n_kv == 8) ? 2 : 1;
        const int64_t units = std::max<int64_t>(1, (int64_t)p.n_seq * p.n_kv * hg);
        const int64_t target = (int64_t)sm_count() * 12 * 2;
        const int64_t splits = std::max<int64_t>(1, (target + units - 1) / units);
        split_rows = std::max<int64_t>(64, ((int64_t)p.max_seq_len + splits - 1) / splits);
        split_rows = (split_rows + 15) / 16 * 16;
    }
    plan.split_rows = (int)std::min<int64_t>(split_rows, INT32_MAX);
    plan.n_splits = (int)std::max<int64_t>(1, ((int64_t)p.max_seq_len + split_rows - 1) / split_rows);
    const size_t rows = (size_t)p.n_seq * p.n_qh;
    plan.off_ml = 0;
    plan.off_o = align256(rows * plan.n_splits * 2 * sizeof(float));
    plan.bytes = plan.off_o + align256(rows * plan.n_splits * 256 * sizeof(float));
    return true;
}

cudaError_t launch_q4_decode(const kvq_q4_problem& p, const Q4Plan& plan, float* out, float* lse,
                             void* ws, uint32_t* dev_status, cudaStream_t s)
{
    if (p.n_seq == 0) return cudaSuccess;
    Q4Args a;
    a.p = p;
    a.split_rows = plan.split_rows;
    a.n_splits = plan.n_splits;
    char* base = static_cast<char*>(ws);
    a.part_ml = reinterpret_cast<float*>(base + plan.off_ml);
    a.part_o = reinterpret_cast<float*>(base + plan.off_o);
    a.out = out;
    a.lse = lse;
    a.status = dev_status;
    const int G = p.n_qh / p.n_kv;
    a.n_hg = G == 8 ? 2 : 1;
    a.n_units = (int64_t)plan.n_splits * p.n_seq * p.n_kv * a.n_hg;
    const dim3 grid((unsigned)((a.n_units + kWarps - 1) / kWarps));
    void (*kern)(Q4Args) = nullptr;
    switch (G) {
        case 1: kern = q4_decode_kernel<1>; break;
        case 2: kern = q4_decode_kernel<2>; break;
        case 4:
        case 8: kern = q4_decode_kernel<4>; break;
        default: return cudaErrorInvalidValue;
    }
    // the shared-memory opt-in is set once per (device, kernel)
    static std::atomic<uint32_t> opted[kMaxDevices];
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    const uint32_t bit = 1u << (G == 1 ? 0 : G == 2 ? 1 : 2);
    if (dev >= kMaxDevices || !(opted[dev].load(std::memory_order_acquire) & bit)) {
        e0 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQ4SmemBytes);
        if (e0 != cudaSuccess) return e0;
        if (dev < kMaxDevices) opted[dev].fetch_or(bit, std::memory_order_release);
    }
    kern<<<grid, 32 * kWarps, kQ4SmemBytes, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t rows = (int64_t)p.n_seq * p.n_qh;
    return launch_dependent(q4_combine_kernel, dim3((unsigned)rows), dim3(32 * kCombineWarps), 0, s, a);
}

}  // namespace kvq
