// kvq_codec.cu — quantize-on-append encoders, the q4_0 paged append and the gathers.
//
// Built with --fmad=false: the byte-exact contract of each codec fixes every rounding,
// so no multiply and add may be fused behind the source's back; each fused
// multiply-add the methods specify is written as __fmaf_rn, each division as
// __fdiv_rn (IEEE), each square root as __fsqrt_rn.
//
// All kernels are memory-streaming: one warp per row, coalesced loads of the fp32
// input, shuffles for the Walsh-Hadamard butterflies and the row reductions, and
// 16-byte stores of the packed output staged through shared memory.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <atomic>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kCodecThreads = 256;
constexpr int kCodecWarps = kCodecThreads / 32;

inline int grid_for(int64_t work_items, int per_block)
{
    int64_t g = (work_items + per_block - 1) / per_block;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return (int)g;
}

// ------------------------------------------------------------------------------------
// fp8 (KV8) per-row encode — colibri PR #399, Summary and Commit 1: scale = amax/448,
// codes = e4m3 nearest-even of x / scale, satfinite.
// ------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d)
{
    // cvt.rn.satfinite.e4m3x2.f32: nearest-even, saturating to +-448 (element .x -> low byte)
    uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

// LANES lanes per row (1 <= LANES <= 32, power of two), VPL float4 per lane:
// dim = 4 * VPL * LANES.  Requires 16-byte aligned x rows and 4-byte aligned code rows.
// Warp `warp` of `n_warps` takes every n_warps-th group of 32 / LANES rows.
template <int LANES, int VPL>
__device__ __forceinline__ void encode_fp8_vec_rows(const float* __restrict__ x, int64_t rows, int64_t ldx,
                                                    uint8_t* __restrict__ codes, int64_t ldc,
                                                    float* __restrict__ scales, int64_t warp, int64_t n_warps)
{
    constexpr int kRowsPerWarp = 32 / LANES;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LANES;
    const int l = lane % LANES;
    for (int64_t r0 = warp * kRowsPerWarp; r0 < rows; r0 += n_warps * kRowsPerWarp) {
        const int64_t r = r0 + sub;
        const bool valid = r < rows;
        float4 v[VPL];
        float amax = 0.0f;
        if (valid) {
            const float4* xr = reinterpret_cast<const float4*>(x + r * ldx);
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                v[k] = __ldcs(xr + k * LANES + l);
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[k].x), fabsf(v[k].y)),
                                         fmaxf(fabsf(v[k].z), fabsf(v[k].w))));
            }
        }
#pragma unroll
        for (int o = LANES / 2; o >= 1; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        if (!valid) continue;
        const float s = __fdiv_rn(amax, 448.0f);
        uint32_t* cr = reinterpret_cast<uint32_t*>(codes + r * ldc);
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            uint32_t w = 0;
            if (amax != 0.0f)
                w = e4m3x4(__fdiv_rn(v[k].x, s), __fdiv_rn(v[k].y, s),
                           __fdiv_rn(v[k].z, s), __fdiv_rn(v[k].w, s));
            cr[k * LANES + l] = w;
        }
        if (l == 0) scales[r] = s;
    }
}

template <int LANES, int VPL>
__global__ void __launch_bounds__(kCodecThreads)
encode_fp8_vec_kernel(const float* __restrict__ x, int64_t rows, int64_t ldx,
                      uint8_t* __restrict__ codes, int64_t ldc, float* __restrict__ scales)
{
    encode_fp8_vec_rows<LANES, VPL>(x, rows, ldx, codes, ldc, scales,
                                    (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5,
                                    ((int64_t)gridDim.x * blockDim.x) >> 5);
}

// Any dim / alignment: one warp per row, two passes over the row.
__global__ void __launch_bounds__(kCodecThreads)
encode_fp8_generic_kernel(const float* __restrict__ x, int64_t rows, int dim, int64_t ldx,
                          uint8_t* __restrict__ codes, int64_t ldc, float* __restrict__ scales)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = warp; r < rows; r += n_warps) {
        const float* xr = x + r * ldx;
        float amax = 0.0f;
        for (int i = lane; i < dim; i += 32) amax = fmaxf(amax, fabsf(xr[i]));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        const float s = __fdiv_rn(amax, 448.0f);
        uint8_t* cr = codes + r * ldc;
        for (int i = lane; i < dim; i += 32) {
            uint8_t c = 0;
            if (amax != 0.0f)
                c = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(xr[i], s), __NV_SATFINITE, __NV_E4M3);
            cr[i] = c;
        }
        if (lane == 0) scales[r] = s;
    }
}

// ------------------------------------------------------------------------------------
// Rotated-int4 (TQ4) encode — colibri PR #399, "Why rotated-int4 for the 4-bit tier".
// ------------------------------------------------------------------------------------
__constant__ float c_tq4_thr[15] = {
    kTq4Thresholds[0], kTq4Thresholds[1], kTq4Thresholds[2], kTq4Thresholds[3],
    kTq4Thresholds[4], kTq4Thresholds[5], kTq4Thresholds[6], kTq4Thresholds[7],
    kTq4Thresholds[8], kTq4Thresholds[9], kTq4Thresholds[10], kTq4Thresholds[11],
    kTq4Thresholds[12], kTq4Thresholds[13], kTq4Thresholds[14]};

// The rotated row of the TQ tiers (every width): y = c * FWHT(s (.) x) with element
// k * 32 + lane in y[k], and its radius: per-lane fused sums of squares, then the xor
// butterfly, then the IEEE square root (the pinned reduction order).
template <int VPL>
__device__ __forceinline__ float tq_rotate_row(const float* __restrict__ xr, uint32_t neg, int lane,
                                               float c, float (&y)[VPL])
{
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
        const float v = __ldcs(xr + k * 32 + lane);
        y[k] = ((neg >> k) & 1u) ? -v : v;
    }
    fwht_warp<VPL>(y, lane);
#pragma unroll
    for (int k = 0; k < VPL; ++k) y[k] = __fmul_rn(y[k], c);
    float acc = 0.0f;
#pragma unroll
    for (int k = 0; k < VPL; ++k) acc = __fmaf_rn(y[k], y[k], acc);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, o));
    return __fsqrt_rn(acc);
}

template <int VPL>   // dim = 32 * VPL
__global__ void __launch_bounds__(kCodecThreads)
encode_tq4_kernel(const float* __restrict__ x, int64_t rows, int64_t ldx,
                  const uint32_t* __restrict__ sign_bits, uint8_t* __restrict__ packed,
                  int64_t ldp, float* __restrict__ radius, float c, bool vec_store)
{
    constexpr int kBytes = 16 * VPL;             // dim / 2
    __shared__ float s_thr[16];
    __shared__ __align__(16) uint8_t s_out[kCodecWarps][kBytes];
    if (threadIdx.x < 15) s_thr[threadIdx.x] = c_tq4_thr[threadIdx.x];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    uint32_t neg = 0;                            // bit k: element k*32+lane has sign -1
#pragma unroll
    for (int k = 0; k < VPL; ++k) neg |= ((__ldg(sign_bits + k) >> lane) & 1u) << k;

    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = warp; r < rows; r += n_warps) {
        float y[VPL];
        const float rad = tq_rotate_row<VPL>(x + r * ldx, neg, lane, c, y);
        const float sigma = __fmul_rn(rad, c);
        uint8_t* pr = packed + r * ldp;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            int code = 0;
            if (rad != 0.0f) {
                const float u = __fdiv_rn(y[k], sigma);
                code = (u >= s_thr[7]) ? 8 : 0;           // count of thresholds <= u
                code += (u >= s_thr[code + 3]) ? 4 : 0;
                code += (u >= s_thr[code + 1]) ? 2 : 0;
                code += (u >= s_thr[code]) ? 1 : 0;
            }
            const int hi = __shfl_down_sync(kFull, code, 1);
            if ((lane & 1) == 0) {
                const uint8_t b = (uint8_t)(code | (hi << 4));
                if (vec_store) s_out[wib][k * 16 + (lane >> 1)] = b;
                else pr[k * 16 + (lane >> 1)] = b;
            }
        }
        if (vec_store) {
            __syncwarp();
            if (lane < kBytes / 16)
                reinterpret_cast<uint4*>(pr)[lane] = reinterpret_cast<const uint4*>(s_out[wib])[lane];
            __syncwarp();
        }
        if (lane == 0) radius[r] = rad;
    }
}

// ------------------------------------------------------------------------------------
// The rotated tiers at 3 and 6 bits (colibri PR #399: KV_TQ=6, and 3 bits): the same row
// transform and radius as TQ4, a 2^b-level codebook, and codes packed as a little-endian
// bit stream (code i at bits b*i .. b*i + b - 1 of the row).  24 / b consecutive codes fill
// 3 bytes: lanes combine them with a shuffle tree and the first lane of each group writes
// the 3 bytes into shared memory, which the warp copies out with 16-byte stores.
// ------------------------------------------------------------------------------------

__constant__ TqCodebook<8> c_tq3 = kTq3;
__constant__ TqCodebook<64> c_tq6 = kTq6;

// 64 levels: instead of a six-step bisection, u is placed in one of 257 buckets
// b = round-to-even(32 u + 128) (one fma against 1.5 * 2^23, exact), clamped to [0, 256];
// kTq6Base[b] counts the thresholds below the bucket's lowest possible u (32 u + 128 =
// b - 1/2), and no bucket, edges included, holds more than one threshold (checked below),
// so the code is kTq6Base[b] + (u >= thr[kTq6Base[b]]).  thr[63] is +inf padding.
struct Tq6Buckets {
    uint8_t base[257];
};

constexpr Tq6Buckets tq6_buckets()
{
    Tq6Buckets r{};
    for (int b = 0; b <= 256; ++b) {
        int n = 0;
        for (int k = 0; k < 63; ++k)
            if (kTq6.thr[k] * 32.0f + 128.0f < (float)b - 0.5f) ++n;
        r.base[b] = (uint8_t)n;
    }
    return r;
}

constexpr bool tq6_buckets_hold_one_threshold()
{
    for (int b = 0; b <= 256; ++b) {
        int n = 0;
        for (int k = 0; k < 63; ++k) {
            const float v = kTq6.thr[k] * 32.0f + 128.0f;
            if (v >= (float)b - 0.5f && v <= (float)b + 0.5f) ++n;
        }
        if (n > 1) return false;
    }
    // the clamped end buckets hold no threshold beyond their range
    return kTq6.thr[0] * 32.0f + 128.0f > 0.5f && kTq6.thr[62] * 32.0f + 128.0f < 255.5f;
}
static_assert(tq6_buckets_hold_one_threshold(), "6-bit bucket table needs a finer grid");

constexpr Tq6Buckets kTq6Buckets = tq6_buckets();
__constant__ Tq6Buckets c_tq6_buckets = kTq6Buckets;

template <int BITS>
__device__ __forceinline__ const float* tq_thresholds()
{
    if constexpr (BITS == 3) return c_tq3.thr;
    else return c_tq6.thr;
}

// ------------------------------------------------------------------------------------
// Rotated-tier encode of 512-wide rows, the MLA latent, at 3, 4 or 6 bits, with fewer
// instructions a row than the general kernels (same bytes):
//  * lane l loads elements 16 l .. 16 l + 15 with 16-byte loads; the FWHT stages h = 1..8
//    run in its registers; one transpose through shared memory (element i at i + i/16,
//    conflict-free both ways) gives lane (bit 8 of i, bits 0-3) registers over bits 4-7,
//    so stages h = 16..128 run in registers too and only h = 256 is a shuffle.  The stage
//    order and every rounding are those of the pinned transform.
//  * the radius keeps the pinned order: partial l (i mod 32) sums i = l, l + 32, ...
//    ascending; its first eight terms sit in lane (0, l mod 16), the last eight in lane
//    (1, l mod 16), which continues the lower lane's sum; the xor butterfly follows.
//  * the code counts the thresholds at or below u = y / sigma.  u' = y * rcp(sigma) (both
//    correctly rounded) is within 4.1e-6 of u (|u| <= sqrt 512).  Buckets of width 1/S,
//    b = rn(S u' + B), hold at most one threshold and every threshold lies at least 1e-3
//    from a bucket edge (checked at compile time below), so u and u' share a bucket and
//    the code is base[b] + (u' >= thr[b]) unless u' is within 1e-5 of thr[b]; then the
//    IEEE quotient decides against the same threshold.  A bucket is one 32-bit word: the
//    thresholds are midpoints of binary16 values, so the low 6 bits of their fp32
//    patterns are zero (checked at compile time) and hold base[b]; a bucket without a
//    threshold holds the largest finite float with those bits cleared.
//  * 4 bits: two codes a byte; 3 and 6 bits: 24 / b consecutive codes (consecutive lanes)
//    combine into 3 bytes with a shuffle tree, code i at bits b i of the row's stream.
// ------------------------------------------------------------------------------------
constexpr float kTqNear = 1e-5f;
constexpr uint32_t kTqBaseMask = 63u;          // bits of a bucket word that hold base[b]
constexpr uint32_t kTqNoThreshold = 0x7F7FFFC0u;   // FLT_MAX with the base bits cleared

// the low `nbits` bits of the fp32 pattern of t are zero (t normal or zero)
constexpr bool tq_low_bits_zero(float t, int nbits)
{
    if (t == 0.0f) return true;
    double v = t < 0.0f ? -(double)t : (double)t;
    while (v >= 16777216.0) v *= 0.5;          // the significand as an integer in [2^23, 2^24)
    while (v < 8388608.0) v *= 2.0;
    return (long long)v % (1LL << nbits) == 0;
}
template <int N>
constexpr bool tq_thresholds_packable(const float (&thr)[N])
{
    for (int k = 0; k < N; ++k)
        if (!tq_low_bits_zero(thr[k], 6)) return false;
    return N <= (int)kTqBaseMask;
}
static_assert(tq_thresholds_packable(kTq3.thr) && tq_thresholds_packable(kTq4Thresholds) &&
              tq_thresholds_packable(kTq6.thr), "thresholds leave 6 low bits for the bucket base");

template <int BITS> struct Tq512Grid;
template <> struct Tq512Grid<3> { static constexpr int n = 17;  static constexpr float scale = 4.0f;  static constexpr float off = 8.0f; };
template <> struct Tq512Grid<4> { static constexpr int n = 320; static constexpr float scale = 7.0f;  static constexpr float off = 160.0f; };
template <> struct Tq512Grid<6> { static constexpr int n = 129; static constexpr float scale = 16.0f; static constexpr float off = 64.0f; };

// every threshold strictly inside the unclamped buckets, at least `margin` (in u) from a
// bucket edge, and no two thresholds in one bucket
template <int N>
constexpr bool tq512_grid_ok(const float (&thr)[N], float scale, float off, int nb, double margin)
{
    long long prev = -1;
    for (int k = 0; k < N; ++k) {
        const double v = (double)thr[k] * scale + off;
        if (v <= 0.5 + margin * scale || v >= nb - 1.5 - margin * scale) return false;
        const double f = v - (double)(long long)v;
        const double d = f > 0.5 ? f - 0.5 : 0.5 - f;
        if (d < margin * scale) return false;
        const long long bucket = (long long)(v + 0.5);
        if (bucket == prev) return false;
        prev = bucket;
    }
    return true;
}
static_assert(tq512_grid_ok(kTq3.thr, Tq512Grid<3>::scale, Tq512Grid<3>::off, Tq512Grid<3>::n, 1e-3), "3-bit grid");
static_assert(tq512_grid_ok(kTq4Thresholds, Tq512Grid<4>::scale, Tq512Grid<4>::off, Tq512Grid<4>::n, 1e-3), "4-bit grid");
static_assert(tq512_grid_ok(kTq6.thr, Tq512Grid<6>::scale, Tq512Grid<6>::off, Tq512Grid<6>::n, 1e-3), "6-bit grid");

template <int BITS>
__device__ __forceinline__ const float* tq512_thresholds()
{
    if constexpr (BITS == 3) return c_tq3.thr;
    else if constexpr (BITS == 4) return c_tq4_thr;
    else return c_tq6.thr;
}

// Rows warp, warp + n_warps, ... of the grid's warps; every thread of the CTA calls it
// (the bucket table is built by the CTA)
template <int BITS>
__device__ __forceinline__ void encode_tq512_rows(const float* __restrict__ x, int64_t rows, int64_t ldx,
                                                  const uint32_t* __restrict__ sign_bits,
                                                  uint8_t* __restrict__ packed, int64_t ldp,
                                                  float* __restrict__ radius, bool vec_store,
                                                  int64_t warp, int64_t n_warps)
{
    using G = Tq512Grid<BITS>;
    constexpr int kNThr = (1 << BITS) - 1;
    constexpr int kRowBytes = 64 * BITS;         // 512 codes of BITS bits
    __shared__ uint32_t s_tab[G::n];
    __shared__ float s_t[kCodecWarps][544];
    __shared__ __align__(16) uint8_t s_out[kCodecWarps][kRowBytes];
    __shared__ __align__(16) uint8_t s_code[kCodecWarps][528];
    const float* thr_c = tq512_thresholds<BITS>();
    const int lane = threadIdx.x & 31;
    // each warp walks its rows with the next row's loads in flight during this row's work;
    // the first row's loads are issued before the bucket table is built
    float4 nx[4];
    if (warp < rows) {
        const float4* src = reinterpret_cast<const float4*>(x + warp * ldx) + 4 * lane;
#pragma unroll
        for (int q = 0; q < 4; ++q) nx[q] = __ldcs(src + q);
    }
    for (int b = threadIdx.x; b < G::n; b += blockDim.x) {
        const float lo = ((float)b - G::off - 0.5f) / G::scale;
        const float hi = ((float)b - G::off + 0.5f) / G::scale;
        uint32_t base = 0, t = kTqNoThreshold;
        for (int k = 0; k < kNThr; ++k) {
            base += thr_c[k] < lo;
            if (thr_c[k] >= lo && thr_c[k] < hi) t = __float_as_uint(thr_c[k]);
        }
        s_tab[b] = t | base;
    }
    __syncthreads();
    const int wib = threadIdx.x >> 5;
    const uint32_t neg16 = (__ldg(sign_bits + (lane >> 1)) >> (16 * (lane & 1))) & 0xFFFFu;
    const float c = tq4_inv_sqrt(512);
    const float sgn256 = (lane & 16) ? -1.0f : 1.0f;      // upper half of the h = 256 stage
    float* st = s_t[wib];
    for (int64_t r = warp; r < rows; r += n_warps) {
        float v[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[4 * q] = nx[q].x; v[4 * q + 1] = nx[q].y; v[4 * q + 2] = nx[q].z; v[4 * q + 3] = nx[q].w;
        }
        if (r + n_warps < rows) {
            const float4* src = reinterpret_cast<const float4*>(x + (r + n_warps) * ldx) + 4 * lane;
#pragma unroll
            for (int q = 0; q < 4; ++q) nx[q] = __ldcs(src + q);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j)                       // s_i x_i: flip the sign bit
            v[j] = __uint_as_float(__float_as_uint(v[j]) ^ (((neg16 >> j) & 1u) << 31));
#pragma unroll
        for (int h = 1; h < 16; h <<= 1) {                 // stages h = 1, 2, 4, 8
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if ((j & h) == 0) {
                    const float a = v[j], b = v[j + h];
                    v[j] = __fadd_rn(a, b);
                    v[j + h] = __fsub_rn(a, b);
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) st[17 * lane + j] = v[j];
        __syncwarp();
        // lane L: elements (L >> 4) * 256 + k * 16 + (L & 15), k = 0..15 (register k)
        const int rb = (lane >> 4) * 272 + (lane & 15);
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = st[rb + 17 * k];
        __syncwarp();
#pragma unroll
        for (int h = 1; h < 16; h <<= 1) {                 // stages h = 16, 32, 64, 128
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                if ((k & h) == 0) {
                    const float a = v[k], b = v[k + h];
                    v[k] = __fadd_rn(a, b);
                    v[k + h] = __fsub_rn(a, b);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {                     // stage h = 256, then y = w * c
            const float pv = __shfl_xor_sync(kFull, v[k], 16);
            v[k] = __fmul_rn(__fmaf_rn(sgn256, v[k], pv), c);
        }
        // radius: partial l = ((k & 1) << 4) | (lane & 15); lane's own terms m = k >> 1
        // (+ 8 in the upper half), ascending; the upper half continues the lower's sums
        float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
            a0 = __fmaf_rn(v[k], v[k], a0);
            a1 = __fmaf_rn(v[k + 1], v[k + 1], a1);
        }
        float b0 = __shfl_up_sync(kFull, a0, 16), b1 = __shfl_up_sync(kFull, a1, 16);
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
            b0 = __fmaf_rn(v[k], v[k], b0);
            b1 = __fmaf_rn(v[k + 1], v[k + 1], b1);
        }
        float acc = __fadd_rn(b0, b1);                     // o = 16
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(kFull, acc, o));
        const float rad = __fsqrt_rn(__shfl_sync(kFull, acc, 16));
        const float sigma = __fmul_rn(rad, c);
        const float inv = __frcp_rn(sigma);
        const bool exact_row = !(sigma >= 0x1p-120f);      // tiny sigma: divide every element
        // the code from u' = y * rcp(sigma) and the bucket of u', one byte per element into
        // s_code (element order, elements 256.. 16 bytes further on, so that the two
        // half-warps' byte stores of a register fall in different banks); elements within
        // reach of their bucket's threshold (bit k of `near`) are decided again by the IEEE
        // quotient, which shares the bucket (its threshold is 1e-3 from the edges), except
        // in a row of tiny sigma, where u' is not used at all.  For those decisions a warp
        // with such an element puts y in the (now free) transpose buffer.
        uint8_t* cb = s_code[wib];
        const int eb = (lane >> 4) * 272 + (lane & 15);    // byte of register k: eb + 16 k
        const int cq = lane + (lane >> 4);                 // 16-byte piece of elements 16 lane ..
        uint32_t near = 0;
        auto bucket_of = [&](float u1) {
            const float bf = __fmaf_rn(u1, G::scale, 12582912.0f + G::off);
            return s_tab[min(max(__float_as_int(bf) - 0x4B400000, 0), G::n - 1)];
        };
        if (rad == 0.0f) {                                 // an all-zero row codes to 0
            reinterpret_cast<uint4*>(cb)[cq] = make_uint4(0u, 0u, 0u, 0u);
        } else {
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float u1 = __fmul_rn(v[k], inv);
                const uint32_t e = bucket_of(u1);
                const float thr = __uint_as_float(e & ~kTqBaseMask);
                cb[eb + 16 * k] = (uint8_t)((e & kTqBaseMask) + (u1 >= thr ? 1u : 0u));
                near |= (fabsf(__fsub_rn(u1, thr)) <= kTqNear ? 1u : 0u) << k;
            }
            if (exact_row) near = 0xFFFFu;
        }
        if (__any_sync(kFull, near != 0)) {
#pragma unroll
            for (int k = 0; k < 16; ++k) st[rb + 17 * k] = v[k];
#pragma unroll 1
            for (int k = 0; k < 16; ++k) {
                if ((near >> k) & 1u) {
                    const float y = st[rb + 17 * k];
                    const float u = __fdiv_rn(y, sigma);
                    int c;
                    if (exact_row) {
                        c = 0;
                        for (int t = 0; t < kNThr; ++t) c += (u >= thr_c[t]) ? 1 : 0;
                    } else {
                        const uint32_t e = bucket_of(__fmul_rn(y, inv));
                        c = (int)(e & kTqBaseMask) + (u >= __uint_as_float(e & ~kTqBaseMask) ? 1 : 0);
                    }
                    cb[eb + 16 * k] = (uint8_t)c;
                }
            }
        }
        __syncwarp();
        // lane l packs elements 16l .. 16l + 15: code i at bits BITS i .. of the row
        // (little-endian), i.e. BITS * 2 bytes at byte 2 BITS l
        uint8_t* out = s_out[wib];
        {
            const uint4 c16 = reinterpret_cast<const uint4*>(cb)[cq];
            if constexpr (BITS == 4) {
                const uint32_t t0 = c16.x | (c16.x >> 4), t1 = c16.y | (c16.y >> 4);
                const uint32_t t2 = c16.z | (c16.z >> 4), t3 = c16.w | (c16.w >> 4);
                reinterpret_cast<uint2*>(out)[lane] =
                    make_uint2(__byte_perm(t0, t1, 0x6420), __byte_perm(t2, t3, 0x6420));
            } else {
                const uint32_t cw[4] = {c16.x, c16.y, c16.z, c16.w};
                uint32_t g[4];                              // codes 4j .. 4j + 3 as 4 BITS bits
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    g[j] = (cw[j] & 0xFFu) | ((cw[j] >> 8) & 0xFFu) << BITS |
                           ((cw[j] >> 16) & 0xFFu) << (2 * BITS) | (cw[j] >> 24) << (3 * BITS);
                if constexpr (BITS == 6) {                  // four 24-bit groups: 12 bytes
                    uint32_t* o = reinterpret_cast<uint32_t*>(out + 12 * lane);
                    o[0] = g[0] | g[1] << 24;
                    o[1] = g[1] >> 8 | g[2] << 16;
                    o[2] = g[2] >> 16 | g[3] << 8;
                } else {                                    // four 12-bit groups: 6 bytes
                    uint16_t* o = reinterpret_cast<uint16_t*>(out + 6 * lane);
                    o[0] = (uint16_t)(g[0] | g[1] << 12);
                    o[1] = (uint16_t)(g[1] >> 4 | g[2] << 8);
                    o[2] = (uint16_t)(g[2] >> 8 | g[3] << 4);
                }
            }
        }
        __syncwarp();
        uint8_t* pr = packed + r * ldp;
        if (vec_store) {
            if (lane < kRowBytes / 16) reinterpret_cast<uint4*>(pr)[lane] = reinterpret_cast<const uint4*>(out)[lane];
        } else {
            for (int q = lane; q < kRowBytes; q += 32) pr[q] = out[q];
        }
        __syncwarp();
        if (lane == 0) radius[r] = rad;
    }
}

template <int BITS>
__global__ void __launch_bounds__(kCodecThreads)
encode_tq512_kernel(const float* __restrict__ x, int64_t rows, int64_t ldx,
                    const uint32_t* __restrict__ sign_bits, uint8_t* __restrict__ packed,
                    int64_t ldp, float* __restrict__ radius, bool vec_store)
{
    encode_tq512_rows<BITS>(x, rows, ldx, sign_bits, packed, ldp, radius, vec_store,
                            (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5,
                            ((int64_t)gridDim.x * blockDim.x) >> 5);
}

// ------------------------------------------------------------------------------------
// Quantize-on-append of MLA rows in one launch: blockIdx.y = 0 encodes the latent rows
// (512 dims; BITS = 8: fp8, else the rotated tier at BITS bits), blockIdx.y = 1 the rope
// keys (64 dims, fp8), with the device code of the separate encoders (the same bytes).
// Both sets of CTAs run at once; a per-token append is one launch instead of two.
// ------------------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(kCodecThreads)
encode_mla_kernel(const float* __restrict__ c_lat, int64_t ldx, const float* __restrict__ k_rope,
                  int64_t ldr, int64_t rows, const uint32_t* __restrict__ sign_bits,
                  uint8_t* __restrict__ lat, int64_t ldl, float* __restrict__ lat_scale,
                  uint8_t* __restrict__ rope, int64_t ldc, float* __restrict__ rope_scale, bool vec_store)
{
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    if (blockIdx.y == 1) {
        encode_fp8_vec_rows<4, 4>(k_rope, rows, ldr, rope, ldc, rope_scale, warp, n_warps);
    } else {
        if constexpr (BITS == 8)
            encode_fp8_vec_rows<32, 4>(c_lat, rows, ldx, lat, ldl, lat_scale, warp, n_warps);
        else
            encode_tq512_rows<BITS>(c_lat, rows, ldx, sign_bits, lat, ldl, lat_scale, vec_store, warp, n_warps);
    }
}

template <int VPL, int BITS>   // dim = 32 * VPL
__global__ void __launch_bounds__(kCodecThreads, 4)
encode_tqb_kernel(const float* __restrict__ x, int64_t rows, int64_t ldx,
                  const uint32_t* __restrict__ sign_bits, uint8_t* __restrict__ packed,
                  int64_t ldp, float* __restrict__ radius, float c, bool vec_store)
{
    constexpr int kL = 1 << BITS;
    constexpr int kBytes = 4 * VPL * BITS;       // dim * BITS / 8
    constexpr int kG = 24 / BITS;                // codes per 3 bytes
    constexpr bool kVecOk = kBytes % 16 == 0;
    __shared__ float s_thr[kL];
    __shared__ uint8_t s_base[BITS == 6 ? 257 : 1];
    __shared__ __align__(16) uint8_t s_out[kCodecWarps][kBytes];
    for (int i = threadIdx.x; i < kL; i += blockDim.x)
        s_thr[i] = i < kL - 1 ? tq_thresholds<BITS>()[i] : INFINITY;
    if constexpr (BITS == 6)
        for (int i = threadIdx.x; i < 257; i += blockDim.x) s_base[i] = c_tq6_buckets.base[i];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    uint32_t neg = 0;
#pragma unroll
    for (int k = 0; k < VPL; ++k) neg |= ((__ldg(sign_bits + k) >> lane) & 1u) << k;
    const bool vec = kVecOk && vec_store;

    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = warp; r < rows; r += n_warps) {
        float y[VPL];
        const float rad = tq_rotate_row<VPL>(x + r * ldx, neg, lane, c, y);
        const float sigma = __fmul_rn(rad, c);
        uint8_t* pr = packed + r * ldp;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            uint32_t code = 0;
            if (rad != 0.0f) {
                const float u = __fdiv_rn(y[k], sigma);
                if constexpr (BITS == 6) {
                    const int b = __float_as_int(fmaf(u, 32.0f, 128.0f + 12582912.0f)) - 0x4B400000;
                    code = s_base[min(max(b, 0), 256)];
                    code += (u >= s_thr[code]) ? 1u : 0u;
                } else {
                    // count of thresholds <= u, by bisection over the sorted thresholds
#pragma unroll
                    for (int step = kL / 2; step >= 1; step >>= 1)
                        code += (u >= s_thr[code + step - 1]) ? step : 0;
                }
            }
            uint32_t v = code;
#pragma unroll
            for (int w = 1; w < kG; w <<= 1) v |= __shfl_down_sync(kFull, v, w) << (BITS * w);
            if (lane % kG == 0) {
                const int off = (k * 32 + lane) * BITS / 8;
                uint8_t* dst = vec ? s_out[wib] + off : pr + off;
                dst[0] = (uint8_t)v;
                dst[1] = (uint8_t)(v >> 8);
                dst[2] = (uint8_t)(v >> 16);
            }
        }
        if (vec) {
            __syncwarp();
            for (int i = lane; i < kBytes / 16; i += 32)
                reinterpret_cast<uint4*>(pr)[i] = reinterpret_cast<const uint4*>(s_out[wib])[i];
            __syncwarp();
        }
        if (lane == 0) radius[r] = rad;
    }
}

// ------------------------------------------------------------------------------------
// q4_0 — Strata PR #2533, kv_q4.metal port commit: fwht256 (one warp a row, 8 values a
// lane, orthonormal 1/16), q4_group / q4_store with the |x| tie rule, the fp16 scale,
// int(fma(x, id, 8.5)) truncating toward zero.
// ------------------------------------------------------------------------------------

// "a is preferred over b": larger |.|, then larger value, then +0 over -0.  A total
// order, so a butterfly reduction gives the same winner in every lane.
__device__ __forceinline__ bool q4_prefer(float a, float b)
{
    const float fa = fabsf(a), fb = fabsf(b);
    if (fa != fb) return fa > fb;
    if (a != b) return a > b;
    return !signbit(a) && signbit(b);
}

// q4_prefer as an integer order: key(a) > key(b) exactly when a is preferred over b, for
// every a, b that are not NaN: |a| in the upper 31 bits, "not negative" in bit 0 (a
// larger |.| first; among equal |.| the positive one, or +0 over -0).  A NaN's key lies
// above that of +inf (0xFF000001).
__device__ __forceinline__ uint32_t q4_key(float a)
{
    const uint32_t u = __float_as_uint(a);
    return ((u & 0x7FFFFFFFu) << 1) | (~u >> 31);
}

// cell of (sequence s, position pos), or -1 (and the status bit) when outside
__device__ __forceinline__ int64_t q4_cell(const int32_t* __restrict__ page_table, int max_pages,
                                           int page_size, int64_t n_cells, int s, int pos)
{
    if (pos < 0) return -1;
    const int page = pos / page_size;
    if (page >= max_pages) return -1;
    const int64_t pid = page_table[(int64_t)s * max_pages + page];
    const int64_t cell = pid * page_size + pos % page_size;
    if (pid < 0 || cell >= n_cells) return -1;
    return cell;
}

// FWHT256 of a row held as 8 consecutive elements per lane (element 8 * lane + k in
// z[k]): stages h = 1, 2, 4 inside the lane, h = 8 .. 128 across lanes (xor h / 8), in
// the order h = 1, 2, ..., 128; each butterfly (a, b) -> (a + b, a - b) in fp32.  Every
// butterfly of a stage is independent, so this layout gives the same bits as any other.
__device__ __forceinline__ void fwht256_lane8(float (&z)[8], int lane)
{
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if ((k & h) == 0) {
                const float a = z[k], b = z[k + h];
                z[k] = __fadd_rn(a, b);
                z[k + h] = __fsub_rn(a, b);
            }
        }
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const float sgn = (lane & m) ? -1.0f : 1.0f;   // a + b or a - b as fma(s, own, partner)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float p = __shfl_xor_sync(kFull, z[k], m);
            z[k] = __fmaf_rn(sgn, z[k], p);
        }
    }
}

// One warp per (sequence, token, K/V, head) row of 256, 8 elements per lane; block b of
// 32 elements is lanes 4b .. 4b + 3.  The next row's loads are issued before this row's
// arithmetic (16-byte loads when k and v allow them).
// One row of 256 values, 8 consecutive ones a lane (element 8 * lane + k), rotated
// (z = FWHT_256(x) / 16, stages h = 1..128) and stored as 8 q4_0 blocks of 18 bytes at
// dst (16-byte aligned), staged through the warp's 144-byte s_row.
__device__ __forceinline__ void q4_store_row(float (&z)[8], int lane, uint8_t* s_row, uint8_t* dst)
{
    fwht256_lane8(z, lane);
#pragma unroll
    for (int j = 0; j < 8; ++j) z[j] = __fmul_rn(z[j], 0.0625f);
    // the block's preferred element: the largest key over the block's 4 lanes (every
    // lane of the block gets the same); a block holding a NaN takes the scan of
    // q4_prefer instead, which decides NaN by position like the reference order
    uint32_t key = q4_key(z[0]);
#pragma unroll
    for (int j = 1; j < 8; ++j) key = max(key, q4_key(z[j]));
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) key = max(key, __shfl_xor_sync(kFull, key, o));
    float mval = __uint_as_float(key >> 1);
    if (!(key & 1u)) mval = -mval;
    if (__any_sync(kFull, key > 0xFF000001u)) {
        mval = z[0];
#pragma unroll
        for (int j = 1; j < 8; ++j)
            if (q4_prefer(z[j], mval)) mval = z[j];
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            const float other = __shfl_xor_sync(kFull, mval, o);
            if (q4_prefer(other, mval)) mval = other;
        }
    }
    const float d = __fmul_rn(mval, -0.125f);          // mval / -8, exact
    // 1/d correctly rounded (the reciprocal and the quotient 1/d round the same value)
    const float idv = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
    uint32_t q[8];
    // truncation toward zero; the unsigned conversion takes negatives and NaN to 0
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = min(__float2uint_rz(__fmaf_rn(z[j], idv, 8.5f)), 15u);
    // lanes 4b + p (p = 0, 1) hold codes j = 8p .. 8p + 7 of block b, lanes
    // 4b + p + 2 the codes j + 16 that share their bytes (high nibble)
    uint32_t w0 = q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24);
    uint32_t w1 = q[4] | (q[5] << 8) | (q[6] << 16) | (q[7] << 24);
    const uint32_t u0 = __shfl_down_sync(kFull, w0, 2), u1 = __shfl_down_sync(kFull, w1, 2);
    const int b = lane >> 2, p = lane & 3;
    if (p < 2) {
        w0 |= u0 << 4;
        w1 |= u1 << 4;
        uint8_t* blk = s_row + b * 18;
        uint16_t* hw = reinterpret_cast<uint16_t*>(blk + 2 + 8 * p);   // bytes 2 + 8p ..
        hw[0] = (uint16_t)w0; hw[1] = (uint16_t)(w0 >> 16);
        hw[2] = (uint16_t)w1; hw[3] = (uint16_t)(w1 >> 16);
        if (p == 0) *reinterpret_cast<uint16_t*>(blk) = __half_as_ushort(__float2half_rn(d));
    }
    __syncwarp();
    if (lane < 9) reinterpret_cast<uint4*>(dst)[lane] = reinterpret_cast<const uint4*>(s_row)[lane];
    __syncwarp();
}

template <bool kVec>
__device__ __forceinline__ void load8(const float* p, float4& a, float4& b)
{
    if (kVec) {
        a = __ldcs(reinterpret_cast<const float4*>(p));
        b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    } else {
        a = make_float4(__ldcs(p), __ldcs(p + 1), __ldcs(p + 2), __ldcs(p + 3));
        b = make_float4(__ldcs(p + 4), __ldcs(p + 5), __ldcs(p + 6), __ldcs(p + 7));
    }
}

template <bool kVec>
__global__ void __launch_bounds__(kCodecThreads)
append_q4_kernel(const float* __restrict__ k, const float* __restrict__ v, int n_seq,
                 const int32_t* __restrict__ pos0, int n_tok, int n_heads,
                 const int32_t* __restrict__ page_table, int max_pages, int page_size,
                 int64_t n_cells, uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool,
                 uint32_t* __restrict__ dev_status)
{
    __shared__ __align__(16) uint8_t s_row[kCodecWarps][144];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int64_t n_tokens = (int64_t)n_seq * n_tok;
    const int rows = 2 * n_heads;                     // K heads, then V heads
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    // row r of token tok: (r < n_heads ? k : v) [tok][r % n_heads][256]; lane's 8 values
    auto src_of = [&](int64_t tok, int r) {
        const int kv = r >= n_heads;
        return (kv ? v : k) + (tok * n_heads + (r - kv * n_heads)) * 256 + 8 * lane;
    };
    float4 nx0 = make_float4(0.f, 0.f, 0.f, 0.f), nx1 = nx0;
    if (warp < n_tokens) load8<kVec>(src_of(warp, 0), nx0, nx1);
    for (int64_t tok = warp; tok < n_tokens; tok += n_warps) {
        const int s = (int)(tok / n_tok), t = (int)(tok - (int64_t)s * n_tok);
        const int64_t cell = q4_cell(page_table, max_pages, page_size, n_cells, s, pos0[s] + t);
        if (cell < 0 && lane == 0 && dev_status) atomicOr(dev_status, (unsigned)KVQ_DEV_BAD_PAGE);
        for (int r = 0; r < rows; ++r) {
            float z[8] = {nx0.x, nx0.y, nx0.z, nx0.w, nx1.x, nx1.y, nx1.z, nx1.w};
            // the next row's loads (of this token, or the next token's first row)
            if (r + 1 < rows) load8<kVec>(src_of(tok, r + 1), nx0, nx1);
            else if (tok + n_warps < n_tokens) load8<kVec>(src_of(tok + n_warps, 0), nx0, nx1);
            if (cell < 0) continue;
            const int kv = r >= n_heads;
            q4_store_row(z, lane, s_row[wib],
                         (kv ? v_pool : k_pool) + (cell * n_heads + (r - kv * n_heads)) * 144);
        }
    }
}

// ------------------------------------------------------------------------------------
// Project-and-append producer of the q4_0 pools: a new token's K and V rows are
// y = h . W (W [d_model][n_heads * 256], fp32 or bfloat16, row-major), rotated and stored
// as kvq_append_q4 stores a row, in one launch: no fp32 row is written to memory.
// The sum has a fixed fp32 order: k runs in 64 chunks of L = 4 ceil(d_model / 256)
// consecutive terms (the last ones short or empty); each chunk is one chain
// acc = fmaf(h[k], w[k][c], acc) from acc = 0 in ascending k, and the 64 chunk sums are
// added pairwise, (0 + 1), (2 + 3), ..., then the 32, 16, 8, 4 and 2 results the same way.
// A cluster of 4 CTAs owns one head row (K head or V head) of a group of 8 tokens.  CTA
// rank r takes chunks 16r .. 16r + 15, one a warp, for all 256 columns (lane = 8
// consecutive columns, so a warp reads whole 512- or 1024-byte weight rows) and the 8
// tokens (NP pairs of them: a group of fewer than 8 tokens runs no chains on empty
// ones); the warp stages its weight rows in shared memory by cp.async (two 4 KB batches
// in flight) and the tokens' h values per 64-term window, and runs its fma chains two at
// a time (fma.rn.f32x2, one rounding per lane).  The CTA adds its 16 chunks (the
// first four pairwise levels); rank r then finishes the last two levels over the 4
// ranks' sums for tokens 2r and 2r + 1, read from the cluster's shared memory, and
// rotates and stores those rows.
// ------------------------------------------------------------------------------------
constexpr int kProjTok = 8;                           // tokens per cluster
constexpr int kProjRanks = 4;                         // CTAs per cluster (chunk groups)
constexpr int kProjLocal = 16;                        // chunks per CTA (64 in all), a warp each
constexpr int kProjWarps = kProjLocal;
constexpr int kProjThreads = 32 * kProjWarps;
constexpr int kProjWin = 64;                          // h terms staged per window
constexpr int kProjBatch = 4096;                      // weight bytes a warp stages per batch
constexpr int kProjStages = 2;                        // batches a warp has in its ring
constexpr size_t kProjWBytes = (size_t)kProjWarps * kProjStages * kProjBatch;       // 128 KB
constexpr size_t kProjPBytes = (size_t)kProjLocal * kProjTok * 256 * 4;             // 128 KB
constexpr size_t kProjHBytes = (size_t)kProjWarps * kProjWin * kProjTok * 4;        // 32 KB
constexpr size_t kProjRBytes = (size_t)kProjTok * 256 * 4;                          // 8 KB
static_assert(kProjWBytes >= kProjPBytes, "the weight stages become the chunk sums");
static_assert(kProjRanks * kProjLocal == 64 && 2 * kProjRanks == kProjTok, "64 chunks, 2 tokens a rank");
constexpr size_t kProjSmem = kProjWBytes + kProjHBytes + kProjRBytes + 2 * 144;

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t local_addr, uint32_t rank)
{
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local_addr), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a) : "memory");
    return v;
}

// d.x = fma(a.x, b.x, d.x), d.y = fma(a.y, b.y, d.y): two fp32 fmas, each rounded once
__device__ __forceinline__ void fma2(uint64_t& d, uint64_t a, uint64_t b)
{
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
__device__ __forceinline__ uint64_t dup2(float x)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float lo_of(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_of(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

template <bool kBf16, int NP>
__global__ void __cluster_dims__(kProjRanks, 1, 1) __launch_bounds__(kProjThreads, 1)
project_append_q4_kernel(const float* __restrict__ h, int n_seq, const int32_t* __restrict__ pos0,
                         int n_tok, int d_model, const void* __restrict__ w_k,
                         const void* __restrict__ w_v, int n_heads,
                         const int32_t* __restrict__ page_table, int max_pages, int page_size,
                         int64_t n_cells, uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool,
                         uint32_t* __restrict__ dev_status)
{
    extern __shared__ __align__(16) float proj_smem[];
    float* s_p = proj_smem;                            // [16 chunks][8 tokens][256 columns],
                                                       // the weight stages until then
    float* s_h = proj_smem + kProjWBytes / 4;          // [warp][64 terms][8 tokens]
    float* s_r = s_h + kProjHBytes / 4;                // [8 tokens][256 columns]
    uint8_t* s_row = reinterpret_cast<uint8_t*>(s_r + kProjTok * 256);   // [2][144]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_rank();
    const int unit = blockIdx.x / kProjRanks;          // K heads 0 .. n_heads - 1, then V heads
    const int kv = unit >= n_heads, head = unit - kv * n_heads;
    const int64_t n_tokens = (int64_t)n_seq * n_tok;
    const int64_t tok0 = (int64_t)blockIdx.y * kProjTok;
    const int nt = (int)min((int64_t)kProjTok, n_tokens - tok0);
    const int64_t n_out = (int64_t)n_heads * 256;
    const int L = 4 * ((d_model + 255) / 256);
    const int chunk = kProjLocal * rank + warp;
    const int k0 = min(chunk * L, d_model), k1 = min(k0 + L, d_model);

    // this warp's weight rows: columns head * 256 .. + 255 of rows k0 .. k1 - 1
    constexpr int kElt = kBf16 ? 2 : 4;
    constexpr int kSlab = 256 * kElt;                  // bytes of a row
    constexpr int kRows = kProjBatch / kSlab;          // rows a batch (8 or 4)
    constexpr int kPerRow = kSlab / 16;                // 16-byte pieces a row
    const uint8_t* wsrc = static_cast<const uint8_t*>(kv ? w_v : w_k) + (int64_t)head * 256 * kElt;
    const int64_t row_bytes = n_out * kElt;
    uint8_t* wst = reinterpret_cast<uint8_t*>(s_p) + (size_t)warp * kProjStages * kProjBatch;
    const uint32_t wst_sa = (uint32_t)__cvta_generic_to_shared(wst);
    // rows k .. k + n - 1 into stage st: lane copies the 16-byte pieces lane, lane + 32, ...
    auto issue = [&](int k, int n, int st) {
        const uint32_t dst = wst_sa + st * kProjBatch + 16 * lane;
#pragma unroll
        for (int j = 0; j < kProjBatch / 512; ++j) {
            const int q = 32 * j + lane, row = q / kPerRow;
            if (row < n)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 512 * j),
                             "l"(wsrc + (int64_t)(k + row) * row_bytes + 16 * (q - row * kPerRow))
                             : "memory");
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    // acc[p][j]: tokens 2p (low half) and 2p + 1 (high half) of column 8 lane + j
    uint64_t acc[NP][8];
#pragma unroll
    for (int p = 0; p < NP; ++p)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[p][j] = 0ull;
    float* hw = s_h + warp * (kProjWin * kProjTok);
    for (int kw = k0; kw < k1; kw += kProjWin) {
        const int kn = min(kProjWin, k1 - kw);         // a multiple of 4
        const int nb = (kn + kRows - 1) / kRows;
        issue(kw, min(kRows, kn), 0);
        // stage h[tok0 + t][kw .. kw + kn) as hw[k][t]: lane = (token t, 16-term quarter)
        {
            const int t = lane & 7, kq = 16 * (lane >> 3);
            const float* src = h + (tok0 + min(t, nt - 1)) * d_model + kw + kq;
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (t < nt && kq + i < kn) x = __ldg(reinterpret_cast<const float4*>(src + i));
                hw[(kq + i) * kProjTok + t] = x.x;
                hw[(kq + i + 1) * kProjTok + t] = x.y;
                hw[(kq + i + 2) * kProjTok + t] = x.z;
                hw[(kq + i + 3) * kProjTok + t] = x.w;
            }
        }
        for (int b = 0; b < nb; ++b) {
            const int kb = b * kRows, nr = min(kRows, kn - kb);
            if (b + 1 < nb) {                          // batch b + 1 stays in flight
                issue(kw + kb + kRows, min(kRows, kn - kb - kRows), (b + 1) % kProjStages);
                asm volatile("cp.async.wait_group 1;" ::: "memory");
            } else {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            }
            __syncwarp();                              // batch b (and the h window) visible
            const uint8_t* ws = wst + (b % kProjStages) * kProjBatch + (8 * kElt) * lane;
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                if (r < nr) {
                    float wv[8];
                    if constexpr (kBf16) {
                        const uint4 u = *reinterpret_cast<const uint4*>(ws + r * kSlab);
                        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            wv[2 * j] = __uint_as_float(uw[j] << 16);
                            wv[2 * j + 1] = __uint_as_float(uw[j] & 0xFFFF0000u);
                        }
                    } else {
                        const float4 a = *reinterpret_cast<const float4*>(ws + r * kSlab);
                        const float4 c = *reinterpret_cast<const float4*>(ws + r * kSlab + 16);
                        wv[0] = a.x; wv[1] = a.y; wv[2] = a.z; wv[3] = a.w;
                        wv[4] = c.x; wv[5] = c.y; wv[6] = c.z; wv[7] = c.w;
                    }
                    // the 8 tokens' h of this row as 4 pairs (token 2p low, 2p + 1 high)
                    const ulonglong2* hp = reinterpret_cast<const ulonglong2*>(hw + (kb + r) * kProjTok);
                    uint64_t hv[4];
                    const ulonglong2 h0 = hp[0];
                    hv[0] = h0.x; hv[1] = h0.y;
                    if constexpr (NP > 2) {
                        const ulonglong2 h1 = hp[1];
                        hv[2] = h1.x; hv[3] = h1.y;
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint64_t wd = dup2(wv[j]);
#pragma unroll
                        for (int p = 0; p < NP; ++p) fma2(acc[p][j], hv[p], wd);
                    }
                }
            }
            __syncwarp();                              // stage b % 2 is refilled next
        }
    }
    __syncthreads();                                   // the weight stages become s_p
#pragma unroll
    for (int p = 0; p < NP; ++p) {                     // rows of tokens past 2 NP are not read
        float* d0 = s_p + (warp * kProjTok + 2 * p) * 256 + 8 * lane;
        float* d1 = d0 + 256;
        *reinterpret_cast<float4*>(d0) = make_float4(lo_of(acc[p][0]), lo_of(acc[p][1]), lo_of(acc[p][2]), lo_of(acc[p][3]));
        *reinterpret_cast<float4*>(d0 + 4) = make_float4(lo_of(acc[p][4]), lo_of(acc[p][5]), lo_of(acc[p][6]), lo_of(acc[p][7]));
        *reinterpret_cast<float4*>(d1) = make_float4(hi_of(acc[p][0]), hi_of(acc[p][1]), hi_of(acc[p][2]), hi_of(acc[p][3]));
        *reinterpret_cast<float4*>(d1 + 4) = make_float4(hi_of(acc[p][4]), hi_of(acc[p][5]), hi_of(acc[p][6]), hi_of(acc[p][7]));
    }
    __syncthreads();
    // the first four pairwise levels over this CTA's 16 chunks, per (token, column)
    for (int i = threadIdx.x; i < kProjTok * 256; i += kProjThreads) {
        float p[kProjLocal];
#pragma unroll
        for (int q = 0; q < kProjLocal; ++q) p[q] = s_p[q * kProjTok * 256 + i];
#pragma unroll
        for (int n = kProjLocal; n > 1; n >>= 1)
#pragma unroll
            for (int j = 0; j < n / 2; ++j) p[j] = __fadd_rn(p[2 * j], p[2 * j + 1]);
        s_r[i] = p[0];
    }
    cluster_sync_all();                                // every rank's sums are in place

    // tokens 2r, 2r + 1: the last two levels over the 4 ranks (lane = columns 8 lane ..
    // 8 lane + 7), then the rotation, the q4_0 blocks and the pool row
    if (warp < 2) {
        const int tl = 2 * (int)rank + warp;
        const int64_t tok = tok0 + tl;
        if (tl < nt) {
            const int s = (int)(tok / n_tok), t = (int)(tok - (int64_t)s * n_tok);
            const int64_t cell = q4_cell(page_table, max_pages, page_size, n_cells, s, pos0[s] + t);
            if (cell < 0) {
                if (lane == 0 && dev_status) atomicOr(dev_status, (unsigned)KVQ_DEV_BAD_PAGE);
            } else {
                const uint32_t la = (uint32_t)__cvta_generic_to_shared(s_r + tl * 256 + 8 * lane);
                float v[kProjRanks][8];
#pragma unroll
                for (int q = 0; q < kProjRanks; ++q) {
                    const float4 a = ld_cluster_f4(la, q), b = ld_cluster_f4(la + 16, q);
                    v[q][0] = a.x; v[q][1] = a.y; v[q][2] = a.z; v[q][3] = a.w;
                    v[q][4] = b.x; v[q][5] = b.y; v[q][6] = b.z; v[q][7] = b.w;
                }
                float z[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    z[j] = __fadd_rn(__fadd_rn(v[0][j], v[1][j]), __fadd_rn(v[2][j], v[3][j]));
                q4_store_row(z, lane, s_row + 144 * warp,
                             (kv ? v_pool : k_pool) + (cell * n_heads + head) * 144);
            }
        }
    }
    cluster_sync_all();                                // the peers' reads of s_r are done
}

// gather: rows (s, t, h) -> binary16 [256], (q - 8) * d rounded to nearest even
__global__ void __launch_bounds__(kCodecThreads)
gather_q4_kernel(const uint8_t* __restrict__ pool, int n_seq, const int32_t* __restrict__ pos0,
                 int n_tok, int n_heads, const int32_t* __restrict__ page_table, int max_pages,
                 int page_size, int64_t n_cells, uint16_t* __restrict__ out,
                 uint32_t* __restrict__ dev_status)
{
    constexpr int kHeadsPerPass = 8;                  // 8 x 144 B = 72 pieces of 16 B
    __shared__ __align__(16) uint8_t s_cell[kCodecWarps][kHeadsPerPass * 144];
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int64_t n_tokens = (int64_t)n_seq * n_tok;
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int b = lane >> 2, part = lane & 3;
    for (int64_t tok = warp; tok < n_tokens; tok += n_warps) {
        const int s = (int)(tok / n_tok), t = (int)(tok - (int64_t)s * n_tok);
        const int64_t cell = q4_cell(page_table, max_pages, page_size, n_cells, s, pos0[s] + t);
        if (cell < 0) {
            if (lane == 0 && dev_status) atomicOr(dev_status, (unsigned)KVQ_DEV_BAD_PAGE);
            continue;
        }
        // the token's heads are contiguous in the pool: h0 .. h0 + nh - 1 in one pass
        for (int h0 = 0; h0 < n_heads; h0 += kHeadsPerPass) {
            const int nh = min(kHeadsPerPass, n_heads - h0);
            const uint4* src = reinterpret_cast<const uint4*>(pool + (cell * n_heads + h0) * 144);
            uint4 pc[3];
#pragma unroll
            for (int i = 0; i < 3; ++i)
                if (lane + 32 * i < 9 * nh) pc[i] = __ldcs(src + lane + 32 * i);
#pragma unroll
            for (int i = 0; i < 3; ++i)
                if (lane + 32 * i < 9 * nh) reinterpret_cast<uint4*>(s_cell[wib])[lane + 32 * i] = pc[i];
            __syncwarp();
            for (int hh = 0; hh < nh; ++hh) {
                const uint8_t* blk = s_cell[wib] + hh * 144 + b * 18;
                const float d = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(blk)));
                // codes j = 8 part .. 8 part + 7: low nibbles of bytes 2 + j (j < 16), else
                // high nibbles of bytes 2 + j - 16
                const uint16_t* bytes = reinterpret_cast<const uint16_t*>(blk + 2 + 8 * (part & 1));
                const uint32_t lo4 = (uint32_t)bytes[0] | ((uint32_t)bytes[1] << 16);
                const uint32_t hi4 = (uint32_t)bytes[2] | ((uint32_t)bytes[3] << 16);
                const int sh = part >= 2 ? 4 : 0;
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const uint32_t src4 = e < 4 ? lo4 : hi4;
                    const int q0 = (int)((src4 >> (8 * (e & 3) + sh)) & 15);
                    const int q1 = (int)((src4 >> (8 * ((e + 1) & 3) + sh)) & 15);
                    const unsigned short x0 = __half_as_ushort(__float2half_rn(__fmul_rn((float)(q0 - 8), d)));
                    const unsigned short x1 = __half_as_ushort(__float2half_rn(__fmul_rn((float)(q1 - 8), d)));
                    w[e >> 1] = (uint32_t)x0 | ((uint32_t)x1 << 16);
                }
                uint16_t* dst = out + (tok * n_heads + h0 + hh) * 256 + b * 32 + part * 8;
                __stcs(reinterpret_cast<uint4*>(dst), make_uint4(w[0], w[1], w[2], w[3]));
            }
            __syncwarp();
        }
    }
}

// ------------------------------------------------------------------------------------
// MLA row gather (fp8 / TQ4 caches) — colibri PR #399, Commit 2: rows gathered by
// absolute index for DSA-style sparse attention.
// One warp per gathered row; byte-for-byte copy of every plane.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kCodecThreads)
gather_mla_kernel(kvq_mla_cache src, int lat_bytes, int64_t src_rows,
                  const int32_t* __restrict__ page_table, int max_pages, int page_size,
                  const int32_t* __restrict__ idx, int64_t n_idx,
                  uint8_t* __restrict__ dst_lat, float* __restrict__ dst_lat_scale,
                  uint8_t* __restrict__ dst_rope, float* __restrict__ dst_rope_scale,
                  uint32_t* __restrict__ dev_status)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t j = warp; j < n_idx; j += n_warps) {
        const int64_t t = idx[j];
        int64_t row = -1;
        if (t >= 0 && t < src_rows) {
            if (page_table) {
                const int64_t page = t / page_size;
                const int64_t pid = page < max_pages ? page_table[page] : -1;
                row = (pid < 0) ? -1 : pid * page_size + t % page_size;
            } else {
                row = t;
            }
            if (row >= src.n_rows) row = -1;
        }
        if (row < 0 && lane == 0 && dev_status) atomicOr(dev_status, (unsigned)KVQ_DEV_BAD_INDEX);
        const int n16 = lat_bytes / 16;
        for (int i = lane; i < n16; i += 32) {
            uint4 w = make_uint4(0, 0, 0, 0);
            if (row >= 0) w = reinterpret_cast<const uint4*>(src.lat + row * lat_bytes)[i];
            reinterpret_cast<uint4*>(dst_lat + j * lat_bytes)[i] = w;
        }
        if (lane < 4) {
            uint4 w = make_uint4(0, 0, 0, 0);
            if (row >= 0) w = reinterpret_cast<const uint4*>(src.rope + row * 64)[lane];
            reinterpret_cast<uint4*>(dst_rope + j * 64)[lane] = w;
        }
        if (lane == 0) {
            dst_lat_scale[j] = row >= 0 ? src.lat_scale[row] : 0.0f;
            dst_rope_scale[j] = row >= 0 ? src.rope_scale[row] : 0.0f;
        }
    }
}

}  // namespace

// ====================================================================================
// launchers
// ====================================================================================

cudaError_t launch_encode_fp8(const float* x, int64_t rows, int dim, int64_t ldx,
                              uint8_t* codes, int64_t ldc, float* scales, cudaStream_t s)
{
    if (rows == 0) return cudaSuccess;
    const bool x16 = ((uintptr_t)x % 16 == 0) && (ldx % 4 == 0);
    const bool c4 = ((uintptr_t)codes % 4 == 0) && (ldc % 4 == 0);
    const int rows_per_block_warp = kCodecWarps;
#define KVQ_FP8_CASE(D, LANES, VPL)                                                        \
    if (dim == D && x16 && c4) {                                                           \
        constexpr int kRpw = 32 / LANES;                                                   \
        encode_fp8_vec_kernel<LANES, VPL><<<grid_for(rows, rows_per_block_warp * kRpw),   \
                                            kCodecThreads, 0, s>>>(x, rows, ldx, codes, ldc, scales); \
        return cudaGetLastError();                                                         \
    }
    KVQ_FP8_CASE(64, 4, 4)          // 8 rows a warp (with 2, too few loads were in flight)
    KVQ_FP8_CASE(128, 32, 1)
    KVQ_FP8_CASE(256, 32, 2)
    KVQ_FP8_CASE(512, 32, 4)
    KVQ_FP8_CASE(576, 16, 9)
    KVQ_FP8_CASE(1024, 32, 8)
#undef KVQ_FP8_CASE
    encode_fp8_generic_kernel<<<grid_for(rows, rows_per_block_warp), kCodecThreads, 0, s>>>(
        x, rows, dim, ldx, codes, ldc, scales);
    return cudaGetLastError();
}

// one wave of the 512-wide rotated-tier encoder: as many CTAs of eight warps as fit on
// every SM at once, each warp many rows (a second, partial wave would double the time of
// its CTAs)
template <int BITS>
cudaError_t launch_tq512(const float* x, int64_t rows, int64_t ldx, const uint32_t* sign_bits,
                         uint8_t* packed, int64_t ldp, float* radius, bool vec, cudaStream_t s)
{
    static std::atomic<int> per_sm{0};
    int n = per_sm.load();
    if (n <= 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, encode_tq512_kernel<BITS>, kCodecThreads, 0) !=
                cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = 1;
        }
        per_sm.store(n);
    }
    const int g = (int)std::max<int64_t>(1, std::min<int64_t>((rows + kCodecWarps - 1) / kCodecWarps,
                                                              (int64_t)sm_count() * n));
    encode_tq512_kernel<BITS><<<g, kCodecThreads, 0, s>>>(x, rows, ldx, sign_bits, packed, ldp, radius, vec);
    return cudaGetLastError();
}

cudaError_t launch_encode_tq4(const float* x, int64_t rows, int dim, int64_t ldx,
                              const uint32_t* sign_bits, uint8_t* packed, int64_t ldp,
                              float* radius, cudaStream_t s)
{
    if (rows == 0) return cudaSuccess;
    const float c = tq4_inv_sqrt(dim);
    const bool vec = ((uintptr_t)packed % 16 == 0) && (ldp % 16 == 0);
    const int g = grid_for(rows, kCodecWarps);
    switch (dim) {
        case 64:   encode_tq4_kernel<2><<<g, kCodecThreads, 0, s>>>(x, rows, ldx, sign_bits, packed, ldp, radius, c, vec); break;
        case 128:  encode_tq4_kernel<4><<<g, kCodecThreads, 0, s>>>(x, rows, ldx, sign_bits, packed, ldp, radius, c, vec); break;
        case 256:  encode_tq4_kernel<8><<<g, kCodecThreads, 0, s>>>(x, rows, ldx, sign_bits, packed, ldp, radius, c, vec); break;
        case 512:
            if ((uintptr_t)x % 16 == 0 && ldx % 4 == 0)
                return launch_tq512<4>(x, rows, ldx, sign_bits, packed, ldp, radius, vec, s);
            else
                encode_tq4_kernel<16><<<g, kCodecThreads, 0, s>>>(x, rows, ldx, sign_bits, packed, ldp, radius, c, vec);
            break;
        case 1024: encode_tq4_kernel<32><<<g, kCodecThreads, 0, s>>>(x, rows, ldx, sign_bits, packed, ldp, radius, c, vec); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_encode_mla_fused(const float* c_lat, int64_t ldx, const float* k_rope, int64_t ldr,
                                    int64_t rows, const uint32_t* sign_bits, uint8_t* lat, int64_t ldl,
                                    float* lat_scale, uint8_t* rope, int64_t ldc, float* rope_scale,
                                    bool vec, cudaStream_t s)
{
    // the latent CTAs sized as the separate encoder would be (one wave of the rotated
    // encoder, by this kernel's occupancy); the rope CTAs share the count and stride
    int64_t g;
    if constexpr (BITS == 8) {
        g = grid_for(rows, kCodecWarps);
    } else {
        static std::atomic<int> per_sm{0};
        int n = per_sm.load();
        if (n <= 0) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, encode_mla_kernel<BITS>, kCodecThreads, 0) !=
                    cudaSuccess || n <= 0) {
                (void)cudaGetLastError();
                n = 1;
            }
            per_sm.store(n);
        }
        g = std::max<int64_t>(1, std::min<int64_t>((rows + kCodecWarps - 1) / kCodecWarps, (int64_t)sm_count() * n));
    }
    encode_mla_kernel<BITS><<<dim3((unsigned)g, 2), kCodecThreads, 0, s>>>(
        c_lat, ldx, k_rope, ldr, rows, sign_bits, lat, ldl, lat_scale, rope, ldc, rope_scale, vec);
    return cudaGetLastError();
}

cudaError_t launch_encode_mla(const float* c_lat, int64_t ldx, const float* k_rope, int64_t ldr,
                              int64_t rows, int fmt, const uint32_t* sign_bits, uint8_t* lat,
                              int64_t ldl, float* lat_scale, uint8_t* rope, int64_t ldc,
                              float* rope_scale, cudaStream_t s)
{
    if (rows == 0) return cudaSuccess;
    const int bits = fmt == KVQ_FMT_FP8 ? 8 : rotated_bits(fmt);
    // the one-launch form needs what the separate encoders' fast paths need: 16-byte
    // aligned input rows, 4-byte aligned fp8 code rows; otherwise the two encoders run
    const bool x16 = (uintptr_t)c_lat % 16 == 0 && ldx % 4 == 0 && (uintptr_t)k_rope % 16 == 0 && ldr % 4 == 0;
    const bool c4 = (uintptr_t)rope % 4 == 0 && ldc % 4 == 0 &&
                    (bits != 8 || ((uintptr_t)lat % 4 == 0 && ldl % 4 == 0));
    if (!x16 || !c4) {
        cudaError_t e = bits == 8 ? launch_encode_fp8(c_lat, rows, kDLat, ldx, lat, ldl, lat_scale, s)
                                  : launch_encode_tq(c_lat, rows, kDLat, ldx, bits, sign_bits, lat, ldl, lat_scale, s);
        if (e != cudaSuccess) return e;
        return launch_encode_fp8(k_rope, rows, kDRope, ldr, rope, ldc, rope_scale, s);
    }
    const bool vec = ((uintptr_t)lat % 16 == 0) && (ldl % 16 == 0);
    switch (bits) {
        case 8: return launch_encode_mla_fused<8>(c_lat, ldx, k_rope, ldr, rows, sign_bits, lat, ldl, lat_scale, rope, ldc, rope_scale, vec, s);
        case 4: return launch_encode_mla_fused<4>(c_lat, ldx, k_rope, ldr, rows, sign_bits, lat, ldl, lat_scale, rope, ldc, rope_scale, vec, s);
        case 3: return launch_encode_mla_fused<3>(c_lat, ldx, k_rope, ldr, rows, sign_bits, lat, ldl, lat_scale, rope, ldc, rope_scale, vec, s);
        case 6: return launch_encode_mla_fused<6>(c_lat, ldx, k_rope, ldr, rows, sign_bits, lat, ldl, lat_scale, rope, ldc, rope_scale, vec, s);
        default: return cudaErrorInvalidValue;
    }
}

void tq_codebook_values(int bits, float* centroids, float* thresholds)
{
    const int L = 1 << bits;
    for (int k = 0; k < L; ++k) {
        centroids[k] = bits == 4 ? kTq4Centroids[k] : bits == 3 ? kTq3.cb[k] : kTq6.cb[k];
    }
    for (int k = 0; k + 1 < L; ++k)
        thresholds[k] = bits == 4 ? kTq4Thresholds[k] : bits == 3 ? kTq3.thr[k] : kTq6.thr[k];
}

cudaError_t launch_encode_tq(const float* x, int64_t rows, int dim, int64_t ldx, int bits,
                             const uint32_t* sign_bits, uint8_t* packed, int64_t ldp,
                             float* radius, cudaStream_t s)
{
    if (bits == 4) return launch_encode_tq4(x, rows, dim, ldx, sign_bits, packed, ldp, radius, s);
    if (rows == 0) return cudaSuccess;
    const float c = tq4_inv_sqrt(dim);
    const bool vec = ((uintptr_t)packed % 16 == 0) && (ldp % 16 == 0);
    const int g = grid_for(rows, kCodecWarps);
#define KVQ_TQB(VPL, B) encode_tqb_kernel<VPL, B><<<g, kCodecThreads, 0, s>>>(x, rows, ldx, sign_bits, packed, ldp, radius, c, vec)
#define KVQ_TQB_DIMS(B)                                   \
    switch (dim) {                                        \
        case 64:   KVQ_TQB(2, B); break;                  \
        case 128:  KVQ_TQB(4, B); break;                  \
        case 256:  KVQ_TQB(8, B); break;                  \
        case 512:  KVQ_TQB(16, B); break;                 \
        case 1024: KVQ_TQB(32, B); break;                 \
        default: return cudaErrorInvalidValue;            \
    }
    if (dim == 512 && (uintptr_t)x % 16 == 0 && ldx % 4 == 0) {
        if (bits == 3) return launch_tq512<3>(x, rows, ldx, sign_bits, packed, ldp, radius, vec, s);
        if (bits == 6) return launch_tq512<6>(x, rows, ldx, sign_bits, packed, ldp, radius, vec, s);
    }
    if (bits == 3) {
        KVQ_TQB_DIMS(3)
    } else if (bits == 6) {
        KVQ_TQB_DIMS(6)
    } else {
        return cudaErrorInvalidValue;
    }
#undef KVQ_TQB_DIMS
#undef KVQ_TQB
    return cudaGetLastError();
}

cudaError_t launch_append_q4(const float* k, const float* v, int n_seq, const int32_t* pos0,
                             int n_tok, int n_heads, const int32_t* page_table, int max_pages,
                             int page_size, int64_t n_cells, uint8_t* k_pool, uint8_t* v_pool,
                             uint32_t* dev_status, cudaStream_t s)
{
    const int64_t n_tokens = (int64_t)n_seq * n_tok;
    if (n_tokens == 0 || n_heads == 0) return cudaSuccess;
    const bool vec = (uintptr_t)k % 16 == 0 && (uintptr_t)v % 16 == 0;
    if (vec)
        append_q4_kernel<true><<<grid_for(n_tokens, kCodecWarps), kCodecThreads, 0, s>>>(
            k, v, n_seq, pos0, n_tok, n_heads, page_table, max_pages, page_size, n_cells,
            k_pool, v_pool, dev_status);
    else
        append_q4_kernel<false><<<grid_for(n_tokens, kCodecWarps), kCodecThreads, 0, s>>>(
            k, v, n_seq, pos0, n_tok, n_heads, page_table, max_pages, page_size, n_cells,
            k_pool, v_pool, dev_status);
    return cudaGetLastError();
}

cudaError_t launch_project_append_q4(const float* h, int n_seq, const int32_t* pos0, int n_tok,
                                     int d_model, const void* w_k, const void* w_v, bool w_bf16,
                                     int n_heads, const int32_t* page_table, int max_pages,
                                     int page_size, int64_t n_cells, uint8_t* k_pool,
                                     uint8_t* v_pool, uint32_t* dev_status, cudaStream_t s)
{
    const int64_t n_tokens = (int64_t)n_seq * n_tok;
    if (n_tokens == 0 || n_heads == 0) return cudaSuccess;
    using Kern = void (*)(const float*, int, const int32_t*, int, int, const void*, const void*, int,
                          const int32_t*, int, int, int64_t, uint8_t*, uint8_t*, uint32_t*);
    // token pairs a group computes: 4, or fewer when all tokens fit in one short group
    const int np = (int)std::min<int64_t>(kProjTok / 2, (n_tokens + 1) / 2);
    static const Kern kKern[2][4] = {
        {project_append_q4_kernel<false, 1>, project_append_q4_kernel<false, 2>,
         project_append_q4_kernel<false, 3>, project_append_q4_kernel<false, 4>},
        {project_append_q4_kernel<true, 1>, project_append_q4_kernel<true, 2>,
         project_append_q4_kernel<true, 3>, project_append_q4_kernel<true, 4>}};
    const Kern kern = kKern[w_bf16 ? 1 : 0][np - 1];
    // the shared-memory opt-in, once per (device, kernel)
    static std::atomic<uint32_t> opted[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint32_t bit = 1u << ((w_bf16 ? 4 : 0) + np - 1);
    if (dev >= 64 || !(opted[dev].load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kProjSmem);
        if (e != cudaSuccess) return e;
        if (dev < 64) opted[dev].fetch_or(bit, std::memory_order_release);
    }
    const dim3 grid((unsigned)(kProjRanks * 2 * n_heads), (unsigned)((n_tokens + kProjTok - 1) / kProjTok));
    kern<<<grid, kProjThreads, kProjSmem, s>>>(h, n_seq, pos0, n_tok, d_model, w_k, w_v, n_heads,
                                              page_table, max_pages, page_size, n_cells, k_pool,
                                              v_pool, dev_status);
    return cudaGetLastError();
}

cudaError_t launch_gather_q4(const kvq_gather_desc& d, cudaStream_t s)
{
    const int64_t n_tokens = (int64_t)d.n_seq * d.n_tok;
    if (n_tokens == 0 || d.n_heads == 0) return cudaSuccess;
    gather_q4_kernel<<<grid_for(n_tokens, kCodecWarps), kCodecThreads, 0, s>>>(
        d.q4_pool, d.n_seq, d.pos0, d.n_tok, d.n_heads, d.page_table, d.max_pages,
        d.page_size, d.n_cells, d.q4_out, d.dev_status);
    return cudaGetLastError();
}

cudaError_t launch_gather_mla(const kvq_gather_desc& d, cudaStream_t s)
{
    if (d.n_idx == 0) return cudaSuccess;
    const int lat_bytes = d.format == KVQ_FMT_FP8 ? kDLat : kDLat * rotated_bits(d.format) / 8;
    gather_mla_kernel<<<grid_for(d.n_idx, kCodecWarps), kCodecThreads, 0, s>>>(
        d.mla_src, lat_bytes, d.mla_src_rows, d.page_table, d.max_pages, d.page_size, d.idx,
        d.n_idx, d.dst_lat, d.dst_lat_scale, d.dst_rope, d.dst_rope_scale, d.dev_status);
    return cudaGetLastError();
}

}  // namespace kvq
