// kvq_tc_common.cuh — device helpers shared by the tensor-core decode kernels
// (kvq_decode_tc.cu, kvq_decode_tc16.cu): row bookkeeping of a split, exact conversion
// of e4m3 and TQ4 codes to binary16, cp.async / TMA copy wrappers, warp reductions,
// and the host-side tensor-map encoder for the code planes.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "kvq_internal.cuh"
#include "kvq_sm100.cuh"

namespace kvq {
namespace tc {

using namespace sm100;

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ int seq_fmt_of(const kvq_mla_problem& p, int s)
{
    return p.seq_fmt ? p.seq_fmt[s] : p.fmt;
}

__device__ __forceinline__ int64_t pool_row_of(const kvq_mla_problem& p, int s, int64_t t)
{
    if (!p.block_table) return (int64_t)s * p.seq_stride_rows + t;
    const int64_t page = t / p.page_size;
    if (page >= p.max_pages) return -1;
    const int64_t pid = p.block_table[(int64_t)s * p.max_pages + page];
    if (pid < 0) return -1;
    return pid * p.page_size + t % p.page_size;
}

// byte offset of 16-byte chunk c (0..7) of row r in a 128B-swizzled [rows x 64] slab
__device__ __forceinline__ uint32_t sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// four e4m3 codes (one 32-bit word) -> two half2 words (exact); the pattern S.1111.111,
// which the encoder never writes, reads as 0
__device__ __forceinline__ void e4m3x4_to_half(uint32_t w, uint32_t& lo, uint32_t& hi)
{
    // (b & 0x7F) + 1 has bit 7 set exactly when the low seven bits of b are all set;
    // prmt's sign mode (selector 8 + i) spreads that bit over byte i, which then clears it
    const uint32_t t = (w & 0x7F7F7F7Fu) + 0x01010101u;
    uint32_t m;
    asm("prmt.b32 %0, %1, 0, 0xBA98;" : "=r"(m) : "r"(t));
    w &= ~m;
    // low byte -> low half, as the two halves of one register
    asm("{.reg .b16 l, h; mov.b32 {l, h}, %2; cvt.rn.f16x2.e4m3x2 %0, l; cvt.rn.f16x2.e4m3x2 %1, h;}"
        : "=r"(lo), "=r"(hi) : "r"(w));
}

// Row bookkeeping shared by producer and softmax threads: the pool row of candidate j
// of this CTA's (sequence, query), or -1 when not admissible (flags bad data).
struct RowCtx {
    const kvq_mla_problem* p;
    int s, q, L;
    int64_t r1, lim;
    const kvq_mla_cache* C;
    uint32_t* status;
    __device__ int64_t row(int64_t j, bool flag) const
    {
        if (j >= r1) return -1;
        const int64_t tl = p->idx ? (int64_t)p->idx[((int64_t)s * p->n_q + q) * p->top_k + j] : j;
        if (tl < 0 || tl >= L) {
            if (flag && status) atomicOr(status, (unsigned)KVQ_DEV_BAD_INDEX);
            return -1;
        }
        if (tl > lim) return -1;
        const int64_t r = pool_row_of(*p, s, tl);
        if (r < 0 || r >= C->n_rows) {
            if (flag && status) atomicOr(status, (unsigned)KVQ_DEV_BAD_PAGE);
            return -1;
        }
        return r;
    }
};

// true in exactly one lane of the (converged) warp
__device__ __forceinline__ bool elect_one()
{
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// 16 bytes global -> shared without registers (zero-filled when `bytes` is 0); L2
// fetches the aligned 256 bytes around them (the rest of the row's codes follow soon);
// completion is tracked per thread in commit groups
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t bytes)
{
    asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// 2-D tiled TMA load of the box at (x, y) of `map` into shared memory; its bytes count
// against the transaction count of `bar`
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// L2 prefetch of the box at (x, y) of `map` (no shared memory, no completion)
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// The codebook is symmetric (code 15 - k is code k with the sign flipped) and its upper
// half is positive; the byte tables below rely on both.
constexpr bool tq4_codebook_symmetric()
{
    for (int k = 0; k < 8; ++k) {
        if (kTq4CentroidBits[15 - k] != (kTq4CentroidBits[k] ^ 0x8000u)) return false;
        if (kTq4CentroidBits[8 + k] & 0x8000u) return false;
    }
    return true;
}
static_assert(tq4_codebook_symmetric(), "TQ4 codebook must be symmetric");

// byte `hi` (0: low byte, 1: high byte) of the binary16 magnitudes m[4*part .. 4*part+3]
constexpr uint32_t tq4_mag_bytes(int hi, int part)
{
    uint32_t r = 0;
    for (int b = 0; b < 4; ++b) {
        const uint32_t h = kTq4CentroidBits[8 + 4 * part + b];
        r |= (hi ? (h >> 8) : (h & 0xFFu)) << (8 * b);
    }
    return r;
}

// eight TQ4 codes (code i in nibble i of w) -> four half2 words of centroids
__device__ __forceinline__ void tq4x8_to_half(uint32_t w, uint32_t* h)
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

// codes -> 32 fp16 values (half hq of a 64-code chunk): fp8 chunks hold 64 bytes in
// raw[0..3], TQ4 chunks 32 bytes in raw[0..1]
__device__ __forceinline__ void codes_to_half(const uint4 (&raw)[4], int hq, bool fp8, uint32_t (&h)[16])
{
    if (fp8) {
#pragma unroll
        for (int v = 0; v < 2; ++v) {
            const uint4 w = raw[2 * hq + v];
            e4m3x4_to_half(w.x, h[8 * v + 0], h[8 * v + 1]);
            e4m3x4_to_half(w.y, h[8 * v + 2], h[8 * v + 3]);
            e4m3x4_to_half(w.z, h[8 * v + 4], h[8 * v + 5]);
            e4m3x4_to_half(w.w, h[8 * v + 6], h[8 * v + 7]);
        }
    } else {
        const uint4 w = raw[hq];
        tq4x8_to_half(w.x, h + 0);
        tq4x8_to_half(w.y, h + 4);
        tq4x8_to_half(w.z, h + 8);
        tq4x8_to_half(w.w, h + 12);
    }
}

// 64 codes of b = 3 or 6 bits (a little-endian bit stream: code i at bits b i .. b i +
// b - 1 of the chunk's 24 or 48 bytes, in the words raw[0].x, .y, ...) -> 32 half2 words
// of centroids, looked up in a shared-memory table of 2^b binary16 values.  A table of at
// most 64 binary16 values fills at most one 32-bit word per bank, so lanes that hit the
// same bank read the same word: the lookups are free of bank conflicts for any codes.
template <int B>
__device__ __forceinline__ void tqb_codes_to_half(const uint4 (&raw)[4], const uint16_t* tab,
                                                  uint32_t (&h)[32])
{
    const uint32_t w[12] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w, raw[1].x, raw[1].y,
                            raw[1].z, raw[1].w, raw[2].x, raw[2].y, raw[2].z, raw[2].w};
    constexpr uint32_t kMask = (1u << B) - 1u;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        uint32_t v[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int bit = B * (2 * c + e), wi = bit >> 5, sh = bit & 31;
            const uint32_t code = (sh + B <= 32 ? (w[wi] >> sh) : __funnelshift_r(w[wi], w[wi + 1], sh)) & kMask;
            v[e] = tab[code];
        }
        h[c] = v[0] | (v[1] << 16);
    }
}

// max (or sum) over the warp's 32 lanes of each of NV values (NV = 4, 8, 16 or 32), transposed:
// on return v[0] of lane l holds the result for value index l % NV.  The stages that
// halve the value count exchange halves between lane pairs (NV - 1 shuffles in all);
// with NV < 32 the remaining lane bits are folded with plain xor shuffles of v[0].
template <bool kMax, int NV>
__device__ __forceinline__ void warp_reduce_transpose(float (&v)[NV], int lane)
{
    static_assert(NV == 4 || NV == 8 || NV == 16 || NV == 32, "4, 8, 16 or 32 values");
#pragma unroll
    for (int w = NV / 2; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
            const float send = up ? v[j] : v[j + w];
            const float keep = up ? v[j + w] : v[j];
            const float got = __shfl_xor_sync(kFull, send, w);
            v[j] = kMax ? fmaxf(keep, got) : keep + got;
        }
    }
#pragma unroll
    for (int w = NV; w < 32; w <<= 1) {
        const float got = __shfl_xor_sync(kFull, v[0], w);
        v[0] = kMax ? fmaxf(v[0], got) : v[0] + got;
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link to libcuda)
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            ptr = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }();
    return fn;
}

// [n_rows x row_bytes] bytes, boxes of [box_rows x box_bytes] (128-byte boxes
// 128B-swizzled, 64-byte boxes 64B-swizzled, 32-byte boxes 32B-swizzled, 48-byte boxes
// unswizzled); rows past n_rows read as 0
inline bool make_code_map(CUtensorMap* m, const uint8_t* plane, int64_t n_rows, int row_bytes, int box_bytes,
                          int box_rows = 128)
{
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || !plane || n_rows < 1 || n_rows > INT32_MAX) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)n_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(plane), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE,
               box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
               : box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
               : box_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------------------------
// Q image of a tensor-core decode with GQ heads a CTA: per (seq, query, head group) the
// 9 swizzled K-major slabs [2 GQ rows x 64 k] fp16 that the score MMA reads as B.  Rows
// 0..GQ-1 hold the hi halves of the group's heads, rows GQ..2GQ-1 the lo halves
// (lo = fp16(q - hi), so hi + lo carries ~22 bits of q); k < 512 comes from q_lat
// (for the rotated tiers rotated first, (1/sqrt 512) FWHT_512(s (.) q) in fp32), k >= 512
// from q_rope.  Heads past n_heads are zero rows.  Grid-stride over (row, group) with
// one warp each.
// ------------------------------------------------------------------------------------
template <int GQ>
__device__ __forceinline__ void build_q_image(const kvq_mla_problem& p, int n_hg, uint8_t* q_img)
{
    constexpr int kSlab = 2 * GQ * 128;
    constexpr int kImg = 9 * kSlab;
    const int lane = threadIdx.x & 31;
    const int64_t n_items = (int64_t)p.n_seq * p.n_q * n_hg * GQ;
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    uint32_t neg = 0;                                       // signs of elements k*32+lane
    if (p.tq4_signs) {
#pragma unroll
        for (int k = 0; k < 16; ++k) neg |= ((p.tq4_signs[k] >> lane) & 1u) << k;
    }
    const float c512 = tq4_inv_sqrt(kDLat);
    for (int64_t it = warp; it < n_items; it += n_warps) {
        const int n = (int)(it % GQ);                        // head within group
        const int64_t grp = it / GQ;                         // (s, q, hg)
        const int hg = (int)(grp % n_hg);
        const int64_t sq = grp / n_hg;                       // s * n_q + q
        const int s = (int)(sq / p.n_q);
        const int h = hg * GQ + n;
        const bool rot = rotated_format(seq_fmt_of(p, s));
        uint8_t* img = q_img + grp * (int64_t)kImg;
        float y[16];
        float r2[2] = {0.0f, 0.0f};
        if (h < p.n_heads) {
            const int64_t r = sq * p.n_heads + h;
#pragma unroll
            for (int j = 0; j < 16; ++j) y[j] = p.q_lat[r * kDLat + j * 32 + lane];
            r2[0] = p.q_rope[r * kDRope + 2 * lane];
            r2[1] = p.q_rope[r * kDRope + 2 * lane + 1];
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) y[j] = 0.0f;
        }
        if (rot) {                                           // warp-uniform
#pragma unroll
            for (int j = 0; j < 16; ++j) y[j] = ((neg >> j) & 1u) ? -y[j] : y[j];
            fwht_warp<16>(y, lane);
#pragma unroll
            for (int j = 0; j < 16; ++j) y[j] *= c512;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int k = j * 32 + lane, slab = k >> 6, kk = k & 63;
            const __half hi = __float2half_rn(y[j]);
            const __half lo = __float2half_rn(y[j] - __half2float(hi));
            uint8_t* base = img + slab * kSlab + (kk & 7) * 2;
            *reinterpret_cast<__half*>(base + sw128(n, kk >> 3)) = hi;
            *reinterpret_cast<__half*>(base + sw128(n + GQ, kk >> 3)) = lo;
        }
        {
            const __half2 hi = __floats2half2_rn(r2[0], r2[1]);
            const float2 hf = __half22float2(hi);
            const __half2 lo = __floats2half2_rn(r2[0] - hf.x, r2[1] - hf.y);
            const int c = lane >> 2, wd = lane & 3;          // k = 512 + 2*lane (+1)
            uint8_t* slab_base = img + 8 * kSlab;
            *reinterpret_cast<__half2*>(slab_base + sw128(n, c) + 4 * wd) = hi;
            *reinterpret_cast<__half2*>(slab_base + sw128(n + GQ, c) + 4 * wd) = lo;
        }
    }
}

}  // namespace tc
}  // namespace kvq
