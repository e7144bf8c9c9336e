// kvq_q4_decode.cu — decode attention over the paged q4_0 pools (grouped-query,
// head_dim 256): Strata PR #2533, the qsa decode commit.  The query is rotated by the
// orthonormal FWHT256 (the rotation the stored K and V rows carry), each block is
// dequantised as (nibble - 8) * f32(d), and the merged output is rotated back before
// the optional sigmoid gate.
//
// A few query heads share each KV head (G = n_qh / n_kv <= 8), so a row carries
// 2 G (256 + 256) flops for 288 bytes: CUDA-core work, bound by streaming the pools.
// One warp per (split, sequence, KV head); lane l owns dims 8l .. 8l + 7 of the
// 256-wide rows, which are elements 8p .. 8p + 7 of block b = l / 4 (p = l % 4): the
// low nibbles of bytes 2 + 8p .. 9 + 8p for p < 2, the high nibbles of bytes
// 2 + 8(p - 2) .. for p >= 2.  Rows go in groups of R = 32 / G, so the R x G partial
// scores of a group are 32 values and one transposing butterfly hands each lane one
// full score.  Each row's bytes are staged through shared memory with 16-byte loads,
// the next group's loads in flight while the current group is reduced.  Split-T
// partials (m, l, o in the rotated domain, log2 units) are merged by a combine kernel
// that also rotates back and gates.
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kRowBytes = 144;           // 8 blocks of 18 bytes

struct Q4Args {
    kvq_q4_problem p;
    int split_rows, n_splits;
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

// the 8 codes of this lane in a staged row, as (code - 8) floats, and the block scale
__device__ __forceinline__ float lane_codes(const uint8_t* row, int lane, float (&x)[8])
{
    const int b = lane >> 2, p = lane & 3;
    const uint8_t* blk = row + 18 * b;
    const float d = __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(blk)));
    const uint16_t* w = reinterpret_cast<const uint16_t*>(blk + 2 + 8 * (p & 1));
    const uint32_t lo = (uint32_t)w[0] | ((uint32_t)w[1] << 16);
    const uint32_t hi = (uint32_t)w[2] | ((uint32_t)w[3] << 16);
    const int sh = p >= 2 ? 4 : 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t word = k < 4 ? lo : hi;
        const uint32_t code = (word >> (8 * (k & 3) + sh)) & 15u;
        // 2^23 + code, minus 2^23 + 8: exact
        x[k] = __uint_as_float(0x4B000000u | code) - 8388616.0f;
    }
    return d;
}

// sum over the warp's lanes of each of 32 values, transposed: lane l ends with value l
__device__ __forceinline__ float reduce_transpose32(float (&v)[32], int lane)
{
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
            const float send = up ? v[j] : v[j + w];
            const float keep = up ? v[j + w] : v[j];
            v[j] = keep + __shfl_xor_sync(kFull, send, w);
        }
    }
    return v[0];
}

template <int G>
__global__ void __launch_bounds__(32) q4_decode_kernel(const __grid_constant__ Q4Args a)
{
    constexpr int R = 32 / G;                        // rows per group
    constexpr int kPieces = 2 * R * (kRowBytes / 16);    // K and V rows, 16-byte pieces
    constexpr int kPerLane = (kPieces + 31) / 32;
    __shared__ __align__(16) uint8_t s_rows[2 * R * kRowBytes];
    grid_dependents_launch();                        // the combine may start launching
    const kvq_q4_problem& p = a.p;
    const int split = blockIdx.x, s = blockIdx.y, kvh = blockIdx.z;
    const int lane = threadIdx.x;
    const int L = min(max(p.seq_len[s], 0), p.max_seq_len);
    const int64_t r0 = (int64_t)split * a.split_rows;
    const int64_t r1 = min(r0 + (int64_t)a.split_rows, (int64_t)L);
    const int64_t head0 = (int64_t)s * p.n_qh + (int64_t)kvh * G;
    if (r0 >= r1) {
        if (lane < G) {
            const int64_t sl = (head0 + lane) * a.n_splits + split;
            a.part_ml[sl * 2] = -INFINITY;
            a.part_ml[sl * 2 + 1] = 0.0f;
        }
        return;
    }
    // rotated queries of the G heads, pre-scaled into log2 units: 8 dims per lane
    float qr[G][8];
    const float qs = p.sm_scale * kLog2e * (1.0f / 16.0f);
#pragma unroll
    for (int j = 0; j < G; ++j) {
        const float4* qp = reinterpret_cast<const float4*>(p.q + (head0 + j) * 256 + 8 * lane);
        const float4 x0 = qp[0], x1 = qp[1];
        float z[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        fwht256_lane8(z, lane);
#pragma unroll
        for (int k = 0; k < 8; ++k) qr[j][k] = z[k] * qs;
    }
    float o[G][8];
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
        for (int k = 0; k < 8; ++k) o[j][k] = 0.0f;
    float m_run = -INFINITY, l_run = 0.0f;           // of head (lane % G)

    // pool cell of position t, or -1 (flagged)
    auto cell_of = [&](int64_t t) -> int64_t {
        if (t >= r1) return -1;
        const int64_t page = t / p.page_size;
        const int64_t pid = page < p.max_pages ? p.page_table[(int64_t)s * p.max_pages + page] : -1;
        const int64_t cell = pid * p.page_size + t % p.page_size;
        if (pid < 0 || cell >= p.n_cells) {
            if (a.status) atomicOr(a.status, (unsigned)KVQ_DEV_BAD_PAGE);
            return -1;
        }
        return cell;
    };
    // this lane's pieces of a group's rows (K rows 0..R-1, then V rows), zero for
    // masked rows
    auto load_group = [&](int64_t t0, uint4 (&pc)[kPerLane], int64_t& my_cell) {
        my_cell = lane < R ? cell_of(t0 + lane) : -1;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            const int idx = lane + 32 * i;
            const int row = idx / 9, piece = idx - row * 9;
            const int r = row % R;
            const int64_t cell = __shfl_sync(kFull, my_cell, r);
            pc[i] = make_uint4(0u, 0u, 0u, 0u);
            if (idx < kPieces && cell >= 0) {
                const uint8_t* pool = row < R ? p.k_pool : p.v_pool;
                pc[i] = __ldcs(reinterpret_cast<const uint4*>(pool + (cell * p.n_kv + kvh) * kRowBytes) + piece);
            }
        }
    };
    uint4 nxt[kPerLane];
    int64_t ncell;
    load_group(r0, nxt, ncell);
    for (int64_t t0 = r0; t0 < r1; t0 += R) {
        const int64_t cur_cell = ncell;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i)
            if (lane + 32 * i < kPieces) reinterpret_cast<uint4*>(s_rows)[lane + 32 * i] = nxt[i];
        if (t0 + R < r1) load_group(t0 + R, nxt, ncell);
        __syncwarp();
        // scores: partial dot products of this lane's 8 dims, one per (row, head)
        float part[32];
        float dk[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float x[8];
            dk[r] = lane_codes(s_rows + r * kRowBytes, lane, x);
#pragma unroll
            for (int j = 0; j < G; ++j) {
                float acc = 0.0f;
#pragma unroll
                for (int k = 0; k < 8; ++k) acc = fmaf(qr[j][k], x[k], acc);
                part[r * G + j] = acc * dk[r];
            }
        }
        float sc = reduce_transpose32(part, lane);   // row lane / G, head lane % G
        const bool valid = __shfl_sync(kFull, cur_cell, lane / G) >= 0;
        sc = valid ? sc : -INFINITY;
        // online softmax per head over the R rows (lanes of equal lane % G)
        float mx = sc;
#pragma unroll
        for (int w = G; w < 32; w <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, w));
        const float m_new = fmaxf(m_run, mx);
        const float pw = (sc == -INFINITY) ? 0.0f : exp2f(sc - m_new);
        const float alpha = (m_run == -INFINITY) ? 0.0f : exp2f(m_run - m_new);
        float ps = pw;
#pragma unroll
        for (int w = G; w < 32; w <<= 1) ps += __shfl_xor_sync(kFull, ps, w);
        l_run = l_run * alpha + ps;
        m_run = m_new;
        // context: o[j] = alpha_j o[j] + sum_r p[r][j] d_v[r] (code - 8)
#pragma unroll
        for (int j = 0; j < G; ++j) {
            const float al = __shfl_sync(kFull, alpha, j);
#pragma unroll
            for (int k = 0; k < 8; ++k) o[j][k] *= al;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float x[8];
            const float dv = lane_codes(s_rows + (R + r) * kRowBytes, lane, x);
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const float pj = __shfl_sync(kFull, pw, r * G + j) * dv;
#pragma unroll
                for (int k = 0; k < 8; ++k) o[j][k] = fmaf(pj, x[k], o[j][k]);
            }
        }
        __syncwarp();
    }
    // partials: (m, l) of head j from lane j, o of all heads from every lane
    if (lane < G) {
        const int64_t sl = (head0 + lane) * a.n_splits + split;
        a.part_ml[sl * 2] = m_run;
        a.part_ml[sl * 2 + 1] = l_run;
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
        float4* dst = reinterpret_cast<float4*>(a.part_o + ((head0 + j) * a.n_splits + split) * 256 + 8 * lane);
        dst[0] = make_float4(o[j][0], o[j][1], o[j][2], o[j][3]);
        dst[1] = make_float4(o[j][4], o[j][5], o[j][6], o[j][7]);
    }
}

// one warp per (sequence, query head): merge the splits, rotate back, gate
__global__ void __launch_bounds__(256) q4_combine_kernel(const __grid_constant__ Q4Args a)
{
    const kvq_q4_problem& p = a.p;
    const int lane = threadIdx.x & 31;
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (row >= (int64_t)p.n_seq * p.n_qh) return;
    const int s = (int)(row / p.n_qh);
    const int L = min(max(p.seq_len[s], 0), p.max_seq_len);
    const int ns = (int)min((int64_t)a.n_splits, ((int64_t)L + a.split_rows - 1) / a.split_rows);
    grid_dependency_wait();                          // the partials of the decode kernel
    const float* ml = a.part_ml + row * a.n_splits * 2;
    float M = -INFINITY;
    for (int S = 0; S < ns; ++S)
        if (ml[2 * S + 1] > 0.0f) M = fmaxf(M, ml[2 * S]);
    float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float Lt = 0.0f;
    for (int S = 0; S < ns; ++S) {
        const float lS = ml[2 * S + 1];
        if (!(lS > 0.0f)) continue;
        const float w = exp2f(ml[2 * S] - M);
        Lt += w * lS;
        const float4* src = reinterpret_cast<const float4*>(a.part_o + (row * a.n_splits + S) * 256 + 8 * lane);
        const float4 x0 = src[0], x1 = src[1];
        z[0] = fmaf(w, x0.x, z[0]); z[1] = fmaf(w, x0.y, z[1]);
        z[2] = fmaf(w, x0.z, z[2]); z[3] = fmaf(w, x0.w, z[3]);
        z[4] = fmaf(w, x1.x, z[4]); z[5] = fmaf(w, x1.y, z[5]);
        z[6] = fmaf(w, x1.z, z[6]); z[7] = fmaf(w, x1.w, z[7]);
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
        // about 32 warps per SM over all (sequence, KV head) units
        const int64_t units = std::max<int64_t>(1, (int64_t)p.n_seq * p.n_kv);
        const int64_t target = (int64_t)kNumSMs * 32;
        int64_t splits = std::max<int64_t>(1, (target + units - 1) / units);
        split_rows = std::max<int64_t>(64, ((int64_t)p.max_seq_len + splits - 1) / splits);
        split_rows = (split_rows + 31) / 32 * 32;
    }
    plan.split_rows = (int)split_rows;
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
    const dim3 grid(plan.n_splits, p.n_seq, p.n_kv);
    switch (p.n_qh / p.n_kv) {
        case 1: q4_decode_kernel<1><<<grid, 32, 0, s>>>(a); break;
        case 2: q4_decode_kernel<2><<<grid, 32, 0, s>>>(a); break;
        case 4: q4_decode_kernel<4><<<grid, 32, 0, s>>>(a); break;
        case 8: q4_decode_kernel<8><<<grid, 32, 0, s>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t rows = (int64_t)p.n_seq * p.n_qh;
    return launch_dependent(q4_combine_kernel, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, s, a);
}

}  // namespace kvq
