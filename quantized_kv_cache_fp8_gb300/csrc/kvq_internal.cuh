// kvq_internal.cuh — declarations shared by the translation units of libkvq.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>
#include <cstddef>
#include <utility>

#include "kvq.h"
#include "kvq_tq_codebooks.cuh"

namespace kvq {

constexpr int kDLat = 512;
constexpr int kDRope = 64;
// SM count of a GB300, used only where no device can be queried (host-only size queries
// on a machine without a GPU); every launch plans with sm_count().
constexpr int kDefaultSMs = 152;

// The number of SMs of the current device (cudaDevAttrMultiProcessorCount), queried once
// per device and cached; kDefaultSMs when there is no device.
int sm_count();

// The limit, in ns, of the bounded device waits in the tensor-core decode kernels'
// pipelines (kvq_set_wait_limit_ns; 2 s by default).  Their final drains always allow
// the default, so that an aborted CTA still lands every copy and MMA it issued.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
uint64_t wait_limit_ns();

// fp32(1/sqrt(n)) for the supported TQ4 widths, correctly rounded.
__host__ __device__ inline float tq4_inv_sqrt(int n)
{
    switch (n) {
        case 64: return 0.125f;
        case 128: return 0x1.6a09e6p-4f;   // bits 0x3DB504F3
        case 256: return 0.0625f;
        case 512: return 0x1.6a09e6p-5f;   // bits 0x3D3504F3
        default: return 0.03125f;          // 1024
    }
}

// The TQ4 codebook: the 16-level Lloyd-Max quantiser of N(0,1) (the fixed point of
// "thresholds are midpoints, centroids are cell means"), each centroid rounded to the
// nearest binary16 value.  Stored as binary16 bit patterns, ascending.
constexpr uint16_t kTq4CentroidBits[16] = {
    0xC177, 0xC023, 0xBE79, 0xBD06, 0xBB8A, 0xB941, 0xB635, 0xB01C,
    0x301C, 0x3635, 0x3941, 0x3B8A, 0x3D06, 0x3E79, 0x4023, 0x4177};

// The same centroids as exact fp32 values, and the 15 thresholds (midpoints of
// adjacent centroids, exact in fp32).
constexpr float kTq4Centroids[16] = {
    -0x1.5dcp+1f, -0x1.08cp+1f, -0x1.9e4p+0f, -0x1.418p+0f, -0x1.e28p-1f, -0x1.504p-1f,
    -0x1.8d4p-2f, -0x1.07p-3f, 0x1.07p-3f, 0x1.8d4p-2f, 0x1.504p-1f, 0x1.e28p-1f,
    0x1.418p+0f, 0x1.9e4p+0f, 0x1.08cp+1f, 0x1.5dcp+1f};
constexpr float kTq4Thresholds[15] = {
    -0x1.334p+1f, -0x1.d7ep+0f, -0x1.6fep+0f, -0x1.196p+0f, -0x1.996p-1f, -0x1.0b7p-1f,
    -0x1.086p-2f, 0.0f, 0x1.086p-2f, 0x1.0b7p-1f, 0x1.996p-1f, 0x1.196p+0f, 0x1.6fep+0f,
    0x1.d7ep+0f, 0x1.334p+1f};

// The rotated tiers at 3 and 6 bits: the generated binary16 centroids (see
// gen_tq_codebooks.py), their exact fp32 values and the midpoints, at compile time.
constexpr float f16_bits_value(uint16_t h)
{
    const int e = (h >> 10) & 31, m = h & 1023;
    float v = e == 0 ? (float)m / 1024.0f * (1.0f / 16384.0f) : (1.0f + (float)m / 1024.0f);
    for (int i = 15; i < e; ++i) v *= 2.0f;
    for (int i = e; i < 15 && e != 0; ++i) v *= 0.5f;
    return (h & 0x8000) ? -v : v;
}

template <int N>
struct TqCodebook {
    float cb[N];
    float thr[N - 1];
};

template <int N>
constexpr TqCodebook<N> tq_codebook_of(const uint16_t (&bits)[N])
{
    TqCodebook<N> r{};
    for (int k = 0; k < N; ++k) r.cb[k] = f16_bits_value(bits[k]);
    for (int k = 0; k + 1 < N; ++k) r.thr[k] = (r.cb[k] + r.cb[k + 1]) * 0.5f;
    return r;
}

constexpr TqCodebook<8> kTq3 = tq_codebook_of(kTq3CentroidBits);
constexpr TqCodebook<64> kTq6 = tq_codebook_of(kTq6CentroidBits);

__host__ __device__ constexpr bool rotated_format(int fmt)
{
    return fmt == KVQ_FMT_TQ4 || fmt == KVQ_FMT_TQ6 || fmt == KVQ_FMT_TQ3;
}
__host__ __device__ constexpr int rotated_bits(int fmt)
{
    return fmt == KVQ_FMT_TQ3 ? 3 : fmt == KVQ_FMT_TQ6 ? 6 : 4;
}

// ------------------------------------------------------------------------------------
// Walsh-Hadamard butterflies over a warp-distributed row: element i = k * 32 + lane,
// VPL registers per lane.  Stages run in the order h = 1, 2, ..., 32 * VPL / 2: the
// five lane stages (shuffles) first, then the register stages.  Each butterfly is
// (a, b) -> (a + b, a - b) in fp32.  A lane stage computes its half as one fused
// multiply-add with a +-1 multiplier, fma(s, own, partner): the product is exact, so the
// single rounding gives the same bits as the add or subtract, with no lane-dependent
// branch.
// ------------------------------------------------------------------------------------
template <int VPL>
__device__ __forceinline__ void fwht_warp(float (&y)[VPL], int lane)
{
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const float sgn = (lane & m) ? -1.0f : 1.0f;   // upper lane: partner - own
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const float p = __shfl_xor_sync(0xffffffffu, y[k], m);
            y[k] = __fmaf_rn(sgn, y[k], p);
        }
    }
#pragma unroll
    for (int hk = 1; hk < VPL; hk <<= 1) {
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            if ((k & hk) == 0) {
                const float a = y[k], b = y[k + hk];
                y[k] = __fadd_rn(a, b);
                y[k + hk] = __fsub_rn(a, b);
            }
        }
    }
}

// ---- dependent launches ----------------------------------------------------------------
// A kernel launched by launch_dependent() may start while the kernel before it in the
// stream is still running; before it touches that kernel's output it calls
// grid_dependency_wait(), which returns once the earlier kernel has completed and its
// writes are visible.  A kernel calls grid_dependents_launch() to let the next kernel
// start early.  Both are no-ops when no such launch is involved.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Record a one-line reason for kvq_last_error() and return `status`.
int set_last_error(int status, const char* fmt, ...);

// The host-side checks of the decode entry points, shared by kvq_mla_decode and
// kvq_mla_decode_noalloc so that each reports failures under its own name:
// fault_injected: the status kvq_set_fault armed for `entry`, else 0;
// validate_mla_decode_call: the problem and the out / lse pointers (no CUDA call);
// mla_decode_checked: those checks, the workspace checks, then the launches.
int fault_injected(const char* entry);
int validate_mla_decode_call(const kvq_mla_problem* p, const float* out, const float* lse,
                             const char* entry);
int mla_decode_checked(const kvq_mla_problem* p, float* out, float* lse, void* workspace,
                       size_t ws_bytes, uint32_t* dev_status, cudaStream_t stream,
                       const char* entry);

// ---- launchers (host), each enqueues on `s` and returns the launch error ----------
cudaError_t launch_encode_fp8(const float* x, int64_t rows, int dim, int64_t ldx,
                              uint8_t* codes, int64_t ldc, float* scales, cudaStream_t s);
cudaError_t launch_encode_tq4(const float* x, int64_t rows, int dim, int64_t ldx,
                              const uint32_t* sign_bits, uint8_t* packed, int64_t ldp,
                              float* radius, cudaStream_t s);
// rotated tiers at b = 3, 4, 6 bits: b = 4 is launch_encode_tq4
cudaError_t launch_encode_tq(const float* x, int64_t rows, int dim, int64_t ldx, int bits,
                             const uint32_t* sign_bits, uint8_t* packed, int64_t ldp,
                             float* radius, cudaStream_t s);
// a row's latent (fp8 or rotated, by fmt) and rope key (fp8), one launch when aligned
cudaError_t launch_encode_mla(const float* c_lat, int64_t ldx, const float* k_rope, int64_t ldr,
                              int64_t rows, int fmt, const uint32_t* sign_bits, uint8_t* lat,
                              int64_t ldl, float* lat_scale, uint8_t* rope, int64_t ldc,
                              float* rope_scale, cudaStream_t s);
// the stored codebook of width b (2^b centroids, 2^b - 1 thresholds), host side
void tq_codebook_values(int bits, float* centroids, float* thresholds);
cudaError_t launch_append_q4(const float* k, const float* v, int n_seq, const int32_t* pos0,
                             int n_tok, int n_heads, const int32_t* page_table, int max_pages,
                             int page_size, int64_t n_cells, uint8_t* k_pool, uint8_t* v_pool,
                             uint32_t* dev_status, cudaStream_t s);
cudaError_t launch_project_append_q4(const float* h, int n_seq, const int32_t* pos0, int n_tok,
                                     int d_model, const void* w_k, const void* w_v, bool w_bf16,
                                     int n_heads, const int32_t* page_table, int max_pages,
                                     int page_size, int64_t n_cells, uint8_t* k_pool,
                                     uint8_t* v_pool, uint32_t* dev_status, cudaStream_t s);
cudaError_t launch_gather_q4(const kvq_gather_desc& d, cudaStream_t s);
cudaError_t launch_gather_mla(const kvq_gather_desc& d, cudaStream_t s);

struct DecodePlan {
    bool tcf8 = false;      // tensor-core (tcgen05 kind::f8f6f4) kernel of the fp8 tier, 16 heads a CTA
    bool tc16 = false;      // tensor-core (tcgen05) kernel, 16 heads a CTA, codes converted once
    bool tc = false;        // tensor-core (tcgen05) kernel, 32 heads a CTA
    bool mma = false;       // warp-level MMA kernel (blocks of 16 heads)
    bool premix = false;    // tc / tc16 put the unrotation's stages h = 128, 256 into the
                            // rotated rows' partials; the combine takes four quarters a row
    bool by_fmt = false;    // a batch of fp8 and TQ4 sequences: the fp8 ones on the e4m3
                            // kernel, the TQ4 ones on the 32-head kernel (tc is set too)
    int split_rows = 0;     // candidate rows per split
    int n_splits = 0;       // splits per (seq, query) at most
    int n_cand_max = 0;     // candidate rows of the longest (seq, query)
    int head_block = 0;     // heads per CTA
    size_t off_qrot = 0, off_qimg = 0, off_ml = 0, off_o = 0, bytes = 0;
};
bool plan_decode(const kvq_mla_problem& p, DecodePlan& plan);
cudaError_t launch_mla_decode(const kvq_mla_problem& p, const DecodePlan& plan, float* out,
                              float* lse, void* ws, uint32_t* dev_status, cudaStream_t s);
size_t tc_q_image_bytes(const kvq_mla_problem& p);
size_t tc16_q_image_bytes(const kvq_mla_problem& p);
// fmt_split: the kernel reads the sequences of its own tier only and leaves the others'
// partials to the kernel of the other tier (the e4m3 kernel skips non-fp8 sequences, the
// 32-head kernel fp8 ones)
cudaError_t launch_mla_decode_tcf8(const kvq_mla_problem& p, const DecodePlan& plan, float* part_ml,
                                   float* part_o, uint32_t* dev_status, cudaStream_t s, bool fmt_split);
cudaError_t launch_mla_decode_tc16(const kvq_mla_problem& p, const DecodePlan& plan, void* q_img,
                                   float* part_ml, float* part_o, uint32_t* dev_status, cudaStream_t s);
cudaError_t launch_mla_decode_tc(const kvq_mla_problem& p, const DecodePlan& plan,
                                 const float* q_rot, void* q_img, float* part_ml, float* part_o,
                                 uint32_t* dev_status, cudaStream_t s, bool fmt_split);

// the warp-level MMA decode (kvq_decode_mma.cu)
int mma_head_block();
void plan_mma_splits(const kvq_mla_problem& p, int64_t n_cand, int64_t& split_rows);
cudaError_t launch_mla_decode_mma(const kvq_mla_problem& p, const DecodePlan& plan, float* part_ml,
                                  float* part_o, uint32_t* dev_status, cudaStream_t s);

struct Q4Plan {
    int split_rows = 0;     // positions per split
    int n_splits = 0;       // splits per (seq, KV head)
    size_t off_ml = 0, off_o = 0, bytes = 0;
};
bool plan_q4_decode(const kvq_q4_problem& p, Q4Plan& plan);
cudaError_t launch_q4_decode(const kvq_q4_problem& p, const Q4Plan& plan, float* out, float* lse,
                             void* ws, uint32_t* dev_status, cudaStream_t s);

}  // namespace kvq
