// kvq_noalloc.cu — kvq_mla_decode_noalloc: the decode with its scratch in a fixed device
// array owned by the library, for callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not available or not allowed at
// decode time, for example inside a memory pool or custom allocator that already owns
// the whole device, a latency-critical loop that must never enter the allocator, or an
// embedding that is only handed pre-placed input and output buffers.  Such callers
// cannot provide the workspace kvq_mla_decode asks for.
//
// The scratch is `g_decode_scratch`, a file-scope __device__ array of
// kNoallocScratchBytes; every GPU that loads the library holds it until the process
// exits.  In host code that name is only a host-side stand-in, not a device address, so
// the first call on each device (with that device current) looks up the real address
// with cudaGetSymbolAddress and caches it.  The decode writes every scratch byte before
// reading it, so nothing needs clearing between calls; but all calls share the one
// array, so calls that overlap on the GPU (two streams, two host threads) race and must
// be serialised by the caller.
#include <cstdarg>
#include <mutex>

#include "kvq_internal.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(64) << 20;   // 64 MiB

__device__ __align__(256) unsigned char g_decode_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

}  // namespace

extern "C" int kvq_mla_decode_noalloc(const kvq_mla_problem* p, float* out, float* lse,
                                      uint32_t* dev_status, kvq_stream_t stream)
{
    const char* E = "kvq_mla_decode_noalloc";
    // every host-side check comes first, under this entry's name, so that a refused or
    // empty call touches no device (no symbol lookup, nothing enqueued)
    if (int st = kvq::fault_injected(E)) return st;
    if (int st = kvq::validate_mla_decode_call(p, out, lse, E)) return st;
    if (p->n_seq == 0) return KVQ_OK;
    const size_t need = kvq_mla_decode_workspace(p);
    if (need > kNoallocScratchBytes)
        return kvq::set_last_error(KVQ_EWORKSPACE,
                                   "%s: this problem needs %zu bytes of scratch but the fixed "
                                   "array holds %zu; use kvq_mla_decode with a workspace",
                                   E, need, kNoallocScratchBytes);
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return kvq::set_last_error(KVQ_ECUDA, "%s: %s", E, cudaGetErrorString(e));
    if (device < 0 || device >= 64)
        return kvq::set_last_error(KVQ_EINVAL, "%s: device index %d out of range", E, device);
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        if (!g_scratch_ptr[device]) {
            void* ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
            if (e != cudaSuccess)
                return kvq::set_last_error(KVQ_ECUDA, "%s: cudaGetSymbolAddress: %s", E,
                                           cudaGetErrorString(e));
            g_scratch_ptr[device] = ptr;
        }
        scratch = g_scratch_ptr[device];
    }
    return kvq::mla_decode_checked(p, out, lse, scratch, kNoallocScratchBytes, dev_status,
                                   (cudaStream_t)stream, E);
}
