// sdv_static.cu -- sdv_verify_multidraft_static: SpecTr-GBV verification
// whose scratch lives in a fixed device array owned by the library, for
// callers that cannot allocate device memory.
//
// Who needs this: a plugin inside a host framework that owns all device
// memory and hands the plugin only its input and output buffers; code
// running inside a custom device allocator's own hooks, where allocating
// would re-enter the allocator; and latency-critical serving loops that
// forbid cudaMalloc because it can synchronise the device and stall other
// streams.  Such callers pass inputs and outputs as usual; the scratch the
// kernels need (the per-slot node records, the trie owner table and the
// per-request status) comes from g_scratch below.
#include <mutex>

#include <cuda.h>

#include "sdv_internal.h"

namespace {

// Every GPU that loads this library reserves these bytes until the
// process exits.
constexpr size_t kStaticScratchBytes = (size_t)SDV_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
    void* addr;               // device address of g_scratch
    unsigned long long ctx;   // id of the context it belongs to (0: unknown)
};
Cached g_addr[kMaxDevices] = {};  // per device

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (the device's primary
// context for runtime callers), or false when there is none yet or the
// driver lacks the query.  The id changes when the context is destroyed
// and created again (cudaDeviceReset), and the array's address with it.
bool context_id(unsigned long long* id)
{
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static bool looked = false;
    if (!looked) {  // called with g_mu held
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
        cudaGetLastError();
        looked = true;
    }
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_scratch on the current device.  The host-side
// symbol g_scratch is not a device address; only the pointer
// cudaGetSymbolAddress returns may be handed to a kernel.  It is looked up
// once per device and context, with that device current: on the first
// call, and again on the first call after the context was reset.
int scratch_address(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return SDV_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    Cached& c = g_addr[dev];
    unsigned long long id = 0;
    const bool have_id = context_id(&id);
    if (!c.addr || (have_id && c.ctx != id)) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return SDV_ERR_CUDA;
        }
        c.addr = p;
        // the lookup made the context current if it was not yet
        c.ctx = context_id(&id) ? id : 0;
    }
    *out = c.addr;
    return SDV_OK;
}

}  // namespace

extern "C" int sdv_verify_multidraft_static(
    int B, int K, int L, int V, long long row_stride, int dtype, float temperature, const void* target_logits,
    const void* draft_logits, const int* draft_tokens, const int* lengths, const float* accept_u,
    const float* sample_u, int* accept_len, int* accept_draft, int* out_token, float* accept_prob,
    float* residual_mass, int* device_status, void* cuda_stream)
{
    const size_t need = sdv_workspace_bytes(SDV_MODE_MULTIDRAFT, B, K, L, V);
    if (need > kStaticScratchBytes) return SDV_ERR_WORKSPACE;  // problem too large for the fixed scratch
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != SDV_OK) return rc;
    // nothing in the scratch has to start at zero: every call writes each
    // record before it reads it
    return sdv_verify_multidraft(B, K, L, V, row_stride, dtype, temperature, target_logits, draft_logits,
                                 draft_tokens, lengths, accept_u, sample_u, accept_len, accept_draft, out_token,
                                 accept_prob, residual_mass, device_status, scratch, kStaticScratchBytes,
                                 cuda_stream);
}
