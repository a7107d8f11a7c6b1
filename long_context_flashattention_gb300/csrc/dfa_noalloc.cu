// dfa_noalloc.cu -- dfa_attn_bwd_noalloc: the attention backward for callers
// that cannot allocate device memory.
//
// dfa_attn_bwd needs scratch memory (an fp32 dQ accumulator, the per-row D
// values and a status word) in a caller-supplied workspace.  Some callers have
// no way to obtain one: code running where cudaMalloc is not allowed or not
// wanted (a host callback, a plugin that only receives tensor pointers from
// its framework, a latency-critical loop that forbids allocation after
// start-up).  This entry point takes its scratch from a fixed array in device
// memory that belongs to the library instead.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes: every
// GPU that loads the library holds it until the process exits.  Its device
// address is looked up once per device context (cudaGetSymbolAddress, with
// that device current) on the first call made in that context; that first
// call should therefore come before any stream capture.  A context that ends
// (cudaDeviceReset) takes the array with it: the next call, in the new
// context, looks the address up again, because the cache is keyed on the
// context's unique id.  Every call on a device shares the one array, which
// keeps the last call's contents: calls that overlap on the GPU (different
// streams, no ordering between them) race on it.
#include <cstdint>
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/dfa.h"

namespace dfa {
dfa_status set_error(dfa_status s, const char* fmt, ...);
}

static constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB

// The scratch itself.  In host code this name is only a stand-in for the
// device variable: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr size_t kStatusBytes = 256;
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (0 if it cannot be read),
// through the driver entry points the runtime exposes.
unsigned long long current_context_id()
{
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault,
                                             &qa) == cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
                cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            get_current = (CtxGetCurrentFn)a;
            get_id = (CtxGetIdFn)b;
        }
        looked_up = true;
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx &&
        get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

}  // namespace

extern "C" dfa_status dfa_attn_bwd_noalloc(const dfa_attn_desc* desc, const void* q,
                                           const void* k, const void* v, const void* o,
                                           const void* dout, const float* lse, void* dq,
                                           void* dk, void* dv, void* stream)
{
    // Argument errors first, with no work queued: dfa_attn_bwd checks the
    // descriptor and the pointers before the workspace, so without one it
    // returns DFA_ERR_WORKSPACE exactly when everything else is valid.
    const dfa_status pre =
        dfa_attn_bwd(desc, q, k, v, o, dout, lse, dq, dk, dv, nullptr, 0, stream);
    if (pre != DFA_ERR_WORKSPACE)
        return pre;
    // scratch this problem needs: the workspace of dfa_attn_bwd (status word,
    // fp32 dQ accumulator, per-row records, and with query blocking fp32 dK
    // and dV)
    const size_t need = dfa_workspace_size(desc, DFA_OP_BWD);
    if (need > kNoAllocScratchBytes)
        return dfa::set_error(DFA_ERR_WORKSPACE,
                              "dfa_attn_bwd_noalloc: this problem needs %zu bytes of scratch, "
                              "above the fixed %zu", need, kNoAllocScratchBytes);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return dfa::set_error(DFA_ERR_CUDA, "dfa_attn_bwd_noalloc: no usable current device");
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        const unsigned long long ctx = current_context_id();
        if (!g_scratch_ptr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
            void* ptr = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess || !ptr)
                return dfa::set_error(DFA_ERR_CUDA, "dfa_attn_bwd_noalloc: scratch lookup: %s",
                                      cudaGetErrorString(e));
            g_scratch_ptr[dev] = ptr;
            g_scratch_ctx[dev] = ctx;
        }
        scratch = g_scratch_ptr[dev];
    }
    // The status word must start at zero; the dQ accumulator and the records
    // are rewritten by the backward's own preprocess step.
    const cudaError_t e = cudaMemsetAsync(scratch, 0, kStatusBytes, (cudaStream_t)stream);
    if (e != cudaSuccess)
        return dfa::set_error(DFA_ERR_CUDA, "dfa_attn_bwd_noalloc: %s", cudaGetErrorString(e));
    return dfa_attn_bwd(desc, q, k, v, o, dout, lse, dq, dk, dv, scratch, kNoAllocScratchBytes,
                        stream);
}
