// ce_merge_chunks_noalloc: the vocabulary-chunked CE for callers that cannot allocate device
// memory for the call.
//
// Some callers own no device allocator of their own for per-call scratch: a host program
// that drives this library through the C ABI alone and has no memory manager for
// short-lived device buffers, or an engine whose device memory is one arena reserved at
// start-up by another component, from which nothing may be carved for a single op.  For
// them this entry point takes the per-(chunk, row) statistics of ce_merge_chunks from a
// fixed array that the library defines in device memory, instead of from a caller-provided
// workspace.  Inputs and outputs are still the caller's.
//
// The array is a file-scope __device__ variable: every GPU on which the library's module is
// loaded holds its 4 MiB until the process exits.  Host code cannot use the array's name as
// a device address (in host code it names a host-side stand-in), so the device address is
// looked up once per device with cudaGetSymbolAddress, with that device current, and passed
// to the kernels.  The lookup is remembered together with the unique id of the device's
// current context: after a device reset the context, the loaded module and the array are new,
// and the next call looks the address up again.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "vce.h"
#include "vce_host.h"

namespace {

// One float4 (max, sum-exp, target logit, owner) per (chunk, row): k * T entries at most.
constexpr long long kScratchEntries = VCE_NOALLOC_MAX_CHUNK_ROWS;
static __device__ __align__(256) float4 g_chunk_stats_scratch[kScratchEntries];

struct ScratchEntry {
    unsigned long long ctx_id;   // unique id of the context the address belongs to (0: none yet)
    float* addr;
};
ScratchEntry g_scratch[vce::kMaxDevices];
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The unique id of the calling thread's current context (process-wide unique, never reused),
// through the driver entry points the runtime hands out; false if it cannot be read.
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    if (!get_current || !get_id) {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) != cudaSuccess ||
            qa != cudaDriverEntryPointSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) != cudaSuccess ||
            qb != cudaDriverEntryPointSuccess)
            return false;
        get_current = reinterpret_cast<CtxGetCurrentFn>(a);
        get_id = reinterpret_cast<CtxGetIdFn>(b);
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

// The array's device address on the current device; the first call for a device (and the
// first after a reset of it) looks it up.
int scratch_address(float** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= vce::kMaxDevices) return VCE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchEntry& e = g_scratch[dev];
    unsigned long long id = 0;
    const bool have_ctx = current_context_id(&id);
    if (!have_ctx || e.ctx_id != id || !e.addr) {
        // (with no context current on this thread yet, the lookup makes the device's primary
        // context current)
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_chunk_stats_scratch) != cudaSuccess || p == nullptr) return VCE_ERR_CUDA;
        if (!have_ctx && !current_context_id(&id)) return VCE_ERR_CUDA;
        e.addr = static_cast<float*>(p);
        e.ctx_id = id;
    }
    *out = e.addr;
    return VCE_OK;
}

}  // namespace

extern "C" int ce_merge_chunks_noalloc(int k, const void* const* chunk_logits, const int64_t* chunk_width,
                                       const int64_t* chunk_ld, vce_dtype dt, int64_t T, const int64_t* labels,
                                       int64_t ignore_index, vce_reduction red, float* loss_rows, float* loss_out,
                                       float* row_stats, const float* grad_output, void* const* chunk_grads,
                                       const int64_t* chunk_grad_ld, vce_dtype grad_dt, int32_t* status,
                                       vce_stream_t s) {
    if (k < 1 || k > VCE_MAX_CHUNKS) return VCE_ERR_ARG;
    if (T < 0) return VCE_ERR_SHAPE;
    if ((long long)k * T > kScratchEntries) return VCE_ERR_SCRATCH_LIMIT;
    float* scratch = nullptr;
    if (T > 0) {
        const int rc = scratch_address(&scratch);
        if (rc != VCE_OK) return rc;
    }
    // Every (chunk, row) entry the kernels read is written earlier in the same call, so the
    // contents left by a previous call need no clearing.
    return ce_merge_chunks(k, chunk_logits, chunk_width, chunk_ld, dt, T, labels, ignore_index, red, loss_rows,
                           loss_out, row_stats, grad_output, chunk_grads, chunk_grad_ld, grad_dt, scratch, status, s);
}
