// Library-wide entry points (version, status text, status read-back) and the cached
// device queries the launchers use.
#include <cuda_runtime.h>

#include <atomic>

#include "vce.h"
#include "vce_check.cuh"
#include "vce_host.h"

namespace vce {

namespace {
std::atomic<int> g_sms[kMaxDevices];
thread_local int g_last_cuda = 0;   // the last failed CUDA result an entry point saw on this thread
std::atomic<int> g_arch[kMaxDevices];   // 0 unknown, 1 ok, -1 not sm_100-family

int current_device() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
    return d;
}
}  // namespace

cudaError_t record_cuda(cudaError_t e) {
    if (e != cudaSuccess) g_last_cuda = (int)e;
    return e;
}

int device_sm_count() {
    const int d = current_device();
    if (d < 0) return 1;
    int n = g_sms[d].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n < 1) n = 1;
    g_sms[d].store(n, std::memory_order_relaxed);
    return n;
}

int require_sm100() {
    const int d = current_device();
    if (d < 0) return VCE_ERR_CUDA;
    int a = g_arch[d].load(std::memory_order_relaxed);
    if (a == 0) {
        int major = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess) return VCE_ERR_CUDA;
        a = (major == 10) ? 1 : -1;
        g_arch[d].store(a, std::memory_order_relaxed);
    }
    return a == 1 ? VCE_OK : VCE_ERR_DEVICE;
}

}  // namespace vce

extern "C" int vce_abi_version(void) { return VCE_ABI_VERSION; }

extern "C" size_t vce_row_stats_floats(void) { return VCE_ROW_STATS; }

extern "C" const char* vce_status_string(int status) {
    switch (status) {
        case VCE_OK: return "ok";
        case VCE_ERR_LABEL: return "a label is neither ignore_index nor in [0, V)";
        case VCE_ERR_NULL: return "a required pointer is NULL";
        case VCE_ERR_DTYPE: return "unknown or unsupported dtype or reduction";
        case VCE_ERR_SHAPE: return "invalid or overflowing size";
        case VCE_ERR_LD: return "leading dimension smaller than the row length";
        case VCE_ERR_ALIGN: return "misaligned pointer";
        case VCE_ERR_WORKSPACE: return "workspace missing or too small";
        case VCE_ERR_CUDA: return "a CUDA runtime call failed";
        case VCE_ERR_ARG: return "invalid argument";
        case VCE_ERR_DEVICE: return "the current device is not an sm_100-family GPU";
        case VCE_ERR_SCRATCH_LIMIT: return "k * T exceeds the built-in scratch of ce_merge_chunks_noalloc";
        case 100: return "the two CTAs of a GEMM pair were given different tensor-memory columns";
        case 101: return "a GEMM pipeline wait for a free shared-memory stage gave up";
        case 102: return "a GEMM pipeline wait for a loaded shared-memory stage gave up";
        case 103: return "a GEMM pipeline wait for a free accumulator gave up";
        case 104: return "a GEMM pipeline wait for a finished accumulator gave up";
        case 105: return "a CE stage-ring wait for a free shared-memory stage gave up";
        case 106: return "a CE stage-ring wait for a loaded shared-memory stage gave up";
        case 107: return "a one-pass CE wait for the cluster's row statistics gave up";
        case 108: return "a CE stage-ring wait for the warps' partial row statistics gave up";
        case 109: return "a one-pass CE wait for a row's gradient coefficients gave up";
        case 110: return "a CE forward wait for free statistics slots gave up";
        case 111: return "a CE forward ring was launched with consumer groups for rows too long for them";
        case 112: return "a CE forward wait for the batch's label count gave up";
        case 121: return "debug check: a row index outside [0, T)";
        case 122: return "debug check: a column range outside its row or chunk";
        case 123: return "debug check: a chunk or segment index outside its table";
        case 124: return "debug check: a stage or ring slot outside the ring";
        case 125: return "debug check: a GEMM output tile outside the output";
        default: return "unknown status";
    }
}

extern "C" int vce_get_status(const int32_t* status, vce_stream_t s, int32_t* host_out) {
    if (!status || !host_out) return VCE_ERR_NULL;
    if (cudaMemcpyAsync(host_out, status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return VCE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return VCE_ERR_CUDA;
    return VCE_OK;
}

extern "C" int vce_debug_checks(void) { return vce::dbg::kEnabled ? 1 : 0; }

extern "C" int vce_debug_status(int32_t* host_out) {
    if (!host_out) return VCE_ERR_NULL;
    *host_out = 0;
    if (!vce::dbg::kEnabled) return VCE_OK;
    if (cudaDeviceSynchronize() != cudaSuccess) return VCE_ERR_CUDA;
    int (*const readers[])(int32_t*) = {vce::debug_word_ce_fwd,   vce::debug_word_ce_bwd, vce::debug_word_ce_fwd_ring,
                                        vce::debug_word_ce_bwd_ring, vce::debug_word_ce_ring, vce::debug_word_ce_fused,
                                        vce::debug_word_lce,      vce::debug_word_gemm_hooks};
    for (auto rd : readers) {
        int32_t w = 0;
        if (rd(&w) != 0) return VCE_ERR_CUDA;
        if (*host_out == 0) *host_out = w;   // the first code found; every word is cleared
    }
    return VCE_OK;
}

extern "C" int vce_last_cuda_error(void) {
    int e = vce::g_last_cuda;
    vce::g_last_cuda = 0;
    const cudaError_t rt = cudaGetLastError();   // also clears the runtime's own record
    return e ? e : (int)rt;
}

extern "C" const char* vce_cuda_error_name(int code) { return cudaGetErrorName((cudaError_t)code); }
