// dapd_noalloc.cu -- dlm_dapd_graph_mis_noalloc: the DAPD call for callers
// that cannot allocate device memory.  Its scratch (the attention pass's
// fixed-point sums, read back by the selection kernel) lives in an array
// inside the library instead of a caller workspace.
//
// Who needs it: a serving engine whose allocator reserved nearly all of HBM
// at start-up (KV-cache pools) and hands out nothing on the decode path; a
// plug-in inside a host framework that owns every device allocation and
// gives the plug-in only its tensors; a decode loop that must not pay
// cudaMalloc's implicit device synchronisation.  They own the inputs and
// outputs, but cannot supply a workspace.
//
// The array below exists once on every GPU that loads libdlm and stays until
// the process exits.  In host code its name stands for the symbol only, not
// for a device address: the address handed to the kernels comes from
// cudaGetSymbolAddress, looked up with the device current and kept per CUDA
// context, so a device reset (which ends the context and its copy of the
// array) leads to a fresh lookup on the next call.
#include <cuda.h>

#include <mutex>

#include "dlm.h"
#include "launch.h"

namespace {

constexpr size_t kScratchBytes = DLM_DAPD_NOALLOC_MAX_BYTES;
static __device__ __align__(256) unsigned char g_dapd_scratch[kScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct DriverFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver() {
    static std::once_flag once;
    static DriverFns f;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    return f;
}

// Id of the current CUDA context (0 when there is none or it cannot be read);
// ids are never reused within a process.
unsigned long long current_context_id() {
    const DriverFns& d = driver();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (d.get_current && d.get_id && d.get_current(&ctx) == CUDA_SUCCESS && ctx && d.get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

constexpr int kMaxDevices = 64;
struct Cached {
    unsigned long long ctx_id;
    void* addr;
};
Cached g_cache[kMaxDevices] = {};
std::mutex g_mu;

// Device address of g_dapd_scratch in the current device's context.  The
// lookup runs with that device current on the first call in each context.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    const unsigned long long id = current_context_id();
    if (id == 0 || g_cache[dev].addr == nullptr || g_cache[dev].ctx_id != id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dapd_scratch);
        if (e != cudaSuccess) return e;
        g_cache[dev].addr = p;
        g_cache[dev].ctx_id = current_context_id();  // the lookup may have made the context current
    }
    *out = g_cache[dev].addr;
    return cudaSuccess;
}

}  // namespace

extern "C" dlm_status dlm_dapd_graph_mis_noalloc(const void* attn, dlm_dtype dtype, int32_t batch, int32_t n_layers,
                                                 int32_t n_heads, int64_t stride_b, int64_t stride_l,
                                                 int64_t stride_h, int64_t stride_row, int32_t block_start,
                                                 int32_t blk, const uint8_t* masked, const float* conf,
                                                 const dlm_dapd_params* params, uint8_t* selected,
                                                 int32_t* n_selected, float* s_out, float* dtilde_out,
                                                 int32_t* deg_out, uint32_t* dev_status, dlm_stream_t stream) {
    // sizes the array cannot hold are refused before anything touches the GPU
    if (batch < 0 || blk < 1 || blk > DLM_MAX_BLK) return DLM_ERR_INVALID_ARG;
    if (batch == 0) return DLM_OK;
    if (dlm_dapd_workspace_size(batch, blk) > kScratchBytes) return DLM_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return DLM_ERR_CUDA;
    // the workspace call with the library's array in place of a caller's
    // workspace: same checks, same kernels
    return dlm_dapd_graph_mis(attn, dtype, batch, n_layers, n_heads, stride_b, stride_l, stride_h, stride_row,
                              block_start, blk, masked, conf, params, selected, n_selected, s_out, dtilde_out,
                              deg_out, scratch, kScratchBytes, dev_status, stream);
}
