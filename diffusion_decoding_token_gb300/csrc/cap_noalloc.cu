// cap_noalloc.cu -- dlm_cap_select_noalloc: CAP-Decoding whose scratch lives
// inside the library, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a serving runtime whose allocator has
// reserved all of HBM up front (its KV-cache pool) and hands out nothing on the
// decode path; a plug-in that runs inside a host framework which owns every
// device allocation; a latency-critical loop that must not pay cudaMalloc's
// implicit device synchronisation.  They still own their inputs and outputs,
// but they cannot provide the CAP workspace.  This entry point uses a
// file-scope device array instead.
//
// The array below exists once per GPU that loads libdlm and stays allocated
// until the process exits.  In host code its name is only a host-side stand-in
// for the symbol, not a device address, so the address passed to the kernels
// is looked up with cudaGetSymbolAddress, once per device, with that device
// current.
#include <mutex>

#include "launch.h"

namespace {

constexpr size_t kScratchBytes = DLM_CAP_NOALLOC_MAX_BYTES;
static __device__ __align__(256) unsigned char g_cap_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of g_cap_scratch on the current device; the first call on a
// device performs the lookup (with that device current) and caches it.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_cap_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" dlm_status dlm_cap_select_noalloc(const void* logits, dlm_dtype dtype, int64_t vocab,
                                             int64_t row_stride, const int32_t* row_index, int64_t n_rows,
                                             const int32_t* argmax, const float* conf, const float* lse,
                                             const uint8_t* masked, const int32_t* scope_len,
                                             int32_t batch, int32_t blk, const dlm_cap_params* params,
                                             uint8_t* selected, int32_t* n_selected, float* D_out,
                                             uint32_t* dev_status, dlm_stream_t stream) {
    if (dtype != DLM_F32 && dtype != DLM_BF16 && dtype != DLM_F16) return DLM_ERR_UNSUPPORTED;
    if (!params || batch < 0 || batch > DLM_MAX_BATCH || blk < 1 || blk > DLM_MAX_BLK || vocab < 1 || row_stride < vocab ||
        params->p_max < 1 || params->p_max > DLM_MAX_BLK ||
        (params->high_tier_unconditional != 0 && params->high_tier_unconditional != 1))
        return DLM_ERR_INVALID_ARG;
    if (batch == 0) return DLM_OK;
    if (n_rows < 1 || (!row_index && n_rows < (int64_t)batch * blk)) return DLM_ERR_INVALID_ARG;
    if (!logits || !argmax || !conf || !lse || !masked || !selected || !n_selected) return DLM_ERR_INVALID_ARG;
    // the library-owned scratch has a fixed size: larger problems are refused
    if (dlm::cap_workspace_bytes(batch, params->p_max) > kScratchBytes) return DLM_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return DLM_ERR_CUDA;
    dlm::CapArgs a{};
    a.logits = logits;
    a.dtype = dtype;
    a.vocab = vocab;
    a.row_stride = row_stride;
    a.argmax = argmax;
    a.conf = conf;
    a.lse = lse;
    a.masked = masked;
    a.scope_len = scope_len;
    a.row_index = row_index;
    a.n_rows = n_rows;
    a.batch = batch;
    a.blk = blk;
    a.tau_low = params->tau_low;
    a.tau_high = params->tau_high;
    a.gamma = params->gamma;
    a.p_max = params->p_max;
    a.high_tier_unconditional = params->high_tier_unconditional;
    a.selected = selected;
    a.n_selected = n_selected;
    a.D_out = D_out;
    a.dev_status = dev_status;
    dlm::cap_carve(a, scratch);
    const cudaError_t e = dlm::launch_cap(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DLM_OK : DLM_ERR_CUDA;
}
