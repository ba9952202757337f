// svpa_noalloc.cu -- paged verification attention for callers that may not
// allocate device memory.
//
// svpa_paged_verify_attn needs a caller-provided workspace (split-KV partial
// results and the scheduler/ticket words).  Some callers cannot provide one:
// code that runs inside a host framework which owns every device allocation
// and forbids cudaMalloc/cudaFree on its hot path (an allocation there can
// synchronise the device and fragments the framework's memory pool), or
// plugin code that is handed only input and output buffers.  This entry
// point takes its scratch from a fixed-size array that lives in the library
// itself (a file-scope __device__ array, kScratchBytes bytes on every GPU that
// loads the library, held until the process exits), and never calls
// cudaMalloc, cudaFree or any allocating routine.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/svpa.h"
#include "svpa_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

// The scratch array.  In host code this name is only a handle for
// cudaGetSymbolAddress, never a device address.
static __device__ __align__(256) unsigned char g_svpa_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices];  // device address of g_svpa_scratch, per device

// Look up (once per device, with that device current) the device address of
// the scratch array.  With CUDA's lazy module loading (the default), this
// first lookup is also what loads the library's module on that device, and
// loading it reserves the 32 MiB array there: the one time this entry point
// makes the driver reserve memory.  The cached address belongs to the
// runtime's primary context of each device; contexts made through the driver
// API are not supported.
svpa_status scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SVPA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SVPA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_svpa_scratch) != cudaSuccess || !p) return SVPA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SVPA_OK;
}

}  // namespace

extern "C" {

svpa_status svpa_paged_verify_attn_noalloc(const svpa_attn_params *p, const void *q, const void *k_pool,
                                           const void *v_pool, const float *k_scale, const float *v_scale,
                                           const int32_t *block_table, const int32_t *context_lens,
                                           const uint64_t *ancestor_mask, void *out, float *lse,
                                           int32_t *error_flag, void *stream) {
    svpa::NvtxRange nvtx_range("svpa_paged_verify_attn_noalloc");
    size_t need = 0;
    svpa_status s = svpa_attn_workspace_size(p, &need);
    if (s != SVPA_OK) return s;
    if (need > kScratchBytes) return SVPA_ERR_WORKSPACE;  // the shape needs more than the fixed array
    if (p->batch == 0) return SVPA_OK;
    // every check of the workspace entry point but the workspace itself, so
    // that a rejected call has enqueued nothing (not even the clear below)
    s = svpa::check_attn_call(p, q, k_pool, v_pool, k_scale, v_scale, block_table, context_lens, ancestor_mask,
                              out, error_flag);
    if (s != SVPA_OK) return s;
    void *ws = nullptr;
    s = scratch_for_current_device(&ws);
    if (s != SVPA_OK) return s;
    // The scheduler counters and per-(sequence, kv head) tickets at the head
    // of the scratch must start at zero; the array keeps whatever the last
    // call left, so clear them on the caller's stream.
    const size_t tickets = ((size_t)p->batch * p->num_kv_heads * sizeof(int32_t) + 255) / 256 * 256;
    const size_t head = 256 + tickets;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, head < need ? head : need, st) != cudaSuccess) return SVPA_ERR_CUDA;
    return svpa_paged_verify_attn(p, q, k_pool, v_pool, k_scale, v_scale, block_table, context_lens,
                                  ancestor_mask, out, lse, ws, kScratchBytes, error_flag, stream);
}

}  // extern "C"
