// Decode without a caller-provided workspace, for callers that cannot allocate
// device memory at the point where they run attention: code that must not call
// cudaMalloc (a custom allocator owns all device memory, a real-time path cannot
// take the allocator's lock or latency, or an embedding runtime forbids it).
//
// The split-KV kernel's scratch (partial softmax states of split sequences, the
// page-count prefix sum and the plan) lives in one file-scope device array of
// fixed size instead.  Every GPU that loads this library holds that array until
// the process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/sinkattn.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = SINKATTN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Device-resident scratch shared by every call on a device.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_mu;

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device, looked up once per
// device (the host-side symbol itself is not a device address).
int scratch_address(void **out) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) {
        sinkattn::record_cuda_error(e, "cudaGetDevice");
        return SINKATTN_ERR_CUDA;
    }
    if (device < 0 || device >= kMaxDevices) return SINKATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[device]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || !p) {
            sinkattn::record_cuda_error(e, "cudaGetSymbolAddress");
            return SINKATTN_ERR_CUDA;
        }
        g_scratch_ptr[device] = p;
    }
    *out = g_scratch_ptr[device];
    return SINKATTN_OK;
}

}  // namespace

extern "C" int sinkattn_decode_noalloc(const void *q, const void *k_pages, const void *v_pages,
                                       const int32_t *block_table, const int32_t *seq_lens,
                                       const float *sinks, float scale, void *out, float *lse,
                                       const sinkattn_paged_desc *desc, uint32_t *status,
                                       sinkattn_stream_t stream) {
    size_t need = 0;
    int rc = sinkattn_decode_workspace_size(desc, &need);
    if (rc) return rc;
    if (need > kScratchBytes) return SINKATTN_ERR_WORKSPACE_TOO_SMALL;
    // every argument sinkattn_decode checks is checked here first, so a rejected call
    // enqueues nothing (not even the status clear below) and leaves *status as it was
    if (desc->num_seqs > 0) {
        if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !out)
            return SINKATTN_ERR_INVALID_ARG;
        if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) ||
            !aligned(block_table, 4) || !aligned(seq_lens, 4) || (sinks && !aligned(sinks, 4)) ||
            (lse && !aligned(lse, 4)))
            return SINKATTN_ERR_INVALID_ARG;
    }
    if (status && !aligned(status, 4)) return SINKATTN_ERR_INVALID_ARG;
    void *scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (desc->num_seqs == 0) {  // an empty batch: nothing runs, its status is clear
        if (status) {
            cudaError_t e = cudaMemsetAsync(status, 0, sizeof(uint32_t), s);
            if (e != cudaSuccess) {
                sinkattn::record_cuda_error(e, "status clear");
                return SINKATTN_ERR_CUDA;
            }
        }
        return SINKATTN_OK;
    }
    // The status word is the only scratch that must start at zero; everything
    // else the merge reads is written earlier in this call by the split-KV kernel.
    cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) {
        sinkattn::record_cuda_error(e, "scratch status clear");
        return SINKATTN_ERR_CUDA;
    }
    rc = sinkattn_decode(q, k_pages, v_pages, block_table, seq_lens, sinks, scale, out, lse, desc,
                         scratch, kScratchBytes, stream);
    if (rc) return rc;
    if (status) {
        e = cudaMemcpyAsync(status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) {
            sinkattn::record_cuda_error(e, "status copy");
            return SINKATTN_ERR_CUDA;
        }
    }
    return SINKATTN_OK;
}
