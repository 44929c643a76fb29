// Paged KV append: scatter new K/V rows into HND pages (TensorSharp
// docs/models/gptoss.md, section 3: K and V are appended to the cache before the
// attention).  A pure copy, bound by HBM bandwidth: one thread moves one
// 16-byte vector; consecutive threads move consecutive vectors of a row, so both
// the reads of k/v and the writes of a (page, head, slot) row are coalesced.
#include "internal.h"
#include "ptx.cuh"

namespace sinkattn {

namespace {

__global__ void __launch_bounds__(256) append_kv_kernel(const AppendArgs a) {
    const int vec_per_row = a.D / 8;  // 16-byte vectors per (token, head) row
    const int64_t total = (int64_t)a.T * a.Hkv * vec_per_row;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(idx % vec_per_row);
        const int64_t tg = idx / vec_per_row;
        const int g = (int)(tg % a.Hkv);
        const int t = (int)(tg / a.Hkv);
        // request holding token t: the last i with cu_seqlens[i] <= t
        int lo = 0, hi = a.n - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.cu_seqlens[mid] <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int c0 = a.cu_seqlens[lo], c1 = a.cu_seqlens[lo + 1];
        if (t < c0 || t >= c1) {
            set_status(a.status, SINKATTN_STATUS_BAD_CU_SEQLENS);
            continue;
        }
        const int64_t pos = (int64_t)a.start_pos[lo] + (t - c0);
        if (pos < 0 || pos / kPageSize >= a.max_pages) {
            set_status(a.status, SINKATTN_STATUS_BAD_LENGTH);
            continue;
        }
        const int pg = a.block_table[(int64_t)lo * a.max_pages + pos / kPageSize];
        if (pg < 0 || pg >= a.num_pages) {
            set_status(a.status, SINKATTN_STATUS_BAD_PAGE);
            continue;
        }
        const int64_t src = (tg * a.D) + c * 8;  // element offset in k / v
        const int64_t dst = ((((int64_t)pg * a.Hkv + g) * kPageSize) + pos % kPageSize) * a.D + c * 8;
        const uint4 kv = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(a.k) + src);
        const uint4 vv = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(a.v) + src);
        *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.k_pages) + dst) = kv;
        *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.v_pages) + dst) = vv;
    }
}

}  // namespace

cudaError_t launch_append_kv(const AppendArgs &a, cudaStream_t stream) {
    const int64_t total = (int64_t)a.T * a.Hkv * (a.D / 8);
    if (total == 0) return cudaSuccess;
    int device = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    const int64_t want = (total + 255) / 256;
    const int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    append_kv_kernel<<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sinkattn
