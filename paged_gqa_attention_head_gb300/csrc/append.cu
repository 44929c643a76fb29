// Paged KV append: scatter new K/V rows into HND pages (TensorSharp
// docs/models/gptoss.md, section 3: K and V are appended to the cache before the
// attention).  A pure copy, bound by HBM bandwidth: one thread moves one
// 16-byte vector; consecutive threads move consecutive vectors of a row, so both
// the reads of k/v and the writes of a (page, head, slot) row are coalesced.
//
// Into an FP8 E4M3 cache each element x becomes the E4M3 code nearest to
// x / scale[g] (IEEE single-precision division; nearest, ties to even; finite
// overflow saturates to +-448, NaN stays NaN): one thread reads 8 bf16 (16 bytes)
// and writes 8 codes (8 bytes).
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"

namespace sinkattn {

namespace {

// Four bf16 (two packed pairs) -> four E4M3 codes of x / s, lowest element in the low byte.
__device__ __forceinline__ uint32_t quantize4(uint2 bf, float s) {
    const float x0 = __uint_as_float(bf.x << 16), x1 = __uint_as_float(bf.x & 0xFFFF0000u);
    const float x2 = __uint_as_float(bf.y << 16), x3 = __uint_as_float(bf.y & 0xFFFF0000u);
    const uint32_t c01 = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(x0, s), __fdiv_rn(x1, s)),
                                                  __NV_SATFINITE, __NV_E4M3);
    const uint32_t c23 = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(x2, s), __fdiv_rn(x3, s)),
                                                  __NV_SATFINITE, __NV_E4M3);
    return (c01 & 0xFFFFu) | (c23 << 16);
}

template <bool kFp8>
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
        if (kFp8) {
            const float ks = a.k_scale ? a.k_scale[g] : 1.f, vs = a.v_scale ? a.v_scale[g] : 1.f;
            *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(a.k_pages) + dst) =
                make_uint2(quantize4(make_uint2(kv.x, kv.y), ks), quantize4(make_uint2(kv.z, kv.w), ks));
            *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(a.v_pages) + dst) =
                make_uint2(quantize4(make_uint2(vv.x, vv.y), vs), quantize4(make_uint2(vv.z, vv.w), vs));
        } else {
            *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.k_pages) + dst) = kv;
            *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.v_pages) + dst) = vv;
        }
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
    if (a.fp8)
        append_kv_kernel<true><<<grid, 256, 0, stream>>>(a);
    else
        append_kv_kernel<false><<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sinkattn
