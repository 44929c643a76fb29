// Paged KV append: scatter new K/V rows into HND pages (TensorSharp
// docs/models/gptoss.md, section 3: K and V are appended to the cache before the
// attention).  A pure copy, bound by HBM bandwidth: one warp moves one token (its
// K and V rows of every KV head); consecutive lanes move consecutive 16-byte
// vectors, so both the reads of k/v and the writes of a (page, head, slot) row are
// coalesced.
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

// One warp per token (grid-stride over tokens).  Each block first copies cu_seqlens and
// start_pos into shared memory (when the batch has at most kStageReqs requests), so that
// finding a token's request and position costs no global round trip.  The warp then loads
// the token's K and V rows (Hkv x D contiguous bf16 each, coalesced 16-byte vectors, kPer
// per lane per pass) - those loads depend on nothing - and only then looks up the token's
// request (a binary search over cu_seqlens, the same for every lane), its position and its
// page, so the one dependent global load left (the block-table entry) overlaps the data
// loads; then each lane stores its vectors to (page, head, slot) rows of the pages.
constexpr int kAppendWarps = 8;   // warps per 256-thread block
constexpr int kPer = 2;           // 16-byte vectors per lane and pass, of K and of V each
constexpr int kStageReqs = 1024;  // requests whose cu_seqlens / start_pos a block stages

template <bool kFp8>
__global__ void __launch_bounds__(256) append_kv_kernel(const AppendArgs a) {
    __shared__ int s_cu[kStageReqs + 1];
    __shared__ int s_start[kStageReqs];
    const bool staged = a.n <= kStageReqs;
    if (staged) {
        for (int i = threadIdx.x; i <= a.n; i += blockDim.x) {
            s_cu[i] = a.cu_seqlens[i];
            if (i < a.n) s_start[i] = a.start_pos[i];
        }
    }
    __syncthreads();
    const int *cu = staged ? s_cu : a.cu_seqlens;
    const int *sp = staged ? s_start : a.start_pos;
    const int lane = threadIdx.x & 31;
    const int vec_per_row = a.D / 8;              // 16-byte vectors per (token, head) row
    const int vec_per_tok = a.Hkv * vec_per_row;  // per token, of K and of V each
    const int nwarps = gridDim.x * kAppendWarps;
    for (int t = blockIdx.x * kAppendWarps + (threadIdx.x >> 5); t < a.T; t += nwarps) {
        const uint4 *krow = reinterpret_cast<const uint4 *>(
            reinterpret_cast<const __nv_bfloat16 *>(a.k) + (int64_t)t * a.Hkv * a.D);
        const uint4 *vrow = reinterpret_cast<const uint4 *>(
            reinterpret_cast<const __nv_bfloat16 *>(a.v) + (int64_t)t * a.Hkv * a.D);
        bool looked_up = false, skip = false;
        int64_t page_base = 0;  // element offset of (page, head 0, slot) in the pages
        for (int base = 0; base < vec_per_tok; base += 32 * kPer) {
            uint4 kx[kPer], vx[kPer];
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                const int v = base + e * 32 + lane;
                if (v < vec_per_tok) {
                    kx[e] = krow[v];
                    vx[e] = vrow[v];
                }
            }
            if (!looked_up) {
                looked_up = true;
                // request holding token t: the last i with cu_seqlens[i] <= t
                int lo = 0, hi = a.n - 1;
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (cu[mid] <= t)
                        lo = mid;
                    else
                        hi = mid - 1;
                }
                const int c0 = cu[lo], c1 = cu[lo + 1];
                uint32_t bad = 0;
                int64_t pos = 0;
                if (t < c0 || t >= c1) {
                    bad = SINKATTN_STATUS_BAD_CU_SEQLENS;
                } else {
                    pos = (int64_t)sp[lo] + (t - c0);
                    if (pos < 0 || pos / kPageSize >= a.max_pages) bad = SINKATTN_STATUS_BAD_LENGTH;
                }
                int pg = -1;
                if (!bad) {
                    pg = a.block_table[(int64_t)lo * a.max_pages + pos / kPageSize];
                    if (pg < 0 || pg >= a.num_pages) bad = SINKATTN_STATUS_BAD_PAGE;
                }
                if (bad) {
                    if (lane == 0) set_status(a.status, bad);
                    skip = true;
                } else {
                    page_base = ((int64_t)pg * a.Hkv * kPageSize + pos % kPageSize) * a.D;
                }
            }
            if (skip) break;  // warp-uniform
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                const int v = base + e * 32 + lane;
                if (v < vec_per_tok) {
                    const int g = v / vec_per_row, c = v % vec_per_row;
                    const int64_t dst = page_base + (int64_t)g * kPageSize * a.D + c * 8;
                    if (kFp8) {
                        const float ks = a.k_scale ? a.k_scale[g] : 1.f, vs = a.v_scale ? a.v_scale[g] : 1.f;
                        *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(a.k_pages) + dst) =
                            make_uint2(quantize4(make_uint2(kx[e].x, kx[e].y), ks),
                                       quantize4(make_uint2(kx[e].z, kx[e].w), ks));
                        *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(a.v_pages) + dst) =
                            make_uint2(quantize4(make_uint2(vx[e].x, vx[e].y), vs),
                                       quantize4(make_uint2(vx[e].z, vx[e].w), vs));
                    } else {
                        *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.k_pages) + dst) = kx[e];
                        *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.v_pages) + dst) = vx[e];
                    }
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_append_kv(const AppendArgs &a, cudaStream_t stream) {
    if (a.T <= 0 || a.Hkv <= 0) return cudaSuccess;
    int device = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    // one warp per token, up to 8 blocks (64 warps) per SM; the warps stride over the rest
    const int64_t want = ((int64_t)a.T + kAppendWarps - 1) / kAppendWarps;
    const int grid = (int)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    if (a.fp8)
        append_kv_kernel<true><<<grid, 32 * kAppendWarps, 0, stream>>>(a);
    else
        append_kv_kernel<false><<<grid, 32 * kAppendWarps, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sinkattn
