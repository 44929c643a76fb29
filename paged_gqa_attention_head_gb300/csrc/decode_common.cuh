// Pieces of the split-KV decode plan shared by the bf16 and the FP8 decode kernels:
// the per-sequence page counts and their prefix sum (the list of (sequence, KV head,
// page) units every warp takes an equal contiguous range of) and the cursor that
// walks that list.
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace sinkattn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMinUnitsPerWarp = 4;  // pages per warp at least (keeps partials few)

// Over the 8 lanes that share lane & 3: one column of an m16n8 accumulator (its rows are
// spread over lane >> 2 and the two register halves).
__device__ __forceinline__ float col_max(float x) {
    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
    return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
}
__device__ __forceinline__ float col_sum(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 8);
    return x + __shfl_xor_sync(0xffffffffu, x, 16);
}

// Transpose of an 8x8 matrix of 16-bit elements held in MMA fragment layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Lengths (validated, clamped), the first page each sequence's query sees (0, or the
// page of its first key inside a sliding window) and the exclusive prefix sum of the
// work units of each sequence (kPPU consecutive visible pages per unit), into shared
// memory.  128 threads.
template <int kPPU = 1>
__device__ void scan_pages(const DecodeArgs &a, int *s_prefix, int *s_len, int *s_first) {
    __shared__ int s_warp_tot[4];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int per_t = (a.B + 127) / 128;
    const int b0 = min(a.B, tid * per_t), b1 = min(a.B, b0 + per_t);
    const int cap = a.max_pages * kPageSize;
    auto units = [](int L, int first) {
        return ((L + kPageSize - 1) / kPageSize - first + kPPU - 1) / kPPU;
    };
    int local = 0;
    for (int b = b0; b < b1; ++b) {
        int L = a.seq_lens[b];
        if (L < 0 || L > cap) {
            set_status(a.status, SINKATTN_STATUS_BAD_LENGTH);
            L = L < 0 ? 0 : cap;
        }
        s_len[b] = L;
        const int first = (a.window > 0 && L > a.window) ? (L - a.window) / kPageSize : 0;
        s_first[b] = first;
        local += units(L, first);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp_tot[wid] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < wid; ++w) run += s_warp_tot[w];
    for (int b = b0; b < b1; ++b) {
        s_prefix[b] = run;
        run += units(s_len[b], s_first[b]);
    }
    if (tid == 0) s_prefix[a.B] = s_warp_tot[0] + s_warp_tot[1] + s_warp_tot[2] + s_warp_tot[3];
    __syncthreads();
}

// Position in the unit list: sequence b, KV head g, unit p of the sequence.
struct Cursor {
    int b, g, p, pb;  // pb = units of sequence b
};

}  // namespace
}  // namespace sinkattn
