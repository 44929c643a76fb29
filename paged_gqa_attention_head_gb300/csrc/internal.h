// Internal interfaces between the C ABI (api.cpp) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sinkattn {

// Remember the CUDA error behind a SINKATTN_ERR_CUDA return and the call that
// produced it (per host thread).
void record_cuda_error(cudaError_t e, const char *where);

constexpr int kPageSize = 16;
constexpr uint32_t kStatusBytes = 256;  // workspace header holding the status word

// Give-up time of a pipeline wait for a descriptor (wait_limit_us; 0 = 2 s).
inline uint64_t wait_limit_ns(int32_t us) { return us > 0 ? (uint64_t)us * 1000ull : 2000000000ull; }

// Arguments of the two decode kernels (plain device pointers and sizes).
struct DecodeArgs {
    const void *q;               // bf16 [B, Hq, D]
    const int32_t *block_table;  // [B, max_pages]
    const int32_t *seq_lens;     // [B]
    const float *sinks;          // [Hq] or nullptr
    float scale_log2;            // scale * log2(e)
    void *out;                   // bf16 [B, Hq, D]
    float *lse;                  // [B, Hq] or nullptr
    int B, Hq, Hkv, G, num_pages, max_pages;
    int window;             // sliding window (keys at the last `window` positions); 0: none
    int total_warps;        // warps of the split-KV grid
    int max_sms_cap;        // SMs the sliding-window grid may use; 0: all
    uint64_t wait_limit_ns; // give-up time of a pipeline wait
    uint32_t *status;       // workspace header
    int32_t *ws_prefix;     // [B + 1] pages-per-sequence prefix sum (written by CTA 0)
    int64_t *ws_plan;       // [2]: total page units, page units per warp
    float *part_ml;         // [slots, G, 2] partial (max, sum), log2 domain
    float *part_acc;        // [slots, G, D] partial unnormalised outputs
    const float *k_scale;   // FP8 cache: [Hkv] per-KV-head scales, or nullptr (1)
    const float *v_scale;
    const void *k_new;      // decode with append: bf16 [B, Hkv, D] new rows, or nullptr
    const void *v_new;
    void *k_pages_w;        // the cache the new rows are written into (decode with append)
    void *v_pages_w;
    // Decode with append and rotary embedding (rope_on != 0): q and the new key are rotated
    // at the new token's position before use.  Per pair i < D/2 the YaRN-scaled frequency
    // theta_i as a float pair rope_hi[i] + rope_lo[i] (hi the nearest float, lo the rest),
    // and the magnitude factor rope_mscale applied to both outputs of a pair.
    int rope_on;
    float rope_mscale;
    float rope_hi[64];
    float rope_lo[64];
    bool start_early;  // split-KV kernel: a programmatic dependent of the kernel before it
};

// Grid and shared memory of the split-KV decode kernel for head_dim D and
// batch B on `device`.  Deterministic for a given (device, D, B).
cudaError_t decode_launch_shape(int D, int B, int G, int device, int *ctas, int *warps_per_cta,
                                int *smem_bytes, int *ring_bytes);
cudaError_t launch_decode_splitkv(int D, const DecodeArgs &a, const CUtensorMap &kmap,
                                  const CUtensorMap &vmap, int ctas, int smem_bytes,
                                  cudaStream_t stream);
cudaError_t launch_decode_merge(int D, const DecodeArgs &a, cudaStream_t stream);

// Sliding-window decode in one launch (no merge, no workspace partials): used by the decode
// entry points when decode_window_fits(window).
bool decode_window_fits(int window);
cudaError_t launch_decode_window(int D, const DecodeArgs &a, const CUtensorMap &kmap,
                                 const CUtensorMap &vmap, cudaStream_t stream);

// The same for the decode over an FP8 E4M3 cache (uint8 tensor maps, one box per page).
cudaError_t decode_fp8_launch_shape(int D, int G, int B, int device, int *ctas, int *warps_per_cta,
                                    int *smem_bytes);
cudaError_t launch_decode_fp8(int D, const DecodeArgs &a, const CUtensorMap &kmap,
                              const CUtensorMap &vmap, int ctas, int smem_bytes, cudaStream_t stream);

struct AppendArgs {
    const void *k, *v;  // bf16 [T, Hkv, D]
    const int32_t *cu_seqlens;
    const int32_t *block_table;
    const int32_t *start_pos;
    void *k_pages, *v_pages;  // bf16, or uint8 E4M3 codes when fp8
    int T, n, Hkv, D, num_pages, max_pages;
    uint32_t *status;
    bool fp8;                          // quantise to E4M3 codes
    const float *k_scale, *v_scale;    // fp8: [Hkv] per-KV-head scales, or nullptr (1)
};
cudaError_t launch_append_kv(const AppendArgs &a, cudaStream_t stream);

struct PrefillArgs {
    const int32_t *cu_seqlens;  // [n + 1]
    const int32_t *prefix_block_table;  // [n, max_pages] or nullptr
    const int32_t *prefix_lens;         // [n] or nullptr
    const void *k_pages, *v_pages;      // prefix pages (plain loads of ragged pages)
    const float *sinks;
    float scale_log2;
    void *out;   // bf16 [T, Hq, D]
    float *lse;  // [T, Hq] or nullptr
    int T, n, Hq, Hkv, G, D, num_pages, max_pages;
    int window;  // sliding window (keys at the query's last `window` positions); 0: none
    int max_sms;  // SMs the persistent grid may use; 0: all
    uint64_t wait_limit_ns;      // give-up time of a pipeline wait
    uint64_t wait_limit_cycles;  // the same in SM cycles (2 per ns)
    uint32_t *status;
    bool fp8_prefix;                   // the prefix pages are FP8 E4M3 codes (uint8)
    bool causal;                       // false: every query sees its whole request (no prefix, no window)
    bool launch_dependents;            // the next kernel on the stream may start at once
    uint32_t *sched;                   // [2] in the workspace header: next item, CTAs done (zero between calls)
    const float *k_scale, *v_scale;    // FP8 prefix: [Hkv] per-KV-head scales, or nullptr (1)
};
// Tensor maps: q [T, Hq, D], k/v [T, Hkv, D] (new tokens), kp/vp prefix pages.
cudaError_t launch_prefill(const PrefillArgs &a, const CUtensorMap &qmap, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, const CUtensorMap &kpmap,
                           const CUtensorMap &vpmap, cudaStream_t stream);

}  // namespace sinkattn
