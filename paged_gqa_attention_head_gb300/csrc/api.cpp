// C ABI of libsinkattn (declared in include/sinkattn.h): argument checks,
// workspace layout, TMA tensor-map encoding and kernel launches.  No device
// memory is allocated here; scratch lives in the caller's workspace.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "../../include/sinkattn.h"
#include "internal.h"

using namespace sinkattn;

namespace {

constexpr size_t kAlign = 256;
// Page copies the bf16 split-KV grid keeps in flight at most (its CTAs' copy rings).
constexpr size_t kDecodeInflightBytes = size_t(18) << 20;

size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

thread_local cudaError_t g_last_cuda_error = cudaSuccess;
thread_local const char *g_last_cuda_where = "";
thread_local char g_last_cuda_text[160];

int cuda_rc(cudaError_t e, const char *where = "") {
    if (e == cudaSuccess) return SINKATTN_OK;
    g_last_cuda_error = e;
    g_last_cuda_where = where;
    return SINKATTN_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tensor of `rank` dims (innermost first); bf16 with 128-byte swizzled boxes unless
// told otherwise.
int encode_map(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
               const cuuint64_t *strides_bytes, const cuuint32_t *box,
               CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto enc = tensor_map_encoder();
    if (!enc) return SINKATTN_ERR_CUDA;
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(m, dtype, (cuuint32_t)rank, const_cast<void *>(base), dims, strides_bytes, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SINKATTN_OK : SINKATTN_ERR_INVALID_ARG;
}

// FP8 pages [num_pages, Hkv, 16, D] of uint8 codes: one box is a whole (page, head),
// 16 rows of D bytes, swizzled by 64 bytes (D = 64) or 128 bytes (D = 128).
// swizzled: the decode's layout (64-byte swizzle at D = 64, 128-byte at D = 128); else rows
// of D bytes one after the other (the prefill's staging of FP8 prefix pages).
int encode_pages_map_fp8(CUtensorMap *m, const void *pages, int num_pages, int Hkv, int D,
                         bool swizzled = true) {
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)kPageSize, (cuuint64_t)Hkv,
                                (cuuint64_t)(num_pages > 0 ? num_pages : 1)};
    const cuuint64_t strides[3] = {(cuuint64_t)D, (cuuint64_t)kPageSize * D,
                                   (cuuint64_t)Hkv * kPageSize * D};
    const cuuint32_t box[4] = {(cuuint32_t)D, (cuuint32_t)kPageSize, 1, 1};
    return encode_map(m, pages, 4, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                      !swizzled ? CU_TENSOR_MAP_SWIZZLE_NONE
                                : (D == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B));
}

// Pages [num_pages, Hkv, 16, D]: dims {D, 16, Hkv, num_pages}; a box is one
// (page, head) row block of 16 tokens x 64 elements.
int encode_pages_map(CUtensorMap *m, const void *pages, int num_pages, int Hkv, int D) {
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)kPageSize, (cuuint64_t)Hkv,
                                (cuuint64_t)(num_pages > 0 ? num_pages : 1)};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)kPageSize * D * 2,
                                   (cuuint64_t)Hkv * kPageSize * D * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)kPageSize, 1, 1};
    return encode_map(m, pages, 4, dims, strides, box);
}

// Rows [T, H, D]: dims {D, H, T}; a box is `rows` consecutive tokens of one head.
int encode_rows_map(CUtensorMap *m, const void *base, int T, int H, int D, int rows) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
    return encode_map(m, base, 3, dims, strides, box);
}

int check_heads(const sinkattn_paged_desc *d) {
    if (!d) return SINKATTN_ERR_INVALID_ARG;
    if (d->num_seqs < 0 || d->num_qo_heads <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 ||
        d->num_pages < 0 || d->max_pages_per_seq < 0 || d->max_sms < 0 || d->wait_limit_us < 0)
        return SINKATTN_ERR_INVALID_ARG;
    if (d->flags & ~(SINKATTN_FLAG_LAUNCH_NEXT_EARLY | SINKATTN_FLAG_START_EARLY)) return SINKATTN_ERR_INVALID_ARG;
    if (d->num_qo_heads % d->num_kv_heads) return SINKATTN_ERR_INVALID_ARG;
    const int G = d->num_qo_heads / d->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return SINKATTN_ERR_UNSUPPORTED;
    if (d->head_dim != 64 && d->head_dim != 128) return SINKATTN_ERR_UNSUPPORTED;
    if (d->page_size != kPageSize) return SINKATTN_ERR_UNSUPPORTED;
    return SINKATTN_OK;
}

int check_decode_desc(const sinkattn_paged_desc *d) {
    int rc = check_heads(d);
    if (rc) return rc;
    if (d->num_pages < 1 || d->max_pages_per_seq < 1) return SINKATTN_ERR_INVALID_ARG;
    // page-unit offsets are 32-bit inside the kernels
    if ((int64_t)d->num_seqs * d->max_pages_per_seq * d->num_kv_heads >= (int64_t)INT32_MAX)
        return SINKATTN_ERR_UNSUPPORTED;
    if ((int64_t)d->num_seqs * d->num_kv_heads >= (int64_t)INT32_MAX / 2) return SINKATTN_ERR_UNSUPPORTED;
    return SINKATTN_OK;
}

// One workspace layout serves both split-KV kernels (bf16 and FP8 cache): the
// partial-state slots are sized for the larger of their grids, so the merge reads
// the same offsets after either.
struct DecodeLayout {
    size_t prefix, plan, ml, acc, total;
    int ctas, warps_per_cta, smem, total_warps;     // bf16 cache kernel
    int ctas8, warps_per_cta8, smem8, total_warps8;  // FP8 cache kernel
};

int decode_layout(const sinkattn_paged_desc *d, DecodeLayout *L) {
    int device = 0;
    int rc = cuda_rc(cudaGetDevice(&device), "cudaGetDevice");
    if (rc) return rc;
    const int G = d->num_qo_heads / d->num_kv_heads;
    int ring = 0;  // bytes of page copies one bf16 split-KV CTA keeps in flight
    rc = cuda_rc(decode_launch_shape(d->head_dim, d->num_seqs, G, device, &L->ctas, &L->warps_per_cta,
                                     &L->smem, &ring),
                 "decode launch shape");
    if (rc) return rc;
    rc = cuda_rc(decode_fp8_launch_shape(d->head_dim, G, d->num_seqs, device, &L->ctas8,
                                         &L->warps_per_cta8, &L->smem8),
                 "fp8 decode launch shape");
    if (rc) return rc;
    // Both grids are (SMs x CTAs per SM); keep the CTAs per SM, on fewer SMs' worth of CTAs
    // where max_sms asks for it.  The bf16 split-KV grid also stops at kDecodeInflightBytes of
    // page copies in flight: with every SM at full occupancy its rings hold 25-29 MB, and HBM
    // delivered 2-5 % less than with ~18 MB (measured on GB300 for the long-context, Qwen3-shape
    // and gpt-oss decode batches: best at 104-120 SMs' worth of five 32 KB CTAs at head_dim 64,
    // 96 SMs' worth of three 64 KB CTAs at 128; the block scheduler still spreads the CTAs over
    // every SM).
    int sms = 0;
    rc = cuda_rc(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device),
                 "cudaDeviceGetAttribute");
    if (rc) return rc;
    if (sms > 0) {
        const int per_sm = L->ctas / sms, per_sm8 = L->ctas8 / sms;
        int use = sms, use8 = sms;
        if (d->max_sms > 0 && d->max_sms < sms) use = use8 = d->max_sms;
        L->ctas = per_sm * use;
        L->ctas8 = per_sm8 * use8;
        const int most = ring > 0 ? (int)(kDecodeInflightBytes / ring) : L->ctas;
        if (L->ctas > most) L->ctas = most;
    }
    L->total_warps = L->ctas * L->warps_per_cta;
    L->total_warps8 = L->ctas8 * L->warps_per_cta8;
    const int most = L->total_warps > L->total_warps8 ? L->total_warps : L->total_warps8;
    const size_t slots = (size_t)most + (size_t)d->num_seqs * d->num_kv_heads;
    size_t off = kStatusBytes;
    L->prefix = off;
    off += align_up(((size_t)d->num_seqs + 1) * 4);
    L->plan = off;
    off += kAlign;
    L->ml = off;
    off += align_up(slots * G * 2 * sizeof(float));
    L->acc = off;
    off += slots * G * d->head_dim * sizeof(float);
    L->total = align_up(off);
    return SINKATTN_OK;
}


struct DecodePrep {
    DecodeArgs args;
    DecodeLayout layout;
};

int prepare_decode(const void *q, const int32_t *block_table, const int32_t *seq_lens,
                   const float *sinks, float scale, void *out, float *lse,
                   const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                   DecodePrep *P) {
    int rc = check_decode_desc(desc);
    if (rc) return rc;
    if (!q || !block_table || !seq_lens || !out || !workspace) return SINKATTN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, kAlign) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4) || (sinks && !aligned(sinks, 4)) ||
        (lse && !aligned(lse, 4)))
        return SINKATTN_ERR_INVALID_ARG;
    rc = decode_layout(desc, &P->layout);
    if (rc) return rc;
    if (ws_bytes < P->layout.total) return SINKATTN_ERR_WORKSPACE_TOO_SMALL;
    DecodeArgs &a = P->args;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.q = q;
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.sinks = sinks;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.out = out;
    a.lse = lse;
    a.B = desc->num_seqs;
    a.Hq = desc->num_qo_heads;
    a.Hkv = desc->num_kv_heads;
    a.G = desc->num_qo_heads / desc->num_kv_heads;
    a.num_pages = desc->num_pages;
    a.max_pages = desc->max_pages_per_seq;
    a.window = desc->window > 0 ? desc->window : 0;
    a.total_warps = P->layout.total_warps;
    a.max_sms_cap = desc->max_sms;
    a.wait_limit_ns = wait_limit_ns(desc->wait_limit_us);
    a.status = reinterpret_cast<uint32_t *>(ws);
    a.ws_prefix = reinterpret_cast<int32_t *>(ws + P->layout.prefix);
    a.ws_plan = reinterpret_cast<int64_t *>(ws + P->layout.plan);
    a.part_ml = reinterpret_cast<float *>(ws + P->layout.ml);
    a.part_acc = reinterpret_cast<float *>(ws + P->layout.acc);
    a.k_scale = nullptr;
    a.v_scale = nullptr;
    a.k_new = nullptr;
    a.v_new = nullptr;
    a.k_pages_w = nullptr;
    a.v_pages_w = nullptr;
    a.rope_on = 0;
    a.start_early = (desc->flags & SINKATTN_FLAG_START_EARLY) != 0;
    a.rope_mscale = 1.f;
    return SINKATTN_OK;
}

// The YaRN-scaled frequency of every rotary pair (the formulas of sinkattn_rope_desc in
// include/sinkattn.h), in double on the host - they depend on the parameters only - and
// handed to the kernel as float pairs hi + lo.  Parameter checks first.
bool rope_ok(const sinkattn_rope_desc *r) {
    return r && r->base > 1.0 && r->base < INFINITY && r->factor >= 1.0 && r->factor < INFINITY &&
           r->original_context > 0 && r->beta_slow > 0.0 && r->beta_fast > r->beta_slow &&
           r->beta_fast < INFINITY;
}

int rope_table(const sinkattn_rope_desc *r, int D, DecodeArgs *a) {
    if (!rope_ok(r)) return SINKATTN_ERR_INVALID_ARG;
    if (D / 2 > 64) return SINKATTN_ERR_UNSUPPORTED;
    const double two_pi = 6.283185307179586476925286766559;
    const double lnb = log(r->base);
    double lo = floor(D * log(r->original_context / (two_pi * r->beta_fast)) / (2.0 * lnb));
    double hi = ceil(D * log(r->original_context / (two_pi * r->beta_slow)) / (2.0 * lnb));
    if (lo < 0.0) lo = 0.0;
    if (hi > D - 1) hi = D - 1;
    const double span = (hi - lo) > 0.001 ? (hi - lo) : 0.001;
    for (int i = 0; i < D / 2; ++i) {
        const double w = pow(r->base, -2.0 * i / D);
        double y = (i - lo) / span;
        y = y < 0.0 ? 0.0 : (y > 1.0 ? 1.0 : y);
        const double th = (1.0 - y) * w + y * (w / r->factor);
        a->rope_hi[i] = (float)th;
        a->rope_lo[i] = (float)(th - (double)a->rope_hi[i]);
    }
    a->rope_mscale = (float)(1.0 + 0.1 * log(r->factor));
    a->rope_on = 1;
    return SINKATTN_OK;
}

// A decode's launches once its arguments are prepared: the one-launch plan for a short
// sliding window, else the split-KV kernel and the merge.
int launch_decode_pair(const DecodePrep &P, const CUtensorMap &kmap, const CUtensorMap &vmap,
                       const sinkattn_paged_desc *desc, cudaStream_t stream, const char *what) {
    if (decode_window_fits(desc->window))
        return cuda_rc(launch_decode_window(desc->head_dim, P.args, kmap, vmap, stream), "sliding-window decode launch");
    int rc = cuda_rc(launch_decode_splitkv(desc->head_dim, P.args, kmap, vmap, P.layout.ctas, P.layout.smem, stream),
                     what);
    if (rc) return rc;
    return cuda_rc(launch_decode_merge(desc->head_dim, P.args, stream), "merge launch");
}

int append_common(const void *k, const void *v, const int32_t *cu_seqlens, int32_t total_tokens,
                  const int32_t *block_table, const int32_t *start_pos, void *k_pages,
                  void *v_pages, const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                  bool fp8, const float *k_scale, const float *v_scale, sinkattn_stream_t stream) {
    int rc = check_heads(desc);
    if (rc) return rc;
    if (total_tokens < 0) return SINKATTN_ERR_INVALID_ARG;
    if (desc->num_seqs == 0 || total_tokens == 0) return SINKATTN_OK;  // no tokens: a no-op
    if (!k || !v || !cu_seqlens || !block_table || !start_pos || !k_pages || !v_pages)
        return SINKATTN_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) ||
        !aligned(cu_seqlens, 4) || !aligned(block_table, 4) || !aligned(start_pos, 4) ||
        (k_scale && !aligned(k_scale, 4)) || (v_scale && !aligned(v_scale, 4)))
        return SINKATTN_ERR_INVALID_ARG;
    if (workspace && (ws_bytes < kStatusBytes || !aligned(workspace, kAlign)))
        return SINKATTN_ERR_INVALID_ARG;
    if (desc->num_pages < 1 || desc->max_pages_per_seq < 1) return SINKATTN_ERR_INVALID_ARG;
    if (desc->num_seqs == 0 || total_tokens == 0) return SINKATTN_OK;
    AppendArgs a;
    a.k = k;
    a.v = v;
    a.cu_seqlens = cu_seqlens;
    a.block_table = block_table;
    a.start_pos = start_pos;
    a.k_pages = k_pages;
    a.v_pages = v_pages;
    a.T = total_tokens;
    a.n = desc->num_seqs;
    a.Hkv = desc->num_kv_heads;
    a.D = desc->head_dim;
    a.num_pages = desc->num_pages;
    a.max_pages = desc->max_pages_per_seq;
    a.status = static_cast<uint32_t *>(workspace);
    a.fp8 = fp8;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    return cuda_rc(launch_append_kv(a, (cudaStream_t)stream), "append launch");
}

}  // namespace

void sinkattn::record_cuda_error(cudaError_t e, const char *where) { cuda_rc(e, where); }

extern "C" {

const char *sinkattn_last_cuda_error(void) {
    if (g_last_cuda_error == cudaSuccess) return "no error";
    snprintf(g_last_cuda_text, sizeof g_last_cuda_text, "%s in %s", cudaGetErrorName(g_last_cuda_error),
             g_last_cuda_where);
    return g_last_cuda_text;
}

const char *sinkattn_error_string(int code) {
    switch (code) {
        case SINKATTN_OK: return "ok";
        case SINKATTN_ERR_INVALID_ARG: return "invalid argument";
        case SINKATTN_ERR_UNSUPPORTED: return "unsupported configuration";
        case SINKATTN_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case SINKATTN_ERR_CUDA: return "CUDA runtime error";
        default: return "unknown error";
    }
}

int sinkattn_version(void) { return 10200; }

int sinkattn_decode_workspace_size(const sinkattn_paged_desc *desc, size_t *bytes) {
    if (!bytes) return SINKATTN_ERR_INVALID_ARG;
    int rc = check_decode_desc(desc);
    if (rc) return rc;
    DecodeLayout L;
    rc = decode_layout(desc, &L);
    if (rc) return rc;
    *bytes = L.total;
    return SINKATTN_OK;
}

int sinkattn_workspace_init(void *workspace, size_t ws_bytes, sinkattn_stream_t stream) {
    if (!workspace || ws_bytes < kStatusBytes || !aligned(workspace, kAlign))
        return SINKATTN_ERR_INVALID_ARG;
    return cuda_rc(cudaMemsetAsync(workspace, 0, kStatusBytes, (cudaStream_t)stream), "cudaMemsetAsync");
}

int sinkattn_decode_splitkv(const void *q, const void *k_pages, const void *v_pages,
                            const int32_t *block_table, const int32_t *seq_lens,
                            const float *sinks, float scale, void *out, float *lse,
                            const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                            sinkattn_stream_t stream) {
    // an empty batch is a no-op (its data pointers may be NULL)
    if (desc && desc->num_seqs == 0) return check_decode_desc(desc);
    DecodePrep P;
    int rc = prepare_decode(q, block_table, seq_lens, sinks, scale, out, lse, desc, workspace,
                            ws_bytes, &P);
    if (rc) return rc;
    if (!k_pages || !v_pages || !aligned(k_pages, 16) || !aligned(v_pages, 16))
        return SINKATTN_ERR_INVALID_ARG;
    if (desc->num_seqs == 0) return SINKATTN_OK;
    CUtensorMap kmap, vmap;
    rc = encode_pages_map(&kmap, k_pages, desc->num_pages, desc->num_kv_heads, desc->head_dim);
    if (rc) return rc;
    rc = encode_pages_map(&vmap, v_pages, desc->num_pages, desc->num_kv_heads, desc->head_dim);
    if (rc) return rc;
    return cuda_rc(launch_decode_splitkv(desc->head_dim, P.args, kmap, vmap, P.layout.ctas,
                                         P.layout.smem, (cudaStream_t)stream),
                   "split-KV decode launch");
}

int sinkattn_decode_merge(const int32_t *seq_lens, const float *sinks, void *out, float *lse,
                          const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                          sinkattn_stream_t stream) {
    if (desc && desc->num_seqs == 0) return check_decode_desc(desc);  // an empty batch
    DecodePrep P;
    // the merge reads the plan written by the split-KV kernel; q and the block
    // table are not used, so stand-in non-null pointers pass the checks
    int rc = prepare_decode(out, seq_lens, seq_lens, sinks, 1.f, out, lse, desc, workspace,
                            ws_bytes, &P);
    if (rc) return rc;
    if (desc->num_seqs == 0) return SINKATTN_OK;
    return cuda_rc(launch_decode_merge(desc->head_dim, P.args, (cudaStream_t)stream), "merge launch");
}

int sinkattn_decode(const void *q, const void *k_pages, const void *v_pages,
                    const int32_t *block_table, const int32_t *seq_lens, const float *sinks,
                    float scale, void *out, float *lse, const sinkattn_paged_desc *desc,
                    void *workspace, size_t ws_bytes, sinkattn_stream_t stream) {
    if (desc && desc->num_seqs > 0 && decode_window_fits(desc->window)) {
        // a short sliding window: the one-launch plan
        DecodePrep P;
        int rc = prepare_decode(q, block_table, seq_lens, sinks, scale, out, lse, desc, workspace,
                                ws_bytes, &P);
        if (rc) return rc;
        if (!k_pages || !v_pages || !aligned(k_pages, 16) || !aligned(v_pages, 16))
            return SINKATTN_ERR_INVALID_ARG;
        CUtensorMap kmap, vmap;
        rc = encode_pages_map(&kmap, k_pages, desc->num_pages, desc->num_kv_heads, desc->head_dim);
        if (rc) return rc;
        rc = encode_pages_map(&vmap, v_pages, desc->num_pages, desc->num_kv_heads, desc->head_dim);
        if (rc) return rc;
        return cuda_rc(launch_decode_window(desc->head_dim, P.args, kmap, vmap, (cudaStream_t)stream),
                       "sliding-window decode launch");
    }
    int rc = sinkattn_decode_splitkv(q, k_pages, v_pages, block_table, seq_lens, sinks, scale, out,
                                     lse, desc, workspace, ws_bytes, stream);
    if (rc) return rc;
    return sinkattn_decode_merge(seq_lens, sinks, out, lse, desc, workspace, ws_bytes, stream);
}

int sinkattn_decode_append(const void *q, const void *k_new, const void *v_new, void *k_pages,
                           void *v_pages, const int32_t *block_table, const int32_t *seq_lens,
                           const float *sinks, float scale, void *out, float *lse,
                           const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                           sinkattn_stream_t stream) {
    // an empty batch is a no-op (its data pointers may be NULL)
    if (desc && desc->num_seqs == 0) return check_decode_desc(desc);
    // the new rows and the cache: checked before anything touches the device
    if (!k_pages || !v_pages || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !k_new || !v_new ||
        !aligned(k_new, 16) || !aligned(v_new, 16))
        return SINKATTN_ERR_INVALID_ARG;
    DecodePrep P;
    int rc = prepare_decode(q, block_table, seq_lens, sinks, scale, out, lse, desc, workspace,
                            ws_bytes, &P);
    if (rc) return rc;
    CUtensorMap kmap, vmap;
    rc = encode_pages_map(&kmap, k_pages, desc->num_pages, desc->num_kv_heads, desc->head_dim);
    if (rc) return rc;
    rc = encode_pages_map(&vmap, v_pages, desc->num_pages, desc->num_kv_heads, desc->head_dim);
    if (rc) return rc;
    P.args.k_new = k_new;
    P.args.v_new = v_new;
    P.args.k_pages_w = k_pages;
    P.args.v_pages_w = v_pages;
    return launch_decode_pair(P, kmap, vmap, desc, (cudaStream_t)stream, "split-KV decode with append launch");
}

int sinkattn_decode_append_rope(const void *q, const void *k_new, const void *v_new, void *k_pages,
                                void *v_pages, const int32_t *block_table, const int32_t *seq_lens,
                                const float *sinks, float scale, const sinkattn_rope_desc *rope,
                                void *out, float *lse, const sinkattn_paged_desc *desc,
                                void *workspace, size_t ws_bytes, sinkattn_stream_t stream) {
    // an empty batch is a no-op (its data pointers may be NULL)
    if (desc && desc->num_seqs == 0) return check_decode_desc(desc);
    if (!k_pages || !v_pages || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !k_new || !v_new ||
        !aligned(k_new, 16) || !aligned(v_new, 16) || !rope_ok(rope))
        return SINKATTN_ERR_INVALID_ARG;
    DecodePrep P;
    int rc = prepare_decode(q, block_table, seq_lens, sinks, scale, out, lse, desc, workspace,
                            ws_bytes, &P);
    if (rc) return rc;
    // positions up to max_pages * 16 - 1 must be exact floats for the angle reduction
    if ((int64_t)desc->max_pages_per_seq * kPageSize > (int64_t)1 << 24) return SINKATTN_ERR_UNSUPPORTED;
    rc = rope_table(rope, desc->head_dim, &P.args);
    if (rc) return rc;
    CUtensorMap kmap, vmap;
    rc = encode_pages_map(&kmap, k_pages, desc->num_pages, desc->num_kv_heads, desc->head_dim);
    if (rc) return rc;
    rc = encode_pages_map(&vmap, v_pages, desc->num_pages, desc->num_kv_heads, desc->head_dim);
    if (rc) return rc;
    P.args.k_new = k_new;
    P.args.v_new = v_new;
    P.args.k_pages_w = k_pages;
    P.args.v_pages_w = v_pages;
    return launch_decode_pair(P, kmap, vmap, desc, (cudaStream_t)stream,
                              "split-KV decode with rotary embedding and append launch");
}

int sinkattn_decode_fp8_splitkv(const void *q, const void *k_pages, const void *v_pages,
                                const float *k_scale, const float *v_scale,
                                const int32_t *block_table, const int32_t *seq_lens,
                                const float *sinks, float scale, void *out, float *lse,
                                const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                                sinkattn_stream_t stream) {
    // an empty batch is a no-op (its data pointers may be NULL)
    if (desc && desc->num_seqs == 0) return check_decode_desc(desc);
    DecodePrep P;
    int rc = prepare_decode(q, block_table, seq_lens, sinks, scale, out, lse, desc, workspace,
                            ws_bytes, &P);
    if (rc) return rc;
    if (!k_pages || !v_pages || !aligned(k_pages, 16) || !aligned(v_pages, 16) ||
        (k_scale && !aligned(k_scale, 4)) || (v_scale && !aligned(v_scale, 4)))
        return SINKATTN_ERR_INVALID_ARG;
    if (desc->num_seqs == 0) return SINKATTN_OK;
    CUtensorMap kmap, vmap;
    rc = encode_pages_map_fp8(&kmap, k_pages, desc->num_pages, desc->num_kv_heads, desc->head_dim);
    if (rc) return rc;
    rc = encode_pages_map_fp8(&vmap, v_pages, desc->num_pages, desc->num_kv_heads, desc->head_dim);
    if (rc) return rc;
    P.args.k_scale = k_scale;
    P.args.v_scale = v_scale;
    P.args.total_warps = P.layout.total_warps8;
    return cuda_rc(launch_decode_fp8(desc->head_dim, P.args, kmap, vmap, P.layout.ctas8,
                                     P.layout.smem8, (cudaStream_t)stream),
                   "fp8 split-KV decode launch");
}

int sinkattn_decode_fp8(const void *q, const void *k_pages, const void *v_pages,
                        const float *k_scale, const float *v_scale, const int32_t *block_table,
                        const int32_t *seq_lens, const float *sinks, float scale, void *out,
                        float *lse, const sinkattn_paged_desc *desc, void *workspace,
                        size_t ws_bytes, sinkattn_stream_t stream) {
    int rc = sinkattn_decode_fp8_splitkv(q, k_pages, v_pages, k_scale, v_scale, block_table,
                                         seq_lens, sinks, scale, out, lse, desc, workspace,
                                         ws_bytes, stream);
    if (rc) return rc;
    return sinkattn_decode_merge(seq_lens, sinks, out, lse, desc, workspace, ws_bytes, stream);
}

int sinkattn_prefill_workspace_size(const sinkattn_paged_desc *desc, size_t *bytes) {
    if (!bytes) return SINKATTN_ERR_INVALID_ARG;
    int rc = check_heads(desc);
    if (rc) return rc;
    *bytes = kStatusBytes;
    return SINKATTN_OK;
}

namespace {
int prefill_common(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                   int32_t total_tokens, const void *k_pages, const void *v_pages,
                   const int32_t *prefix_block_table, const int32_t *prefix_lens, const float *sinks,
                   float scale, void *out, float *lse, const sinkattn_paged_desc *desc, void *workspace,
                   size_t ws_bytes, bool fp8, const float *k_scale, const float *v_scale,
                   bool causal, sinkattn_stream_t stream) {
    int rc = check_heads(desc);
    if (rc) return rc;
    if (!causal && desc->window > 0) return SINKATTN_ERR_INVALID_ARG;
    if (total_tokens < 0) return SINKATTN_ERR_INVALID_ARG;
    if (desc->num_seqs == 0 || total_tokens == 0) return SINKATTN_OK;  // no tokens: a no-op
    if (!(scale > 0.f) || !(scale < INFINITY)) return SINKATTN_ERR_INVALID_ARG;
    if (!q || !k || !v || !cu_seqlens || !out || !workspace) return SINKATTN_ERR_INVALID_ARG;
    if (ws_bytes < kStatusBytes) return SINKATTN_ERR_WORKSPACE_TOO_SMALL;
    // out: 32-byte stores of the output rows
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 32) ||
        !aligned(workspace, kAlign) || !aligned(cu_seqlens, 4) || (sinks && !aligned(sinks, 4)) ||
        (lse && !aligned(lse, 4)))
        return SINKATTN_ERR_INVALID_ARG;
    const bool has_prefix = k_pages || v_pages || prefix_block_table || prefix_lens;
    if (has_prefix) {
        if (!k_pages || !v_pages || !prefix_block_table || !prefix_lens) return SINKATTN_ERR_INVALID_ARG;
        if (!aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(prefix_block_table, 4) ||
            !aligned(prefix_lens, 4))
            return SINKATTN_ERR_INVALID_ARG;
        if (desc->num_pages < 1 || desc->max_pages_per_seq < 1) return SINKATTN_ERR_INVALID_ARG;
    }
    if (desc->num_seqs == 0 || total_tokens == 0) return SINKATTN_OK;
    const int D = desc->head_dim, Hq = desc->num_qo_heads, Hkv = desc->num_kv_heads;
    CUtensorMap qmap, kmap, vmap, kpmap, vpmap;
    if ((rc = encode_rows_map(&qmap, q, total_tokens, Hq, D, 128))) return rc;
    if ((rc = encode_rows_map(&kmap, k, total_tokens, Hkv, D, 128))) return rc;
    if ((rc = encode_rows_map(&vmap, v, total_tokens, Hkv, D, 128))) return rc;
    if (fp8 && !has_prefix) return SINKATTN_ERR_INVALID_ARG;
    if ((k_scale && !aligned(k_scale, 4)) || (v_scale && !aligned(v_scale, 4))) return SINKATTN_ERR_INVALID_ARG;
    if (has_prefix && fp8) {
        if ((rc = encode_pages_map_fp8(&kpmap, k_pages, desc->num_pages, Hkv, D, false))) return rc;
        if ((rc = encode_pages_map_fp8(&vpmap, v_pages, desc->num_pages, Hkv, D, false))) return rc;
    } else if (has_prefix) {
        if ((rc = encode_pages_map(&kpmap, k_pages, desc->num_pages, Hkv, D))) return rc;
        if ((rc = encode_pages_map(&vpmap, v_pages, desc->num_pages, Hkv, D))) return rc;
    } else {
        kpmap = kmap;  // unused
        vpmap = vmap;
    }
    PrefillArgs a;
    a.cu_seqlens = cu_seqlens;
    a.prefix_block_table = has_prefix ? prefix_block_table : nullptr;
    a.prefix_lens = has_prefix ? prefix_lens : nullptr;
    a.k_pages = has_prefix ? k_pages : nullptr;
    a.v_pages = has_prefix ? v_pages : nullptr;
    a.sinks = sinks;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.out = out;
    a.lse = lse;
    a.T = total_tokens;
    a.n = desc->num_seqs;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.D = D;
    a.num_pages = has_prefix ? desc->num_pages : 0;
    a.max_pages = has_prefix ? desc->max_pages_per_seq : 0;
    a.window = desc->window > 0 ? desc->window : 0;
    a.max_sms = desc->max_sms;
    a.wait_limit_ns = wait_limit_ns(desc->wait_limit_us);
    a.wait_limit_cycles = a.wait_limit_ns * 2;  // SM cycles, at least the limit up to 2 GHz
    a.status = static_cast<uint32_t *>(workspace);
    a.fp8_prefix = fp8;
    a.causal = causal;
    a.launch_dependents = (desc->flags & SINKATTN_FLAG_LAUNCH_NEXT_EARLY) != 0;
    a.sched = static_cast<uint32_t *>(workspace) + 16;  // header bytes 64..71
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    cudaError_t e = launch_prefill(a, qmap, kmap, vmap, kpmap, vpmap, (cudaStream_t)stream);
    if (e == cudaErrorNotSupported) return SINKATTN_ERR_UNSUPPORTED;
    return cuda_rc(e, "prefill launch");
}
}  // namespace

int sinkattn_prefill(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                     int32_t total_tokens, const void *k_pages, const void *v_pages,
                     const int32_t *prefix_block_table, const int32_t *prefix_lens,
                     const float *sinks, float scale, void *out, float *lse,
                     const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                     sinkattn_stream_t stream) {
    return prefill_common(q, k, v, cu_seqlens, total_tokens, k_pages, v_pages, prefix_block_table,
                          prefix_lens, sinks, scale, out, lse, desc, workspace, ws_bytes, false, nullptr,
                          nullptr, true, stream);
}

int sinkattn_prefill_noncausal(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                               int32_t total_tokens, const float *sinks, float scale, void *out,
                               float *lse, const sinkattn_paged_desc *desc, void *workspace,
                               size_t ws_bytes, sinkattn_stream_t stream) {
    return prefill_common(q, k, v, cu_seqlens, total_tokens, nullptr, nullptr, nullptr, nullptr, sinks,
                          scale, out, lse, desc, workspace, ws_bytes, false, nullptr, nullptr, false,
                          stream);
}

int sinkattn_prefill_fp8(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                         int32_t total_tokens, const void *k_pages, const void *v_pages,
                         const float *k_scale, const float *v_scale,
                         const int32_t *prefix_block_table, const int32_t *prefix_lens,
                         const float *sinks, float scale, void *out, float *lse,
                         const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                         sinkattn_stream_t stream) {
    return prefill_common(q, k, v, cu_seqlens, total_tokens, k_pages, v_pages, prefix_block_table,
                          prefix_lens, sinks, scale, out, lse, desc, workspace, ws_bytes, true, k_scale,
                          v_scale, true, stream);
}

int sinkattn_append_kv(const void *k, const void *v, const int32_t *cu_seqlens,
                       int32_t total_tokens, const int32_t *block_table,
                       const int32_t *start_pos, void *k_pages, void *v_pages,
                       const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                       sinkattn_stream_t stream) {
    return append_common(k, v, cu_seqlens, total_tokens, block_table, start_pos, k_pages, v_pages,
                         desc, workspace, ws_bytes, false, nullptr, nullptr, stream);
}

int sinkattn_append_kv_fp8(const void *k, const void *v, const float *k_scale,
                           const float *v_scale, const int32_t *cu_seqlens, int32_t total_tokens,
                           const int32_t *block_table, const int32_t *start_pos, void *k_pages,
                           void *v_pages, const sinkattn_paged_desc *desc, void *workspace,
                           size_t ws_bytes, sinkattn_stream_t stream) {
    return append_common(k, v, cu_seqlens, total_tokens, block_table, start_pos, k_pages, v_pages,
                         desc, workspace, ws_bytes, true, k_scale, v_scale, stream);
}

int sinkattn_get_status(void *workspace, uint32_t *status_out, sinkattn_stream_t stream) {
    if (!workspace || !status_out || !aligned(workspace, kAlign)) return SINKATTN_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t v = 0;
    int rc = cuda_rc(cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s), "status read");
    if (!rc) rc = cuda_rc(cudaMemsetAsync(workspace, 0, sizeof v, s), "status clear");
    if (!rc) rc = cuda_rc(cudaStreamSynchronize(s), "cudaStreamSynchronize");
    if (rc) return rc;
    *status_out = v;
    return SINKATTN_OK;
}

}  // extern "C"
