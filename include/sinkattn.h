/*
 * sinkattn.h - C ABI of libsinkattn: paged grouped-query attention with per-head
 * attention sinks on GB300 (sm_103a).
 *
 * What is computed.  For query head h, its KV head g = h / (Hq / Hkv), a query
 * vector q and the keys J the query may see:
 *     s_j = scale * <q, k_j>
 *     m   = max(sink_h, max_j s_j)
 *     out = sum_j e^(s_j - m) v_j / (e^(sink_h - m) + sum_j e^(s_j - m))
 *     lse = m + ln(e^(sink_h - m) + sum_j e^(s_j - m))        (natural log)
 * The sink is a per-head learned logit that takes part in the softmax as a
 * virtual token with zero key and zero value ("GPT-OSS on Day 0", section "Sink
 * Attention"; TensorSharp docs/models/gptoss.md, section 3 "Forward graph" and
 * section 4.1 "Attention").  The sink is used as given (it is not multiplied by
 * `scale`).  sinks == NULL means every sink is -inf: plain GQA attention.
 * A query that sees no key and has no sink gets out = 0 and lse = -inf.
 *
 * KV cache layout (HND, "Hosting Qwen on Blackwell", KV-cache paragraph of the
 * "Prefill" part: heads leading, the tokens of a page contiguous):
 *     k_pages, v_pages: bf16 [num_pages, num_kv_heads, page_size, head_dim]
 *     token j of sequence b is slot j % page_size of page block_table[b][j / page_size]
 *     block_table: int32 [num_seqs, max_pages_per_seq], row-major
 *
 * Supported: bf16 data (and FP8 E4M3 KV caches for decode, append and the prefix of a
 * chunked prefill, see below),
 * fp32 sinks, head_dim 64 or 128, page_size 16, num_qo_heads / num_kv_heads in
 * {1, 2, 4, 8, 16}.
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers into memory the caller owns; the
 *     library never allocates or frees inside a compute call.  Scratch space
 *     comes from a caller-provided device workspace whose size is queried first.
 *     Pointers must be 16-byte aligned; tensors are dense and row-major.
 *   - Work is enqueued on `stream` (a cudaStream_t); calls return after enqueueing.
 *     Launch shapes depend only on host arguments and the device, never on device
 *     data, so the calls can be recorded into CUDA graphs.
 *   - The return value is a sinkattn_error code.  Invalid host arguments are
 *     rejected before anything is enqueued.  Nothing is printed; nothing traps.
 *   - Problems that only the device can see (a block-table entry outside
 *     [0, num_pages), a length beyond the block table, a malformed cu_seqlens)
 *     make the kernels skip the offending access and set a bit in a status word
 *     that lives in the workspace; read it with sinkattn_get_status.  Outputs of
 *     the affected rows are then unspecified (but no memory outside the given
 *     buffers is touched).
 *   - Empty work: a decode with num_seqs == 0, or a prefill or append with
 *     num_seqs == 0 or total_tokens == 0, returns SINKATTN_OK at once after the
 *     descriptor's shapes are checked; its data pointers may then be NULL.
 */
#ifndef SINKATTN_H
#define SINKATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *sinkattn_stream_t;

typedef enum sinkattn_error {
    SINKATTN_OK = 0,
    SINKATTN_ERR_INVALID_ARG = 1,         /* a NULL/misaligned pointer or inconsistent size */
    SINKATTN_ERR_UNSUPPORTED = 2,         /* valid but not implemented (dtype, head_dim, group) */
    SINKATTN_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes below the size query's answer */
    SINKATTN_ERR_CUDA = 4                 /* a CUDA runtime call failed */
} sinkattn_error;

/* Bits of the device status word (sinkattn_get_status). */
#define SINKATTN_STATUS_BAD_PAGE 0x1u       /* block-table entry outside [0, num_pages) */
#define SINKATTN_STATUS_BAD_LENGTH 0x2u     /* a length < 0 or > max_pages_per_seq * page_size */
#define SINKATTN_STATUS_BAD_CU_SEQLENS 0x4u /* cu_seqlens not non-decreasing from 0 to total */
#define SINKATTN_STATUS_WAIT_TIMEOUT 0x8u   /* a pipeline wait hit its iteration limit */
#define SINKATTN_STATUS_VALUE_RANGE 0x10u   /* prefill: a V value with |v| >= 2^22 or not finite */

/* Shapes of a paged KV cache and of the heads that read it. */
typedef struct sinkattn_paged_desc {
    int32_t num_seqs;          /* B: sequences (decode) or requests (prefill) */
    int32_t num_qo_heads;      /* Hq */
    int32_t num_kv_heads;      /* Hkv; Hq % Hkv == 0 */
    int32_t head_dim;          /* D: 64 or 128 */
    int32_t page_size;         /* P: 16 */
    int32_t num_pages;         /* pages in k_pages / v_pages (may be 0 for a prefill without prefix) */
    int32_t max_pages_per_seq; /* columns of the block table */
    int32_t window;            /* sliding window W (decode and prefill): a query at
                                * position pos sees only the keys at positions
                                * pos - W < j <= pos (gptoss.md section 4: a 128-token
                                * window on alternating layers, passed per call);
                                * 0 or negative: no window */
    int32_t max_sms;           /* SMs the persistent grids may use (split-KV decode and
                                * prefill): 0 = all of them; n > 0 = at most n, leaving the
                                * rest to kernels the caller runs at the same time on other
                                * streams (for example a decode batch beside a chunked
                                * prefill).  Negative: SINKATTN_ERR_INVALID_ARG.  No page
                                * has this: it is a scheduling control of this library.  It
                                * changes which warp does which part of a decode, so decode
                                * sums may round differently than with all SMs; prefill
                                * results do not depend on it.  The decode workspace size
                                * query takes it into account (a smaller grid needs fewer
                                * partial-state slots).  With 0, or a large value, the
                                * split-KV decode's grid still stops where its CTAs' copy
                                * rings hold about 18 MB of page reads in flight (about
                                * three quarters of GB300's SMs' worth of CTAs), where HBM
                                * measured fastest. */
    int32_t wait_limit_us;     /* watchdog of the kernels' pipeline waits (decode, FP8
                                * decode, prefill), in microseconds: a wait that has not
                                * completed after this long gives up, the kernel sets
                                * SINKATTN_STATUS_WAIT_TIMEOUT, lets the copies and MMAs
                                * it already issued finish, and returns (outputs are then
                                * unspecified).  0 = the default, 2 seconds; negative:
                                * SINKATTN_ERR_INVALID_ARG.  1 is the testing setting of
                                * that path: the decode kernels' waits then give up unless
                                * already complete when first tested (the first one never is:
                                * its copy from HBM is in flight), and the prefill gives up
                                * right after issuing its first copies. */
    int32_t flags;             /* 0, or an OR of the SINKATTN_FLAG_* bits below; other bits:
                                * SINKATTN_ERR_INVALID_ARG. */
} sinkattn_paged_desc;

/* Overlap of a prefill and the decode launched after it on the same stream (programmatic
 * dependent launch).  A prefill given SINKATTN_FLAG_LAUNCH_NEXT_EARLY lets the next kernel on
 * its stream start as soon as the prefill's own CTAs are running; a split-KV decode given
 * SINKATTN_FLAG_START_EARLY is launched so that it may start then (otherwise, or after any
 * other kernel, it starts when the kernel before it has completed).  With max_sms set so that
 * the two grids fit side by side (the prefill's S SMs, the decode's on the other SMs), the two
 * calls run at once on one stream, and the CTAs of each land on SMs of their own.  The decode
 * must read nothing the prefill writes (the prefill writes only its out and lse).  The merge
 * after the split-KV decode, and every later kernel on the stream, still wait for both.
 * The one-launch sliding-window decode and the FP8 decode ignore SINKATTN_FLAG_START_EARLY. */
#define SINKATTN_FLAG_LAUNCH_NEXT_EARLY 0x1
#define SINKATTN_FLAG_START_EARLY 0x2

/* Human-readable name of an error code (static string). */
const char *sinkattn_error_string(int code);

/* Library version as 10000 * major + 100 * minor + patch. */
int sinkattn_version(void);

/* Name of the CUDA runtime error behind the most recent SINKATTN_ERR_CUDA returned to
 * the calling host thread (static string; "no error" if there was none). */
const char *sinkattn_last_cuda_error(void);

/* ------------------------------------------------------------------ decode --
 * Split-KV decode ("GPT-OSS on Day 0", section "Sink Attention": the attention is
 * parallelised over heads and along the KV length, the partial softmax states are
 * combined, and the sink enters exactly once).  One query token per sequence; it
 * attends all seq_lens[b] cached tokens (the current token's K/V already appended).
 *
 * Workspace: query its size for a descriptor, then pass at least that many bytes,
 * 256-byte aligned.  The first 256 bytes are a header holding the status word; it
 * must be zero before the first call (sinkattn_workspace_init, or a memset).  The
 * size depends on the descriptor and on the number of SMs of the CURRENT device.
 * Calls that share one workspace must be ordered on the GPU (same stream, or
 * synchronised); overlapping calls on one workspace race.
 */
int sinkattn_decode_workspace_size(const sinkattn_paged_desc *desc, size_t *bytes);

/* Zero the workspace header (status word) on `stream`. */
int sinkattn_workspace_init(void *workspace, size_t ws_bytes, sinkattn_stream_t stream);

/*
 * q:           bf16 [B, Hq, D]
 * k_pages/v_pages: bf16 [num_pages, Hkv, 16, D]   (HND, see top of file)
 * block_table: int32 [B, max_pages_per_seq]; only the first ceil(seq_lens[b]/16)
 *              entries of row b are read
 * seq_lens:    int32 [B], each in [0, max_pages_per_seq * 16]
 * sinks:       fp32 [Hq] or NULL (= -inf, no sink)
 * scale:       multiplies q.k (typically 1/sqrt(D))
 * out:         bf16 [B, Hq, D]                       (written)
 * lse:         fp32 [B, Hq] natural-log normaliser including the sink, or NULL
 * workspace:   device scratch of ws_bytes (>= sinkattn_decode_workspace_size)
 *
 * Equivalent to sinkattn_decode_splitkv followed by sinkattn_decode_merge.  With a short
 * sliding window (0 < desc->window <= 2032: every (sequence, KV head) then sees at most
 * 128 pages) it runs a one-launch plan instead - one CTA per (sequence, KV head), its
 * warps splitting the visible pages, their partial states merged in shared memory, no
 * merge launch - whose results agree with the two-kernel plan within rounding (the sums
 * are split differently) and do not depend on the grid; sinkattn_decode_append and
 * sinkattn_decode_append_rope do the same.
 */
int sinkattn_decode(const void *q, const void *k_pages, const void *v_pages,
                    const int32_t *block_table, const int32_t *seq_lens, const float *sinks,
                    float scale, void *out, float *lse, const sinkattn_paged_desc *desc,
                    void *workspace, size_t ws_bytes, sinkattn_stream_t stream);

/* First kernel of sinkattn_decode: every page of every (sequence, KV head) is read
 * once; the work is cut into equal page ranges, one per warp of a persistent grid.
 * A (sequence, KV head) read entirely by one warp gets its final out/lse here (sink
 * folded in); the others leave sink-free partial states (m, l, acc) in the workspace.
 * Same arguments as sinkattn_decode. */
int sinkattn_decode_splitkv(const void *q, const void *k_pages, const void *v_pages,
                            const int32_t *block_table, const int32_t *seq_lens,
                            const float *sinks, float scale, void *out, float *lse,
                            const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                            sinkattn_stream_t stream);

/* Second kernel of sinkattn_decode: log-sum-exp merge of the partial states of each
 * split (sequence, KV head) with the sink term added once:
 *     M = max(sink, max_s m_s);  den = e^(sink - M) + sum_s l_s e^(m_s - M)
 *     out = sum_s acc_s e^(m_s - M) / den;  lse = M + ln den
 * Must follow sinkattn_decode_splitkv on the same workspace with the same
 * seq_lens, sinks and descriptor.  Also writes out = 0, lse = sink for empty
 * sequences. */
int sinkattn_decode_merge(const int32_t *seq_lens, const float *sinks, void *out, float *lse,
                          const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                          sinkattn_stream_t stream);

/* Decode step with its K/V append: each sequence's new token (the step's query token) is
 * written into the cache and then attended, in the order of TensorSharp
 * docs/models/gptoss.md, section 3 "Forward graph" (append K and V to the cache, then
 * attention over it), without a launch of its own: the warp that reads a sequence's last
 * page puts the new row into its copy of the page and into the cache.
 *
 * k_new, v_new: bf16 [B, Hkv, D], 16-byte aligned: row (b, g) is the new token of
 *              sequence b for KV head g
 * seq_lens:    as for sinkattn_decode, COUNTING the new token: it sits at position
 *              seq_lens[b] - 1, i.e. page block_table[b][(seq_lens[b] - 1) / 16], slot
 *              (seq_lens[b] - 1) % 16.  A sequence with seq_lens[b] = 0 has no new token
 *              (nothing is written; out = 0, lse = sink).
 * k_pages, v_pages: the cache; the new rows are written into it (each (page, KV head,
 *              slot) by exactly one thread; no other byte changes).  A block-table entry
 *              outside [0, num_pages) sets SINKATTN_STATUS_BAD_PAGE and writes nothing; so does
 *              a length beyond max_pages_per_seq * 16 (SINKATTN_STATUS_BAD_LENGTH).
 * Other arguments, workspace and errors as for sinkattn_decode (and the sliding window
 * and SM budget of the descriptor apply).  The result equals sinkattn_append_kv of the
 * same rows at start positions seq_lens - 1 followed by sinkattn_decode, bit for bit.
 * Sequences must not share the page their new token goes to.
 */
int sinkattn_decode_append(const void *q, const void *k_new, const void *v_new, void *k_pages,
                           void *v_pages, const int32_t *block_table, const int32_t *seq_lens,
                           const float *sinks, float scale, void *out, float *lse,
                           const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                           sinkattn_stream_t stream);

/* Rotary position embedding of gpt-oss: NeoX layout with YaRN frequency scaling
 * (TensorSharp docs/models/gptoss.md, section 3 "Forward graph": RoPE_NeoX with YaRN
 * scaling, original context 4096, freqScale = 1 / RopeScale, beta_fast 32, beta_slow 1;
 * "GPT-OSS on Day 0": YaRN position encoding as in DeepSeek-V3).  For head_dim D, pair i
 * (i < D/2) is elements i and i + D/2.  Its base frequency w_i = base^(-2i/D); with the
 * correction dims c(r) = D ln(original_context / (2 pi r)) / (2 ln base),
 * lo = max(0, floor(c(beta_fast))), hi = min(D - 1, ceil(c(beta_slow))) and the ramp
 * y_i = clamp((i - lo) / max(0.001, hi - lo), 0, 1), the pair turns at the rate
 * theta_i = (1 - y_i) w_i + y_i w_i / factor; at position p, with a = p theta_i,
 *     x'[i]       = mscale (x[i] cos a - x[i + D/2] sin a)
 *     x'[i + D/2] = mscale (x[i + D/2] cos a + x[i] sin a),    mscale = 1 + 0.1 ln(factor).
 * factor = 1 is plain NeoX RoPE. */
typedef struct sinkattn_rope_desc {
    double base;              /* frequency base (> 1), e.g. 150000 for gpt-oss */
    double factor;            /* YaRN scale factor (RopeScale) >= 1 */
    int32_t original_context; /* context length before scaling (> 0), 4096 for gpt-oss */
    double beta_fast;         /* > beta_slow > 0; 32 for gpt-oss */
    double beta_slow;         /* 1 for gpt-oss */
} sinkattn_rope_desc;

/* Decode step with rotary embedding and K/V append, in the order of gptoss.md section 3
 * (RoPE on Q and K, append K and V to the cache, attention): q [B, Hq, D] and k_new
 * [B, Hkv, D] arrive NOT rotated; both are rotated at the new token's position
 * seq_lens[b] - 1 and rounded to bf16, the rotated key and v_new are written to the cache
 * at that position, and the rotated query attends the seq_lens[b] cached tokens - all in
 * the launches of sinkattn_decode_append (no extra launch).  The rotation angles are
 * reduced in float arithmetic that carries each theta_i as two floats, so positions up to
 * 2^24 keep the angle within ~1e-6 rad; a rotated element can then differ from the bf16
 * rounding of the exact rotation by one bf16 step when it lies within ~1e-7 (relative) of
 * a rounding boundary.
 * rope: the rotation's parameters (host pointer, read during the call only); positions
 * (max_pages_per_seq * 16) must stay below 2^24 (else SINKATTN_ERR_UNSUPPORTED).
 * Other arguments, results and errors as for sinkattn_decode_append. */
int sinkattn_decode_append_rope(const void *q, const void *k_new, const void *v_new, void *k_pages,
                                void *v_pages, const int32_t *block_table, const int32_t *seq_lens,
                                const float *sinks, float scale, const sinkattn_rope_desc *rope,
                                void *out, float *lse, const sinkattn_paged_desc *desc,
                                void *workspace, size_t ws_bytes, sinkattn_stream_t stream);

/* -------------------------------------------------------- FP8 E4M3 KV cache --
 * A KV cache of one byte per element.  The pages name an FP8 serving precision
 * ("GPT-OSS on Day 0", section "GPT-OSS on Hopper") and an 8-bit KV-cache type
 * (TensorSharp gptoss.md section 10, "Memory and KV cache strategy") without a scale
 * convention; this library's convention:
 *   - each element is an OCP FP8 E4M3 code (sign, 4 exponent bits with bias 7,
 *     3 mantissa bits; no infinities; 0x7F / 0xFF are NaN; largest finite 448);
 *   - its value is scale[g] * e4m3(code), with one fp32 scale per KV head g, one
 *     array for K (k_scale) and one for V (v_scale), each fp32 [Hkv] on the device;
 *     NULL means every scale is 1.  Scales must be positive and finite.
 * Pages keep the HND layout: uint8 [num_pages, Hkv, 16, D].
 *
 * sinkattn_decode_fp8: the decode above over such a cache (same q, block_table,
 * seq_lens, sinks, scale, out, lse, descriptor, window and status behaviour).  The
 * product q.k is formed with q converted to fp16: |q| entries must be below 65504
 * (values below 2^-14 lose precision as fp16 subnormals).  The probabilities enter
 * the P.V product rounded to fp16 (relative error <= 2^-11 each), so an output's
 * absolute error is bounded by about 2^-11 * max |v| over its keys plus the bf16
 * rounding of the output; lse is not affected.  NaN codes in visible keys give
 * unspecified outputs.  The workspace is the
 * decode workspace (sinkattn_decode_workspace_size covers both caches), and
 * sinkattn_decode_merge completes sinkattn_decode_fp8_splitkv exactly as it
 * completes sinkattn_decode_splitkv.
 */
int sinkattn_decode_fp8(const void *q, const void *k_pages, const void *v_pages,
                        const float *k_scale, const float *v_scale, const int32_t *block_table,
                        const int32_t *seq_lens, const float *sinks, float scale, void *out,
                        float *lse, const sinkattn_paged_desc *desc, void *workspace,
                        size_t ws_bytes, sinkattn_stream_t stream);

/* First kernel of sinkattn_decode_fp8 (the split-KV pass; see sinkattn_decode_splitkv). */
int sinkattn_decode_fp8_splitkv(const void *q, const void *k_pages, const void *v_pages,
                                const float *k_scale, const float *v_scale,
                                const int32_t *block_table, const int32_t *seq_lens,
                                const float *sinks, float scale, void *out, float *lse,
                                const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                                sinkattn_stream_t stream);

/* sinkattn_append_kv into an FP8 cache: bf16 rows k, v [T, Hkv, D] are quantised,
 * element x of KV head g to the E4M3 code nearest to x / scale[g] (the division in
 * IEEE single precision; ties to the even code; finite values beyond 448 and
 * infinities saturate to +-448; NaN stays NaN), and written to the same slots
 * sinkattn_append_kv would write.  k_pages, v_pages: uint8 [num_pages, Hkv, 16, D]. */
int sinkattn_append_kv_fp8(const void *k, const void *v, const float *k_scale,
                           const float *v_scale, const int32_t *cu_seqlens, int32_t total_tokens,
                           const int32_t *block_table, const int32_t *start_pos, void *k_pages,
                           void *v_pages, const sinkattn_paged_desc *desc, void *workspace,
                           size_t ws_bytes, sinkattn_stream_t stream);

/* ------------------------------------------------------- decode, no allocation --
 * No counterpart on the source pages: an addition for callers that cannot allocate
 * device memory where they run attention - code whose device memory is owned by
 * another allocator, latency-critical paths that must not call cudaMalloc, or hosts
 * that forbid allocation after start-up.  It computes exactly what sinkattn_decode
 * computes, but its scratch is a fixed array inside the library instead of a
 * caller-provided workspace; the caller still passes every input and output.
 *
 * Limit: the scratch array holds SINKATTN_NOALLOC_SCRATCH_BYTES (32 MiB).  Shapes
 * whose sinkattn_decode_workspace_size exceeds it are rejected with
 * SINKATTN_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.  Every GPU that loads
 * the library holds the array until the process exits.
 *
 * The first call on a device looks up the array's device address (once per device,
 * with that device current).  With CUDA's lazy module loading (the default) that
 * lookup is also what loads the library's device code and so places the 32 MiB array
 * in device memory: the driver allocates it inside that first call.  Callers that must
 * not see any allocation after start-up therefore make one call at start-up (an empty
 * batch, num_seqs = 0, is enough), and that first call must come before any stream
 * capture.  Later calls allocate nothing and call no allocating routine.  Arguments
 * are checked before anything is enqueued; a rejected call leaves *status untouched.
 * All calls on a
 * device share the one array and it keeps the previous call's contents, so calls
 * that overlap on the GPU (different streams without ordering, or different host
 * threads) race; order them on one stream or synchronise.
 *
 * status: device pointer to one uint32, or NULL.  When given, it receives the
 * SINKATTN_STATUS_* bits of this call (overwritten, not OR-ed), in stream order.
 */
#define SINKATTN_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

int sinkattn_decode_noalloc(const void *q, const void *k_pages, const void *v_pages,
                            const int32_t *block_table, const int32_t *seq_lens,
                            const float *sinks, float scale, void *out, float *lse,
                            const sinkattn_paged_desc *desc, uint32_t *status,
                            sinkattn_stream_t stream);

/* ----------------------------------------------------------------- prefill --
 * Causal prefill over packed ragged sequences ("Fast embeddings on GPUs", section
 * on kernels: ragged inputs without padding, paged prefill), optionally after a
 * paged prefix (chunked prefill).  Query t of request i (0 <= t < new_len_i) sits at
 * absolute position prefix_len_i + t and attends every prefix token plus new tokens
 * 0..t of the same request (causal mask of gptoss.md section 3, aligned to the end).
 * QK^T and PV run on the tcgen05 tensor cores with TMEM accumulators; the online
 * softmax's running max and denominator start from the sink.  The P.V product takes
 * P and V in fp16 (11-bit significand, fp32 accumulation): each V tile is scaled by a
 * power of two into fp16 range, which covers |v| < 2^22; larger or non-finite values
 * set SINKATTN_STATUS_VALUE_RANGE (their outputs are then unspecified).
 *
 * q:          bf16 [T, Hq, D]   (T = total_tokens = cu_seqlens[num_seqs])
 * k, v:       bf16 [T, Hkv, D]  (the new tokens' keys and values)
 * cu_seqlens: int32 [num_seqs + 1], cu_seqlens[0] = 0, non-decreasing
 * k_pages, v_pages, prefix_block_table [num_seqs, max_pages_per_seq], prefix_lens
 *             [num_seqs]: the paged prefix; all four NULL for a plain causal prefill
 * sinks, scale, lse: as for decode, with lse [T, Hq]; scale must be positive and finite
 * out:        bf16 [T, Hq, D], 32-byte aligned (the other data pointers 16-byte aligned)
 * desc:       num_seqs, heads, head_dim, page_size; num_pages and max_pages_per_seq
 *             describe the prefix pages (ignored without a prefix)
 * workspace:  at least sinkattn_prefill_workspace_size bytes: the 256-byte header only,
 *             holding the status word and the counters the persistent grid takes its work
 *             items from.  Zero it once before the first call (sinkattn_workspace_init);
 *             every call leaves the counters at zero.  Calls that share one workspace must
 *             be ordered on the GPU (same stream, or synchronised).
 */
int sinkattn_prefill_workspace_size(const sinkattn_paged_desc *desc, size_t *bytes);

int sinkattn_prefill(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                     int32_t total_tokens, const void *k_pages, const void *v_pages,
                     const int32_t *prefix_block_table, const int32_t *prefix_lens,
                     const float *sinks, float scale, void *out, float *lse,
                     const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                     sinkattn_stream_t stream);

/* Non-causal prefill over packed ragged sequences, without a KV cache: the attention of an
 * embedding (encoder) model served through ragged kernels that instantiate no KV cache
 * ("Fast embeddings on GPUs", section on attention kernels).  The pages give no mask for it;
 * this is the plain bidirectional reading: query t of request i attends every token of
 * request i (cu_seqlens[i] <= j < cu_seqlens[i+1]), before and after it, and nothing else.
 * The same tcgen05 kernel as sinkattn_prefill, with the diagonal mask replaced by the
 * request's end; sinks, fp16 P.V and SINKATTN_STATUS_VALUE_RANGE as there.
 *
 * q, k, v, cu_seqlens, sinks, scale, out, lse: as for sinkattn_prefill (no prefix)
 * desc:       num_seqs, heads, head_dim, page_size; num_pages and max_pages_per_seq are
 *             ignored; window must be <= 0 (SINKATTN_ERR_INVALID_ARG otherwise)
 * workspace:  at least sinkattn_prefill_workspace_size bytes (status header only)
 * Errors as for sinkattn_prefill. */
int sinkattn_prefill_noncausal(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                               int32_t total_tokens, const float *sinks, float scale, void *out,
                               float *lse, const sinkattn_paged_desc *desc, void *workspace,
                               size_t ws_bytes, sinkattn_stream_t stream);

/* Chunked prefill over an FP8 E4M3 paged prefix: sinkattn_prefill with the prefix pages
 * in the FP8 cache convention above (uint8 codes [num_pages, Hkv, 16, D], value =
 * scale[g] * e4m3(code); k_scale / v_scale fp32 [Hkv] on the device, NULL = 1, positive
 * and finite).  The new tokens' k, v stay bf16 (a serving step appends them to the FP8 cache
 * with sinkattn_append_kv_fp8 for later steps).  The prefix tiles are copied as codes and
 * converted in shared memory: K exactly to bf16 code values, the K scale multiplying those
 * tiles' scores.  V: with v_scale = m * 2^e (m in [1, 2), -12 <= e <= 6, i.e. 2^-12 <= v_scale
 * < 128) to code * 2^e, exact in fp16, the softmax multiplying those keys' P by m; other scales
 * to fp16 of value * 2^-k, one k per KV head from the format's largest value (448 * v_scale <
 * 2^15 * 2^k; k > 7 sets SINKATTN_STATUS_VALUE_RANGE), relative rounding <= 2^-11.  NaN codes in
 * visible keys give unspecified outputs.  All four prefix
 * pointers and the prefix lengths are required; other arguments, workspace and errors as
 * for sinkattn_prefill. */
int sinkattn_prefill_fp8(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                         int32_t total_tokens, const void *k_pages, const void *v_pages,
                         const float *k_scale, const float *v_scale,
                         const int32_t *prefix_block_table, const int32_t *prefix_lens,
                         const float *sinks, float scale, void *out, float *lse,
                         const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                         sinkattn_stream_t stream);

/* ------------------------------------------------------------------ append --
 * Write new K/V rows into the paged cache (each layer stores its K and V there before its
 * attention, gptoss.md section 3).  Token t of request i (cu_seqlens[i] <= t <
 * cu_seqlens[i+1]) goes to position pos = start_pos[i] + t - cu_seqlens[i], i.e. slot
 * pos % 16 of page block_table[i][pos / 16], for every KV head.  A bit-exact copy.
 *
 * k, v:        bf16 [T, Hkv, D]
 * cu_seqlens:  int32 [num_seqs + 1]
 * block_table: int32 [num_seqs, max_pages_per_seq]
 * start_pos:   int32 [num_seqs], tokens already in each sequence's pages
 * k_pages, v_pages: bf16 [num_pages, Hkv, 16, D], updated in place
 * workspace:   optional (may be NULL): if given (>= 256 bytes), rows whose
 *              destination is out of range set status bits there; they are skipped
 *              either way.
 */
int sinkattn_append_kv(const void *k, const void *v, const int32_t *cu_seqlens,
                       int32_t total_tokens, const int32_t *block_table,
                       const int32_t *start_pos, void *k_pages, void *v_pages,
                       const sinkattn_paged_desc *desc, void *workspace, size_t ws_bytes,
                       sinkattn_stream_t stream);

/* ------------------------------------------------------------------ status --
 * Read the status word of a workspace and clear it (synchronous: waits for the work
 * already enqueued on `stream`).  *status_out gets an OR of SINKATTN_STATUS_* bits
 * accumulated since the last read; 0 means no device-side problem was seen. */
int sinkattn_get_status(void *workspace, uint32_t *status_out, sinkattn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SINKATTN_H */
