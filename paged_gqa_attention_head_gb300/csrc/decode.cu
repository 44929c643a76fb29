// Split-KV paged decode with per-head sinks, and the log-sum-exp merge.
//
// Method ("GPT-OSS on Day 0", section "Sink Attention"): the attention of one
// query token is parallelised over heads and along the KV length; each piece
// keeps an online-softmax state (running max m, running sum l, unnormalised
// output acc) and the pieces are combined afterwards; the sink logit is counted
// exactly once.  KV pages are HND ("Hosting Qwen on Blackwell", KV-cache
// layout): one (page, KV head) is 16 contiguous rows of head_dim bf16.
//
// GB300 design.  Decode reads every KV byte once and does ~8-16 flop per byte,
// so it is bound by HBM bandwidth.  The work is the list of all (sequence,
// KV head, page) units in order; a persistent grid cuts that list into equal
// contiguous ranges, one per warp, so every warp moves the same number of bytes
// whatever the length mix.  Each warp streams its pages through a private ring
// of shared-memory stages filled by TMA (4-D tensor maps over the page pool,
// 128-byte swizzle; the grid is as many 4-warp CTAs as fit on every SM), and
// computes all G query heads of the KV head with
// m16n8k16 tensor-core MMAs (heads on the M axis, 16 tokens of a page on N).
// A (sequence, KV head) that one warp covers entirely is finished in place with
// the sink folded in; otherwise the warp leaves a sink-free partial state and
// the merge kernel combines the pieces and adds the sink.
//
// Decode with append (the step's new K/V row of each sequence is first written to
// the cache, then attended; TensorSharp docs/models/gptoss.md, section 3 "Forward
// graph"): exactly one warp reads the last page of each (sequence, KV head).  Once
// that page's copy has landed, the warp writes the new row, taken from the inputs,
// over its slot in the shared-memory stage (the copy read the slot before the row
// existed) and into the cache, so the append needs no launch of its own.
//
// Decode with append and rotary embedding (TensorSharp gptoss.md, section 3: Q and K go
// through RoPE_NeoX with YaRN scaling, then K/V are appended, then attention): the warp
// that starts a (sequence, KV head) segment rotates the G query rows it loads into its
// MMA registers, and the warp that appends the new key rotates it before writing it, both
// at the new token's position L - 1.  Pair i (elements i and i + D/2) turns by the angle
// p * theta_i, reduced modulo 2 pi in float arithmetic that carries theta_i as a float
// pair (see rope_cs), and both outputs are scaled by the YaRN magnitude; the rotated
// values are rounded to bf16 like any query or cached key.
#include <float.h>

#include <mutex>
#include <vector>

#include "decode_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace sinkattn {

namespace {

template <int D>
struct DecodeCfg {
    static constexpr int kWarps = 4;
    static constexpr int kThreads = kWarps * 32;
    // Ring depth per warp.  An SM keeps ~192 KB of pages in flight either way; shallow
    // rings let more warps share it (D=64: 3 x 4 KB per warp, four 4-warp CTAs per SM;
    // D=128: 2 x 8 KB, three CTAs, bounded by registers), and the per-warp work on a page
    // (ldmatrix, MMAs, softmax), not HBM, is what more warps hide: measured 6 -> 3 stages
    // at D=64 raised a 256-sequence long-context batch from 6.04 to 6.57 TB/s.
    static constexpr int kStages = D == 64 ? 3 : 2;
    static constexpr int kHalves = D / 64;               // 128-byte column blocks per row
    static constexpr int kPageBytes = kPageSize * D * 2;  // one (page, head) of K or of V
    static constexpr int kStageBytes = 2 * kPageBytes;
    static constexpr int kWarpBytes = kStages * kStageBytes;
    static constexpr int kKSteps = D / 16;
    static constexpr int kNTiles = D / 8;
};

template <int D>
int decode_smem_bytes(int B) {
    using C = DecodeCfg<D>;
    return 1024 /* alignment slack */ + C::kWarps * C::kWarpBytes +
           C::kWarps * C::kStages * (8 + 4 + 4 + 4) + (3 * B + 1) * 4;
}

// 2 pi as three floats for Cody and Waite's reduction: the first has 8 significant bits
// (201 / 32), the second is the float nearest to the rest, the third the float nearest to
// what remains after that.
constexpr float kTwoPi1 = 6.28125f;
constexpr float kTwoPi2 = 1.9353071693331003e-3f;
constexpr float kTwoPi3 = 1.0253376273028358e-11f;
constexpr float kInvTwoPi = 0.15915493667125702f;

// (cos, sin) of the angle p * (hi + lo), both times ms.  p is an integer position below
// 2^24 (exact in float).  The product is split exactly, p * hi = a_hi + a_err (one FMA),
// so the angle is a_hi + a_lo with a_lo = p * lo + a_err; the whole turns k = rint(a / 2 pi)
// come off in three FMAs against the three parts of 2 pi (k * kTwoPi1 is exact, and so is
// the first difference), which keeps the reduced angle within ~1e-6 rad of the exact one,
// where a float product p * theta alone would be off by up to ~1e-2 rad at p = 131072.
__device__ __forceinline__ float2 rope_cs(float p, float hi, float lo, float ms) {
    const float a_hi = p * hi;
    const float a_err = fmaf(p, hi, -a_hi);
    const float a_lo = fmaf(p, lo, a_err);
    const float k = rintf(a_hi * kInvTwoPi);
    float r = fmaf(-k, kTwoPi1, a_hi);
    r = fmaf(-k, kTwoPi2, r);
    r = fmaf(-k, kTwoPi3, r);
    r += a_lo;
    float s, c;
    sincosf(r, &s, &c);
    return make_float2(c * ms, s * ms);
}

// Rotate one pair of packed bf16 pairs: lo_w holds elements (i, i + 1), hi_w elements
// (i + D/2, i + 1 + D/2); cs0 / cs1 are the (cos, sin) of pairs i and i + 1.
__device__ __forceinline__ void rope_pairs(uint32_t &lo_w, uint32_t &hi_w, float2 cs0, float2 cs1) {
    const float l0 = __uint_as_float(lo_w << 16), l1 = __uint_as_float(lo_w & 0xFFFF0000u);
    const float h0 = __uint_as_float(hi_w << 16), h1 = __uint_as_float(hi_w & 0xFFFF0000u);
    lo_w = pack_bf16x2(fmaf(l0, cs0.x, -(h0 * cs0.y)), fmaf(l1, cs1.x, -(h1 * cs1.y)));
    hi_w = pack_bf16x2(fmaf(h0, cs0.x, l0 * cs0.y), fmaf(h1, cs1.x, l1 * cs1.y));
}


// ---------------------------------------------------------------- per-warp page work
// Shared by the split-KV kernel and the sliding-window kernel.  A warp holds the G query
// rows of one (sequence, KV head) as m16n8k16 A fragments (rows = heads, padded to 16),
// and an online-softmax state: running max m0 / m1 and per-lane partial sums l0 / l1 of
// rows gr and gr + 8 (log2 domain), unnormalised output acc (rows gr, gr + 8; columns
// n * 8 + tc, tc + 1).

// Rows nv..15 of a V stage past the sequence end (or of a skipped page) may hold
// anything, even NaN; P is 0 there but 0 * NaN is not 0, so clear them.
template <int D>
__device__ __forceinline__ void clear_v_tail(uint8_t *vb, int nv, int lane) {
    using C = DecodeCfg<D>;
    const int nrow = kPageSize - nv, per_half = nrow * 8;
    for (int i = lane; i < per_half * C::kHalves; i += 32) {
        const int h = i / per_half, j = i % per_half;
        *reinterpret_cast<uint4 *>(vb + h * 2048 + (nv + j / 8) * 128 + (j % 8) * 16) = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
}

// Decode with append: the new K/V row of (b, g) - the token at position L - 1, slot
// (L - 1) % 16 of physical page pg - taken from the inputs (the key rotated first with
// kRope), written over its slot in the stage (the copy read the slot before the row
// existed) and into the cache.  Warp-uniform; every lane calls it.
template <int D, bool kRope>
__device__ __forceinline__ void append_row(const DecodeArgs &a, int b, int g, int L, int pg, uint8_t *kb,
                                           uint8_t *vb, int lane) {
    constexpr int kChunks = D / 8;  // 16-byte chunks of one row
    const int slot = (L - 1) % kPageSize;
    const bool isv = lane >= kChunks;
    const int ck = lane % kChunks;
    const int64_t row = ((int64_t)b * a.Hkv + g) * D + ck * 8;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (lane < 2 * kChunks)
        w = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(isv ? a.v_new : a.k_new) + row);
    if (kRope) {
        // NeoX pairs: chunk ck (elements 8ck .. 8ck + 7) with chunk ck ^ (kChunks / 2)
        uint4 o;
        o.x = __shfl_xor_sync(0xffffffffu, w.x, kChunks / 2);
        o.y = __shfl_xor_sync(0xffffffffu, w.y, kChunks / 2);
        o.z = __shfl_xor_sync(0xffffffffu, w.z, kChunks / 2);
        o.w = __shfl_xor_sync(0xffffffffu, w.w, kChunks / 2);
        if (lane < kChunks) {
            const bool upper = ck >= kChunks / 2;  // this lane holds elements >= D/2
            const int i0 = (ck % (kChunks / 2)) * 8;
            const float p = (float)(L - 1);
            uint32_t *ow = reinterpret_cast<uint32_t *>(&w);
            const uint32_t *pw = reinterpret_cast<const uint32_t *>(&o);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 cs0 = rope_cs(p, a.rope_hi[i0 + 2 * e], a.rope_lo[i0 + 2 * e], a.rope_mscale);
                const float2 cs1 = rope_cs(p, a.rope_hi[i0 + 2 * e + 1], a.rope_lo[i0 + 2 * e + 1], a.rope_mscale);
                uint32_t lo_w = upper ? pw[e] : ow[e], hi_w = upper ? ow[e] : pw[e];
                rope_pairs(lo_w, hi_w, cs0, cs1);
                ow[e] = upper ? hi_w : lo_w;
            }
        }
    }
    if (lane < 2 * kChunks) {
        *reinterpret_cast<uint4 *>((isv ? vb : kb) + (ck >> 3) * 2048 + sw128(slot, ck & 7)) = w;
        const int64_t dst = (((int64_t)pg * a.Hkv + g) * kPageSize + slot) * D + ck * 8;
        *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(isv ? a.v_pages_w : a.k_pages_w) + dst) = w;
    }
    __syncwarp();
}

// The G query rows of (b, g) as A fragments; with kRope rotated at position L - 1.
template <int D, bool kRope>
__device__ __forceinline__ void load_q(const DecodeArgs &a, int b, int g, int L, uint32_t (&qa)[D / 16][4],
                                       int lane) {
    constexpr int kK = D / 16;
    const int gr = lane >> 2, tc = (lane & 3) * 2;
    const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(a.q) + ((int64_t)b * a.Hq + (int64_t)g * a.G) * D;
#pragma unroll
    for (int kk = 0; kk < kK; ++kk) {
        const int col = kk * 16 + tc;
        const bool r0 = gr < a.G, r1 = gr + 8 < a.G;
        qa[kk][0] = r0 ? *reinterpret_cast<const uint32_t *>(qg + gr * D + col) : 0u;
        qa[kk][1] = r1 ? *reinterpret_cast<const uint32_t *>(qg + (gr + 8) * D + col) : 0u;
        qa[kk][2] = r0 ? *reinterpret_cast<const uint32_t *>(qg + gr * D + col + 8) : 0u;
        qa[kk][3] = r1 ? *reinterpret_cast<const uint32_t *>(qg + (gr + 8) * D + col + 8) : 0u;
    }
    if (kRope) {
        // the query rows turn at the new token's position: column c < D/2 (register step
        // kk) pairs with column c + D/2 (step kk + kK / 2)
        const float p = (float)(L > 0 ? L - 1 : 0);
#pragma unroll
        for (int kk = 0; kk < kK / 2; ++kk)
#pragma unroll
            for (int x = 0; x < 2; ++x) {  // columns col, col + 1 (x = 0) or col + 8, col + 9
                const int i0 = kk * 16 + tc + x * 8;
                const float2 cs0 = rope_cs(p, a.rope_hi[i0], a.rope_lo[i0], a.rope_mscale);
                const float2 cs1 = rope_cs(p, a.rope_hi[i0 + 1], a.rope_lo[i0 + 1], a.rope_mscale);
                rope_pairs(qa[kk][2 * x], qa[kk + kK / 2][2 * x], cs0, cs1);          // row gr
                rope_pairs(qa[kk][2 * x + 1], qa[kk + kK / 2][2 * x + 1], cs0, cs1);  // row gr + 8
            }
    }
}

// One page: S = Q K^T for its 16 tokens (keys klo .. nv - 1 visible), the online-softmax
// update and O += P V.
template <int D, bool kWindow>
__device__ __forceinline__ void page_step(const DecodeArgs &a, const uint8_t *kb, const uint8_t *vb, int nv,
                                          int klo, const uint32_t (&qa)[D / 16][4], float (&acc)[D / 8][4],
                                          float &m0, float &m1, float &l0, float &l1, int lane) {
    constexpr int kK = D / 16, kN = D / 8;
    const int tc = (lane & 3) * 2;
    const int lm = lane >> 3, lr = lane & 7;  // ldmatrix: matrix index, row within it
    // S = Q K^T for the 16 tokens of this page (two n-tiles of 8 tokens)
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const uint32_t kbase = smem_u32(kb);
#pragma unroll
    for (int kk = 0; kk < kK; ++kk) {
        const int tok = (lm >> 1) * 8 + lr, chunk = kk * 2 + (lm & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + (chunk >> 3) * 2048 + sw128(tok, chunk & 7), b0, b1, b2, b3);
        mma_16816(s[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
        mma_16816(s[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
    }
#pragma unroll
    for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int tok = n * 8 + tc + (i & 1);
            s[n][i] = (tok < nv && (!kWindow || tok >= klo)) ? s[n][i] * a.scale_log2 : -INFINITY;
        }
    const float mx0 = quad_max(fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1])));
    const float mx1 = quad_max(fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3])));
    // the running max is raised only when a score passes it by more than 8 (log2 units), so
    // P = exp2(s - m) <= 2^8 and most pages leave the accumulators as they are
    if (__any_sync(0xffffffffu, mx0 > m0 + 8.f || mx1 > m1 + 8.f)) {
        const float mn0 = mx0 > m0 + 8.f ? mx0 : m0, mn1 = mx1 > m1 + 8.f ? mx1 : m1;
        const float al0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - mn0);
        const float al1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int n = 0; n < kN; ++n) {
            acc[n][0] *= al0;
            acc[n][1] *= al0;
            acc[n][2] *= al1;
            acc[n][3] *= al1;
        }
        l0 *= al0;
        l1 *= al1;
    }
    const float base0 = m0 == -INFINITY ? 0.f : m0, base1 = m1 == -INFINITY ? 0.f : m1;
    float p[2][4];
#pragma unroll
    for (int n = 0; n < 2; ++n) {
        p[n][0] = fast_exp2(s[n][0] - base0);
        p[n][1] = fast_exp2(s[n][1] - base0);
        p[n][2] = fast_exp2(s[n][2] - base1);
        p[n][3] = fast_exp2(s[n][3] - base1);
    }
    l0 += (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
    l1 += (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
    // P = P_hi + P_lo, both bf16: the rounding of P to bf16 alone (relative 2^-9)
    // is too coarse for short sequences, the pair keeps ~16 bits
    uint32_t ph[4], pl[4];
    {
        const float pv[4][2] = {{p[0][0], p[0][1]}, {p[0][2], p[0][3]}, {p[1][0], p[1][1]}, {p[1][2], p[1][3]}};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            ph[e] = pack_bf16x2(pv[e][0], pv[e][1]);
            pl[e] = pack_bf16x2(pv[e][0] - __uint_as_float(ph[e] << 16), pv[e][1] - __uint_as_float(ph[e] & 0xFFFF0000u));
        }
    }
    // O += P V: V rows are tokens (the k axis), columns head_dim (n axis)
    const uint32_t vbase = smem_u32(vb);
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
        const int tok = (lm & 1) * 8 + lr, chunk = c * 2 + (lm >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + (chunk >> 3) * 2048 + sw128(tok, chunk & 7), b0, b1, b2, b3);
        mma_16816(acc[2 * c], ph[0], ph[1], ph[2], ph[3], b0, b1);
        mma_16816(acc[2 * c + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
        mma_16816(acc[2 * c], pl[0], pl[1], pl[2], pl[3], b0, b1);
        mma_16816(acc[2 * c + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
    }
}

// The final out / lse rows of (b, g) from a state that covers every visible key: the sink
// joins the max and the denominator.  L0 / L1 are the row sums (quad-reduced).
template <int D>
__device__ __forceinline__ void finish_rows(const DecodeArgs &a, int b, int g, const float (&acc)[D / 8][4],
                                            float m0, float m1, float L0, float L1, int lane) {
    const int gr = lane >> 2, tc = (lane & 3) * 2;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int r = gr + half * 8;
        if (r < a.G) {
            const int h = g * a.G + r;
            const float m = half ? m1 : m0, l = half ? L1 : L0;
            const float sk = a.sinks ? a.sinks[h] * kLog2e : -INFINITY;
            const float M = fmaxf(m, sk);
            float scl = 0.f, lse2 = -INFINITY;
            if (M != -INFINITY) {
                const float wm = m == -INFINITY ? 0.f : exp2f(m - M);
                const float den = l * wm + (sk == -INFINITY ? 0.f : exp2f(sk - M));
                scl = wm / den;
                lse2 = M + log2f(den);
            }
            __nv_bfloat16 *og = reinterpret_cast<__nv_bfloat16 *>(a.out) + ((int64_t)b * a.Hq + h) * D;
#pragma unroll
            for (int n = 0; n < D / 8; ++n)
                *reinterpret_cast<uint32_t *>(og + n * 8 + tc) =
                    pack_bf16x2(acc[n][2 * half] * scl, acc[n][2 * half + 1] * scl);
            if (a.lse && (lane & 3) == 0) a.lse[(int64_t)b * a.Hq + h] = lse2 * kLn2;
        }
    }
}

// kWindow: a sliding window is given (a.window > 0); the kernel without it carries no
// window arithmetic.  kAppend: the new K/V rows a.k_new / a.v_new are appended (see above).
// kRope (with kAppend): q and the new key are rotated first (see above).
template <int D, bool kWindow, bool kAppend = false, bool kRope = false>
__global__ void __launch_bounds__(DecodeCfg<D>::kThreads)
    decode_splitkv_kernel(const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap, const __grid_constant__ DecodeArgs a) {
    static_assert(kAppend || !kRope, "the rotary variant is a decode with append");
    using C = DecodeCfg<D>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kWarps * C::kWarpBytes);
    int *s_nvalid = reinterpret_cast<int *>(bars + C::kWarps * S);
    int *s_lo = s_nvalid + C::kWarps * S;  // [warp][stage] first key of the page in the window
    int *s_prefix = s_lo + C::kWarps * S;
    int *s_len = s_prefix + a.B + 1;
    int *s_first = s_len + a.B;
    int *s_pg = s_first + a.B;  // [warp][stage] physical page of the stage (appending kernel)

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    if (lane < S) mbar_init(&bars[wid * S + lane], 1);
    fence_mbar_init();
    scan_pages(a, s_prefix, s_len, s_first);  // contains __syncthreads

    const int64_t T = (int64_t)a.Hkv * s_prefix[a.B];
    int64_t per = (T + a.total_warps - 1) / a.total_warps;
    if (per < kMinUnitsPerWarp) per = kMinUnitsPerWarp;
    if (blockIdx.x == 0) {
        for (int b = tid; b <= a.B; b += blockDim.x) a.ws_prefix[b] = s_prefix[b];
        if (tid == 0) {
            a.ws_plan[0] = T;
            a.ws_plan[1] = per;
        }
    }
    const int wglob = blockIdx.x * C::kWarps + wid;
    const int64_t u_begin = (int64_t)wglob * per;
    if (u_begin >= T) return;  // warp-uniform; no block-wide barrier follows
    const int n_units = (int)min(per, T - u_begin);

    uint8_t *wbuf = smem + wid * C::kWarpBytes;
    uint64_t *wbar = bars + wid * S;
    int *wnv = s_nvalid + wid * S;
    int *wlo = s_lo + wid * S;
    int *wpg = s_pg + wid * S;

    // locate the first unit: the last sequence whose first unit is <= u_begin
    Cursor cur;
    {
        int lo = 0, hi = a.B - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if ((int64_t)a.Hkv * s_prefix[mid] <= u_begin)
                lo = mid;
            else
                hi = mid - 1;
        }
        cur.b = lo;
        cur.pb = s_prefix[lo + 1] - s_prefix[lo];
        const int64_t local = u_begin - (int64_t)a.Hkv * s_prefix[lo];
        cur.g = (int)(local / cur.pb);
        cur.p = (int)(local % cur.pb);
    }
    auto advance = [&](Cursor &c) {
        if (++c.p == c.pb) {
            c.p = 0;
            if (++c.g == a.Hkv) {
                c.g = 0;
                do {
                    ++c.b;
                    c.pb = c.b < a.B ? s_prefix[c.b + 1] - s_prefix[c.b] : 1;
                } while (c.b < a.B && c.pb == 0);
            }
        }
    };

    // Block-table window: lane l holds entry p0 + l of sequence win_b.
    int win_b = -1, win_p0 = 0, win_val = -1;
    auto page_of = [&](const Cursor &c) -> int {
        const int p0 = c.p & ~31;
        if (c.b != win_b || p0 != win_p0) {
            win_b = c.b;
            win_p0 = p0;
            const int pp = p0 + lane;
            const int first = kWindow ? s_first[c.b] : 0;
            win_val = pp < c.pb ? a.block_table[(int64_t)c.b * a.max_pages + first + pp] : -1;
        }
        return __shfl_sync(0xffffffffu, win_val, c.p - p0);
    };

    const uint64_t policy = l2_policy_evict_first();
    auto produce = [&](int stage, const Cursor &c) {
        const int pg = page_of(c);
        const bool ok = pg >= 0 && pg < a.num_pages;
        if (lane == 0) {
            const int page = (kWindow ? s_first[c.b] : 0) + c.p;  // page index within the sequence
            const int nv = ok ? min(kPageSize, s_len[c.b] - kPageSize * page) : 0;
            wnv[stage] = nv;
            // keys before the sliding window in this page are hidden
            if (kWindow) wlo[stage] = max(0, s_len[c.b] - a.window - kPageSize * page);
            if (kAppend) wpg[stage] = pg;
            uint64_t *bar = &wbar[stage];
            uint8_t *kb = wbuf + stage * C::kStageBytes;
            uint8_t *vb = kb + C::kPageBytes;
            if (ok) {
                mbar_arrive_expect_tx(bar, C::kStageBytes);
#pragma unroll
                for (int x = 0; x < C::kHalves; ++x) {
                    tma_load_4d_hint(kb + x * 2048, &kmap, bar, x * 64, 0, c.g, pg, policy);
                    tma_load_4d_hint(vb + x * 2048, &vmap, bar, x * 64, 0, c.g, pg, policy);
                }
            } else {
                set_status(a.status, SINKATTN_STATUS_BAD_PAGE);
                mbar_arrive(bar);
            }
        }
    };

    Cursor pc = cur;
    const int n_pro = min(S, n_units);
    for (int u = 0; u < n_pro; ++u) {
        produce(u, pc);
        advance(pc);
    }

    // per-lane fragment coordinates
    const int gr = lane >> 2;        // row (query head) of c0/c1; +8 for c2/c3
    const int tc = (lane & 3) * 2;   // first column of this lane's pair

    uint32_t qa[C::kKSteps][4];
    float acc[C::kNTiles][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    int seg_p0 = cur.p;
    bool seg_start = true;

    for (int u = 0; u < n_units; ++u) {
        const int stage = u % S;
        if (!__all_sync(0xffffffffu, mbar_wait_sleep(&wbar[stage], (uint32_t)((u / S) & 1), a.wait_limit_ns))) {
            // give up (all lanes together: the outcome is voted): record it, let the copies
            // already issued land, leave
            if (lane == 0) set_status(a.status, SINKATTN_STATUS_WAIT_TIMEOUT);
            for (int v = u; v < min(n_units, u + S); ++v)
                mbar_wait(&wbar[v % S], (uint32_t)((v / S) & 1), kDrainLimitNs);
            return;
        }
        uint8_t *kb = wbuf + stage * C::kStageBytes;
        uint8_t *vb = kb + C::kPageBytes;
        const int nv = wnv[stage];
        const int klo = kWindow ? wlo[stage] : 0;
        if (nv < kPageSize) clear_v_tail<D>(vb, nv, lane);
        if (kAppend) {
            // the unit holding the sequence's last token (its new one, at L - 1): that row
            // comes from the inputs, into the stage and into the cache (nv > 0: a valid page;
            // a length beyond the block table, clamped above, has no slot: nothing is written)
            const int L = s_len[cur.b];
            const int page = (kWindow ? s_first[cur.b] : 0) + cur.p;
            if (nv > 0 && page == (L - 1) / kPageSize && a.seq_lens[cur.b] == L)
                append_row<D, kRope>(a, cur.b, cur.g, L, wpg[stage], kb, vb, lane);
        }
        if (seg_start) {
            load_q<D, kRope>(a, cur.b, cur.g, s_len[cur.b], qa, lane);
#pragma unroll
            for (int n = 0; n < C::kNTiles; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
            seg_p0 = cur.p;
            seg_start = false;
        }
        page_step<D, kWindow>(a, kb, vb, nv, klo, qa, acc, m0, m1, l0, l1, lane);

        const bool seg_end = (cur.p == cur.pb - 1) || (u == n_units - 1);
        if (seg_end) {
            const float L0 = quad_sum(l0), L1 = quad_sum(l1);
            const bool whole = seg_p0 == 0 && cur.p == cur.pb - 1;
            if (whole) {
                finish_rows<D>(a, cur.b, cur.g, acc, m0, m1, L0, L1, lane);
            } else {
                const int64_t slot = (int64_t)wglob + (int64_t)cur.b * a.Hkv + cur.g;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int r = gr + half * 8;
                    if (r < a.G) {
                        const int64_t row = slot * a.G + r;
                        float *pa = a.part_acc + row * D;
#pragma unroll
                        for (int n = 0; n < C::kNTiles; ++n)
                            *reinterpret_cast<float2 *>(pa + n * 8 + tc) =
                                make_float2(acc[n][2 * half], acc[n][2 * half + 1]);
                        if ((lane & 3) == 0)
                            *reinterpret_cast<float2 *>(a.part_ml + row * 2) =
                                make_float2(half ? m1 : m0, half ? L1 : L0);
                    }
                }
            }
            seg_start = true;
        }
        advance(cur);

        // every lane's reads and V-row clears of this stage are ordered before
        // the TMA that lane 0 issues into it next
        fence_proxy_async_smem();
        __syncwarp();
        if (u + S < n_units) {
            produce(stage, pc);
            advance(pc);
        }
    }
}


// ---------------------------------------------------------------- sliding-window decode
// With a window W every (sequence, KV head) sees at most ceil(W / 16) + 1 pages, so the
// pieces are short and about equal.  One launch does it all: a CTA takes one (sequence,
// KV head) at a time (persistent over the list), each of its 4 warps a quarter of that
// item's visible pages (all of a quarter's copies in flight at once when it fits the ring),
// and the warps' partial states - each written into the warp's own copy ring, idle by then -
// are merged in shared memory with the sink: no merge launch and no partial states in the
// workspace (which then only holds the status word).  Used when a quarter is at most 32
// pages (W <= 2032 at page size 16).
constexpr int kWinWarps = 4;
constexpr int kWinMaxPagesPerWarp = 32;

template <int D>
struct WinCfg {
    using C = DecodeCfg<D>;
    static constexpr int kStages = C::kStages;
    static constexpr int kOffBars = kWinWarps * C::kWarpBytes;                      // after the rings
    static constexpr int kOffInts = kOffBars + kWinWarps * kStages * 8;             // nv, lo, pg per stage
    static constexpr int kOffMl = kOffInts + 3 * kWinWarps * kStages * 4;           // [warp][16][2] fp32
    static constexpr int kSmemBytes = 1024 + kOffMl + kWinWarps * 16 * 2 * 4;
    // a warp's partial output [16][D] fp32 goes into its own ring, idle by then
    static_assert(16 * D * 4 <= C::kWarpBytes, "partial state fits the ring");
};

template <int D, bool kAppend, bool kRope>
__global__ void __launch_bounds__(kWinWarps * 32)
    decode_window_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                         const __grid_constant__ DecodeArgs a) {
    static_assert(kAppend || !kRope, "the rotary variant is a decode with append");
    using C = DecodeCfg<D>;
    using W = WinCfg<D>;
    constexpr int S = W::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint64_t *wbar = reinterpret_cast<uint64_t *>(smem + W::kOffBars) + wid * S;
    int *wnv = reinterpret_cast<int *>(smem + W::kOffInts) + wid * S;
    int *wlo = wnv + kWinWarps * S;
    int *wpg = wlo + kWinWarps * S;
    float *s_ml = reinterpret_cast<float *>(smem + W::kOffMl);
    uint8_t *wbuf = smem + wid * C::kWarpBytes;
    if (tid == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    if (lane < S) mbar_init(&wbar[lane], 1);
    fence_mbar_init();
    __syncthreads();

    const int gr = lane >> 2, tc = (lane & 3) * 2;
    const uint64_t policy = l2_policy_evict_first();
    const int cap = a.max_pages * kPageSize;
    const int items = a.B * a.Hkv;
    uint32_t uc = 0;    // pages this warp has streamed so far (ring position)
    bool dead = false;  // a wait of this warp gave up: it only takes part in the barriers now
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int b = item / a.Hkv, g = item - b * a.Hkv;
        int L = a.seq_lens[b];
        if (L < 0 || L > cap) {
            if (tid == 0 && g == 0) set_status(a.status, SINKATTN_STATUS_BAD_LENGTH);
            L = L < 0 ? 0 : cap;
        }
        const int first = L > a.window ? (L - a.window) / kPageSize : 0;
        const int npg = (L + kPageSize - 1) / kPageSize - first;
        const int per = (npg + kWinWarps - 1) / kWinWarps;
        const int p0 = min(npg, wid * per);
        int n = dead ? 0 : min(npg, p0 + per) - p0;
        if (per > kWinMaxPagesPerWarp) {  // the host keeps W small enough; never read past a lane
            if (tid == 0) set_status(a.status, SINKATTN_STATUS_BAD_LENGTH);
            n = 0;
        }
        // block-table entries of this warp's pages: lane j holds page first + p0 + j
        const int ent = lane < n ? a.block_table[(int64_t)b * a.max_pages + first + p0 + lane] : -1;
        auto produce = [&](int j) {
            const int pg = __shfl_sync(0xffffffffu, ent, j);
            const int stage = (int)((uc + j) % S);
            if (lane == 0) {
                const bool ok = pg >= 0 && pg < a.num_pages;
                const int page = first + p0 + j;  // page index within the sequence
                wnv[stage] = ok ? min(kPageSize, L - kPageSize * page) : 0;
                wlo[stage] = max(0, L - a.window - kPageSize * page);  // keys before the window
                wpg[stage] = pg;
                uint64_t *bar = &wbar[stage];
                uint8_t *kb = wbuf + stage * C::kStageBytes;
                uint8_t *vb = kb + C::kPageBytes;
                if (ok) {
                    mbar_arrive_expect_tx(bar, C::kStageBytes);
#pragma unroll
                    for (int x = 0; x < C::kHalves; ++x) {
                        tma_load_4d_hint(kb + x * 2048, &kmap, bar, x * 64, 0, g, pg, policy);
                        tma_load_4d_hint(vb + x * 2048, &vmap, bar, x * 64, 0, g, pg, policy);
                    }
                } else {
                    set_status(a.status, SINKATTN_STATUS_BAD_PAGE);
                    mbar_arrive(bar);
                }
            }
        };
        for (int j = 0; j < min(S, n); ++j) produce(j);

        uint32_t qa[C::kKSteps][4];
        float acc[C::kNTiles][4];
#pragma unroll
        for (int c = 0; c < C::kNTiles; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        if (n > 0) load_q<D, kRope>(a, b, g, L, qa, lane);
        for (int j = 0; j < n; ++j) {
            const int stage = (int)((uc + j) % S);
            if (!__all_sync(0xffffffffu,
                            mbar_wait_sleep(&wbar[stage], (uint32_t)(((uc + j) / S) & 1), a.wait_limit_ns))) {
                // give up (all lanes together): record it, let this warp's copies in flight
                // land, and do no more work in this launch
                if (lane == 0) set_status(a.status, SINKATTN_STATUS_WAIT_TIMEOUT);
                for (int v = j; v < min(n, j + S); ++v)
                    mbar_wait(&wbar[(uc + v) % S], (uint32_t)(((uc + v) / S) & 1), kDrainLimitNs);
                dead = true;
                m0 = m1 = -INFINITY;
                break;
            }
            uint8_t *kb = wbuf + stage * C::kStageBytes;
            uint8_t *vb = kb + C::kPageBytes;
            const int nv = wnv[stage];
            if (nv < kPageSize) clear_v_tail<D>(vb, nv, lane);
            if (kAppend) {
                // the page holding the sequence's new token (position L - 1): that row comes
                // from the inputs (a length beyond the table, clamped above, has no slot)
                if (nv > 0 && first + p0 + j == (L - 1) / kPageSize && a.seq_lens[b] == L)
                    append_row<D, kRope>(a, b, g, L, wpg[stage], kb, vb, lane);
            }
            page_step<D, true>(a, kb, vb, nv, wlo[stage], qa, acc, m0, m1, l0, l1, lane);
            // every lane's reads and V-row clears of this stage are ordered before the TMA
            // that lane 0 issues into it next
            fence_proxy_async_smem();
            __syncwarp();
            if (j + S < n) produce(j + S);
        }
        if (!dead) uc += n;
        // this warp's partial state (sink-free) into shared memory
        const float L0 = quad_sum(l0), L1 = quad_sum(l1);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int r = gr + half * 8;
            if (r < a.G) {
                float *pa = reinterpret_cast<float *>(wbuf) + r * D;
#pragma unroll
                for (int c = 0; c < C::kNTiles; ++c)
                    *reinterpret_cast<float2 *>(pa + c * 8 + tc) = make_float2(acc[c][2 * half], acc[c][2 * half + 1]);
                if ((lane & 3) == 0)
                    *reinterpret_cast<float2 *>(s_ml + (wid * 16 + r) * 2) =
                        make_float2(half ? m1 : m0, half ? L1 : L0);
            }
        }
        __syncthreads();
        // merge the four partial states and fold in the sink
        constexpr int kQuads = D / 4;
        for (int i = tid; i < a.G * kQuads; i += kWinWarps * 32) {
            const int r = i / kQuads, d4 = i - r * kQuads, h = g * a.G + r;
            const float sk = a.sinks ? a.sinks[h] * kLog2e : -INFINITY;
            float M = sk;
#pragma unroll
            for (int w = 0; w < kWinWarps; ++w) M = fmaxf(M, s_ml[(w * 16 + r) * 2]);
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            float lse2 = -INFINITY;
            if (M != -INFINITY) {
                float den = sk == -INFINITY ? 0.f : exp2f(sk - M);
#pragma unroll
                for (int w = 0; w < kWinWarps; ++w) {
                    const float2 ml = *reinterpret_cast<const float2 *>(s_ml + (w * 16 + r) * 2);
                    if (ml.x == -INFINITY) continue;
                    const float e = exp2f(ml.x - M);
                    den += ml.y * e;
                    const float4 v =
                        *reinterpret_cast<const float4 *>(smem + w * C::kWarpBytes + ((r * D + d4 * 4) << 2));
                    o.x += e * v.x;
                    o.y += e * v.y;
                    o.z += e * v.z;
                    o.w += e * v.w;
                }
                const float inv = 1.f / den;
                o.x *= inv;
                o.y *= inv;
                o.z *= inv;
                o.w *= inv;
                lse2 = M + log2f(den);
            }
            __nv_bfloat16 *og = reinterpret_cast<__nv_bfloat16 *>(a.out) + ((int64_t)b * a.Hq + h) * D;
            *reinterpret_cast<uint2 *>(og + d4 * 4) = make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
            if (a.lse && d4 == 0) a.lse[(int64_t)b * a.Hq + h] = lse2 * kLn2;
        }
        // the partial states were read from the rings, which the next item's copies refill
        fence_proxy_async_smem();
        __syncthreads();
    }
}

// One CTA per (sequence, KV head): combine the partial states of a split
// sequence and add the sink; write out = 0, lse = sink for empty sequences.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeArgs a) {
    const int b = blockIdx.x / a.Hkv, g = blockIdx.x % a.Hkv;
    const int p0 = a.ws_prefix[b], pb = a.ws_prefix[b + 1] - p0;
    const int G = a.G;
    __nv_bfloat16 *og = reinterpret_cast<__nv_bfloat16 *>(a.out) + ((int64_t)b * a.Hq + (int64_t)g * G) * D;
    if (pb == 0) {
        for (int i = threadIdx.x; i < G * D; i += blockDim.x) og[i] = __float2bfloat16(0.f);
        if (a.lse)
            for (int r = threadIdx.x; r < G; r += blockDim.x)
                a.lse[(int64_t)b * a.Hq + g * G + r] = a.sinks ? a.sinks[g * G + r] : -INFINITY;
        return;
    }
    const int64_t start = (int64_t)a.Hkv * p0 + (int64_t)g * pb, last = start + pb - 1;
    const int64_t per = a.ws_plan[1];
    const int64_t w_lo = start / per, w_hi = last / per;
    if (w_lo == w_hi) return;  // finished by the split-KV kernel
    const int nsplit = (int)(w_hi - w_lo + 1);
    const int64_t slot0 = w_lo + (int64_t)b * a.Hkv + g;
    constexpr int kQuads = D / 4;
    for (int i = threadIdx.x; i < G * kQuads; i += blockDim.x) {
        const int r = i / kQuads, d4 = i % kQuads, h = g * G + r;
        const float sk = a.sinks ? a.sinks[h] * kLog2e : -INFINITY;
        float M = sk;
        for (int s = 0; s < nsplit; ++s) M = fmaxf(M, a.part_ml[((slot0 + s) * G + r) * 2]);
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        float lse2 = -INFINITY;
        if (M != -INFINITY) {
            float den = sk == -INFINITY ? 0.f : exp2f(sk - M);
            for (int s = 0; s < nsplit; ++s) {
                const int64_t row = (slot0 + s) * G + r;
                const float2 ml = *reinterpret_cast<const float2 *>(a.part_ml + row * 2);
                if (ml.x == -INFINITY) continue;
                const float w = exp2f(ml.x - M);
                den += ml.y * w;
                const float4 v = *reinterpret_cast<const float4 *>(a.part_acc + row * D + d4 * 4);
                o.x += w * v.x;
                o.y += w * v.y;
                o.z += w * v.z;
                o.w += w * v.w;
            }
            const float inv = 1.f / den;
            o.x *= inv;
            o.y *= inv;
            o.z *= inv;
            o.w *= inv;
            lse2 = M + log2f(den);
        }
        uint2 packed = make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
        *reinterpret_cast<uint2 *>(og + r * D + d4 * 4) = packed;
        if (a.lse && d4 == 0) a.lse[(int64_t)b * a.Hq + h] = lse2 * kLn2;
    }
}

template <int D>
cudaError_t shape_for(int B, int device, int *ctas, int *warps, int *smem) {
    using C = DecodeCfg<D>;
    const int bytes = decode_smem_bytes<D>(B);
    // The kernel's dynamic shared-memory ceiling is one setting per kernel, shared
    // by every batch size: raise it to the device maximum (the occupancy below
    // still uses this batch's real size).
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e != cudaSuccess) return e;
    // every variant (with and without a window, with and without append and rotation) gets
    // the same grid:
    // the split plan and the
    // workspace layout depend on it
    int sms = 0, occ = 1 << 30;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    const void *kernels[6] = {reinterpret_cast<const void *>(decode_splitkv_kernel<D, false>),
                              reinterpret_cast<const void *>(decode_splitkv_kernel<D, true>),
                              reinterpret_cast<const void *>(decode_splitkv_kernel<D, false, true>),
                              reinterpret_cast<const void *>(decode_splitkv_kernel<D, true, true>),
                              reinterpret_cast<const void *>(decode_splitkv_kernel<D, false, true, true>),
                              reinterpret_cast<const void *>(decode_splitkv_kernel<D, true, true, true>)};
    for (const void *k : kernels) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, k);
        if (e != cudaSuccess) return e;
        const int ceiling = optin - (int)fa.sharedSizeBytes;  // dynamic + static <= opt-in maximum
        if (bytes > ceiling) return cudaErrorInvalidConfiguration;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, ceiling);
        if (e != cudaSuccess) return e;
        int o = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, k, C::kThreads, bytes);
        if (e != cudaSuccess) return e;
        occ = min(occ, o);
    }
    if (occ < 1) return cudaErrorInvalidConfiguration;
    *ctas = sms * occ;
    *warps = C::kWarps;
    *smem = bytes;
    return cudaSuccess;
}

}  // namespace

cudaError_t decode_launch_shape(int D, int B, int device, int *ctas, int *warps_per_cta,
                                int *smem_bytes) {
    // occupancy queries cost microseconds; remember the answer per (device, D, B)
    struct Entry {
        int device, D, B, ctas, warps, smem;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry &e : cache)
            if (e.device == device && e.D == D && e.B == B) {
                *ctas = e.ctas;
                *warps_per_cta = e.warps;
                *smem_bytes = e.smem;
                return cudaSuccess;
            }
    }
    cudaError_t e;
    if (D == 64)
        e = shape_for<64>(B, device, ctas, warps_per_cta, smem_bytes);
    else if (D == 128)
        e = shape_for<128>(B, device, ctas, warps_per_cta, smem_bytes);
    else
        return cudaErrorInvalidValue;
    if (e == cudaSuccess) {
        std::lock_guard<std::mutex> lock(mu);
        if (cache.size() > 256) cache.clear();
        cache.push_back({device, D, B, *ctas, *warps_per_cta, *smem_bytes});
    }
    return e;
}

namespace {
// One launch of a split-KV kernel; with a.start_early it is a programmatic dependent of the
// kernel before it on the stream (it may start once that kernel lets it).
template <int D, bool kWindow, bool kAppend = false, bool kRope = false>
cudaError_t launch_splitkv_d(const DecodeArgs &a, const CUtensorMap &kmap, const CUtensorMap &vmap, int ctas,
                             int smem_bytes, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(DecodeCfg<D>::kThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.start_early ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_splitkv_kernel<D, kWindow, kAppend, kRope>, kmap, vmap, a);
}
}  // namespace

cudaError_t launch_decode_splitkv(int D, const DecodeArgs &a, const CUtensorMap &kmap,
                                  const CUtensorMap &vmap, int ctas, int smem_bytes,
                                  cudaStream_t stream) {
    const bool w = a.window > 0;
    if (a.k_new && a.rope_on) {  // decode with rotary embedding and append: same grid and plan
        if (D == 64)
            return w ? launch_splitkv_d<64, true, true, true>(a, kmap, vmap, ctas, smem_bytes, stream)
                     : launch_splitkv_d<64, false, true, true>(a, kmap, vmap, ctas, smem_bytes, stream);
        return w ? launch_splitkv_d<128, true, true, true>(a, kmap, vmap, ctas, smem_bytes, stream)
                 : launch_splitkv_d<128, false, true, true>(a, kmap, vmap, ctas, smem_bytes, stream);
    }
    if (a.k_new) {  // decode with append: same grid and plan
        if (D == 64)
            return w ? launch_splitkv_d<64, true, true>(a, kmap, vmap, ctas, smem_bytes, stream)
                     : launch_splitkv_d<64, false, true>(a, kmap, vmap, ctas, smem_bytes, stream);
        return w ? launch_splitkv_d<128, true, true>(a, kmap, vmap, ctas, smem_bytes, stream)
                 : launch_splitkv_d<128, false, true>(a, kmap, vmap, ctas, smem_bytes, stream);
    }
    if (D == 64)
        return w ? launch_splitkv_d<64, true>(a, kmap, vmap, ctas, smem_bytes, stream)
                 : launch_splitkv_d<64, false>(a, kmap, vmap, ctas, smem_bytes, stream);
    return w ? launch_splitkv_d<128, true>(a, kmap, vmap, ctas, smem_bytes, stream)
             : launch_splitkv_d<128, false>(a, kmap, vmap, ctas, smem_bytes, stream);
}

namespace {
template <int D, bool kAppend, bool kRope>
cudaError_t launch_window_d(const DecodeArgs &a, const CUtensorMap &kmap, const CUtensorMap &vmap,
                            cudaStream_t stream) {
    constexpr int bytes = WinCfg<D>::kSmemBytes;
    auto kern = decode_window_kernel<D, kAppend, kRope>;
    // occupancy per (device, variant), asked once
    static int occ_of[64] = {};
    int device = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess) return e;
    int occ = device < 64 ? occ_of[device] : 0;
    if (occ == 0) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess)
            return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kWinWarps * 32, bytes)) != cudaSuccess)
            return e;
        if (occ < 1) return cudaErrorInvalidConfiguration;
        if (device < 64) occ_of[device] = occ;
    } else if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess) {
        return e;
    }
    if (a.max_sms_cap > 0 && a.max_sms_cap < sms) sms = a.max_sms_cap;
    const int64_t items = (int64_t)a.B * a.Hkv;
    const int grid = (int)(items < (int64_t)sms * occ ? items : (int64_t)sms * occ);
    if (grid == 0) return cudaSuccess;
    kern<<<grid, kWinWarps * 32, bytes, stream>>>(kmap, vmap, a);
    return cudaGetLastError();
}
}  // namespace

bool decode_window_fits(int window) { return window > 0 && window <= kWinWarps * kWinMaxPagesPerWarp * kPageSize - 15; }

cudaError_t launch_decode_window(int D, const DecodeArgs &a, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                 cudaStream_t stream) {
    const bool app = a.k_new != nullptr, rope = app && a.rope_on;
    if (D == 64)
        return rope ? launch_window_d<64, true, true>(a, kmap, vmap, stream)
                    : app ? launch_window_d<64, true, false>(a, kmap, vmap, stream)
                          : launch_window_d<64, false, false>(a, kmap, vmap, stream);
    if (D == 128)
        return rope ? launch_window_d<128, true, true>(a, kmap, vmap, stream)
                    : app ? launch_window_d<128, true, false>(a, kmap, vmap, stream)
                          : launch_window_d<128, false, false>(a, kmap, vmap, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_merge(int D, const DecodeArgs &a, cudaStream_t stream) {
    const unsigned grid = (unsigned)a.B * (unsigned)a.Hkv;
    if (grid == 0) return cudaSuccess;
    if (D == 64)
        decode_merge_kernel<64><<<grid, 128, 0, stream>>>(a);
    else
        decode_merge_kernel<128><<<grid, 128, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace sinkattn
