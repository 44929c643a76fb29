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
// computes all G query heads of the KV head with m16n8k16 tensor-core MMAs taken
// transposed: S^T = K Q^T (the 16 tokens of a page on the M axis) and O^T = V^T P^T
// (head_dim on M), the heads on the N axis in tiles of 8, so that a group of up to 8
// heads is not padded to the 16 rows of an A operand.
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
    // Ring depth per warp.  Shallow rings let more warps share an SM's shared memory, and
    // the per-warp work on a page (ldmatrix, MMAs, softmax), not HBM, is what more warps
    // hide: measured at D=64, 6 -> 3 stages (8 -> 16 warps an SM) raised a 256-sequence
    // long-context batch from 6.04 to 6.57 TB/s, and 3 -> 2 stages (16 -> 20 warps, with the
    // transposed MMAs' lower register count) from 6.98 to 7.21 TB/s.  D=64: 2 x 4 KB per
    // warp, five 4-warp CTAs per SM for groups of up to 8 heads (four for 16, by registers);
    // D=128: 2 x 8 KB, three CTAs.
    static constexpr int kStages = 2;
    static constexpr int kHalves = D / 64;               // 128-byte column blocks per row
    static constexpr int kPageBytes = kPageSize * D * 2;  // one (page, head) of K or of V
    static constexpr int kStageBytes = 2 * kPageBytes;
    static constexpr int kWarpBytes = kStages * kStageBytes;
    static constexpr int kKSteps = D / 16;  // k-steps of S^T over head_dim; m-tiles of O^T
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
// Shared by the split-KV kernel and the sliding-window kernel.  The products are taken
// transposed, S^T = K Q^T and O^T = V^T P^T: a page's 16 tokens are the M axis of the
// first and the head_dim that of the second, and the G query heads of the group the N
// axis of both, in NH tiles of 8 heads (NH = 1 for G <= 8).  A page then costs D/16 MMAs
// per 8 heads for S and 2 D/16 for O (P as a bf16 pair), half of what padding G <= 8
// heads to the 16 rows of an A operand costs.  A warp holds for one (sequence, KV head):
//   qb[kk][nt]   q as B fragments: head 8nt + gr, head_dim columns 16kk + tc, +1 / +8, +9;
//   acc[mt][nt]  the unnormalised O^T: head_dim rows 16mt + gr / +8, heads 8nt + tc, +1;
//   mr[nt][e]    the running max of head 8nt + tc + e (log2 domain, equal in the 8 lanes
//                that share lane & 3), ls[nt][e] this lane's partial sum of its P.

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

// Decode with append: the new K/V row of (b, g) as 16-byte chunks, lane l < D/8 holding
// chunk l of the key and lane D/8 + l chunk l of the value.  Loaded when a warp starts the
// segment that holds the row's page, so the load overlaps the pages before it.
template <int D>
__device__ __forceinline__ uint4 load_new_row(const DecodeArgs &a, int b, int g, int lane) {
    constexpr int kChunks = D / 8;  // 16-byte chunks of one row
    const bool isv = lane >= kChunks;
    const int64_t row = ((int64_t)b * a.Hkv + g) * D + (lane % kChunks) * 8;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (lane < 2 * kChunks)
        w = *reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(isv ? a.v_new : a.k_new) + row);
    return w;
}

// ... and that row - the token at position L - 1, slot (L - 1) % 16 of physical page pg -
// (the key rotated first with kRope) written over its slot in the stage (the copy read the
// slot before the row existed) and into the cache.  Warp-uniform; every lane calls it.
template <int D, bool kRope>
__device__ __forceinline__ void append_row(const DecodeArgs &a, int b, int g, int L, int pg, uint8_t *kb,
                                           uint8_t *vb, uint4 w, int lane) {
    constexpr int kChunks = D / 8;  // 16-byte chunks of one row
    const int slot = (L - 1) % kPageSize;
    const bool isv = lane >= kChunks;
    const int ck = lane % kChunks;
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

// The G query rows of (b, g) as B fragments (heads past G zero); with kRope rotated at
// position L - 1.
template <int D, int NH, bool kRope>
__device__ __forceinline__ void load_q(const DecodeArgs &a, int b, int g, int L, uint32_t (&qb)[D / 16][NH][2],
                                       int lane) {
    constexpr int kK = D / 16;
    const int gr = lane >> 2, tc = (lane & 3) * 2;
    const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(a.q) + ((int64_t)b * a.Hq + (int64_t)g * a.G) * D;
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) {
        const int h = nt * 8 + gr;
        const bool ok = h < a.G;
#pragma unroll
        for (int kk = 0; kk < kK; ++kk) {
            const int col = kk * 16 + tc;
            qb[kk][nt][0] = ok ? *reinterpret_cast<const uint32_t *>(qg + h * D + col) : 0u;
            qb[kk][nt][1] = ok ? *reinterpret_cast<const uint32_t *>(qg + h * D + col + 8) : 0u;
        }
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
#pragma unroll
                for (int nt = 0; nt < NH; ++nt) rope_pairs(qb[kk][nt][x], qb[kk + kK / 2][nt][x], cs0, cs1);
            }
    }
}

// One page: S^T = K Q^T for its 16 tokens (keys klo .. nv - 1 visible), the online-softmax
// update and O^T += V^T P^T.
template <int D, int NH, bool kWindow>
__device__ __forceinline__ void page_step(const DecodeArgs &a, const uint8_t *kb, const uint8_t *vb, int nv,
                                          int klo, const uint32_t (&qb)[D / 16][NH][2],
                                          float (&acc)[D / 16][NH][4], float (&mr)[NH][2], float (&ls)[NH][2],
                                          int lane) {
    constexpr int kK = D / 16;
    const int gr = lane >> 2;
    const int lm = lane >> 3, lr = lane & 7;  // ldmatrix: matrix index, row within it
    // S^T: rows tokens gr / gr + 8, columns heads 8nt + tc, +1
    float s[NH][4];
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    const uint32_t kbase = smem_u32(kb);
#pragma unroll
    for (int kk = 0; kk < kK; ++kk) {
        // A fragments of K: tokens 0-7 / 8-15 (matrices 0, 2 / 1, 3), columns 16kk..+7 / +8..15
        const int tok = (lm & 1) * 8 + lr, chunk = kk * 2 + (lm >> 1);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kbase + (chunk >> 3) * 2048 + sw128(tok, chunk & 7), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NH; ++nt) mma_16816(s[nt], a0, a1, a2, a3, qb[kk][nt][0], qb[kk][nt][1]);
    }
    const bool ok0 = gr < nv && (!kWindow || gr >= klo), ok1 = gr + 8 < nv && (!kWindow || gr + 8 >= klo);
    // the running max of a head is raised only when a score passes it by more than 8 (log2
    // units), so P = exp2(s - m) <= 2^8 and most pages leave the accumulators as they are;
    // whether any score does is voted on first, and only then are the column maxima taken
    bool raise = false;
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) {
        s[nt][0] = ok0 ? s[nt][0] * a.scale_log2 : -INFINITY;
        s[nt][1] = ok0 ? s[nt][1] * a.scale_log2 : -INFINITY;
        s[nt][2] = ok1 ? s[nt][2] * a.scale_log2 : -INFINITY;
        s[nt][3] = ok1 ? s[nt][3] * a.scale_log2 : -INFINITY;
        raise |= fmaxf(s[nt][0], s[nt][2]) > mr[nt][0] + 8.f || fmaxf(s[nt][1], s[nt][3]) > mr[nt][1] + 8.f;
    }
    if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
        for (int nt = 0; nt < NH; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float mx = col_max(fmaxf(s[nt][e], s[nt][2 + e]));
                const float mn = mx > mr[nt][e] + 8.f ? mx : mr[nt][e];
                const float al = mr[nt][e] == -INFINITY ? 0.f : fast_exp2(mr[nt][e] - mn);
                mr[nt][e] = mn;
                ls[nt][e] *= al;
#pragma unroll
                for (int mt = 0; mt < kK; ++mt) {
                    acc[mt][nt][e] *= al;
                    acc[mt][nt][2 + e] *= al;
                }
            }
    }
    // P^T as B fragments of O^T = V^T P^T, P = P_hi + P_lo, both bf16 (the rounding of P to
    // bf16 alone, relative 2^-9, is too coarse for short sequences; the pair keeps ~16 bits):
    // each 8x8 (token, head) block is transposed in registers to (head, token)
    uint32_t bh[NH][2], bl[NH][2];
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) {
        const float base0 = mr[nt][0] == -INFINITY ? 0.f : mr[nt][0];
        const float base1 = mr[nt][1] == -INFINITY ? 0.f : mr[nt][1];
        const float p0 = fast_exp2(s[nt][0] - base0), p1 = fast_exp2(s[nt][1] - base1);
        const float p2 = fast_exp2(s[nt][2] - base0), p3 = fast_exp2(s[nt][3] - base1);
        ls[nt][0] += p0 + p2;
        ls[nt][1] += p1 + p3;
        const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
        const uint32_t l01 = pack_bf16x2(p0 - __uint_as_float(h01 << 16), p1 - __uint_as_float(h01 & 0xFFFF0000u));
        const uint32_t l23 = pack_bf16x2(p2 - __uint_as_float(h23 << 16), p3 - __uint_as_float(h23 & 0xFFFF0000u));
        bh[nt][0] = movmatrix_t(h01);
        bh[nt][1] = movmatrix_t(h23);
        bl[nt][0] = movmatrix_t(l01);
        bl[nt][1] = movmatrix_t(l23);
    }
    // O^T += V^T P^T: A fragments of V^T read transposed from the V rows (tokens 0-7 / 8-15 in
    // matrices 0, 1 / 2, 3; head_dim 16mt..+7 / +8..15)
    const uint32_t vbase = smem_u32(vb);
#pragma unroll
    for (int mt = 0; mt < kK; ++mt) {
        const int tok = (lm >> 1) * 8 + lr, chunk = mt * 2 + (lm & 1);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vbase + (chunk >> 3) * 2048 + sw128(tok, chunk & 7), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NH; ++nt) mma_16816(acc[mt][nt], a0, a1, a2, a3, bh[nt][0], bh[nt][1]);
#pragma unroll
        for (int nt = 0; nt < NH; ++nt) mma_16816(acc[mt][nt], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);
    }
}

// Hands each lane two adjacent head_dim columns of one head: the lanes of gr and gr ^ 1
// (lane ^ 4) swap their values of the other's head, so the even one holds head 8nt + tc,
// the odd one head 8nt + tc + 1, at columns 16mt + 8 half + (gr & ~1), +1.  Every lane
// calls it (warp shuffles); e = gr & 1 is the head the lane keeps.
template <int D, int NH>
__device__ __forceinline__ float2 head_pair(const float (&acc)[D / 16][NH][4], int mt, int nt, int half, int lane) {
    const bool odd = (lane >> 2) & 1;
    const float c0 = acc[mt][nt][2 * half], c1 = acc[mt][nt][2 * half + 1];
    const float got = __shfl_xor_sync(0xffffffffu, odd ? c0 : c1, 4);
    return odd ? make_float2(got, c1) : make_float2(c0, got);
}

// The final out / lse rows of (b, g) from a state that covers every visible key: the sink
// joins the max and the denominator.
template <int D, int NH>
__device__ __forceinline__ void finish_rows(const DecodeArgs &a, int b, int g, const float (&acc)[D / 16][NH][4],
                                            const float (&mr)[NH][2], const float (&ls)[NH][2], int lane) {
    const int gr = lane >> 2, tc = (lane & 3) * 2, e = gr & 1;
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) {
        float scl[2], lse2[2];
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int hl = nt * 8 + tc + x;  // head within the group
            const float l = col_sum(ls[nt][x]), m = mr[nt][x];
            const float sk = a.sinks && hl < a.G ? a.sinks[g * a.G + hl] * kLog2e : -INFINITY;
            const float M = fmaxf(m, sk);
            scl[x] = 0.f;
            lse2[x] = -INFINITY;
            if (M != -INFINITY) {
                const float wm = m == -INFINITY ? 0.f : exp2f(m - M);
                const float den = l * wm + (sk == -INFINITY ? 0.f : exp2f(sk - M));
                scl[x] = wm / den;
                lse2[x] = M + log2f(den);
            }
        }
        const int hl = nt * 8 + tc + e;
        __nv_bfloat16 *og = reinterpret_cast<__nv_bfloat16 *>(a.out) + ((int64_t)b * a.Hq + g * a.G + hl) * D;
        const float sc = e ? scl[1] : scl[0];
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const float2 v = head_pair<D, NH>(acc, mt, nt, half, lane);
                if (hl < a.G)
                    *reinterpret_cast<uint32_t *>(og + mt * 16 + half * 8 + (gr & ~1)) = pack_bf16x2(v.x * sc, v.y * sc);
            }
        if (a.lse && gr == 0)
#pragma unroll
            for (int x = 0; x < 2; ++x)
                if (nt * 8 + tc + x < a.G) a.lse[(int64_t)b * a.Hq + g * a.G + nt * 8 + tc + x] = lse2[x] * kLn2;
    }
}

// The partial state of (sequence, KV head) over part of its pages, unnormalised and without
// the sink, into rows row0 .. row0 + G - 1 (head_dim values, and (m, l) per row).
template <int D, int NH>
__device__ __forceinline__ void write_partial(float *part_acc, float *part_ml, int64_t row0, int G,
                                              const float (&acc)[D / 16][NH][4], const float (&mr)[NH][2],
                                              const float (&ls)[NH][2], int lane) {
    const int gr = lane >> 2, tc = (lane & 3) * 2, e = gr & 1;
#pragma unroll
    for (int nt = 0; nt < NH; ++nt) {
        const float l0 = col_sum(ls[nt][0]), l1 = col_sum(ls[nt][1]);
        const int hl = nt * 8 + tc + e;
        float *pa = part_acc + (row0 + hl) * D;
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const float2 v = head_pair<D, NH>(acc, mt, nt, half, lane);
                if (hl < G) *reinterpret_cast<float2 *>(pa + mt * 16 + half * 8 + (gr & ~1)) = v;
            }
        if (gr == 0) {
            if (nt * 8 + tc < G) *reinterpret_cast<float2 *>(part_ml + (row0 + nt * 8 + tc) * 2) = make_float2(mr[nt][0], l0);
            if (nt * 8 + tc + 1 < G)
                *reinterpret_cast<float2 *>(part_ml + (row0 + nt * 8 + tc + 1) * 2) = make_float2(mr[nt][1], l1);
        }
    }
}

// NH: 8-head tiles of the query group (1 for G <= 8, 2 for G <= 16).  kWindow: a sliding
// window is given (a.window > 0); the kernel without it carries no window arithmetic.
// kAppend: the new K/V rows a.k_new / a.v_new are appended (see above).  kRope (with
// kAppend): q and the new key are rotated first (see above).
template <int D, int NH, bool kWindow, bool kAppend = false, bool kRope = false>
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

    uint32_t qb[C::kKSteps][NH][2];
    float acc[C::kKSteps][NH][4];
    float mr[NH][2], ls[NH][2];
    int seg_p0 = cur.p;
    bool seg_start = true;
    uint4 new_row = make_uint4(0, 0, 0, 0);  // with kAppend: the new K/V row of the segment's last page
    int len_given = -1;                       // ... and its sequence's length as given

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
            // a segment that reaches the last visible page (the one holding L - 1) loads the
            // new row, and the length as given (unclamped), as it starts
            if (seg_start && u + (cur.pb - 1 - cur.p) < n_units) {
                new_row = load_new_row<D>(a, cur.b, cur.g, lane);
                len_given = a.seq_lens[cur.b];
            }
            const int page = (kWindow ? s_first[cur.b] : 0) + cur.p;
            if (nv > 0 && page == (L - 1) / kPageSize && len_given == L)
                append_row<D, kRope>(a, cur.b, cur.g, L, wpg[stage], kb, vb, new_row, lane);
        }
        if (seg_start) {
            load_q<D, NH, kRope>(a, cur.b, cur.g, s_len[cur.b], qb, lane);
#pragma unroll
            for (int mt = 0; mt < C::kKSteps; ++mt)
#pragma unroll
                for (int nt = 0; nt < NH; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
#pragma unroll
            for (int nt = 0; nt < NH; ++nt) {
                mr[nt][0] = mr[nt][1] = -INFINITY;
                ls[nt][0] = ls[nt][1] = 0.f;
            }
            seg_p0 = cur.p;
            seg_start = false;
        }
        page_step<D, NH, kWindow>(a, kb, vb, nv, klo, qb, acc, mr, ls, lane);

        const bool seg_end = (cur.p == cur.pb - 1) || (u == n_units - 1);
        if (seg_end) {
            const bool whole = seg_p0 == 0 && cur.p == cur.pb - 1;
            if (whole) {
                finish_rows<D, NH>(a, cur.b, cur.g, acc, mr, ls, lane);
            } else {
                const int64_t slot = (int64_t)wglob + (int64_t)cur.b * a.Hkv + cur.g;
                write_partial<D, NH>(a.part_acc, a.part_ml, slot * a.G, a.G, acc, mr, ls, lane);
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

template <int D, int NH, bool kAppend, bool kRope>
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

        uint32_t qb[C::kKSteps][NH][2];
        float acc[C::kKSteps][NH][4];
        float mr[NH][2], ls[NH][2];
#pragma unroll
        for (int nt = 0; nt < NH; ++nt) {
#pragma unroll
            for (int mt = 0; mt < C::kKSteps; ++mt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
            mr[nt][0] = mr[nt][1] = -INFINITY;
            ls[nt][0] = ls[nt][1] = 0.f;
        }
        if (n > 0) load_q<D, NH, kRope>(a, b, g, L, qb, lane);
        // the warp with the last visible page (the one holding L - 1) loads the new row now
        const uint4 new_row = kAppend && n > 0 && p0 + n == npg ? load_new_row<D>(a, b, g, lane) : make_uint4(0, 0, 0, 0);
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
#pragma unroll
                for (int nt = 0; nt < NH; ++nt) mr[nt][0] = mr[nt][1] = -INFINITY;
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
                    append_row<D, kRope>(a, b, g, L, wpg[stage], kb, vb, new_row, lane);
            }
            page_step<D, NH, true>(a, kb, vb, nv, wlo[stage], qb, acc, mr, ls, lane);
            // every lane's reads and V-row clears of this stage are ordered before the TMA
            // that lane 0 issues into it next
            fence_proxy_async_smem();
            __syncwarp();
            if (j + S < n) produce(j + S);
        }
        if (!dead) uc += n;
        // this warp's partial state (sink-free) into shared memory: [16][D] fp32 in its ring
        write_partial<D, NH>(reinterpret_cast<float *>(wbuf), s_ml + wid * 16 * 2, 0, a.G, acc, mr, ls, lane);
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
cudaError_t shape_for(int B, int G, int device, int *ctas, int *warps, int *smem, int *ring) {
    using C = DecodeCfg<D>;
    const int bytes = decode_smem_bytes<D>(B);
    // The kernel's dynamic shared-memory ceiling is one setting per kernel, shared
    // by every batch size: raise it to the device maximum (the occupancy below
    // still uses this batch's real size).
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e != cudaSuccess) return e;
    // every variant of one group size (with and without a window, with and without append
    // and rotation) gets the same grid: the split plan and the workspace layout depend on it;
    // groups of up to 8 heads (one 8-head tile) use fewer registers and may fit more CTAs
    int sms = 0, occ = 1 << 30;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    const void *all[12] = {reinterpret_cast<const void *>(decode_splitkv_kernel<D, 1, false>),
                               reinterpret_cast<const void *>(decode_splitkv_kernel<D, 1, true>),
                               reinterpret_cast<const void *>(decode_splitkv_kernel<D, 1, false, true>),
                               reinterpret_cast<const void *>(decode_splitkv_kernel<D, 1, true, true>),
                               reinterpret_cast<const void *>(decode_splitkv_kernel<D, 1, false, true, true>),
                               reinterpret_cast<const void *>(decode_splitkv_kernel<D, 1, true, true, true>),
                               reinterpret_cast<const void *>(decode_splitkv_kernel<D, 2, false>),
                               reinterpret_cast<const void *>(decode_splitkv_kernel<D, 2, true>),
                               reinterpret_cast<const void *>(decode_splitkv_kernel<D, 2, false, true>),
                               reinterpret_cast<const void *>(decode_splitkv_kernel<D, 2, true, true>),
                               reinterpret_cast<const void *>(decode_splitkv_kernel<D, 2, false, true, true>),
                               reinterpret_cast<const void *>(decode_splitkv_kernel<D, 2, true, true, true>)};
    const void *const *kernels = all + (G > 8 ? 6 : 0);  // the variants of this group size
    for (int ki = 0; ki < 6; ++ki) {
        const void *k = kernels[ki];
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
    *ring = C::kWarps * C::kWarpBytes;
    return cudaSuccess;
}

}  // namespace

cudaError_t decode_launch_shape(int D, int B, int G, int device, int *ctas, int *warps_per_cta,
                                int *smem_bytes, int *ring_bytes) {
    // occupancy queries cost microseconds; remember the answer per (device, D, B, head tiles)
    struct Entry {
        int device, D, B, G, ctas, warps, smem, ring;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry &e : cache)
            if (e.device == device && e.D == D && e.B == B && (e.G > 8) == (G > 8)) {
                *ctas = e.ctas;
                *warps_per_cta = e.warps;
                *smem_bytes = e.smem;
                *ring_bytes = e.ring;
                return cudaSuccess;
            }
    }
    cudaError_t e;
    if (D == 64)
        e = shape_for<64>(B, G, device, ctas, warps_per_cta, smem_bytes, ring_bytes);
    else if (D == 128)
        e = shape_for<128>(B, G, device, ctas, warps_per_cta, smem_bytes, ring_bytes);
    else
        return cudaErrorInvalidValue;
    if (e == cudaSuccess) {
        std::lock_guard<std::mutex> lock(mu);
        if (cache.size() > 256) cache.clear();
        cache.push_back({device, D, B, G, *ctas, *warps_per_cta, *smem_bytes, *ring_bytes});
    }
    return e;
}

namespace {
// One launch of a split-KV kernel; with a.start_early it is a programmatic dependent of the
// kernel before it on the stream (it may start once that kernel lets it).
template <int D, bool kWindow, bool kAppend = false, bool kRope = false>
cudaError_t launch_splitkv_d(const DecodeArgs &a, const CUtensorMap &kmap, const CUtensorMap &vmap, int ctas,
                             int smem_bytes, cudaStream_t stream) {
    // one tile of 8 heads for G <= 8, two for G <= 16
    auto kern = a.G > 8 ? decode_splitkv_kernel<D, 2, kWindow, kAppend, kRope>
                        : decode_splitkv_kernel<D, 1, kWindow, kAppend, kRope>;
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
    return cudaLaunchKernelEx(&cfg, kern, kmap, vmap, a);
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
template <int D, int NH, bool kAppend, bool kRope>
cudaError_t launch_window_nh(const DecodeArgs &a, const CUtensorMap &kmap, const CUtensorMap &vmap,
                             cudaStream_t stream) {
    constexpr int bytes = WinCfg<D>::kSmemBytes;
    auto kern = decode_window_kernel<D, NH, kAppend, kRope>;
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
template <int D, bool kAppend, bool kRope>
cudaError_t launch_window_d(const DecodeArgs &a, const CUtensorMap &kmap, const CUtensorMap &vmap,
                            cudaStream_t stream) {
    return a.G > 8 ? launch_window_nh<D, 2, kAppend, kRope>(a, kmap, vmap, stream)
                   : launch_window_nh<D, 1, kAppend, kRope>(a, kmap, vmap, stream);
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
