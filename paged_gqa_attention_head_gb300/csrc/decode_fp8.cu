// Split-KV paged decode with per-head sinks over an FP8 E4M3 KV cache.
//
// Same method and work plan as the bf16 decode ("GPT-OSS on Day 0", section "Sink
// Attention": heads and the KV length are split, partial softmax states are merged,
// the sink counted once; HND pages, "Hosting Qwen on Blackwell", KV-cache layout).
// The cache holds one E4M3 code per element; element value = scale[g] * e4m3(code)
// with one fp32 scale per KV head g for K and one for V (the pages name an FP8
// serving precision, "GPT-OSS on Day 0", "GPT-OSS on Hopper", and an 8-bit KV
// type, TensorSharp gptoss.md section 10, without a scale convention; this is the
// reading taken).  A page of one head is 16 x D bytes, half the bf16 bytes, so the
// kernel does twice the arithmetic per byte read and is laid out to spend less:
//
//   * S^T = K Q^T on m16n8k16 f16 MMAs: the 16 tokens of a page are the M axis and
//     up to 8 query heads of the group the N axis, so a page costs D/16 MMAs per 8
//     heads (the bf16 kernel's Q K^T pads G heads to 16 rows and needs twice that).
//     E4M3 codes convert exactly to f16 (hardware cvt, two per instruction); q is
//     converted bf16 -> f16 once per segment (exact for |q| in [2^-14, 65504]).
//   * The contraction index is permuted so that each lane's K fragment is one run of
//     D/4 contiguous bytes of a token row (one or two 16-byte shared loads).
//   * O^T = V^T P^T: head_dim on M, heads on N, tokens on K.  P^T comes from the S^T
//     accumulator by movmatrix (an 8x8 transpose in registers); the head_dim index is
//     permuted so that each lane's V fragment is D/8 contiguous bytes of four token
//     rows, paired by byte permutes.  P is rounded once to f16 (relative 2^-12; f16
//     has 3 more significand bits than bf16, which is why one term suffices here).
//   * Probabilities are taken as 2^(s - m + 8) (values up to 256) so that small ones
//     stay f16 normals; the partial state carries m - 8 as its reference, which the
//     merge and the in-place finish treat like any other reference.
//   * Token rows are permuted (head_dim 64) and TMA swizzles each page (64-byte
//     swizzle for head_dim 64, 128-byte for 128) so that every shared load above is
//     free of bank conflicts.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>
#include <vector>

#include "decode_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace sinkattn {

namespace {

template <int D>
struct Fp8Cfg {
    static constexpr int kWarps = 4;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kPPU = 2;  // pages per work unit (32 tokens)
    static constexpr int kStages = 2;
    static constexpr int kPageBytes = kPageSize * D;  // one (page, head) of K or of V codes
    static constexpr int kStageBytes = 2 * kPPU * kPageBytes;  // the unit's K pages, then V pages
    static constexpr int kWarpBytes = kStages * kStageBytes;
    static constexpr int kKSteps = D / 16;  // S^T k-steps over head_dim
    static constexpr int kMTiles = D / 16;  // O^T m-tiles over head_dim
    static constexpr int kKWords = D / 16;  // 32-bit words of K a lane reads per token row
    static constexpr int kVWords = D / 32;  // 32-bit words of V a lane reads per token row
};

template <int D>
int fp8_smem_bytes(int B) {
    using C = Fp8Cfg<D>;
    return 1024 /* alignment slack */ + C::kWarps * C::kWarpBytes +
           C::kWarps * C::kStages * (8 + 8 * C::kPPU) + (3 * B + 1) * 4;
}

// Byte offset of byte c of token row r inside a page buffer written by TMA with
// this head_dim's swizzle (64-byte swizzle: 16-byte chunk bits 4-5 XOR address bits
// 7-8; 128-byte swizzle: bits 4-6 XOR bits 7-9; buffers 1024-byte aligned).
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    if (D == 64) return (uint32_t)(r * 64 + ((((c >> 4) ^ (r >> 1)) & 3) << 4) + (c & 15));
    return (uint32_t)(r * 128 + ((((c >> 4) ^ r) & 7) << 4) + (c & 15));
}

// Physical token row of MMA token index k (0..15).  For head_dim 64 the order
// 0,3,1,2,4,7,5,6 (and +8) puts the rows one load instruction touches into distinct
// banks under the 64-byte swizzle; for 128 the identity already does.
template <int D>
__device__ __forceinline__ int tok_row(int k) {
    if (D == 64) return (int)((0x65742130u >> (4 * (k & 7))) & 15u) + (k & 8);
    return k;
}


__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
    return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col)
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}


// NH: 8-head tiles of the query group (1 for G <= 8, 2 for G = 16).  The second bound is the
// CTAs an SM each variant is built for (its register budget; the occupancy each already had):
// left to itself the compiler held the two-tile head_dim-128 variant near 210 registers, and
// with the whole 2-CTA budget (up to 255) it ran the Qwen3-shape FP8 batch 6.6 % faster.
template <int D, int NH, bool kWindow>
__global__ void __launch_bounds__(Fp8Cfg<D>::kThreads, D == 64 ? (NH == 1 ? 4 : 3) : (NH == 1 ? 3 : 2))
    decode_fp8_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
    using C = Fp8Cfg<D>;
    constexpr int S = C::kStages, U = C::kPPU;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kWarps * C::kWarpBytes);
    int *s_nvalid = reinterpret_cast<int *>(bars + C::kWarps * S);  // [warp][stage][page]
    int *s_lo = s_nvalid + C::kWarps * S * U;  // [warp][stage][page] first key in the window
    int *s_prefix = s_lo + C::kWarps * S * U;
    int *s_len = s_prefix + a.B + 1;
    int *s_first = s_len + a.B;

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    if (lane < S) mbar_init(&bars[wid * S + lane], 1);
    fence_mbar_init();
    scan_pages<U>(a, s_prefix, s_len, s_first);  // contains __syncthreads

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
    int *wnv = s_nvalid + wid * S * U;
    int *wlo = s_lo + wid * S * U;

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

    // Block-table window: lane l holds the entry of visible page win_p0 + l of sequence
    // win_b (-1 past its last page).  pp is warp-uniform.
    int win_b = -1, win_p0 = 0, win_val = -1;
    auto page_entry = [&](int b, int first, int npv, int pp) -> int {
        const int p0 = pp & ~31;
        if (b != win_b || p0 != win_p0) {
            win_b = b;
            win_p0 = p0;
            const int q = p0 + lane;
            win_val = q < npv ? a.block_table[(int64_t)b * a.max_pages + first + q] : -1;
        }
        return __shfl_sync(0xffffffffu, win_val, pp - p0);
    };

    const uint64_t policy = l2_policy_evict_first();
    auto produce = [&](int stage, const Cursor &c) {
        const int first = kWindow ? s_first[c.b] : 0;
        const int L = s_len[c.b];
        const int npv = (L + kPageSize - 1) / kPageSize - first;  // pages the query sees
        int pg[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int pp = c.p * U + j;
            pg[j] = pp < npv ? page_entry(c.b, first, npv, pp) : -2;  // -2: no such page
        }
        if (lane == 0) {
            uint8_t *kb = wbuf + stage * C::kStageBytes;
            uint32_t bytes = 0;
            bool bad = false;
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int page = first + c.p * U + j;  // page index within the sequence
                const bool ok = pg[j] >= 0 && pg[j] < a.num_pages;
                bad |= pg[j] != -2 && !ok;
                wnv[stage * U + j] = ok ? min(kPageSize, L - kPageSize * page) : 0;
                // keys before the sliding window in this page are hidden
                if (kWindow) wlo[stage * U + j] = max(0, L - a.window - kPageSize * page);
                if (ok) bytes += 2 * C::kPageBytes;
            }
            if (bad) set_status(a.status, SINKATTN_STATUS_BAD_PAGE);
            uint64_t *bar = &wbar[stage];
            if (bytes) {
                mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
                for (int j = 0; j < U; ++j)
                    if (pg[j] >= 0 && pg[j] < a.num_pages) {
                        tma_load_4d_hint(kb + j * C::kPageBytes, &kmap, bar, 0, 0, c.g, pg[j], policy);
                        tma_load_4d_hint(kb + (U + j) * C::kPageBytes, &vmap, bar, 0, 0, c.g, pg[j],
                                         policy);
                    }
            } else {
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

    const int gr = lane >> 2, t4 = lane & 3;
    // K: this lane's MMA rows are tokens gr and gr + 8; its bytes are [t4 * D/4, +D/4)
    const int rk0 = tok_row<D>(gr), rk1 = rk0 + 8;
    uint32_t koff[2][C::kKWords / 4];
#pragma unroll
    for (int i = 0; i < C::kKWords / 4; ++i) {
        koff[0][i] = swz<D>(rk0, t4 * (D / 4) + 16 * i);
        koff[1][i] = swz<D>(rk1, t4 * (D / 4) + 16 * i);
    }
    // V: tokens 2t, 2t+1, 2t+8, 2t+9 of the MMA's k axis; bytes [gr * D/8, +D/8)
    uint32_t voff[4];
    int vrow[4];
    {
        const int ks[4] = {2 * t4, 2 * t4 + 1, 2 * t4 + 8, 2 * t4 + 9};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            vrow[i] = tok_row<D>(ks[i]);
            voff[i] = swz<D>(vrow[i], gr * (D / 8));
        }
    }

    uint32_t qf[C::kKSteps][NH][2];
    float acc[C::kMTiles][NH][4];
    float mr[NH][2], ls[NH][2];
    float sl = 0.f, vsc = 1.f;
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
        // Take the unit's fragments into registers and hand the stage straight back to the
        // copy engine: the next copy then overlaps this unit's arithmetic, so nearly every
        // stage of the ring is in flight rather than one held per warp while it computes.
        const uint8_t *kb = wbuf + stage * C::kStageBytes;  // K of page j at kb + j * kPageBytes
        const uint8_t *vb = kb + U * C::kPageBytes;         // V of page j at vb + j * kPageBytes
        int nv[U], klo[U];
        uint32_t kw[U][2][C::kKWords];  // K rows gr, gr + 8: the lane's run of D/4 bytes
        uint32_t vw[U][4][C::kVWords];  // V rows of tokens 2t, 2t+1, 2t+8, 2t+9: D/8 bytes
#pragma unroll
        for (int j = 0; j < U; ++j) {
            nv[j] = wnv[stage * U + j];
            klo[j] = kWindow ? wlo[stage * U + j] : 0;
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int i = 0; i < C::kKWords / 4; ++i) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(kb + j * C::kPageBytes + koff[r][i]);
                    kw[j][r][4 * i] = w.x;
                    kw[j][r][4 * i + 1] = w.y;
                    kw[j][r][4 * i + 2] = w.z;
                    kw[j][r][4 * i + 3] = w.w;
                }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint8_t *src = vb + j * C::kPageBytes + voff[i];
                uint32_t w[4] = {0u, 0u, 0u, 0u};
                if (D == 64) {
                    const uint2 x = *reinterpret_cast<const uint2 *>(src);
                    w[0] = x.x;
                    w[1] = x.y;
                } else {
                    const uint4 x = *reinterpret_cast<const uint4 *>(src);
                    w[0] = x.x;
                    w[1] = x.y;
                    w[2] = x.z;
                    w[3] = x.w;
                }
                // rows past the sequence end may hold NaN codes; P is 0 there but 0 * NaN
                // is not 0, so those V rows become zeros
                const bool live = vrow[i] < nv[j];
#pragma unroll
                for (int e = 0; e < C::kVWords; ++e) vw[j][i][e] = live ? w[e] : 0u;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (u + S < n_units) {
            produce(stage, pc);
            advance(pc);
        }

        if (seg_start) {
            const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(a.q) +
                                      ((int64_t)cur.b * a.Hq + (int64_t)cur.g * a.G) * D;
#pragma unroll
            for (int nt = 0; nt < NH; ++nt) {
                const int h = nt * 8 + gr;
#pragma unroll
                for (int i = 0; i < D / 32; ++i) {  // 8 bf16 per 16-byte load
                    uint4 w = make_uint4(0, 0, 0, 0);
                    if (h < a.G)
                        w = *reinterpret_cast<const uint4 *>(qg + h * D + t4 * (D / 4) + 8 * i);
                    // elements 8i .. 8i+7 of the lane's run: k-steps 2i and 2i + 1
                    qf[2 * i][nt][0] = bf16x2_to_f16x2(w.x);
                    qf[2 * i][nt][1] = bf16x2_to_f16x2(w.y);
                    qf[2 * i + 1][nt][0] = bf16x2_to_f16x2(w.z);
                    qf[2 * i + 1][nt][1] = bf16x2_to_f16x2(w.w);
                }
            }
#pragma unroll
            for (int mt = 0; mt < C::kMTiles; ++mt)
#pragma unroll
                for (int nt = 0; nt < NH; ++nt)
                    acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
#pragma unroll
            for (int nt = 0; nt < NH; ++nt) {
                mr[nt][0] = mr[nt][1] = -INFINITY;
                ls[nt][0] = ls[nt][1] = 0.f;
            }
            sl = a.scale_log2 * (a.k_scale ? a.k_scale[cur.g] : 1.f);
            vsc = a.v_scale ? a.v_scale[cur.g] : 1.f;
            seg_p0 = cur.p;
            seg_start = false;
        }

        // S^T = K Q^T per page: rows tokens, columns heads
        float s[U][NH][4];
#pragma unroll
        for (int j = 0; j < U; ++j) {
#pragma unroll
            for (int nt = 0; nt < NH; ++nt) s[j][nt][0] = s[j][nt][1] = s[j][nt][2] = s[j][nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < C::kKSteps; ++kk) {
                const uint32_t a0 = e4m3x2_lo_to_f16x2(kw[j][0][kk]), a2 = e4m3x2_hi_to_f16x2(kw[j][0][kk]);
                const uint32_t a1 = e4m3x2_lo_to_f16x2(kw[j][1][kk]), a3 = e4m3x2_hi_to_f16x2(kw[j][1][kk]);
#pragma unroll
                for (int nt = 0; nt < NH; ++nt)
                    mma_f16_16816(s[j][nt], a0, a1, a2, a3, qf[kk][nt][0], qf[kk][nt][1]);
            }
#pragma unroll
            for (int nt = 0; nt < NH; ++nt) {
                const bool ok0 = rk0 < nv[j] && rk0 >= klo[j], ok1 = rk1 < nv[j] && rk1 >= klo[j];
                s[j][nt][0] = ok0 ? s[j][nt][0] * sl : -INFINITY;
                s[j][nt][1] = ok0 ? s[j][nt][1] * sl : -INFINITY;
                s[j][nt][2] = ok1 ? s[j][nt][2] * sl : -INFINITY;
                s[j][nt][3] = ok1 ? s[j][nt][3] * sl : -INFINITY;
            }
        }
        uint32_t pb[U][NH][2];
#pragma unroll
        for (int nt = 0; nt < NH; ++nt) {
            float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
            for (int j = 0; j < U; ++j) {
                x0 = fmax3(x0, s[j][nt][0], s[j][nt][2]);
                x1 = fmax3(x1, s[j][nt][1], s[j][nt][3]);
            }
            const float mn0 = fmaxf(mr[nt][0], col_max(x0));
            const float mn1 = fmaxf(mr[nt][1], col_max(x1));
            const float r0 = mn0 == -INFINITY ? 0.f : mn0, r1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = fast_exp2(mr[nt][0] - r0), al1 = fast_exp2(mr[nt][1] - r1);
            mr[nt][0] = mn0;
            mr[nt][1] = mn1;
            float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const float p0 = fast_exp2(s[j][nt][0] - (r0 - 8.f)), p1 = fast_exp2(s[j][nt][1] - (r1 - 8.f));
                const float p2 = fast_exp2(s[j][nt][2] - (r0 - 8.f)), p3 = fast_exp2(s[j][nt][3] - (r1 - 8.f));
                sum0 += p0 + p2;
                sum1 += p1 + p3;
                // P^T fragments: transpose (token, head) blocks to (head, token)
                pb[j][nt][0] = movmatrix_t(pack_f16x2(p0, p1));
                pb[j][nt][1] = movmatrix_t(pack_f16x2(p2, p3));
            }
            ls[nt][0] = ls[nt][0] * al0 + sum0;
            ls[nt][1] = ls[nt][1] * al1 + sum1;
#pragma unroll
            for (int mt = 0; mt < C::kMTiles; ++mt) {
                acc[mt][nt][0] *= al0;
                acc[mt][nt][1] *= al1;
                acc[mt][nt][2] *= al0;
                acc[mt][nt][3] *= al1;
            }
        }

        // O^T += V^T P^T, one 16-token k-step per page
#pragma unroll
        for (int j = 0; j < U; ++j) {
            // word layout per token row: [half 0 (rows gr): D/64 words][half 1 (rows gr+8)]
#pragma unroll
            for (int mp = 0; mp < C::kMTiles / 2; ++mp) {  // m-tiles 2mp, 2mp + 1
                const int wi = (mp >> 1), sel = (mp & 1) ? 0x7362 : 0x5140;
                const uint32_t x00 = __byte_perm(vw[j][0][wi], vw[j][1][wi], sel);  // half 0, tokens 2t, 2t+1
                const uint32_t x01 = __byte_perm(vw[j][0][wi + D / 64], vw[j][1][wi + D / 64], sel);  // half 1
                const uint32_t x10 = __byte_perm(vw[j][2][wi], vw[j][3][wi], sel);  // half 0, tokens + 8
                const uint32_t x11 = __byte_perm(vw[j][2][wi + D / 64], vw[j][3][wi + D / 64], sel);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int mt = 2 * mp + e;
                    const uint32_t a0 = e ? e4m3x2_hi_to_f16x2(x00) : e4m3x2_lo_to_f16x2(x00);
                    const uint32_t a1 = e ? e4m3x2_hi_to_f16x2(x01) : e4m3x2_lo_to_f16x2(x01);
                    const uint32_t a2 = e ? e4m3x2_hi_to_f16x2(x10) : e4m3x2_lo_to_f16x2(x10);
                    const uint32_t a3 = e ? e4m3x2_hi_to_f16x2(x11) : e4m3x2_lo_to_f16x2(x11);
#pragma unroll
                    for (int nt = 0; nt < NH; ++nt)
                        mma_f16_16816(acc[mt][nt], a0, a1, a2, a3, pb[j][nt][0], pb[j][nt][1]);
                }
            }
        }

        const bool seg_end = (cur.p == cur.pb - 1) || (u == n_units - 1);
        if (seg_end) {
            const bool whole = seg_p0 == 0 && cur.p == cur.pb - 1;
            const int64_t slot = (int64_t)wglob + (int64_t)cur.b * a.Hkv + cur.g;
#pragma unroll
            for (int nt = 0; nt < NH; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float L = col_sum(ls[nt][e]);
                    const int hc = nt * 8 + 2 * t4 + e;  // column (head in the group)
                    // reference of the state: probabilities were taken against mr - 8
                    const float m = mr[nt][e] == -INFINITY ? -INFINITY : mr[nt][e] - 8.f;
                    if (hc >= a.G) continue;
                    const int h = cur.g * a.G + hc;
                    if (whole) {
                        const float sk = a.sinks ? a.sinks[h] * kLog2e : -INFINITY;
                        const float M = fmaxf(m, sk);
                        float scl = 0.f, lse2 = -INFINITY;
                        if (M != -INFINITY) {
                            const float wm = m == -INFINITY ? 0.f : exp2f(m - M);
                            const float den = L * wm + (sk == -INFINITY ? 0.f : exp2f(sk - M));
                            scl = wm / den * vsc;
                            lse2 = M + log2f(den);
                        }
                        // the lane's D/8 outputs of this head are contiguous: half 0 (MMA
                        // rows gr) then half 1 (rows gr + 8), D/16 each
                        uint32_t w[D / 16];
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                            for (int j = 0; j < D / 32; ++j)
                                w[hf * (D / 32) + j] = pack_bf16x2(acc[2 * j][nt][2 * hf + e] * scl,
                                                                   acc[2 * j + 1][nt][2 * hf + e] * scl);
                        __nv_bfloat16 *og = reinterpret_cast<__nv_bfloat16 *>(a.out) +
                                            ((int64_t)cur.b * a.Hq + h) * D + gr * (D / 8);
#pragma unroll
                        for (int i = 0; i < D / 64; ++i)
                            *reinterpret_cast<uint4 *>(og + 8 * i) =
                                make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                        if (a.lse && gr == 0) a.lse[(int64_t)cur.b * a.Hq + h] = lse2 * kLn2;
                    } else {
                        const int64_t row = slot * a.G + hc;
                        float f[D / 8];
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                            for (int mt = 0; mt < D / 16; ++mt) f[hf * (D / 16) + mt] = acc[mt][nt][2 * hf + e] * vsc;
                        float *pa = a.part_acc + row * D + gr * (D / 8);
#pragma unroll
                        for (int i = 0; i < D / 32; ++i)
                            *reinterpret_cast<float4 *>(pa + 4 * i) =
                                make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
                        if (gr == 0) *reinterpret_cast<float2 *>(a.part_ml + row * 2) = make_float2(m, L);
                    }
                }
            seg_start = true;
        }
        advance(cur);
    }
}

template <int D, int NH>
cudaError_t fp8_shape_for(int B, int device, int *ctas, int *warps, int *smem) {
    using C = Fp8Cfg<D>;
    const int bytes = fp8_smem_bytes<D>(B);
    int optin = 0, sms = 0, occ = 1 << 30;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    const void *kernels[2] = {reinterpret_cast<const void *>(decode_fp8_kernel<D, NH, false>),
                              reinterpret_cast<const void *>(decode_fp8_kernel<D, NH, true>)};
    for (const void *k : kernels) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, k);
        if (e != cudaSuccess) return e;
        const int ceiling = optin - (int)fa.sharedSizeBytes;
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

cudaError_t decode_fp8_launch_shape(int D, int G, int B, int device, int *ctas, int *warps_per_cta,
                                    int *smem_bytes) {
    struct Entry {
        int device, D, NH, B, ctas, warps, smem;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    const int NH = G > 8 ? 2 : 1;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry &e : cache)
            if (e.device == device && e.D == D && e.NH == NH && e.B == B) {
                *ctas = e.ctas;
                *warps_per_cta = e.warps;
                *smem_bytes = e.smem;
                return cudaSuccess;
            }
    }
    cudaError_t e;
    if (D == 64 && NH == 1)
        e = fp8_shape_for<64, 1>(B, device, ctas, warps_per_cta, smem_bytes);
    else if (D == 64)
        e = fp8_shape_for<64, 2>(B, device, ctas, warps_per_cta, smem_bytes);
    else if (D == 128 && NH == 1)
        e = fp8_shape_for<128, 1>(B, device, ctas, warps_per_cta, smem_bytes);
    else if (D == 128)
        e = fp8_shape_for<128, 2>(B, device, ctas, warps_per_cta, smem_bytes);
    else
        return cudaErrorInvalidValue;
    if (e == cudaSuccess) {
        std::lock_guard<std::mutex> lock(mu);
        if (cache.size() > 256) cache.clear();
        cache.push_back({device, D, NH, B, *ctas, *warps_per_cta, *smem_bytes});
    }
    return e;
}

cudaError_t launch_decode_fp8(int D, const DecodeArgs &a, const CUtensorMap &kmap,
                              const CUtensorMap &vmap, int ctas, int smem_bytes, cudaStream_t stream) {
    const bool w = a.window > 0;
    const bool two = a.G > 8;
#define SINKATTN_FP8_LAUNCH(DD, NN, WW) \
    decode_fp8_kernel<DD, NN, WW><<<ctas, Fp8Cfg<DD>::kThreads, smem_bytes, stream>>>(kmap, vmap, a)
    if (D == 64) {
        if (two) {
            if (w) SINKATTN_FP8_LAUNCH(64, 2, true); else SINKATTN_FP8_LAUNCH(64, 2, false);
        } else {
            if (w) SINKATTN_FP8_LAUNCH(64, 1, true); else SINKATTN_FP8_LAUNCH(64, 1, false);
        }
    } else {
        if (two) {
            if (w) SINKATTN_FP8_LAUNCH(128, 2, true); else SINKATTN_FP8_LAUNCH(128, 2, false);
        } else {
            if (w) SINKATTN_FP8_LAUNCH(128, 1, true); else SINKATTN_FP8_LAUNCH(128, 1, false);
        }
    }
#undef SINKATTN_FP8_LAUNCH
    return cudaGetLastError();
}

}  // namespace sinkattn
