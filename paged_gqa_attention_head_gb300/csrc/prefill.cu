// Causal ragged prefill and chunked prefill over a paged prefix, on tcgen05
// tensor cores with TMEM accumulators.
//
// Method: softmax attention with a per-head sink that enters the max and the
// denominator only (TensorSharp docs/models/gptoss.md, section 3 "Forward graph";
// section 4.1: a virtual token with zero K and V), computed as an online softmax
// whose running max starts at the sink and whose running denominator starts at 1
// ("GPT-OSS on Day 0", section "Sink Attention").  Ragged inputs are packed with
// cu_seqlens; a request may continue a paged HND prefix ("Fast embeddings on
// GPUs", attention kernels: ragged, paged prefill; "Hosting Qwen on Blackwell":
// HND pages).  Query t of request i sits at absolute position P_i + t and sees
// every prefix key and new keys 0..t.
//
// GB300 design.  One CTA computes a 128-row query tile of one head against all
// the key tiles it may see (prefix tiles first, then the causal new-token tiles
// up to the diagonal; fully masked tiles are never visited):
//   warp 0      TMA producer: the Q tile once, K and V tiles into a ring of
//               stages (new tokens: one 3-D box of 128 rows; prefix: eight 16-row
//               page boxes through the block table, with a ragged or invalid page
//               copied by the warp and zero-filled)
//   warp 1      allocates TMEM; one thread issues S = Q K^T (M=128, N=128) into
//               one of two TMEM S buffers, then O += P V (M=128, N=D) into TMEM
//   warps 2..5  softmax: each thread owns one query row; reads its S row from
//               TMEM, masks, keeps the running max (rescaling O in TMEM only when
//               the max grows by more than 2^8), writes P into shared memory
//               as two bf16 tiles P_hi + P_lo (128-byte swizzled, the MMA's
//               K-major A layout); O += P_hi V + P_lo V keeps ~16 bits of P
// S for tile j+1 is computed while the softmax works on tile j.
#include <float.h>

#include "internal.h"
#include "ptx.cuh"

namespace sinkattn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P values stay below 2^8
constexpr int kBM = 128;                   // query rows per tile
constexpr int kBN = 128;                   // keys per tile
constexpr int kThreads = 192;              // 6 warps
constexpr uint32_t kTmemCols = 512;

template <int D>
struct PrefillCfg {
    static constexpr int kHalves = D / 64;                 // 128-byte column blocks
    static constexpr int kStages = 2;                      // K/V ring depth
    static constexpr int kPBufs = D == 64 ? 2 : 1;         // P buffers (hi + lo each)
    static constexpr int kQBytes = kBM * D * 2;
    static constexpr int kKVBytes = kBN * D * 2;           // one K (or V) tile
    static constexpr int kPHalf = kBM * kBN * 2;           // P_hi or P_lo of one tile
    static constexpr int kPBytes = 2 * kPHalf;             // P_hi then P_lo
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kQBytes;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffP = kOffV + kStages * kKVBytes;
    static constexpr int kOffBar = kOffP + kPBufs * kPBytes;
    static constexpr int kNumBars = 1 + 3 * kStages + 4 + 2 * kPBufs + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = 1024 + kOffMisc + 64;
    static constexpr uint32_t kColS = 0;      // two S buffers: columns [0,128), [128,256)
    static constexpr uint32_t kColO = 256;    // O: columns [256, 256 + D)
};

struct Bars {
    uint64_t *q_full, *k_full, *v_full, *kv_empty, *s_full, *s_free, *p_full, *p_empty, *drain;
};

// Bounded wait that also gives up as soon as another role has given up.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort,
                                              uint32_t *status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 128; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            set_status(status, SINKATTN_STATUS_WAIT_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Which (request, query block) this CTA works on: query blocks are ranked by
// their index inside the request, largest first (they see the most key tiles),
// so the longest work starts first.  Returns false if the rank is past the end.
__device__ bool locate_tile(const PrefillArgs &a, int rank, int *req, int *qb) {
    int maxnq = 0;
    for (int i = 0; i < a.n; ++i) {
        const int L = a.cu_seqlens[i + 1] - a.cu_seqlens[i];
        maxnq = max(maxnq, (L + kBM - 1) / kBM);
    }
    for (int lev = maxnq - 1; lev >= 0; --lev)
        for (int i = 0; i < a.n; ++i) {
            const int L = a.cu_seqlens[i + 1] - a.cu_seqlens[i];
            if ((L + kBM - 1) / kBM > lev) {
                if (rank == 0) {
                    *req = i;
                    *qb = lev;
                    return true;
                }
                --rank;
            }
        }
    return false;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap kpmap,
                   const __grid_constant__ CUtensorMap vpmap, const PrefillArgs a) {
    using C = PrefillCfg<D>;
    constexpr int NS = C::kStages;
    constexpr int NP = C::kPBufs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *sQ = smem + C::kOffQ;
    uint8_t *sK = smem + C::kOffK;
    uint8_t *sV = smem + C::kOffV;
    uint8_t *sP = smem + C::kOffP;
    uint64_t *bar_base = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    Bars bars;
    bars.q_full = bar_base;
    bars.k_full = bar_base + 1;
    bars.v_full = bars.k_full + NS;
    bars.kv_empty = bars.v_full + NS;
    bars.s_full = bars.kv_empty + NS;
    bars.s_free = bars.s_full + 2;
    bars.p_full = bars.s_free + 2;
    bars.p_empty = bars.p_full + NP;
    bars.drain = bars.p_empty + NP;
    int *misc = reinterpret_cast<int *>(smem + C::kOffMisc);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(misc);  // misc[0]: TMEM base
    volatile int *s_abort = misc + 1;
    int *s_tile = misc + 2;  // request, query block, valid flag

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x % a.Hq;
    const int rank = blockIdx.x / a.Hq;

    if (tid == 0) {
        int req = 0, qb = 0;
        const bool ok = locate_tile(a, rank, &req, &qb);
        s_tile[0] = req;
        s_tile[1] = qb;
        s_tile[2] = ok ? 1 : 0;
        *s_abort = 0;
        mbar_init(bars.q_full, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars.s_full[b], 1);
            mbar_init(&bars.s_free[b], 4);
        }
        for (int b = 0; b < NP; ++b) {
            mbar_init(&bars.p_full[b], 4);
            mbar_init(&bars.p_empty[b], 1);
        }
        mbar_init(bars.drain, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (!s_tile[2]) return;  // CTA-uniform: nothing allocated yet

    const int req = s_tile[0], qb = s_tile[1];
    const int row0 = a.cu_seqlens[req];
    const int L = a.cu_seqlens[req + 1] - row0;
    const int g = h / a.G;
    int P = 0;
    if (a.prefix_lens) {
        P = a.prefix_lens[req];
        const int cap = a.max_pages * kPageSize;
        if (P < 0 || P > cap) {
            if (tid == 0) set_status(a.status, SINKATTN_STATUS_BAD_LENGTH);
            P = P < 0 ? 0 : cap;
        }
    }
    const int n_pre = (P + kBN - 1) / kBN;
    const int n_kv = n_pre + qb + 1;

    if (warp == 1) {
        tc::alloc(s_tmem, kTmemCols);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *s_tmem;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            mbar_arrive_expect_tx(bars.q_full, C::kQBytes);
#pragma unroll
            for (int x = 0; x < C::kHalves; ++x)
                tma_load_3d(sQ + x * 16384, &qmap, bars.q_full, x * 64, h, row0 + qb * kBM);
        }
        for (int j = 0; j < n_kv; ++j) {
            const int s = j % NS;
            if (j >= NS && !wait_or_abort(&bars.kv_empty[s], (uint32_t)(((j / NS) + 1) & 1), s_abort,
                                          a.status))
                break;
            uint8_t *kt = sK + s * C::kKVBytes;
            uint8_t *vt = sV + s * C::kKVBytes;
            if (j < n_pre) {
                // eight pages of 16 tokens; whole valid pages by TMA, the rest by the warp
                const int pt = j;
                uint32_t nfull = 0;
#pragma unroll
                for (int pp = 0; pp < 8; ++pp) {
                    const int page = pt * 8 + pp;
                    const int nrow = min(kPageSize, max(0, P - page * kPageSize));
                    if (nrow > 0) {
                        const int pg = a.prefix_block_table[(int64_t)req * a.max_pages + page];
                        if (pg < 0 || pg >= a.num_pages) {
                            if (lane == 0) set_status(a.status, SINKATTN_STATUS_BAD_PAGE);
                        } else if (nrow == kPageSize) {
                            ++nfull;
                        }
                    }
                }
                if (lane == 0) {
                    mbar_expect_tx(&bars.k_full[s], nfull * kPageSize * D * 2);
                    mbar_expect_tx(&bars.v_full[s], nfull * kPageSize * D * 2);
                }
#pragma unroll 1
                for (int pp = 0; pp < 8; ++pp) {
                    const int page = pt * 8 + pp;
                    const int nrow = min(kPageSize, max(0, P - page * kPageSize));
                    int pg = -1;
                    if (nrow > 0) {
                        pg = a.prefix_block_table[(int64_t)req * a.max_pages + page];
                        if (pg < 0 || pg >= a.num_pages) pg = -1;
                    }
                    if (nrow == kPageSize && pg >= 0) {
                        if (lane == 0) {
#pragma unroll
                            for (int x = 0; x < C::kHalves; ++x) {
                                tma_load_4d(kt + x * 16384 + pp * 2048, &kpmap, &bars.k_full[s], x * 64,
                                            0, g, pg);
                                tma_load_4d(vt + x * 16384 + pp * 2048, &vpmap, &bars.v_full[s], x * 64,
                                            0, g, pg);
                            }
                        }
                    } else {
                        // ragged or invalid page: copy the valid rows, zero the rest
                        const int nv = pg >= 0 ? nrow : 0;
                        const __nv_bfloat16 *kg = reinterpret_cast<const __nv_bfloat16 *>(a.k_pages);
                        const __nv_bfloat16 *vg = reinterpret_cast<const __nv_bfloat16 *>(a.v_pages);
                        for (int e = lane; e < kPageSize * C::kHalves * 8; e += 32) {
                            const int slot = e / (C::kHalves * 8);
                            const int x = (e / 8) % C::kHalves;
                            const int c = e % 8;
                            uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
                            if (slot < nv) {
                                const int64_t off =
                                    (((int64_t)pg * a.Hkv + g) * kPageSize + slot) * D + x * 64 + c * 8;
                                kv = *reinterpret_cast<const uint4 *>(kg + off);
                                vv = *reinterpret_cast<const uint4 *>(vg + off);
                            }
                            const uint32_t o = x * 16384 + sw128(pp * kPageSize + slot, c);
                            *reinterpret_cast<uint4 *>(kt + o) = kv;
                            *reinterpret_cast<uint4 *>(vt + o) = vv;
                        }
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars.k_full[s]);
                    mbar_arrive(&bars.v_full[s]);
                }
            } else if (lane == 0) {
                const int kt_idx = j - n_pre;
                mbar_arrive_expect_tx(&bars.k_full[s], C::kKVBytes);
#pragma unroll
                for (int x = 0; x < C::kHalves; ++x)
                    tma_load_3d(kt + x * 16384, &kmap, &bars.k_full[s], x * 64, g, row0 + kt_idx * kBN);
                mbar_arrive_expect_tx(&bars.v_full[s], C::kKVBytes);
#pragma unroll
                for (int x = 0; x < C::kHalves; ++x)
                    tma_load_3d(vt + x * 16384, &vmap, &bars.v_full[s], x * 64, g, row0 + kt_idx * kBN);
            }
            __syncwarp();
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kBM, kBN, false);
            constexpr uint32_t idesc_o = tc::idesc_bf16_f32(kBM, D, true);
            const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV);
            const uint32_t p_addr = smem_u32(sP);
            bool ok = wait_or_abort(bars.q_full, 0, s_abort, a.status);
            // O += P_hi V + P_lo V: P = P_hi + P_lo carries ~16 bits of each weight
            auto issue_pv = [&](int j) -> bool {
                const int pb = j % NP, s = j % NS;
                if (!wait_or_abort(&bars.p_full[pb], (uint32_t)((j / NP) & 1), s_abort, a.status))
                    return false;
                if (!wait_or_abort(&bars.v_full[s], (uint32_t)((j / NS) & 1), s_abort, a.status))
                    return false;
                tc::fence_after_sync();
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk) {
                        const uint64_t adesc = tc::smem_desc_sw128(
                            p_addr + pb * C::kPBytes + part * C::kPHalf + (kk >> 2) * 16384 + (kk & 3) * 32,
                            16, 1024);
                        const uint64_t bdesc =
                            tc::smem_desc_sw128(v_addr + s * C::kKVBytes + kk * 2048, 16384, 1024);
                        tc::mma_f16_ss(tmem + C::kColO, adesc, bdesc, idesc_o,
                                       (j > 0 || part > 0 || kk > 0) ? 1u : 0u);
                    }
                tc::commit(&bars.p_empty[pb]);
                tc::commit(&bars.kv_empty[s]);
                return true;
            };
            for (int j = 0; ok && j < n_kv; ++j) {
                const int b = j & 1, s = j % NS;
                if (!wait_or_abort(&bars.k_full[s], (uint32_t)((j / NS) & 1), s_abort, a.status)) {
                    ok = false;
                    break;
                }
                if (j >= 2 &&
                    !wait_or_abort(&bars.s_free[b], (uint32_t)(((j - 2) >> 1) & 1), s_abort, a.status)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint64_t adesc = tc::smem_desc_sw128(q_addr + koff, 16, 1024);
                    const uint64_t bdesc = tc::smem_desc_sw128(k_addr + s * C::kKVBytes + koff, 16, 1024);
                    tc::mma_f16_ss(tmem + C::kColS + b * kBN, adesc, bdesc, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc::commit(&bars.s_full[b]);
                if (j >= 1 && !issue_pv(j - 1)) {
                    ok = false;
                    break;
                }
            }
            if (ok) issue_pv(n_kv - 1);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // row of the tile this thread owns
        const int t = qb * kBM + r;         // position among the request's new tokens
        const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
        const float sink2 = a.sinks ? a.sinks[h] * kLog2e : -INFINITY;
        float m_used = sink2;                        // running max, seeded with the sink
        float l = sink2 == -INFINITY ? 0.f : 1.f;    // running denominator: e^(sink - m) = 1
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int b = j & 1;
            if (!wait_or_abort(&bars.s_full[b], (uint32_t)((j >> 1) & 1), s_abort, a.status)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            uint32_t sv[kBN];
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c)
                tc::ld_32x32b_x32(trow + C::kColS + b * kBN + c * 32,
                                  *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.s_free[b]);

            // visible keys of this tile for this row
            int ncols;
            if (j < n_pre)
                ncols = min(kBN, P - j * kBN);
            else if (j - n_pre == qb)
                ncols = r + 1;  // diagonal tile: keys 0..r
            else
                ncols = kBN;
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kBN; ++c)
                if (c < ncols) mx = fmaxf(mx, __uint_as_float(sv[c]));
            const float mt = mx * a.scale_log2;
            if (j == 0) {
                const float mn = fmaxf(m_used, mt);
                l = (m_used == -INFINITY) ? 0.f : l * fast_exp2(m_used - mn);
                m_used = mn;
            } else {
                const bool need = mt > m_used + kRescaleThreshold;
                if (__any_sync(0xffffffffu, need)) {
                    const float mn = fmaxf(m_used, mt);
                    const float alpha = need ? fast_exp2(m_used - mn) : 1.f;
                    if (need) {
                        l *= alpha;
                        m_used = mn;
                    }
                    // O must hold every P.V issued so far before it is rescaled
                    if (!wait_or_abort(&bars.p_empty[(j - 1) % NP], (uint32_t)(((j - 1) / NP) & 1),
                                       s_abort, a.status)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tc::ld_32x32b_x32(trow + C::kColO + c * 32, o);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc::st_32x32b_x32(trow + C::kColO + c * 32, o);
                    }
                    tc::wait_st();
                }
            }
            const float neg = m_used == -INFINITY ? 0.f : -m_used;
            const int pb = j % NP;
            // P buffer pb is free once the P.V of tile j - NP has completed
            if (j >= NP && !wait_or_abort(&bars.p_empty[pb], (uint32_t)(((j / NP) + 1) & 1), s_abort,
                                          a.status)) {
                ok = false;
                break;
            }
            uint8_t *pt = sP + pb * C::kPBytes;
            float sum = 0.f;
            // P is written as P_hi = bf16(p) and P_lo = bf16(p - P_hi); the bf16 rounding
            // of p alone (relative 2^-9) is too coarse for rows with few keys
#pragma unroll
            for (int c8 = 0; c8 < kBN / 8; ++c8) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int c = c8 * 8 + 2 * e;
                    const float p0 =
                        c < ncols ? fast_exp2(fmaf(__uint_as_float(sv[c]), a.scale_log2, neg)) : 0.f;
                    const float p1 =
                        c + 1 < ncols ? fast_exp2(fmaf(__uint_as_float(sv[c + 1]), a.scale_log2, neg)) : 0.f;
                    sum += p0 + p1;
                    hi[e] = pack_bf16x2(p0, p1);
                    lo[e] = pack_bf16x2(p0 - __uint_as_float(hi[e] << 16),
                                        p1 - __uint_as_float(hi[e] & 0xFFFF0000u));
                }
                const uint32_t o = (c8 >> 3) * 16384 + sw128(r, c8 & 7);
                *reinterpret_cast<uint4 *>(pt + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(pt + C::kPHalf + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            l += sum;
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.p_full[pb]);
        }
        // epilogue: O / l for this row
        if (ok && wait_or_abort(&bars.p_empty[(n_kv - 1) % NP], (uint32_t)(((n_kv - 1) / NP) & 1),
                                s_abort, a.status)) {
            tc::fence_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const bool valid = t < L && row0 >= 0 && row0 + t < a.T;
            __nv_bfloat16 *og = reinterpret_cast<__nv_bfloat16 *>(a.out) +
                                ((int64_t)(row0 + t) * a.Hq + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tc::ld_32x32b_x32(trow + C::kColO + c * 32, o);
                tc::wait_ld();
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 v;
                        v.x = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                        v.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                        v.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                        v.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                        *reinterpret_cast<uint4 *>(og + c * 32 + e) = v;
                    }
                }
            }
            if (valid && a.lse)
                a.lse[(int64_t)(row0 + t) * a.Hq + h] =
                    (l > 0.f) ? (m_used + log2f(l)) * kLn2 : -INFINITY;
        }
    }

    // all roles done: wait for the MMAs still in flight after an abort, then free TMEM
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        if (*s_abort && lane == 0) {
            // a final commit arrives once every MMA issued so far has completed
            tc::commit(bars.drain);
            mbar_wait(bars.drain, 0, 100000000ull);
        }
        __syncwarp();
        tc::fence_after_sync();
        tc::dealloc(tmem, kTmemCols);
    }
    if (warp == 0 && *s_abort) {
        // let any TMA copy still in flight land before the CTA's shared memory is released
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 50000000ull) __nanosleep(1000);
    }
}

template <int D>
cudaError_t launch_d(const PrefillArgs &a, const CUtensorMap &qmap, const CUtensorMap &kmap,
                     const CUtensorMap &vmap, const CUtensorMap &kpmap, const CUtensorMap &vpmap,
                     cudaStream_t stream) {
    using C = PrefillCfg<D>;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    // bound on the number of 128-row query blocks: sum_i ceil(L_i / 128) <= T / 128 + n
    const int64_t tiles = (int64_t)(a.T + kBM - 1) / kBM + a.n;
    const int64_t grid = tiles * a.Hq;
    if (grid > INT32_MAX) return cudaErrorInvalidConfiguration;
    prefill_kernel<D><<<(unsigned)grid, kThreads, C::kSmemBytes, stream>>>(qmap, kmap, vmap, kpmap,
                                                                           vpmap, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, const CUtensorMap &qmap, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, const CUtensorMap &kpmap,
                           const CUtensorMap &vpmap, cudaStream_t stream) {
    if (a.D == 64) return launch_d<64>(a, qmap, kmap, vmap, kpmap, vpmap, stream);
    if (a.D == 128) return launch_d<128>(a, qmap, kmap, vmap, kpmap, vpmap, stream);
    return cudaErrorNotSupported;
}

}  // namespace sinkattn
