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
// GB300 design.  A persistent grid (one CTA per SM) walks work items, heaviest
// first.  An item is one 128-row query block of one request for TWO query heads
// of the same KV head (tiles A and B), so every K/V tile in shared memory feeds
// two S = Q K^T products and the two softmax warpgroups run side by side while
// the tensor core alternates between them.  Key tiles: prefix tiles first, then
// the causal new-token tiles up to the diagonal; fully masked tiles are skipped.
//   warp 0      TMA producer: both Q tiles of an item, K and V tiles into a ring
//               of stages (new tokens: one 3-D box of 128 rows; prefix: 16-row page
//               boxes through the block table; a ragged or invalid page is copied
//               by the warp and zero-filled)
//   warp 1      owns TMEM; one thread issues S_x = Q_x K^T (M=128, N=128) and
//               O_x += P_x V (M=128, N=D, P read from TMEM)
//   warps 2..3  idle (they complete warpgroup 0, which hands registers to softmax)
//   warps 4..7  softmax of tile A, warps 8..11 softmax of tile B: one query row per
//               thread; the whole S row is read from TMEM once, P = exp2(s - m) is
//               written back over S as two bf16 halves P_hi + P_lo (bf16 P alone,
//               relative 2^-9, is too coarse for rows with few keys); O is rescaled
//               in TMEM only when the running max grows by more than 2^8.
// TMEM columns per tile x: S/P at [256x, 256x + 128), O at [256x + 128, 256x + 128 + D).
// MMAs issued by one thread complete in order, so when S_x(j) is complete the
// P.V of tile j - 1 has landed in O_x and P_x(j - 1) has been consumed.
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
constexpr int kThreads = 384;              // 12 warps = 3 warpgroups
// Register split: the kernel is built for 168 registers per thread (384 x 168 =
// 64512); warpgroup 0 (producer, MMA, two idle warps) gives up to 72 and the two
// softmax warpgroups take 216: 128 x 72 + 256 x 216 = 64512.  The build checks
// that ptxas used exactly 168.
constexpr uint32_t kRegsLaunch = 168, kRegsSide = 72, kRegsSoftmax = 216;
static_assert(128 * kRegsSide + 256 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr int kLocateMax = 1024;  // requests / levels of the shared-memory tile lookup

template <int D>
struct PrefillCfg {
    static constexpr int kHalves = D / 64;           // 128-byte column blocks
    static constexpr int kStages = D == 64 ? 4 : 2;  // K/V ring depth
    static constexpr int kQBytes = kBM * D * 2;      // one Q tile
    static constexpr int kKVBytes = kBN * D * 2;     // one K (or V) tile
    static constexpr int kOffQ = 0;                  // Q tiles A and B
    static constexpr int kOffK = kOffQ + 2 * kQBytes;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffBar = kOffV + kStages * kKVBytes;
    static constexpr int kNumBars = 2 + 3 * kStages + 8 + 1;
    static constexpr int kOffLoc = kOffBar + ((kNumBars * 8 + 127) / 128) * 128;
    static constexpr int kOffMisc = kOffLoc + 3 * kLocateMax * 4;
    static constexpr int kSmemBytes = 1024 + kOffMisc + 64;
    static constexpr uint32_t kColSP(int x) { return 256u * x; }
    static constexpr uint32_t kColO(int x) { return 256u * x + 128u; }
};

struct Bars {
    uint64_t *q_full, *q_empty, *k_full, *v_full, *kv_empty, *s_full, *p_full, *pv_done, *o_free,
        *drain;
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

// Work list.  Query blocks are ordered by their index inside the request (the
// number of causal key tiles they see), largest first, then by request, then by
// head (pair); items are dealt round-robin to the persistent CTAs.  Set-up, once
// per CTA: s_nq[i] = query blocks of request i; s_cnt[lev] = requests with more
// than lev query blocks; s_cum[lev] = query blocks at levels above lev.
struct WorkList {
    const int *nq, *cnt, *cum;
    int n, levels, tiles, heads_per_item, groups;  // groups = items per query block
    bool fast;
};

__device__ void worklist_setup(const PrefillArgs &a, int *s_nq, int *s_cnt, int *s_cum, int *s_misc,
                               WorkList *wl) {
    const int tid = threadIdx.x;
    const bool fast = a.n <= kLocateMax;
    if (tid == 0) s_misc[0] = 0;
    __syncthreads();
    int mx = 0;
    for (int i = tid; i < a.n; i += blockDim.x) {
        const int L = a.cu_seqlens[i + 1] - a.cu_seqlens[i];
        const int q = L > 0 ? (L + kBM - 1) / kBM : 0;
        if (fast) s_nq[i] = q;
        mx = max(mx, q);
    }
    atomicMax(&s_misc[0], mx);
    __syncthreads();
    const int levels = s_misc[0];
    const bool fast_lv = fast && levels <= kLocateMax;
    if (fast_lv)
        for (int lev = tid; lev < levels; lev += blockDim.x) {
            int c = 0;
            for (int i = 0; i < a.n; ++i) c += s_nq[i] > lev;
            s_cnt[lev] = c;
        }
    __syncthreads();
    if (tid == 0) {
        int tiles = 0;
        if (fast_lv) {
            for (int lev = levels - 1; lev >= 0; --lev) {
                s_cum[lev] = tiles;
                tiles += s_cnt[lev];
            }
        } else {
            for (int i = 0; i < a.n; ++i) {
                const int L = a.cu_seqlens[i + 1] - a.cu_seqlens[i];
                tiles += L > 0 ? (L + kBM - 1) / kBM : 0;
            }
        }
        s_misc[1] = tiles;
    }
    __syncthreads();
    wl->nq = s_nq;
    wl->cnt = s_cnt;
    wl->cum = s_cum;
    wl->n = a.n;
    wl->levels = levels;
    wl->tiles = s_misc[1];
    wl->heads_per_item = a.G >= 2 ? 2 : 1;
    wl->groups = a.Hq / wl->heads_per_item;
    wl->fast = fast_lv;
}

struct Item {
    int req, qb, h0;
};

// Item of a given rank (any thread; reads the set-up tables).
__device__ Item item_of(const PrefillArgs &a, const WorkList &wl, int rank) {
    Item it;
    const int tr = rank / wl.groups;
    it.h0 = (rank % wl.groups) * wl.heads_per_item;
    it.req = 0;
    it.qb = 0;
    if (wl.fast) {
        // the level holding tile rank tr: cum[lev] <= tr < cum[lev] + cnt[lev]; cum
        // decreases as lev grows, so this is the smallest lev with cum[lev] <= tr
        int lo = 0, hi = wl.levels - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (wl.cum[mid] <= tr)
                hi = mid;
            else
                lo = mid + 1;
        }
        int k = tr - wl.cum[lo];
        for (int i = 0; i < wl.n; ++i)
            if (wl.nq[i] > lo && k-- == 0) {
                it.req = i;
                break;
            }
        it.qb = lo;
        return it;
    }
    // slow path: walk levels from the top over global memory
    int mq = 0;
    for (int i = 0; i < a.n; ++i) {
        const int L = a.cu_seqlens[i + 1] - a.cu_seqlens[i];
        mq = max(mq, L > 0 ? (L + kBM - 1) / kBM : 0);
    }
    int r = tr;
    for (int lev = mq - 1; lev >= 0; --lev)
        for (int i = 0; i < a.n; ++i) {
            const int L = a.cu_seqlens[i + 1] - a.cu_seqlens[i];
            if (L > 0 && (L + kBM - 1) / kBM > lev && r-- == 0) {
                it.req = i;
                it.qb = lev;
                return it;
            }
        }
    return it;
}

struct ItemGeom {
    int row0, L, P, n_pre, n_kv, g;
};

__device__ __forceinline__ ItemGeom geom_of(const PrefillArgs &a, const Item &it) {
    ItemGeom q;
    q.row0 = a.cu_seqlens[it.req];
    q.L = a.cu_seqlens[it.req + 1] - q.row0;
    q.P = 0;
    if (a.prefix_lens) {
        q.P = a.prefix_lens[it.req];
        const int cap = a.max_pages * kPageSize;
        q.P = q.P < 0 ? 0 : (q.P > cap ? cap : q.P);
    }
    q.n_pre = (q.P + kBN - 1) / kBN;
    q.n_kv = q.n_pre + it.qb + 1;
    q.g = it.h0 / a.G;
    return q;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap kpmap,
                   const __grid_constant__ CUtensorMap vpmap, const PrefillArgs a) {
    using C = PrefillCfg<D>;
    constexpr int NS = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *sQ = smem + C::kOffQ;
    uint8_t *sK = smem + C::kOffK;
    uint8_t *sV = smem + C::kOffV;
    uint64_t *bb = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    Bars bars;
    bars.q_full = bb;
    bars.q_empty = bb + 1;
    bars.k_full = bb + 2;
    bars.v_full = bars.k_full + NS;
    bars.kv_empty = bars.v_full + NS;
    bars.s_full = bars.kv_empty + NS;
    bars.p_full = bars.s_full + 2;
    bars.pv_done = bars.p_full + 2;
    bars.o_free = bars.pv_done + 2;
    bars.drain = bars.o_free + 2;
    int *s_loc = reinterpret_cast<int *>(smem + C::kOffLoc);
    int *misc = reinterpret_cast<int *>(smem + C::kOffMisc);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(misc);
    volatile int *s_abort = misc + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    WorkList wl;
    worklist_setup(a, s_loc, s_loc + kLocateMax, s_loc + 2 * kLocateMax, misc + 4, &wl);
    const int n_items = wl.tiles * wl.groups;
    if ((int)blockIdx.x >= n_items) return;  // CTA-uniform, before any allocation
    const int ntiles = wl.heads_per_item;    // query tiles per item (1 or 2)

    if (tid == 0) {
        *s_abort = 0;
        mbar_init(bars.q_full, 1);
        mbar_init(bars.q_empty, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.kv_empty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&bars.s_full[x], 1);
            mbar_init(&bars.p_full[x], 4);
            mbar_init(&bars.pv_done[x], 1);
            mbar_init(&bars.o_free[x], 4);
        }
        mbar_init(bars.drain, 1);
        fence_mbar_init();
    }
    if (warp == 1) tc::alloc(s_tmem, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *s_tmem;

    if (warp == 0) {
        // ================================================================ producer
        reg_dealloc<kRegsSide>();
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
        }
        int kv = 0;  // key tiles loaded so far (ring position)
        int k = 0;   // items so far
        bool ok = true;
        for (int rank = blockIdx.x; ok && rank < n_items; rank += gridDim.x, ++k) {
            const Item it = item_of(a, wl, rank);
            const ItemGeom gm = geom_of(a, it);
            if (lane == 0 && a.prefix_lens) {
                const int Praw = a.prefix_lens[it.req];
                if (Praw < 0 || Praw > a.max_pages * kPageSize)
                    set_status(a.status, SINKATTN_STATUS_BAD_LENGTH);
            }
            // Q tiles of this item, once the previous item's last S products are done
            if (k > 0 && !wait_or_abort(bars.q_empty, (uint32_t)((k - 1) & 1), s_abort, a.status)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(bars.q_full, ntiles * C::kQBytes);
                for (int x = 0; x < ntiles; ++x)
#pragma unroll
                    for (int hf = 0; hf < C::kHalves; ++hf)
                        tma_load_3d(sQ + x * C::kQBytes + hf * 16384, &qmap, bars.q_full, hf * 64,
                                    it.h0 + x, gm.row0 + it.qb * kBM);
            }
            for (int j = 0; j < gm.n_kv; ++j, ++kv) {
                const int s = kv % NS, u = kv / NS;
                if (u > 0 &&
                    !wait_or_abort(&bars.kv_empty[s], (uint32_t)((u - 1) & 1), s_abort, a.status)) {
                    ok = false;
                    break;
                }
                uint8_t *kt = sK + s * C::kKVBytes;
                uint8_t *vt = sV + s * C::kKVBytes;
                if (j < gm.n_pre) {
                    // eight pages of 16 tokens; whole valid pages by TMA, the rest by the warp
                    uint32_t nfull = 0;
#pragma unroll
                    for (int pp = 0; pp < 8; ++pp) {
                        const int page = j * 8 + pp;
                        const int nrow = min(kPageSize, max(0, gm.P - page * kPageSize));
                        if (nrow > 0) {
                            const int pg = a.prefix_block_table[(int64_t)it.req * a.max_pages + page];
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
                        const int page = j * 8 + pp;
                        const int nrow = min(kPageSize, max(0, gm.P - page * kPageSize));
                        int pg = -1;
                        if (nrow > 0) {
                            pg = a.prefix_block_table[(int64_t)it.req * a.max_pages + page];
                            if (pg < 0 || pg >= a.num_pages) pg = -1;
                        }
                        if (nrow == kPageSize && pg >= 0) {
                            if (lane == 0) {
#pragma unroll
                                for (int hf = 0; hf < C::kHalves; ++hf) {
                                    tma_load_4d(kt + hf * 16384 + pp * 2048, &kpmap, &bars.k_full[s],
                                                hf * 64, 0, gm.g, pg);
                                    tma_load_4d(vt + hf * 16384 + pp * 2048, &vpmap, &bars.v_full[s],
                                                hf * 64, 0, gm.g, pg);
                                }
                            }
                        } else {
                            // ragged or invalid page: copy the valid rows, zero the rest
                            const int nv = pg >= 0 ? nrow : 0;
                            const __nv_bfloat16 *kg = reinterpret_cast<const __nv_bfloat16 *>(a.k_pages);
                            const __nv_bfloat16 *vg = reinterpret_cast<const __nv_bfloat16 *>(a.v_pages);
                            for (int e = lane; e < kPageSize * C::kHalves * 8; e += 32) {
                                const int slot = e / (C::kHalves * 8);
                                const int hf = (e / 8) % C::kHalves;
                                const int c = e % 8;
                                uint4 kx = make_uint4(0, 0, 0, 0), vx = make_uint4(0, 0, 0, 0);
                                if (slot < nv) {
                                    const int64_t off =
                                        (((int64_t)pg * a.Hkv + gm.g) * kPageSize + slot) * D + hf * 64 + c * 8;
                                    kx = *reinterpret_cast<const uint4 *>(kg + off);
                                    vx = *reinterpret_cast<const uint4 *>(vg + off);
                                }
                                const uint32_t o = hf * 16384 + sw128(pp * kPageSize + slot, c);
                                *reinterpret_cast<uint4 *>(kt + o) = kx;
                                *reinterpret_cast<uint4 *>(vt + o) = vx;
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
                    const int row = gm.row0 + (j - gm.n_pre) * kBN;
                    mbar_arrive_expect_tx(&bars.k_full[s], C::kKVBytes);
#pragma unroll
                    for (int hf = 0; hf < C::kHalves; ++hf)
                        tma_load_3d(kt + hf * 16384, &kmap, &bars.k_full[s], hf * 64, gm.g, row);
                    mbar_arrive_expect_tx(&bars.v_full[s], C::kKVBytes);
#pragma unroll
                    for (int hf = 0; hf < C::kHalves; ++hf)
                        tma_load_3d(vt + hf * 16384, &vmap, &bars.v_full[s], hf * 64, gm.g, row);
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        reg_dealloc<kRegsSide>();
        if (lane == 0) {
            constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kBM, kBN, false);
            constexpr uint32_t idesc_o = tc::idesc_bf16_f32(kBM, D, true);
            const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV);
            int kv = 0;                   // key tiles consumed so far (ring position)
            uint32_t tcount[2] = {0, 0};  // tiles processed per query tile x (barrier phases)
            int k = 0;
            bool ok = true;
            auto issue_s = [&](int x, int s) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    const uint64_t adesc = tc::smem_desc_sw128(q_addr + x * C::kQBytes + off, 16, 1024);
                    const uint64_t bdesc = tc::smem_desc_sw128(k_addr + s * C::kKVBytes + off, 16, 1024);
                    tc::mma_f16_ss(tmem + C::kColSP(x), adesc, bdesc, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc::commit(&bars.s_full[x]);
            };
            for (int rank = blockIdx.x; ok && rank < n_items; rank += gridDim.x, ++k) {
                const Item it = item_of(a, wl, rank);
                const ItemGeom gm = geom_of(a, it);
                if (!wait_or_abort(bars.q_full, (uint32_t)(k & 1), s_abort, a.status)) {
                    ok = false;
                    break;
                }
                // first key tile: S for every query tile
                {
                    const int s = kv % NS, u = kv / NS;
                    if (!wait_or_abort(&bars.k_full[s], (uint32_t)(u & 1), s_abort, a.status)) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    for (int x = 0; x < ntiles; ++x) issue_s(x, s);
                    if (gm.n_kv == 1) tc::commit(bars.q_empty);
                }
                for (int j = 0; ok && j < gm.n_kv; ++j) {
                    const int s = (kv + j) % NS, u = (kv + j) / NS;
                    const int s1 = (kv + j + 1) % NS, u1 = (kv + j + 1) / NS;
                    if (!wait_or_abort(&bars.v_full[s], (uint32_t)(u & 1), s_abort, a.status)) {
                        ok = false;
                        break;
                    }
                    for (int x = 0; x < ntiles; ++x) {
                        if (!wait_or_abort(&bars.p_full[x], tcount[x] & 1, s_abort, a.status)) {
                            ok = false;
                            break;
                        }
                        ++tcount[x];
                        if (j == 0 && k > 0 &&
                            !wait_or_abort(&bars.o_free[x], (uint32_t)((k - 1) & 1), s_abort, a.status)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        // O_x += P_hi V + P_lo V; P chunk c (keys 32c..32c+31): hi in columns
                        // 32c..32c+15, lo in 32c+16..32c+31 of the tile's S/P region
#pragma unroll
                        for (int part = 0; part < 2; ++part)
#pragma unroll
                            for (int kk = 0; kk < kBN / 16; ++kk) {
                                const uint32_t acol =
                                    C::kColSP(x) + 32 * (kk >> 1) + 8 * (kk & 1) + 16 * part;
                                const uint64_t bdesc =
                                    tc::smem_desc_sw128(v_addr + s * C::kKVBytes + kk * 2048, 16384, 1024);
                                tc::mma_f16_ts(tmem + C::kColO(x), tmem + acol, bdesc, idesc_o,
                                               (j > 0 || part > 0 || kk > 0) ? 1u : 0u);
                            }
                        if (j == gm.n_kv - 1) tc::commit(&bars.pv_done[x]);
                        if (j + 1 < gm.n_kv) {
                            if (x == 0 &&
                                !wait_or_abort(&bars.k_full[s1], (uint32_t)(u1 & 1), s_abort, a.status)) {
                                ok = false;
                                break;
                            }
                            tc::fence_after_sync();
                            issue_s(x, s1);
                            if (j + 1 == gm.n_kv - 1 && x == ntiles - 1) tc::commit(bars.q_empty);
                        }
                    }
                    if (!ok) break;
                    tc::commit(&bars.kv_empty[s]);
                }
                kv += gm.n_kv;
            }
        }
        __syncwarp();
    } else if (warp < 4) {
        reg_dealloc<kRegsSide>();  // idle warps of warpgroup 0
    } else {
        // ================================================================ softmax
        reg_alloc<kRegsSoftmax>();
        const int x = (warp - 4) >> 2;  // query tile of this warpgroup
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // tile row of this thread
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t tsp = tmem + lane_base + C::kColSP(x);
        const uint32_t tO = tmem + lane_base + C::kColO(x);
        uint32_t tcount = 0;
        int k = 0;
        bool ok = x < ntiles;
        for (int rank = blockIdx.x; ok && rank < n_items; rank += gridDim.x, ++k) {
            const Item it = item_of(a, wl, rank);
            const ItemGeom gm = geom_of(a, it);
            const int h = it.h0 + x;
            const int t = it.qb * kBM + r;  // position among the request's new tokens
            const float sink2 = a.sinks ? a.sinks[h] * kLog2e : -INFINITY;
            float m_used = sink2;                      // running max, seeded with the sink
            float l = sink2 == -INFINITY ? 0.f : 1.f;  // running denominator: e^(sink - m) = 1
            for (int j = 0; j < gm.n_kv; ++j) {
                if (!wait_or_abort(&bars.s_full[x], tcount & 1, s_abort, a.status)) {
                    ok = false;
                    break;
                }
                ++tcount;
                tc::fence_after_sync();
                int ncols;  // keys of this tile the row may see
                if (j < gm.n_pre)
                    ncols = min(kBN, gm.P - j * kBN);
                else if (j - gm.n_pre == it.qb)
                    ncols = r + 1;  // diagonal tile: keys 0..r
                else
                    ncols = kBN;
                // the whole S row of this tile
                uint32_t sv[kBN];
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c)
                    tc::ld_32x32b_x32(tsp + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
                tc::wait_ld();
                if (ncols < kBN) {  // diagonal, ragged or prefix-tail tile: hide invisible keys
#pragma unroll
                    for (int c = 0; c < kBN; ++c)
                        if (c >= ncols) sv[c] = 0xFF800000u;  // -inf
                }
                float mx8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mx8[e] = __uint_as_float(sv[e]);
#pragma unroll
                for (int c = 8; c < kBN; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], __uint_as_float(sv[c]));
                const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                const float mt = mx * a.scale_log2;
                if (j == 0) {
                    const float mn = fmaxf(m_used, mt);
                    l = (m_used == -INFINITY) ? 0.f : l * fast_exp2(m_used - mn);
                    m_used = mn;
                } else {
                    const bool need = mt > m_used + kRescaleThreshold;
                    if (__any_sync(0xffffffffu, need)) {
                        // O_x holds every earlier P.V: S_x(j) was issued after them
                        const float mn = fmaxf(m_used, mt);
                        const float alpha = need ? fast_exp2(m_used - mn) : 1.f;
                        if (need) {
                            l *= alpha;
                            m_used = mn;
                        }
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t o[32];
                            tc::ld_32x32b_x32(tO + c * 32, o);
                            tc::wait_ld();
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tc::st_32x32b_x32(tO + c * 32, o);
                        }
                    }
                }
                // P = exp2(s * scale - m), written back over S: per 32 keys, 16 columns of
                // P_hi = P with its low 16 bits cleared, then 16 columns of P_lo = bf16(P - P_hi)
                const float neg = m_used == -INFINITY ? 0.f : -m_used;
                float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ch = 0; ch < kBN / 32; ++ch) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int c = ch * 32 + 2 * e;
                        const float p0 = fast_exp2(fmaf(__uint_as_float(sv[c]), a.scale_log2, neg));
                        const float p1 = fast_exp2(fmaf(__uint_as_float(sv[c + 1]), a.scale_log2, neg));
                        sum8[(2 * e) & 7] += p0;
                        sum8[(2 * e + 1) & 7] += p1;
                        const uint32_t t0 = __float_as_uint(p0) & 0xFFFF0000u;
                        const uint32_t t1 = __float_as_uint(p1) & 0xFFFF0000u;
                        hi[e] = (t0 >> 16) | t1;  // exact: both are bf16 values already
                        lo[e] = pack_bf16x2(p0 - __uint_as_float(t0), p1 - __uint_as_float(t1));
                    }
                    tc::st_32x32b_x16(tsp + ch * 32, hi);
                    tc::st_32x32b_x16(tsp + ch * 32 + 16, lo);
                }
                l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.p_full[x]);
            }
            if (!ok) break;
            // epilogue: O / l for this row, once the item's last P.V has landed
            if (!wait_or_abort(&bars.pv_done[x], (uint32_t)(k & 1), s_abort, a.status)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const bool valid = t < gm.L && gm.row0 >= 0 && gm.row0 + t < a.T;
            __nv_bfloat16 *og = reinterpret_cast<__nv_bfloat16 *>(a.out) +
                                ((int64_t)(gm.row0 + t) * a.Hq + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tc::ld_32x32b_x32(tO + c * 32, o);
                tc::wait_ld();
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                        *reinterpret_cast<uint4 *>(og + c * 32 + e) = w;
                    }
                }
            }
            if (valid && a.lse)
                a.lse[(int64_t)(gm.row0 + t) * a.Hq + h] = (l > 0.f) ? (m_used + log2f(l)) * kLn2 : -INFINITY;
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.o_free[x]);
        }
    }

    // all roles done: after an abort wait for MMAs still in flight, then free TMEM
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        if (*s_abort && lane == 0) {
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
    int device = 0, sms = 0;
    if ((e = cudaGetDevice(&device)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess) return e;
    // persistent: one CTA per SM (shared memory and the 512 TMEM columns allow no more)
    prefill_kernel<D><<<sms, kThreads, C::kSmemBytes, stream>>>(qmap, kmap, vmap, kpmap, vpmap, a);
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
