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
// GB300 design.  A persistent grid (one CTA per SM) takes work items, heaviest first,
// from a counter shared by the grid.  An item is one 128-row query block of one request
// for TWO query heads of the same KV head (tiles A and B), so every K/V tile in shared memory feeds
// two S = Q K^T products and the two softmax warpgroups run side by side while
// the tensor core alternates between them.  Key tiles: prefix tiles first, then
// the causal new-token tiles up to the diagonal; fully masked tiles are skipped.
//   warp 0      TMA producer: both Q tiles of an item, K and V tiles into a ring
//               of stages (new tokens: one 3-D box of 128 rows; prefix: 16-row page
//               boxes through the block table; a ragged or invalid page is copied
//               by the warp and zero-filled)
//   warp 1      owns TMEM; issues O_x += P_x V (M=128, N=D, P read from TMEM, fp16)
//   warp 2      issues S_x = Q_x K^T (M=128, N=128, bf16) into the next free S/P buffer
//   warp 3      idle
//   warps 4..7  softmax of tile A, warps 8..11 softmax of tile B: one query row per
//               thread; the whole S row is read from TMEM once, and P = exp2(s - m) * 2^k
//               is written to TMEM in fp16 (bf16 P, relative 2^-9, is too coarse for rows
//               with few keys; fp16 keeps 2^-12).  The running max m is taken from an
//               item's first key tile; later tiles compute P against it at once, and only a
//               row whose P values then sum past 2^8 (a score risen by more than 8 in log2
//               units) takes its maximum, rescales O in TMEM and writes its P again.
//   warps 12..15 convert each V tile in shared memory from bf16 to fp16, one 32-key
//               quarter per warp (one warp per SM sub-partition), each quarter scaled by
//               its own power of two 2^-k that keeps it in fp16 range (k = 0 unless
//               |v| >= 2^15); the softmax multiplies P by 2^k over the same 32 keys.
// TMEM columns.  S products are numbered i = 0, 1, ... over the CTA's lifetime (key tile
// by key tile, query tile x = i % ntiles).  At head_dim 64: two S buffers of 128 columns,
// two P buffers of 64 (fp16 pairs), O_A and O_B of 64.  S(i) goes to S buffer i % 2 as
// soon as the softmax has copied S(i - 2) into registers, and P(i) to P buffer i % 2 once
// the P.V of product i - 2 has completed, so the tensor core computes the next S products
// while the softmax works.  At head_dim 128 (O_A and O_B take 256 columns) P is written
// over S in two S/P buffers, and S(i) waits for the P.V of product i - 2.
#include <float.h>

#include "internal.h"
#include "ptx.cuh"

namespace sinkattn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kPSumLimit = 256.0f;  // P values (times 2^-k) stay at most 2^8
constexpr int kBM = 128;                   // query rows per tile
constexpr int kBN = 128;                   // keys per tile
constexpr int kThreads = 512;              // 16 warps = 4 warpgroups
// Register split: the kernel is built for 128 registers per thread (512 x 128 =
// 65536); warpgroup 0 (producer, MMA issuers) drops to 48, warpgroup 3 (V converters)
// to 32, and the two softmax warpgroups take 216: 128 x 48 + 128 x 32 + 256 x 216 =
// 65536.  The build checks that ptxas used exactly 128.
constexpr uint32_t kRegsLaunch = 128, kRegsSide = 48, kRegsConvert = 32, kRegsSoftmax = 216;
static_assert(128 * kRegsSide + 128 * kRegsConvert + 256 * kRegsSoftmax <= kThreads * kRegsLaunch,
              "register split");
constexpr uint32_t kTmemCols = 512;
constexpr int kLocateMax = 1024;  // requests / levels of the shared-memory tile lookup
// Items reach the CTA's roles through a ring of slots.  Every role is within a few items of
// the producer (it loads a K/V stage only after the P.V that last read it, which follows that
// tile's S product, softmax and V conversion; a Q tile only after the last S product of the
// item before), at most the ring depth of NS <= 4 tiles, so a slot is read by every role before
// the producer posts to it again.
constexpr int kItemRing = 16;

// QB: Q buffers.  Two at head_dim 64 with a sliding window, where items are one or two key
// tiles long: the next item's Q tiles load while the current item's S products still read
// its own (measured: 12 % faster window-128 prefill; 2 % slower causal prefill, whose longer
// items hide the Q load, so one buffer there).
template <int D, int QB = 1>
struct PrefillCfg {
    static constexpr int kHalves = D / 64;           // 128-byte column blocks
    static constexpr int kStages = D == 64 ? 4 : 2;  // K/V ring depth
    static constexpr int kQBytes = kBM * D * 2;      // one Q tile
    static constexpr int kKVBytes = kBN * D * 2;     // one K (or V) tile
    static constexpr int kQBufs = QB;                // Q buffers (items in flight)
    static constexpr int kOffQ = 0;                  // Q tiles A and B of each buffer
    static constexpr int kOffK = kOffQ + kQBufs * 2 * kQBytes;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffBar = kOffV + kStages * kKVBytes;
    static constexpr bool kSplitP = D == 64;         // P in buffers of its own (else over S)
    static constexpr int kSBufs = 2;                 // S buffers (128 columns, fp32)
    static constexpr int kPBufs = 2;                 // P buffers (64 columns of fp16 pairs)
    static constexpr int kNumBars = 2 * kQBufs + 5 * kStages + 2 * kSBufs + 2 * kPBufs + 2 + 1 + kItemRing;
    static constexpr int kOffLoc = kOffBar + ((kNumBars * 8 + 127) / 128) * 128;
    static constexpr int kOffMisc = kOffLoc + 4 * kLocateMax * 4;
    static constexpr int kOffSlot = kOffMisc + 256;  // [kItemRing] ItemSlot, 64 bytes each
    static constexpr int kSmemBytes = 1024 + kOffSlot + kItemRing * 64;
    __host__ __device__ static constexpr uint32_t kColS(int b) { return 128u * b; }
    __host__ __device__ static constexpr uint32_t kColP(int p) {
        return kSplitP ? 128u * kSBufs + 64u * p : 128u * p;
    }
    __host__ __device__ static constexpr uint32_t kColO(int x) {
        return (kSplitP ? 128u * kSBufs + 64u * kPBufs : 128u * kSBufs) + D * x;
    }
    static_assert(kSplitP || kSBufs == kPBufs, "P over S needs one P buffer per S buffer");
    // FP8 prefix pages (E4M3 codes, D bytes a row) are staged inside the stage they are
    // converted into: page p of a tile in the bytes its own converted rows end in, so one
    // warp converts a page in place (keys 16p .. 16p + 15: bf16 / fp16 rows of 128 bytes,
    // one such block per 64 columns).
    __host__ __device__ static constexpr uint32_t kOffFp8Page(int p) {
        return D == 64 ? 2048u * p + 1024u : 16384u + 2048u * p;
    }
    static_assert(kColO(2) <= 512, "TMEM columns");
};

struct Bars {
    uint64_t *q_full, *q_empty, *k_full, *v_full, *v_conv, *k_conv, *kv_empty, *s_full, *s_free,
        *p_full, *pv_done, *o_free, *drain, *item_full;
};

// Bounded wait (limit_cycles SM cycles: the call's wait limit, converted on the host) that also
// gives up as soon as another role has given up.  With kSleep the thread sleeps in the wait
// (for warps off the critical path: it leaves the issue slots to the softmax warps, at ~50
// cycles more wake-up latency).  The lanes of a converged warp test the same barrier in the
// same instruction and read the same flag and clock, so they come to the same answer; the
// MMA-issuing and converter warps also vote on it (warp_wait, the converter loop).  The
// fast path is one blocking probe: measured, a vote inside the wait cost the prefill 18 %,
// a non-blocking first probe 5-20 %, and any branch ahead of the first probe (such as one
// for the testing limit) 25-45 %, so the testing setting is handled by the producer instead.
template <bool kSleep = false>
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort,
                                              uint32_t *status, uint64_t limit_cycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = clock64();
    for (;;) {
        if (kSleep) {
            if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
        } else {
            for (int i = 0; i < 128; ++i)
                if (mbar_try_wait(bar, parity)) return true;
        }
        if (*abort) return false;
        if ((uint64_t)clock64() - t0 >= limit_cycles) {
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


// ---------------------------------------------------------------- FP8 prefix conversion
// Two f16 values (a packed pair) to a bf16 pair (exact for E4M3 values).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
    float lo, hi;
    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, u;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
    return pack_bf16x2(lo, hi);
}
// Two f16 values times sc, rounded to an f16 pair.
__device__ __forceinline__ uint32_t f16x2_scaled(uint32_t h, float sc) {
    float lo, hi;
    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, u;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
    return pack_f16x2(lo * sc, hi * sc);
}

// Two f16 values times a power of two (given as an f16 pair), exact when the results stay
// f16 normals or exact subnormals.
__device__ __forceinline__ uint32_t f16x2_pow2(uint32_t h, uint32_t p2) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(p2));
    return r;
}

// Eight E4M3 codes (two words) to one 16-byte vector: bf16 code values (kMode 0), fp16 code
// values times sc (1), or fp16 code values times the power of two p2 (2).
template <int kMode>
__device__ __forceinline__ uint4 codes8(uint32_t w0, uint32_t w1, float sc, uint32_t p2) {
    const uint32_t h0 = e4m3x2_lo_to_f16x2(w0), h1 = e4m3x2_hi_to_f16x2(w0);
    const uint32_t h2 = e4m3x2_lo_to_f16x2(w1), h3 = e4m3x2_hi_to_f16x2(w1);
    if (kMode == 0) return make_uint4(f16x2_to_bf16x2(h0), f16x2_to_bf16x2(h1), f16x2_to_bf16x2(h2), f16x2_to_bf16x2(h3));
    if (kMode == 2) return make_uint4(f16x2_pow2(h0, p2), f16x2_pow2(h1, p2), f16x2_pow2(h2, p2), f16x2_pow2(h3, p2));
    return make_uint4(f16x2_scaled(h0, sc), f16x2_scaled(h1, sc), f16x2_scaled(h2, sc), f16x2_scaled(h3, sc));
}

// One converter warp's quarter of an FP8 prefix tile (keys 32q .. 32q + 31, pages 2q and
// 2q + 1) from its staged codes to 128-byte swizzled rows in place: bf16 code values for K,
// fp16 code values times sc (kMode 1) or times the power of two p2 (kMode 2) for V.  Every
// lane reads its codes of a page (or half page) before any lane writes, since the rows
// written cover the codes staged.
template <int D, int kMode>
__device__ __forceinline__ void convert_fp8_quarter(uint8_t *t, int q, int lane, float sc, uint32_t p2 = 0) {
    using C = PrefillCfg<D>;
#pragma unroll 1
    for (int i = 0; i < 2; ++i) {
        const int p = 2 * q + i;
        const uint8_t *src = t + C::kOffFp8Page(p);
        if (D == 64) {
            // lane: row r, codes 32h .. 32h + 31 -> 16-byte chunks 4h .. 4h + 3 of row 16p + r
            const int r = lane >> 1, h = lane & 1;
            const uint4 x = *reinterpret_cast<const uint4 *>(src + r * 64 + h * 32);
            const uint4 y = *reinterpret_cast<const uint4 *>(src + r * 64 + h * 32 + 16);
            __syncwarp();
            *reinterpret_cast<uint4 *>(t + sw128(16 * p + r, 4 * h + 0)) = codes8<kMode>(x.x, x.y, sc, p2);
            *reinterpret_cast<uint4 *>(t + sw128(16 * p + r, 4 * h + 1)) = codes8<kMode>(x.z, x.w, sc, p2);
            *reinterpret_cast<uint4 *>(t + sw128(16 * p + r, 4 * h + 2)) = codes8<kMode>(y.x, y.y, sc, p2);
            *reinterpret_cast<uint4 *>(t + sw128(16 * p + r, 4 * h + 3)) = codes8<kMode>(y.z, y.w, sc, p2);
        } else {
            // two passes of eight rows: lane: row r, codes 32 h4 .. 32 h4 + 31 -> column block
            // h4 / 2, chunks 4 (h4 % 2) .. + 3 (the rows of block 1 are where the codes sit)
#pragma unroll 1
            for (int ps = 0; ps < 2; ++ps) {
                const int r = ps * 8 + (lane >> 2), h4 = lane & 3;
                const uint4 x = *reinterpret_cast<const uint4 *>(src + r * 128 + h4 * 32);
                const uint4 y = *reinterpret_cast<const uint4 *>(src + r * 128 + h4 * 32 + 16);
                __syncwarp();
                uint8_t *blk = t + (h4 >> 1) * 16384;
                const int c0 = 4 * (h4 & 1);
                *reinterpret_cast<uint4 *>(blk + sw128(16 * p + r, c0 + 0)) = codes8<kMode>(x.x, x.y, sc, p2);
                *reinterpret_cast<uint4 *>(blk + sw128(16 * p + r, c0 + 1)) = codes8<kMode>(x.z, x.w, sc, p2);
                *reinterpret_cast<uint4 *>(blk + sw128(16 * p + r, c0 + 2)) = codes8<kMode>(y.x, y.y, sc, p2);
                *reinterpret_cast<uint4 *>(blk + sw128(16 * p + r, c0 + 3)) = codes8<kMode>(y.z, y.w, sc, p2);
                __syncwarp();
            }
        }
    }
}

// Work list, in two parts.  (A) Requests with a paged prefix, request by request (each
// request's query blocks from the last to the first, then by head pair): the items that
// read one request's prefix run close together in time and share its pages in L2.
// (B) Requests without a prefix: query blocks ordered by their index inside the request
// (the number of causal key tiles they see), largest first, then by request, then by head
// pair.  Without the causal mask every block of a request sees all of its key tiles: the
// requests are taken from the most blocks to the fewest, each one's blocks in order, then
// by head pair.  The persistent CTAs take items in this order from a counter in the workspace
// header, each as its producer gets to it, so a CTA that ran faster takes more of them.
// Set-up, once per CTA: s_nq[i] = query blocks of request i if it is in part B, else 0;
// s_aend[i] = part-A query blocks of requests 0..i; s_cnt[lev] = part-B requests with more
// than lev query blocks (non-causal: the blocks of the requests of exactly lev + 1 blocks);
// s_cum[lev] = part-B query blocks at levels above lev.
struct WorkList {
    const int *nq, *cnt, *cum, *aend;
    int n, levels, tiles, tiles_a, heads_per_item, groups;  // groups = items per query block
    bool fast;
};

__device__ __forceinline__ int query_blocks(const PrefillArgs &a, int i) {
    const int L = a.cu_seqlens[i + 1] - a.cu_seqlens[i];
    return L > 0 ? (L + kBM - 1) / kBM : 0;
}

__device__ __forceinline__ bool has_prefix(const PrefillArgs &a, int i) {
    return a.prefix_lens != nullptr && a.prefix_lens[i] > 0;
}

__device__ void worklist_setup(const PrefillArgs &a, int *s_nq, int *s_cnt, int *s_cum, int *s_aend,
                               int *s_misc, WorkList *wl) {
    const int tid = threadIdx.x;
    const bool fast = a.n <= kLocateMax;
    if (tid == 0) s_misc[0] = 0;
    __syncthreads();
    int mx = 0;
    for (int i = tid; i < a.n; i += blockDim.x) {
        const int q = query_blocks(a, i);
        const bool pa = has_prefix(a, i);
        if (fast) {
            s_nq[i] = pa ? 0 : q;
            s_aend[i] = pa ? q : 0;  // made inclusive below
        }
        mx = max(mx, pa ? 0 : q);
    }
    atomicMax(&s_misc[0], mx);
    __syncthreads();
    const int levels = s_misc[0];
    const bool fast_lv = fast && levels <= kLocateMax;
    if (fast && tid < 32) {
        // inclusive prefix sum of s_aend by warp 0: lane l sums a contiguous chunk, the
        // chunk totals are scanned across the warp, then each lane adds its offset
        const int per = (a.n + 31) / 32, i0 = min(a.n, tid * per), i1 = min(a.n, i0 + per);
        int run = 0;
        for (int i = i0; i < i1; ++i) {
            run += s_aend[i];
            s_aend[i] = run;
        }
        int incl = run;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, d);
            if (tid >= d) incl += v;
        }
        const int off = incl - run;
        for (int i = i0; i < i1; ++i) s_aend[i] += off;
    }
    if (fast_lv)
        for (int lev = tid; lev < levels; lev += blockDim.x) {
            int c = 0;
            if (a.causal)
                for (int i = 0; i < a.n; ++i) c += s_nq[i] > lev;
            else  // non-causal: level lev holds every block of the requests of lev + 1 blocks
                for (int i = 0; i < a.n; ++i) c += s_nq[i] == lev + 1 ? lev + 1 : 0;
            s_cnt[lev] = c;
        }
    __syncthreads();
    if (tid == 0) {
        int tiles_a = 0, tiles_b = 0;
        if (fast_lv) {
            tiles_a = a.n > 0 ? s_aend[a.n - 1] : 0;
            for (int lev = levels - 1; lev >= 0; --lev) {
                s_cum[lev] = tiles_b;
                tiles_b += s_cnt[lev];
            }
        } else {
            for (int i = 0; i < a.n; ++i) {
                if (has_prefix(a, i))
                    tiles_a += query_blocks(a, i);
                else
                    tiles_b += query_blocks(a, i);
            }
        }
        s_misc[1] = tiles_a + tiles_b;
        s_misc[2] = tiles_a;
    }
    __syncthreads();
    wl->nq = s_nq;
    wl->cnt = s_cnt;
    wl->cum = s_cum;
    wl->aend = s_aend;
    wl->n = a.n;
    wl->levels = levels;
    wl->tiles = s_misc[1];
    wl->tiles_a = s_misc[2];
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
    int tr = rank / wl.groups;
    it.h0 = (rank % wl.groups) * wl.heads_per_item;
    it.req = 0;
    it.qb = 0;
    if (tr < wl.tiles_a) {
        // part A: the request whose query blocks hold tile rank tr, then its blocks from
        // the last one down
        int i = 0, before = 0;
        if (wl.fast) {
            // smallest i with aend[i] > tr (aend does not decrease)
            int lo = 0, hi = wl.n - 1;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (wl.aend[mid] > tr)
                    hi = mid;
                else
                    lo = mid + 1;
            }
            i = lo;
            before = i > 0 ? wl.aend[i - 1] : 0;
            it.qb = wl.aend[i] - 1 - tr;  // blocks of request i: aend[i] - before
        } else {
            for (i = 0; i < a.n; ++i) {
                const int q = has_prefix(a, i) ? query_blocks(a, i) : 0;
                if (tr < before + q) break;
                before += q;
            }
            it.qb = before + query_blocks(a, i) - 1 - tr;
        }
        it.req = i;
        return it;
    }
    tr -= wl.tiles_a;
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
        if (a.causal) {
            for (int i = 0; i < wl.n; ++i)
                if (wl.nq[i] > lo && k-- == 0) {
                    it.req = i;
                    break;
                }
            it.qb = lo;
        } else {
            // the (k / (lo + 1))-th request of lo + 1 blocks, its block k % (lo + 1)
            it.qb = k % (lo + 1);
            k /= lo + 1;
            for (int i = 0; i < wl.n; ++i)
                if (wl.nq[i] == lo + 1 && k-- == 0) {
                    it.req = i;
                    break;
                }
        }
        return it;
    }
    // slow path: walk the levels of part B from the top over global memory
    int mq = 0;
    for (int i = 0; i < a.n; ++i)
        if (!has_prefix(a, i)) mq = max(mq, query_blocks(a, i));
    int r = tr;
    for (int lev = mq - 1; lev >= 0; --lev)
        for (int i = 0; i < a.n; ++i) {
            if (has_prefix(a, i)) continue;
            const int q = query_blocks(a, i);
            if (a.causal ? q > lev && r-- == 0 : q == lev + 1 && r < q) {
                it.req = i;
                it.qb = a.causal ? lev : r;
                return it;
            }
            if (!a.causal && q == lev + 1) r -= q;
        }
    return it;
}

// A CTA has taken its last item: count it; the last CTA of the grid puts the work-list
// counters back to zero for the next call on this workspace (calls on one workspace are
// ordered on the GPU).  Every item fetch of every CTA comes before its count.
__device__ __forceinline__ void cta_done(uint32_t *sched) {
    __threadfence();
    if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
        sched[0] = 0;
        sched[1] = 0;
        __threadfence();
    }
}

// Key tiles of an item: prefix tiles 0..n_pre-1 (keys 128t .. 128t+127 of the prefix),
// then the new-token tiles n_pre + k (keys P + 128k ..), up to the diagonal n_pre + qb.
// A sliding window hides every tile before t0 from all 128 rows: the item visits tiles
// t0 .. n_pre + qb, n_kv of them.  Without the causal mask (an encoder's attention: no
// prefix, no window) the item visits all new-token tiles of its request.
struct ItemGeom {
    int row0, L, P, n_pre, t0, n_kv, g;
};

template <bool kWindow, bool kCausal>
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
    q.t0 = 0;
    if (kWindow) {
        // first key the block's first row sees: its position P + 128 qb, minus W - 1
        const int lb = q.P + it.qb * kBM - a.window + 1;
        if (lb > 0) q.t0 = lb < q.P ? lb / kBN : q.n_pre + (lb - q.P) / kBN;
    }
    // non-causal (no prefix, no window): every new-token tile of the request
    q.n_kv = kCausal ? q.n_pre + it.qb + 1 - q.t0 : (q.L + kBN - 1) / kBN;
    q.g = it.h0 / a.G;
    return q;
}

// What the producer posts for an item: its rank and what the other roles derive from it, so
// that they read it from shared memory instead of computing it again from global memory.
struct alignas(16) ItemSlot {
    int rank;           // >= n_items: no more items
    Item it;
    ItemGeom gm;
    float sink2[2];     // per query tile: sink * log2(e), -inf without sinks
    float kscale, vscale;  // FP8 prefix: the KV head's scales (1 if not given)
};
static_assert(sizeof(ItemSlot) == 64, "item slot");

// kWindow: a sliding window is given (a.window > 0); the kernel without it carries no
// window arithmetic.  kCausal = false: the non-causal variant (no prefix, no window), in
// which each query row sees all keys of its request.  kFp8: the paged prefix is an FP8 E4M3 cache (value = scale[g] *
// e4m3(code)); its tiles are staged as codes and converted in shared memory by the
// converter warps - K to bf16 code values (exact; the K scale joins the score scale of
// those tiles), V to fp16 value * 2^-k like the bf16 V tiles.
template <int D, bool kWindow, bool kFp8, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap kpmap,
                   const __grid_constant__ CUtensorMap vpmap, const PrefillArgs a) {
    using C = PrefillCfg<D, (D == 64 && kWindow) ? 2 : 1>;
    constexpr int NS = C::kStages;
    // the next kernel on the stream may start now (it takes the SMs this grid leaves free)
    if (a.launch_dependents) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int NBS = C::kSBufs, NBP = C::kPBufs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *sQ = smem + C::kOffQ;
    uint8_t *sK = smem + C::kOffK;
    uint8_t *sV = smem + C::kOffV;
    uint64_t *bb = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    Bars bars;
    bars.q_full = bb;                    // [kQBufs] the buffer's Q tiles landed
    bars.q_empty = bb + C::kQBufs;       // [kQBufs] the buffer's last S products are done
    bars.k_full = bb + 2 * C::kQBufs;
    bars.v_full = bars.k_full + NS;
    bars.v_conv = bars.v_full + NS;     // [NS] the stage's V tile is in fp16
    bars.k_conv = bars.v_conv + NS;     // [NS] FP8 prefix: the stage's K tile is in bf16
    bars.kv_empty = bars.k_conv + NS;
    // Every wait below is for the next completion of its barrier or the one before,
    // never older: a parity wait cannot tell phases two apart.
    bars.s_full = bars.kv_empty + NS;      // [NBS] per S buffer: its S product is done
    bars.s_free = bars.s_full + NBS;       // [NBS] per S buffer: the softmax has read it
    bars.p_full = bars.s_free + NBS;       // [NBP] per P buffer: its P is written
    bars.pv_done = bars.p_full + NBP;      // [NBP] per P buffer: the P.V reading it is done
    bars.o_free = bars.pv_done + NBP;      // [2] per query tile: O was read (once per item)
    bars.drain = bars.o_free + 2;
    bars.item_full = bars.drain + 1;     // [kItemRing] per slot: the producer posted an item
    int *s_loc = reinterpret_cast<int *>(smem + C::kOffLoc);
    int *misc = reinterpret_cast<int *>(smem + C::kOffMisc);
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(misc);
    volatile int *s_abort = misc + 1;
    int *s_vscale = misc + 32;  // [NS][4] exponent k of each 32-key quarter of each V tile
    ItemSlot *s_slot = reinterpret_cast<ItemSlot *>(smem + C::kOffSlot);  // the k-th item in slot k % kItemRing

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    WorkList wl;
    worklist_setup(a, s_loc, s_loc + kLocateMax, s_loc + 2 * kLocateMax, s_loc + 3 * kLocateMax, misc + 4,
                   &wl);
    const int n_items = wl.tiles * wl.groups;
    if ((int)blockIdx.x >= n_items) {  // CTA-uniform, before any allocation
        if (tid == 0) cta_done(a.sched);
        return;
    }
    const int ntiles = wl.heads_per_item;    // query tiles per item (1 or 2)

    if (tid == 0) {
        *s_abort = 0;
        for (int qb = 0; qb < C::kQBufs; ++qb) {
            mbar_init(&bars.q_full[qb], 1);
            mbar_init(&bars.q_empty[qb], 1);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.v_conv[s], 4);  // one arrive per converter warp
            mbar_init(&bars.k_conv[s], 4);
            mbar_init(&bars.kv_empty[s], 1);
        }
        for (int b = 0; b < NBS; ++b) {
            mbar_init(&bars.s_full[b], 1);
            mbar_init(&bars.s_free[b], 4);
        }
        for (int p = 0; p < NBP; ++p) {
            mbar_init(&bars.p_full[p], 4);
            mbar_init(&bars.pv_done[p], 1);
        }
        for (int x = 0; x < 2; ++x) mbar_init(&bars.o_free[x], 4);
        mbar_init(bars.drain, 64);  // one commit from every lane of the two MMA-issuing warps
        for (int s = 0; s < kItemRing; ++s) mbar_init(&bars.item_full[s], 1);
        fence_mbar_init();
    }
    // What the producer issued (for the drain after an abort): the Q tiles of items
    // 0..q_issued and the K/V tiles 0..kv_issued-1 of the ring.
    int q_issued = -1, kv_issued = 0;
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
        const bool test_limit = a.wait_limit_ns <= kImmediateLimitNs;
        // the next item from the work-list counter (items in rank order: heaviest first), posted
        // in slot kk % kItemRing for the other roles; a rank >= n_items ends the CTA's work
        auto fetch = [&](int kk) {
            int r = 0;
            if (lane == 0) {
                ItemSlot &sl = s_slot[kk % kItemRing];
                r = min((int)atomicAdd(a.sched, 1u), n_items);
                sl.rank = r;
                if (r < n_items) {
                    sl.it = item_of(a, wl, r);
                    sl.gm = geom_of<kWindow, kCausal>(a, sl.it);
                    for (int x = 0; x < 2; ++x)
                        sl.sink2[x] = a.sinks && x < ntiles ? a.sinks[sl.it.h0 + x] * kLog2e : -INFINITY;
                    sl.kscale = kFp8 && a.k_scale ? a.k_scale[sl.gm.g] : 1.f;
                    sl.vscale = kFp8 && a.v_scale ? a.v_scale[sl.gm.g] : 1.f;
                }
                mbar_arrive(&bars.item_full[kk % kItemRing]);
            }
            __syncwarp();
            return __shfl_sync(0xffffffffu, r, 0);
        };
        for (int rank = fetch(0); ok && rank < n_items; rank = fetch(++k)) {
            const Item it = s_slot[k % kItemRing].it;
            const ItemGeom gm = s_slot[k % kItemRing].gm;
            if (lane == 0 && a.prefix_lens) {
                const int Praw = a.prefix_lens[it.req];
                if (Praw < 0 || Praw > a.max_pages * kPageSize)
                    set_status(a.status, SINKATTN_STATUS_BAD_LENGTH);
            }
            // Q tiles of this item, once the previous item's last S products are done
            const int qbuf = k % C::kQBufs;
            if (k >= C::kQBufs && !wait_or_abort<true>(&bars.q_empty[qbuf], (uint32_t)((k / C::kQBufs - 1) & 1), s_abort,
                                                      a.status, a.wait_limit_cycles)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars.q_full[qbuf], ntiles * C::kQBytes);
                for (int x = 0; x < ntiles; ++x)
#pragma unroll
                    for (int hf = 0; hf < C::kHalves; ++hf)
                        tma_load_3d(sQ + (qbuf * 2 + x) * C::kQBytes + hf * 16384, &qmap, &bars.q_full[qbuf], hf * 64,
                                    it.h0 + x, gm.row0 + it.qb * kBM);
            }
            q_issued = k;
            if (test_limit) {
                // the testing setting of the watchdog: give up here, with the item's Q copy still
                // in flight; the other roles leave at their next wait that does not complete
                if (lane == 0) {
                    *s_abort = 1;
                    set_status(a.status, SINKATTN_STATUS_WAIT_TIMEOUT);
                }
                __syncwarp();
                ok = false;
                break;
            }
            for (int j = 0; j < gm.n_kv; ++j, ++kv) {
                const int s = kv % NS, u = kv / NS;
                const int tt = kWindow ? gm.t0 + j : j;  // key tile
                // prefix tile: lane p < 8 looks up page 8tt + p (issued before the wait below so
                // the load overlaps it); nrow = its valid rows, pg = -1 for a missing page
                int nrow = 0, pg = -1;
                if (tt < gm.n_pre && lane < 8) {
                    const int page = tt * 8 + lane;
                    nrow = min(kPageSize, max(0, gm.P - page * kPageSize));
                    if (nrow > 0) {
                        pg = a.prefix_block_table[(int64_t)it.req * a.max_pages + page];
                        if (pg < 0 || pg >= a.num_pages) {
                            set_status(a.status, SINKATTN_STATUS_BAD_PAGE);
                            pg = -1;
                        }
                    }
                }
                if (u > 0 &&
                    !wait_or_abort<true>(&bars.kv_empty[s], (uint32_t)((u - 1) & 1), s_abort, a.status, a.wait_limit_cycles)) {
                    ok = false;
                    break;
                }
                uint8_t *kt = sK + s * C::kKVBytes;
                uint8_t *vt = sV + s * C::kKVBytes;
                if (kFp8 && tt < gm.n_pre) {
                    // eight FP8 pages of 16 tokens, as codes into their staging places: each
                    // whole valid page by a TMA issued from its own lane (one box of 16 rows x D
                    // bytes), the others by the warp (valid rows copied, the rest code 0 = 0.0)
                    const bool full = nrow == kPageSize && pg >= 0;
                    const uint32_t full_mask = __ballot_sync(0xffffffffu, full);
                    const uint32_t other_mask = __ballot_sync(0xffffffffu, lane < 8 && !full);
                    if (lane == 0) {
                        const uint32_t bytes = (uint32_t)__popc(full_mask) * kPageSize * D;
                        mbar_expect_tx(&bars.k_full[s], bytes);
                        mbar_expect_tx(&bars.v_full[s], bytes);
                    }
                    if (full) {
                        tma_load_4d(kt + C::kOffFp8Page(lane), &kpmap, &bars.k_full[s], 0, 0, gm.g, pg);
                        tma_load_4d(vt + C::kOffFp8Page(lane), &vpmap, &bars.v_full[s], 0, 0, gm.g, pg);
                    }
                    for (uint32_t om = other_mask; om; om &= om - 1) {
                        const int pp = __ffs(om) - 1;
                        const int pgp = __shfl_sync(0xffffffffu, pg, pp);
                        const int nv = pgp >= 0 ? __shfl_sync(0xffffffffu, nrow, pp) : 0;
                        const uint8_t *kg = static_cast<const uint8_t *>(a.k_pages);
                        const uint8_t *vg = static_cast<const uint8_t *>(a.v_pages);
                        constexpr int kVec = D / 16;  // 16-byte vectors per row
                        for (int e = lane; e < kPageSize * kVec; e += 32) {
                            const int slot = e / kVec, c = e % kVec;
                            uint4 kx = make_uint4(0, 0, 0, 0), vx = make_uint4(0, 0, 0, 0);
                            if (slot < nv) {
                                const int64_t off = (((int64_t)pgp * a.Hkv + gm.g) * kPageSize + slot) * D + c * 16;
                                kx = *reinterpret_cast<const uint4 *>(kg + off);
                                vx = *reinterpret_cast<const uint4 *>(vg + off);
                            }
                            const uint32_t o = C::kOffFp8Page(pp) + slot * D + c * 16;
                            *reinterpret_cast<uint4 *>(kt + o) = kx;
                            *reinterpret_cast<uint4 *>(vt + o) = vx;
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&bars.k_full[s]);
                        mbar_arrive(&bars.v_full[s]);
                    }
                } else if (tt < gm.n_pre) {
                    // eight pages of 16 tokens: each whole valid page by a TMA issued from its
                    // own lane, the others (ragged tail, missing page) by the warp
                    const bool full = nrow == kPageSize && pg >= 0;
                    const uint32_t full_mask = __ballot_sync(0xffffffffu, full);
                    const uint32_t other_mask = __ballot_sync(0xffffffffu, lane < 8 && !full);
                    if (lane == 0) {
                        const uint32_t bytes = (uint32_t)__popc(full_mask) * kPageSize * D * 2;
                        mbar_expect_tx(&bars.k_full[s], bytes);
                        mbar_expect_tx(&bars.v_full[s], bytes);
                    }
                    if (full) {
#pragma unroll
                        for (int hf = 0; hf < C::kHalves; ++hf) {
                            tma_load_4d(kt + hf * 16384 + lane * 2048, &kpmap, &bars.k_full[s], hf * 64, 0,
                                        gm.g, pg);
                            tma_load_4d(vt + hf * 16384 + lane * 2048, &vpmap, &bars.v_full[s], hf * 64, 0,
                                        gm.g, pg);
                        }
                    }
                    for (uint32_t om = other_mask; om; om &= om - 1) {
                        // copy the valid rows of page pp (none if missing), zero the rest
                        const int pp = __ffs(om) - 1;
                        const int pgp = __shfl_sync(0xffffffffu, pg, pp);
                        const int nv = pgp >= 0 ? __shfl_sync(0xffffffffu, nrow, pp) : 0;
                        const __nv_bfloat16 *kg = reinterpret_cast<const __nv_bfloat16 *>(a.k_pages);
                        const __nv_bfloat16 *vg = reinterpret_cast<const __nv_bfloat16 *>(a.v_pages);
                        for (int e = lane; e < kPageSize * C::kHalves * 8; e += 32) {
                            const int slot = e / (C::kHalves * 8);
                            const int hf = (e / 8) % C::kHalves;
                            const int c = e % 8;
                            uint4 kx = make_uint4(0, 0, 0, 0), vx = make_uint4(0, 0, 0, 0);
                            if (slot < nv) {
                                const int64_t off =
                                    (((int64_t)pgp * a.Hkv + gm.g) * kPageSize + slot) * D + hf * 64 + c * 8;
                                kx = *reinterpret_cast<const uint4 *>(kg + off);
                                vx = *reinterpret_cast<const uint4 *>(vg + off);
                            }
                            const uint32_t o = hf * 16384 + sw128(pp * kPageSize + slot, c);
                            *reinterpret_cast<uint4 *>(kt + o) = kx;
                            *reinterpret_cast<uint4 *>(vt + o) = vx;
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&bars.k_full[s]);
                        mbar_arrive(&bars.v_full[s]);
                    }
                } else if (lane == 0) {
                    const int row = gm.row0 + (tt - gm.n_pre) * kBN;
                    mbar_arrive_expect_tx(&bars.k_full[s], C::kKVBytes);
#pragma unroll
                    for (int hf = 0; hf < C::kHalves; ++hf)
                        tma_load_3d(kt + hf * 16384, &kmap, &bars.k_full[s], hf * 64, gm.g, row);
                    mbar_arrive_expect_tx(&bars.v_full[s], C::kKVBytes);
#pragma unroll
                    for (int hf = 0; hf < C::kHalves; ++hf)
                        tma_load_3d(vt + hf * 16384, &vmap, &bars.v_full[s], hf * 64, gm.g, row);
                }
                kv_issued = kv + 1;
                __syncwarp();
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ================================================================ MMA issuers
        reg_dealloc<kRegsSide>();
        // Warp 1 issues the P.V products, warp 2 the S products; each runs its loop warp-
        // uniformly and one elected lane issues each MMA group.  S products are numbered
        // i = 0, 1, ... over the CTA's lifetime (key tile by key tile, query tile x = i %
        // ntiles); S(i) goes to S buffer i % NBS and P(i) is read from P buffer i % NBP.
        const bool pv_role = warp == 1;
        constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kBM, kBN, false);
        constexpr uint32_t idesc_o = tc::idesc_f16_f32(kBM, D, true);
        // Descriptors are built once; an operand at byte offset `off` inside a tile only
        // moves the start-address field (bits 0..13, address >> 4), which cannot overflow
        // because every shared address is below 2^18.
        const uint64_t dq = tc::smem_desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk = tc::smem_desc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t dv = tc::smem_desc_sw128(smem_u32(sV), 16384, 1024);
        // all lanes wait; the outcome is made warp-uniform so that no lane is left behind
        // at the elect.sync below when a wait gives up
        auto warp_wait = [&](uint64_t *bar, uint32_t parity) {
            return __all_sync(0xffffffffu, wait_or_abort<true>(bar, parity, s_abort, a.status, a.wait_limit_cycles));
        };
        auto take = [&](int kk) {
            if (!warp_wait(&bars.item_full[kk % kItemRing], (uint32_t)((kk / kItemRing) & 1))) return -1;
            return s_slot[kk % kItemRing].rank;
        };
        int k = 0, j = 0, x = 0, kv = 0;
        int rank = take(0);
        int n_kv = rank >= 0 && rank < n_items ? s_slot[0].gm.n_kv : 0;
        uint32_t i = 0;
        int b = 0, pb = 0;            // i % NBS, i % NBP
        uint32_t use = 0, use_p = 0;  // i / NBS, i / NBP
        bool ok = true;
        while (ok && rank >= 0 && rank < n_items) {
            const int st = kv % NS;
            const uint32_t sp = (uint32_t)((kv / NS) & 1);
            if (pv_role) {
                // O_x += P V in fp16: P (keys 2c, 2c + 1 in column c) in the first 64 columns
                // of the S/P buffer, V scaled into fp16 by the converter warp
                if (!warp_wait(&bars.p_full[pb], use_p & 1)) break;
                if (j == 0 && k > 0 && !warp_wait(&bars.o_free[x], (uint32_t)((k - 1) & 1))) break;
                if (x == 0 && !warp_wait(&bars.v_conv[st], sp)) break;
                const uint64_t v0 = dv + (uint64_t)((st * C::kKVBytes) >> 4);
                const uint32_t tp = tmem + C::kColP(pb), to = tmem + C::kColO(x);
                const uint32_t acc0 = j > 0 ? 1u : 0u;
                if (elect_one()) {
                    tc::fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        tc::mma_f16_ts(to, tp + 8 * kk, v0 + (uint64_t)((kk * 2048) >> 4), idesc_o,
                                       kk > 0 ? 1u : acc0);
                    tc::commit(&bars.pv_done[pb]);
                    if (x == ntiles - 1) tc::commit(&bars.kv_empty[st]);
                }
                __syncwarp();
            } else {
                // S buffer b is free once the softmax has read S(i - NBS) (with P over S:
                // once the P.V of product i - NBS has completed)
                if (use > 0 &&
                    !warp_wait(C::kSplitP ? &bars.s_free[b] : &bars.pv_done[b], (use - 1) & 1))
                    break;
                if (j == 0 && x == 0 && !warp_wait(&bars.q_full[k % C::kQBufs], (uint32_t)((k / C::kQBufs) & 1))) break;
                if (x == 0 && !warp_wait(kFp8 ? &bars.k_conv[st] : &bars.k_full[st], sp)) break;
                const uint64_t q0 = dq + (uint64_t)((((k % C::kQBufs) * 2 + x) * C::kQBytes) >> 4);
                const uint64_t k0 = dk + (uint64_t)((st * C::kKVBytes) >> 4);
                const bool last = j == n_kv - 1 && x == ntiles - 1;
                if (elect_one()) {
                    tc::fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        tc::mma_f16_ss(tmem + C::kColS(b), q0 + off, k0 + off, idesc_s, kk > 0 ? 1u : 0u);
                    }
                    tc::commit(&bars.s_full[b]);
                    if (last) tc::commit(&bars.q_empty[k % C::kQBufs]);  // the item's Q tiles are no longer read
                }
                __syncwarp();
            }
            // next product
            ++i;
            if (++b == NBS) {
                b = 0;
                ++use;
            }
            if (++pb == NBP) {
                pb = 0;
                ++use_p;
            }
            if (++x == ntiles) {
                x = 0;
                ++kv;
                if (++j == n_kv) {
                    j = 0;
                    rank = take(++k);
                    if (rank < 0) break;
                    if (rank < n_items) n_kv = s_slot[k % kItemRing].gm.n_kv;
                }
            }
            continue;
        }
        ok = false;
        (void)ok;
    } else if (warp == 3) {
        reg_dealloc<kRegsSide>();
    } else if (warp >= 12) {
        // ================================================================ V converters
        reg_dealloc<kRegsConvert>();
        // Keys 32q..32q+31 of the V tile, bf16 -> fp16 scaled by 2^-k, in place;
        // k = max(0, e - 14) where 2^e <= max|v| < 2^(e+1) over the quarter, so the
        // quarter stays below 2^15 and P * 2^k below 2^15 (k <= 7).  The quarter is
        // 32 rows x 128 bytes of each 64-column half of the tile.
        const int q = warp - 12;
        int kv = 0, k = 0;
        bool ok = true;
        auto take = [&](int kk) {
            if (!__all_sync(0xffffffffu, wait_or_abort<true>(&bars.item_full[kk % kItemRing], (uint32_t)((kk / kItemRing) & 1),
                                                        s_abort, a.status, a.wait_limit_cycles)))
                return n_items;
            return s_slot[kk % kItemRing].rank;
        };
        for (int rank = take(0); ok && rank < n_items; rank = take(++k)) {
            const ItemGeom gm = s_slot[k % kItemRing].gm;
            // FP8 V: |value| <= 448 * v_scale, so one exponent k per item keeps every converted
            // value below 2^15 (k = 0 for any scale below 73): no per-tile maximum needed
            const float vsc = kFp8 ? s_slot[k % kItemRing].vscale : 1.f;
            // v_scale = m * 2^e8 with m in [1, 2): for -12 <= e8 <= 6 the V codes become
            // code * 2^e8, exact in fp16 and below 2^15, and the softmax multiplies those keys'
            // P by m; other scales take the exponent k below
            const int e8 = (int)((__float_as_uint(vsc) >> 23) & 0xFFu) - 127;
            const bool fold8 = kFp8 && e8 >= -12 && e8 <= 6;
            const uint32_t p2e8 = (uint32_t)(e8 + 15) << 10 | (uint32_t)(e8 + 15) << 26;  // f16 pair 2^e8
            int kexp8 = 0;
            if (kFp8 && !fold8) {
                const float top = 448.f * vsc;
                kexp8 = max(0, (int)((__float_as_uint(top) >> 23) & 0xFFu) - 127 - 14);
                if (!(top < INFINITY) || kexp8 > 7) {
                    if (lane == 0) set_status(a.status, SINKATTN_STATUS_VALUE_RANGE);
                    kexp8 = min(kexp8, 7);
                }
            }
            const float vmul8 = vsc * __uint_as_float((uint32_t)(127 - kexp8) << 23);
            for (int j = 0; j < gm.n_kv; ++j, ++kv) {
                const int st = kv % NS;
                const bool fp8_tile = kFp8 && (kWindow ? gm.t0 + j : j) < gm.n_pre;
                if (kFp8) {
                    // K: the FP8 prefix tiles to bf16 code values (the S products wait for this)
                    if (!__all_sync(0xffffffffu, wait_or_abort<true>(&bars.k_full[st], (uint32_t)((kv / NS) & 1),
                                                                s_abort, a.status, a.wait_limit_cycles))) {
                        ok = false;
                        break;
                    }
                    if (fp8_tile) convert_fp8_quarter<D, 0>(sK + st * C::kKVBytes, q, lane, 1.f);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.k_conv[st]);
                }
                if (!__all_sync(0xffffffffu, wait_or_abort<true>(&bars.v_full[st], (uint32_t)((kv / NS) & 1),
                                                            s_abort, a.status, a.wait_limit_cycles))) {
                    ok = false;
                    break;
                }
                if (fp8_tile) {
                    // V: code * 2^e8 (the softmax takes the rest of the scale), or fp16 of
                    // value * 2^-k, value = scale * e4m3(code), k of the item
                    if (fold8)
                        convert_fp8_quarter<D, 2>(sV + st * C::kKVBytes, q, lane, 1.f, p2e8);
                    else
                        convert_fp8_quarter<D, 1>(sV + st * C::kKVBytes, q, lane, vmul8);
                    if (lane == 0) s_vscale[st * 4 + q] = fold8 ? 0 : kexp8;
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.v_conv[st]);
                    continue;
                }
                uint4 *vt = reinterpret_cast<uint4 *>(sV + st * C::kKVBytes + q * 4096) + lane;
                // this lane's vectors: 8 per 64-column half, 512 bytes apart
                uint32_t mx = 0;  // largest |v| per 16-bit half, as bf16 bits (monotonic in |v|)
#pragma unroll 1
                for (int hf = 0; hf < C::kHalves; ++hf) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const uint4 w = vt[hf * 1024 + e * 32];
                        mx = __vmaxu2(mx, w.x & 0x7FFF7FFFu);
                        mx = __vmaxu2(mx, w.y & 0x7FFF7FFFu);
                        mx = __vmaxu2(mx, w.z & 0x7FFF7FFFu);
                        mx = __vmaxu2(mx, w.w & 0x7FFF7FFFu);
                    }
                }
                mx = __reduce_max_sync(0xffffffffu, max(mx & 0xFFFFu, mx >> 16));
                int kexp = max(0, (int)(mx >> 7) - 127 - 14);
                if (mx >= 0x7F80u || kexp > 7) {
                    if (lane == 0) set_status(a.status, SINKATTN_STATUS_VALUE_RANGE);
                    kexp = min(kexp, 7);
                }
                const float sc = __uint_as_float((uint32_t)(127 - kexp) << 23);  // 2^-k
#pragma unroll 1
                for (int hf = 0; hf < C::kHalves; ++hf) {
                    if (kexp == 0) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            uint4 *pw = vt + hf * 1024 + e * 32;
                            uint4 w = *pw;
                            w.x = pack_f16x2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u));
                            w.y = pack_f16x2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
                            w.z = pack_f16x2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u));
                            w.w = pack_f16x2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u));
                            *pw = w;
                        }
                    } else {
#pragma unroll 2
                        for (int e = 0; e < 8; ++e) {
                            uint4 *pw = vt + hf * 1024 + e * 32;
                            uint4 w = *pw;
                            w.x = pack_f16x2(__uint_as_float(w.x << 16) * sc, __uint_as_float(w.x & 0xFFFF0000u) * sc);
                            w.y = pack_f16x2(__uint_as_float(w.y << 16) * sc, __uint_as_float(w.y & 0xFFFF0000u) * sc);
                            w.z = pack_f16x2(__uint_as_float(w.z << 16) * sc, __uint_as_float(w.z & 0xFFFF0000u) * sc);
                            w.w = pack_f16x2(__uint_as_float(w.w << 16) * sc, __uint_as_float(w.w & 0xFFFF0000u) * sc);
                            *pw = w;
                        }
                    }
                }
                if (lane == 0) s_vscale[st * 4 + q] = kexp;
                fence_proxy_async_smem();  // the P.V MMA reads these through the async proxy
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.v_conv[st]);
            }
        }
    } else {
        // ================================================================ softmax
        reg_alloc<kRegsSoftmax>();
        const int x = (warp - 4) >> 2;  // query tile of this warpgroup
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // tile row of this thread
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_base + C::kColO(x);
        uint32_t tcount = 0;  // key tiles this query tile has processed (over all items)
        int k = 0;
        bool ok = x < ntiles;
        auto take = [&](int kk) {
            if (!wait_or_abort(&bars.item_full[kk % kItemRing], (uint32_t)((kk / kItemRing) & 1), s_abort, a.status,
                               a.wait_limit_cycles))
                return n_items;
            return s_slot[kk % kItemRing].rank;
        };
        for (int rank = ok ? take(0) : n_items; ok && rank < n_items; rank = take(++k)) {
            const Item it = s_slot[k % kItemRing].it;
            const ItemGeom gm = s_slot[k % kItemRing].gm;
            const int h = it.h0 + x;
            const int t = it.qb * kBM + r;  // position among the request's new tokens
            const float sink2 = s_slot[k % kItemRing].sink2[x];
            // score scale of FP8 prefix tiles: their K holds code values, the K scale joins here
            const float sc_pre = kFp8 ? a.scale_log2 * s_slot[k % kItemRing].kscale : a.scale_log2;
            // FP8 prefix V in the converters' power-of-two form: P of those keys times m8, the
            // mantissa of v_scale (m8 in [1, 2), so P * m8 < 2^9 stays in fp16)
            const float vsc8 = kFp8 ? s_slot[k % kItemRing].vscale : 1.f;
            const int e8 = (int)((__float_as_uint(vsc8) >> 23) & 0xFFu) - 127;
            const bool fold8 = kFp8 && e8 >= -12 && e8 <= 6;
            const float m8 = fold8 ? __uint_as_float((__float_as_uint(vsc8) & 0x807FFFFFu) | 0x3F800000u) : 1.f;
            const float add8 = log2f(m8), mul8 = 1.f / m8;
            float m_used = sink2;                      // running max, seeded with the sink
            float l = sink2 == -INFINITY ? 0.f : 1.f;  // running denominator: e^(sink - m) = 1
            for (int j = 0; j < gm.n_kv; ++j) {
                const uint32_t i = tcount * ntiles + x;  // number of this S product
                const int b = i % NBS, pb = i % NBP;
                const uint32_t ts = tmem + lane_base + C::kColS(b);
                const uint32_t tp = tmem + lane_base + C::kColP(pb);
                if (!wait_or_abort(&bars.s_full[b], (i / NBS) & 1, s_abort, a.status, a.wait_limit_cycles)) {
                    ok = false;
                    break;
                }
                ++tcount;
                tc::fence_after_sync();
                const int tt = kWindow ? gm.t0 + j : j;  // key tile
                // keys lo .. ncols-1 of this tile are the row's to see
                int ncols;
                if (!kCausal)
                    ncols = min(kBN, gm.L - tt * kBN);  // the request's ragged end
                else if (tt < gm.n_pre)
                    ncols = min(kBN, gm.P - tt * kBN);
                else if (tt - gm.n_pre == it.qb)
                    ncols = r + 1;  // diagonal tile: keys 0..r
                else
                    ncols = kBN;
                int lo = 0;
                if (kWindow) {  // keys at positions <= (P + t) - W are outside the window
                    const int key0 = tt < gm.n_pre ? tt * kBN : gm.P + (tt - gm.n_pre) * kBN;
                    lo = gm.P + t - a.window + 1 - key0;
                }
                // the whole S row of this tile
                uint32_t sv[kBN];
#pragma unroll
                for (int c = 0; c < kBN / 32; ++c)
                    tc::ld_32x32b_x32(ts + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
                tc::wait_ld();
                if (C::kSplitP) {  // S is in registers: its buffer may take the next S product
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.s_free[b]);
                }
                if (__any_sync(0xffffffffu, ncols < kBN || lo > 0)) {
                    // diagonal, ragged, prefix-tail or window edge: only the 32-key chunks in
                    // which some row of the warp hides a key are masked key by key
#pragma unroll
                    for (int ch = 0; ch < kBN / 32; ++ch) {
                        const int c0 = ch * 32;
                        if (__any_sync(0xffffffffu, ncols < c0 + 32 || lo > c0)) {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (c0 + e >= ncols || c0 + e < lo) sv[c0 + e] = 0xFF800000u;  // -inf
                        }
                    }
                }
                const float sc = kFp8 && tt < gm.n_pre ? sc_pre : a.scale_log2;
                // row max: eight chains of three-input maxima over 16 keys each
                auto row_max = [&]() {
                    float mx8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float *sf = reinterpret_cast<const float *>(sv) + 16 * e;
                        float m = fmax3(sf[0], sf[1], sf[2]);
#pragma unroll
                        for (int t = 3; t < 15; t += 2) m = fmax3(m, sf[t], sf[t + 1]);
                        mx8[e] = fmaxf(m, sf[15]);
                    }
                    return fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                 fmaxf(mx8[6], mx8[7]));
                };
                if (j == 0) {
                    const float mt = row_max() * sc;
                    const float mn = fmaxf(m_used, mt);
                    l = (m_used == -INFINITY) ? 0.f : l * fast_exp2(m_used - mn);
                    m_used = mn;
                }
                // P * 2^k = exp2(s * scale - m + k) in fp16 in the 64 columns of the P buffer
                // (keys 2c, 2c + 1 in column c); 2^-k is the scale of the V quarter holding
                // keys 32ch..32ch+31
                const int vst = (tcount - 1) % NS;
                if (!wait_or_abort(&bars.v_conv[vst], ((tcount - 1) / NS) & 1, s_abort, a.status, a.wait_limit_cycles)) {
                    ok = false;
                    break;
                }
                // the P buffer is free once the P.V of product i - NBP has completed: waited for
                // in emit, after the first chunk's exponentials
                bool pwait = C::kSplitP && i >= (uint32_t)NBP, pfail = false;
                const int4 kq = *reinterpret_cast<const int4 *>(s_vscale + vst * 4);
                const float2 sc2 = make_float2(sc, sc);
                // writes P against the running max m_used; returns the row's sum of P * 2^-k
                const bool f8 = kFp8 && fold8 && tt < gm.n_pre;  // warp-uniform
                auto emit = [&]() {
                    const float neg0 = m_used == -INFINITY ? 0.f : -m_used;
                    float tl = 0.f;
#pragma unroll
                    for (int ch = 0; ch < kBN / 32; ++ch) {
                        const int kc = ch == 0 ? kq.x : ch == 1 ? kq.y : ch == 2 ? kq.z : kq.w;
                        const float neg = neg0 + (f8 ? add8 : (float)kc);
                        const float2 ng2 = make_float2(neg, neg);
                        // running sums of keys c with c % 8 = 2q (.x) and 2q + 1 (.y)
                        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                         make_float2(0.f, 0.f)};
                        uint32_t pp[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int c = ch * 32 + 2 * e;
                            const float2 t2 = ffma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])),
                                                    sc2, ng2);
                            const float p0 = fast_exp2(t2.x);
                            const float p1 = fast_exp2(t2.y);
                            acc[e & 3] = fadd2(acc[e & 3], make_float2(p0, p1));
                            pp[e] = pack_f16x2(p0, p1);
                        }
                        if (ch == 0 && pwait) {
                            pwait = false;
                            if (!wait_or_abort(&bars.pv_done[pb], ((i - NBP) / NBP) & 1, s_abort, a.status,
                                               a.wait_limit_cycles))
                                pfail = true;
                            tc::fence_after_sync();
                        }
                        if (!pfail) tc::st_32x32b_x16(tp + ch * 16, pp);
                        tl += (((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) +
                               ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y))) *
                              (f8 ? mul8 : __uint_as_float((uint32_t)(127 - kc) << 23));
                    }
                    return tl;
                };
                float tl = emit();
                if (pfail) {
                    ok = false;
                    break;
                }
                if (j > 0) {
                    // every P * 2^-k at most 2^8 (so P fits fp16) unless the row's sum passes it
                    const bool need = !(tl <= kPSumLimit) || m_used == -INFINITY;
                    if (__any_sync(0xffffffffu, need)) {
                        // the row max, a rescale of O and l, and P again (the P written above is
                        // overwritten before p_full; rows that need nothing write the same P)
                        const float mt = row_max() * sc;
                        // O_x must hold the P.V of this query tile's previous key tile, product i - ntiles
                        const uint32_t ip = i - ntiles;
                        if (!wait_or_abort(&bars.pv_done[ip % NBP], (ip / NBP) & 1, s_abort, a.status, a.wait_limit_cycles)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        const float mn = fmaxf(m_used, mt);
                        const float alpha = need && mn > m_used ? fast_exp2(m_used - mn) : 1.f;
                        if (need && mn > m_used) {
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
                        tc::wait_st();  // the first P stores land before the second ones
                        tl = emit();
                    }
                }
                l += tl;
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.p_full[pb]);
            }
            if (!ok) break;
            // epilogue: O / l for this row, once the item's last P.V has landed
            const uint32_t il = (tcount - 1) * ntiles + x;  // S product of the last key tile
            if (!wait_or_abort(&bars.pv_done[il % NBP], (il / NBP) & 1, s_abort, a.status, a.wait_limit_cycles)) {
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
                    for (int e = 0; e < 32; e += 16) {
                        uint32_t w[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            w[u] = pack_bf16x2(__uint_as_float(o[e + 2 * u]) * inv, __uint_as_float(o[e + 2 * u + 1]) * inv);
                        st_global_v8(og + c * 32 + e, w);  // 32 bytes; the output rows are 32-byte aligned
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

    // All roles done.  After an abort, before TMEM is freed and the CTA's shared memory is
    // released: every MMA still in flight completes (each lane of the two MMA-issuing warps
    // commits to the drain barrier; a commit arrives once the MMAs its thread issued have
    // completed, at once for a thread that issued none), and every copy the producer issued
    // lands - Q of the last item it loaded, and the last NS tiles of the K/V ring, each stage
    // holding at most one copy that no consumer took (a stage is refilled only after its
    // previous tile was consumed, so the parity of its last use names it).  These waits use
    // their own limit, not the call's: what they wait for always completes.
    tc::fence_before_sync();
    __syncthreads();
    if (*s_abort) {
        if (warp == 1 || warp == 2) {
            tc::commit(bars.drain);
            mbar_wait(bars.drain, 0, kDrainLimitNs);
        } else if (warp == 0) {
            // the Q loads of the last kQBufs items it issued (each either landed or in flight)
            for (int t = q_issued >= C::kQBufs - 1 ? q_issued - C::kQBufs + 1 : 0; t <= q_issued; ++t)
                mbar_wait(&bars.q_full[t % C::kQBufs], (uint32_t)((t / C::kQBufs) & 1), kDrainLimitNs);
            for (int t = kv_issued > NS ? kv_issued - NS : 0; t < kv_issued; ++t) {
                mbar_wait(&bars.k_full[t % NS], (uint32_t)((t / NS) & 1), kDrainLimitNs);
                mbar_wait(&bars.v_full[t % NS], (uint32_t)((t / NS) & 1), kDrainLimitNs);
            }
        }
        tc::fence_before_sync();
        __syncthreads();
    }
    if (warp == 1) {
        tc::fence_after_sync();
        tc::dealloc(tmem, kTmemCols);
    }
    if (tid == 0) cta_done(a.sched);
}

template <int D, bool kWindow, bool kFp8, bool kCausal = true>
cudaError_t launch_d(const PrefillArgs &a, const CUtensorMap &qmap, const CUtensorMap &kmap,
                     const CUtensorMap &vmap, const CUtensorMap &kpmap, const CUtensorMap &vpmap,
                     cudaStream_t stream) {
    using C = PrefillCfg<D, (D == 64 && kWindow) ? 2 : 1>;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, kWindow, kFp8, kCausal>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    int device = 0, sms = 0;
    if ((e = cudaGetDevice(&device)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess) return e;
    // persistent: one CTA per SM (shared memory and the 512 TMEM columns allow no more),
    // on at most max_sms SMs when the caller keeps the others for concurrent work
    if (a.max_sms > 0 && a.max_sms < sms) sms = a.max_sms;
    prefill_kernel<D, kWindow, kFp8, kCausal><<<sms, kThreads, C::kSmemBytes, stream>>>(qmap, kmap, vmap, kpmap, vpmap, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, const CUtensorMap &qmap, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, const CUtensorMap &kpmap,
                           const CUtensorMap &vpmap, cudaStream_t stream) {
    const bool w = a.window > 0;
    if (!a.causal) {  // no prefix, no window
        if (a.fp8_prefix || w || a.prefix_lens) return cudaErrorInvalidValue;
        if (a.D == 64) return launch_d<64, false, false, false>(a, qmap, kmap, vmap, kpmap, vpmap, stream);
        if (a.D == 128) return launch_d<128, false, false, false>(a, qmap, kmap, vmap, kpmap, vpmap, stream);
        return cudaErrorNotSupported;
    }
    if (a.fp8_prefix) {
        if (a.D == 64)
            return w ? launch_d<64, true, true>(a, qmap, kmap, vmap, kpmap, vpmap, stream)
                     : launch_d<64, false, true>(a, qmap, kmap, vmap, kpmap, vpmap, stream);
        if (a.D == 128)
            return w ? launch_d<128, true, true>(a, qmap, kmap, vmap, kpmap, vpmap, stream)
                     : launch_d<128, false, true>(a, qmap, kmap, vmap, kpmap, vpmap, stream);
        return cudaErrorNotSupported;
    }
    if (a.D == 64)
        return w ? launch_d<64, true, false>(a, qmap, kmap, vmap, kpmap, vpmap, stream)
                 : launch_d<64, false, false>(a, qmap, kmap, vmap, kpmap, vpmap, stream);
    if (a.D == 128)
        return w ? launch_d<128, true, false>(a, qmap, kmap, vmap, kpmap, vpmap, stream)
                 : launch_d<128, false, false>(a, qmap, kmap, vmap, kpmap, vpmap, stream);
    return cudaErrorNotSupported;
}

}  // namespace sinkattn
