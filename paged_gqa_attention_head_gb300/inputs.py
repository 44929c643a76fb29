"""Seeded synthetic workloads for paged GQA attention with sinks.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the fp64 CPU oracle (through the tests) and the
CUDA library (through the tests and the benchmark) are fed from here, so the
two sides always see the same bytes.

Recipe (shared by every workload):
  * values: standard normal float32 from numpy's PCG64, rounded to bf16 with
    round-to-nearest-even (torch's float32 -> bfloat16 conversion);
  * per-head sinks: standard normal float32, or None when sinks are disabled;
  * lengths: uniform integers with both ends included, or log-uniform
    L = round(exp(U(ln lo, ln hi)));
  * physical pages: every sequence gets ceil(L / 16) pages; 5 % extra
    "distractor" pages are added; all pages are shuffled by a random
    permutation, so a sequence's pages are scattered through the pool;
  * the unused slots of each sequence's last page, the distractor pages and
    the unused block-table columns are poisoned (NaN values, page index -1) so
    that any read beyond a sequence shows up in the results;
  * FP8 E4M3 caches: per-KV-head scales s_g = (4.5 / 448) * (1 + g / (2 Hkv)),
    codes = torch's float8_e4m3fn cast of the standard normal float32 values
    divided by s_g and clipped to [-448, 448]; poisoned slots hold the NaN code
    0x7F.

Random streams are keyed by (seed, stream id, chunk index) through numpy's
SeedSequence, so a tensor's contents do not depend on the thread count or on
which other tensors were drawn before it.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

PAGE_SIZE = 16
_CHUNK = 1 << 22  # elements per independently seeded chunk
BF16_NAN_BITS = 0x7FC0
E4M3_NAN_CODE = 0x7F

# stream ids: one per kind of tensor so that draws are independent
_S_LENS, _S_Q, _S_K, _S_V, _S_SINK, _S_PERM, _S_KNEW, _S_VNEW, _S_PREFIX = range(9)


def _rng(seed: int, stream: int, chunk: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence(entropy=seed, spawn_key=(stream, chunk)))


def normal_f32(n: int, seed: int, stream: int) -> np.ndarray:
    """n standard-normal float32 values, drawn in seeded chunks (thread-parallel)."""
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(i: int) -> None:
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        _rng(seed, stream, i).standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])

    if nchunks <= 1:
        if n:
            work(0)
    else:
        with ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def normal_bf16(shape, seed: int, stream: int) -> torch.Tensor:
    """Same values as normal_f32(...) rounded to bf16, converted chunk by chunk so
    that large tensors never exist in float32 all at once."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=torch.bfloat16)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(i: int) -> None:
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)
        buf = _rng(seed, stream, i).standard_normal(hi - lo, dtype=np.float32)
        out[lo:hi] = torch.from_numpy(buf).to(torch.bfloat16)

    if nchunks <= 1:
        if n:
            work(0)
    else:
        with ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(work, range(nchunks)))
    return out.reshape(shape)


def fp8_head_scales(num_kv_heads: int) -> torch.Tensor:
    """Per-KV-head scales of the synthetic FP8 caches (float32 [Hkv])."""
    g = torch.arange(num_kv_heads, dtype=torch.float64)
    return ((4.5 / 448.0) * (1.0 + g / (2 * num_kv_heads))).to(torch.float32)


def normal_e4m3(shape, head_scales: torch.Tensor, seed: int, stream: int) -> torch.Tensor:
    """E4M3 codes (uint8) of standard normal float32 values divided by the scale of
    their KV head, for pages [num_pages, Hkv, 16, D]; chunked like normal_bf16."""
    n = int(np.prod(shape)) if len(shape) else 1
    Hkv, row = shape[1], shape[2] * shape[3]
    assert _CHUNK % row == 0
    inv_rows = (1.0 / head_scales.double()).numpy().astype(np.float32)
    out = torch.empty(n, dtype=torch.uint8)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(i: int) -> None:
        lo, hi = i * _CHUNK, min(n, (i + 1) * _CHUNK)  # chunks hold whole rows
        buf = _rng(seed, stream, i).standard_normal(hi - lo, dtype=np.float32).reshape(-1, row)
        head = (np.arange(lo // row, hi // row, dtype=np.int64) % Hkv)
        buf = np.clip(buf * inv_rows[head][:, None], -448.0, 448.0).astype(np.float32)
        out[lo:hi] = torch.from_numpy(buf.reshape(-1)).to(torch.float8_e4m3fn).view(torch.uint8)

    if nchunks <= 1:
        if n:
            work(0)
    else:
        with ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 1)) as ex:
            list(ex.map(work, range(nchunks)))
    return out.reshape(shape)


def poison_rows_(t: torch.Tensor) -> None:
    """Fill a bf16 tensor (view) with NaN; a uint8 (E4M3 code) tensor with the NaN code."""
    if t.dtype == torch.uint8:
        t.fill_(E4M3_NAN_CODE)
    else:
        t.view(torch.int16).fill_(BF16_NAN_BITS)


def draw_lengths(spec, count: int, seed: int) -> list[int]:
    """spec: a list of ints, ("uniform", lo, hi) or ("loguniform", lo, hi)."""
    if isinstance(spec, (list, tuple)) and spec and not isinstance(spec[0], str):
        assert len(spec) == count
        return [int(x) for x in spec]
    kind, lo, hi = spec
    r = _rng(seed, _S_LENS)
    if kind == "uniform":
        return [int(x) for x in r.integers(lo, hi, size=count, endpoint=True)]
    if kind == "loguniform":
        u = r.uniform(math.log(lo), math.log(hi), size=count)
        return [int(min(hi, max(lo, round(math.exp(x))))) for x in u]
    raise ValueError(kind)


@dataclass
class PagedCache:
    """KV pages [num_pages, Hkv, 16, D] (bf16, or uint8 E4M3 codes with per-head
    scales) plus the block table of each sequence."""
    k_pages: torch.Tensor
    v_pages: torch.Tensor
    block_table: torch.Tensor  # [num_seqs, max_pages_per_seq] int32, unused = -1
    lens: torch.Tensor  # [num_seqs] int32 tokens held in the pages
    num_pages: int = 0
    k_scale: Optional[torch.Tensor] = None  # [Hkv] float32 (FP8 caches only)
    v_scale: Optional[torch.Tensor] = None

    @property
    def fp8(self) -> bool:
        return self.k_pages.dtype == torch.uint8


def make_paged_cache(lens: list[int], num_kv_heads: int, head_dim: int, seed: int,
                     distractor_frac: float = 0.05, poison: bool = True,
                     max_pages_per_seq: Optional[int] = None, k_stream: int = _S_K,
                     v_stream: int = _S_V, kv_dtype: str = "bf16",
                     fp8_unit_scales: bool = False) -> PagedCache:
    npages_seq = [(L + PAGE_SIZE - 1) // PAGE_SIZE for L in lens]
    used = sum(npages_seq)
    num_pages = used + int(math.ceil(distractor_frac * used))
    num_pages = max(num_pages, 1)
    maxp = max_pages_per_seq if max_pages_per_seq is not None else max(1, max(npages_seq, default=1))
    perm = _rng(seed, _S_PERM).permutation(num_pages).astype(np.int64)
    shape = (num_pages, num_kv_heads, PAGE_SIZE, head_dim)
    ks = vs = None
    if kv_dtype == "fp8":
        if fp8_unit_scales:  # codes are the N(0,1) values themselves
            ks = vs = torch.ones(num_kv_heads, dtype=torch.float32)
        else:
            ks = fp8_head_scales(num_kv_heads)
            vs = (ks * 1.25).to(torch.float32)
        k_pages = normal_e4m3(shape, ks, seed, k_stream)
        v_pages = normal_e4m3(shape, vs, seed, v_stream)
    else:
        assert kv_dtype == "bf16", kv_dtype
        k_pages = normal_bf16(shape, seed, k_stream)
        v_pages = normal_bf16(shape, seed, v_stream)
    bt = torch.full((len(lens), maxp), -1, dtype=torch.int32)
    cursor = 0
    for b, (L, np_b) in enumerate(zip(lens, npages_seq)):
        pages = perm[cursor:cursor + np_b]
        cursor += np_b
        bt[b, :np_b] = torch.from_numpy(pages.astype(np.int32))
        if poison and np_b and L % PAGE_SIZE:
            last = int(pages[-1])
            poison_rows_(k_pages[last, :, L % PAGE_SIZE:, :])
            poison_rows_(v_pages[last, :, L % PAGE_SIZE:, :])
    if poison and num_pages > used:
        idx = torch.from_numpy(perm[used:])
        for pages in (k_pages, v_pages):
            if kv_dtype == "fp8":
                pages[idx] = E4M3_NAN_CODE
            else:
                pages.view(torch.int16)[idx] = BF16_NAN_BITS
    return PagedCache(k_pages, v_pages, bt, torch.tensor(lens, dtype=torch.int32), num_pages, ks, vs)


@dataclass
class DecodeInputs:
    q: torch.Tensor  # [B, Hq, D] bf16
    cache: PagedCache
    sinks: Optional[torch.Tensor]  # [Hq] float32 or None
    scale: float
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int

    @property
    def seq_lens(self) -> torch.Tensor:
        return self.cache.lens

    def kv_bytes(self, window: int = 0) -> int:
        """Bytes of K and V the attention must read: every cached token (with a sliding
        window, the last `window` of each sequence), both tensors."""
        lens = self.cache.lens.long()
        if window > 0:
            lens = lens.clamp(max=window)
        elem = 1 if self.cache.fp8 else 2
        return int(lens.sum()) * 2 * self.num_kv_heads * self.head_dim * elem


def make_decode(lens_spec, batch: int, num_qo_heads: int, num_kv_heads: int, head_dim: int,
                seed: int = 0, sinks: bool = True, scale: Optional[float] = None,
                poison: bool = True, distractor_frac: float = 0.05,
                kv_dtype: str = "bf16", fp8_unit_scales: bool = False) -> DecodeInputs:
    """kv_dtype "bf16" or "fp8" (E4M3 codes with per-KV-head scales; fp8_unit_scales:
    all scales 1, the codes then encode the N(0,1) values directly)."""
    lens = draw_lengths(lens_spec, batch, seed)
    cache = make_paged_cache(lens, num_kv_heads, head_dim, seed, distractor_frac, poison,
                             kv_dtype=kv_dtype, fp8_unit_scales=fp8_unit_scales)
    q = normal_bf16((batch, num_qo_heads, head_dim), seed, _S_Q)
    s = torch.from_numpy(normal_f32(num_qo_heads, seed, _S_SINK)) if sinks else None
    sc = scale if scale is not None else 1.0 / math.sqrt(head_dim)
    return DecodeInputs(q, cache, s, sc, num_qo_heads, num_kv_heads, head_dim)


def new_rows(batch: int, num_kv_heads: int, head_dim: int, seed: int = 0):
    """The new token's K and V rows of every sequence of a decode step, bf16 [B, Hkv, D]
    ~ N(0, 1) (for the decode with append)."""
    shape = (batch, num_kv_heads, head_dim)
    return normal_bf16(shape, seed + 7919, _S_KNEW), normal_bf16(shape, seed + 7919, _S_VNEW)


@dataclass
class PrefillInputs:
    q: torch.Tensor  # [T, Hq, D] bf16 (new tokens, packed)
    k: torch.Tensor  # [T, Hkv, D]
    v: torch.Tensor  # [T, Hkv, D]
    cu_seqlens: torch.Tensor  # [n+1] int32
    new_lens: list[int]
    prefix: Optional[PagedCache]  # pages already holding each request's prefix
    sinks: Optional[torch.Tensor]
    scale: float
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    prefix_lens: list[int] = field(default_factory=list)

    def causal_pairs(self, window: int = 0) -> int:
        """Number of (query, key) pairs the attention visits: prefix keys plus the causal
        triangle; with a sliding window, min(window, position + 1) keys per query."""
        pre = self.prefix_lens or [0] * len(self.new_lens)
        if window <= 0:
            return sum(L * P + L * (L + 1) // 2 for L, P in zip(self.new_lens, pre))
        total = 0
        for L, P in zip(self.new_lens, pre):
            # query t sees min(window, P + t + 1) keys: the ramp part, then window each
            ramp = max(0, min(L, window - P))  # queries with P + t + 1 <= window
            total += sum(P + t + 1 for t in range(ramp)) + (L - ramp) * window
        return total

    def flops(self, window: int = 0) -> int:
        """2 flops per multiply-add, for Q.K^T and P.V over the visited pairs."""
        return 4 * self.head_dim * self.num_qo_heads * self.causal_pairs(window)

    def noncausal_flops(self) -> int:
        """The same count when every query sees its whole request (L^2 pairs per request)."""
        return 4 * self.head_dim * self.num_qo_heads * sum(L * L for L in self.new_lens)


def make_prefill(new_lens: list[int], num_qo_heads: int, num_kv_heads: int, head_dim: int,
                 seed: int = 0, sinks: bool = True, scale: Optional[float] = None,
                 prefix_lens: Optional[list[int]] = None, poison: bool = True,
                 extra_pages_per_seq: int = 0, prefix_kv_dtype: str = "bf16",
                 fp8_unit_scales: bool = False) -> PrefillInputs:
    """Packed ragged prefill; with prefix_lens, each request already has that many
    tokens in paged HND pages (chunked prefill), bf16 or (prefix_kv_dtype "fp8") E4M3
    codes with per-KV-head scales.  extra_pages_per_seq widens each block-table row so
    the new tokens can be appended after the prefix."""
    T = sum(new_lens)
    cu = torch.zeros(len(new_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(new_lens, dtype=torch.int64), 0).to(torch.int32)
    q = normal_bf16((T, num_qo_heads, head_dim), seed, _S_Q)
    k = normal_bf16((T, num_kv_heads, head_dim), seed, _S_KNEW)
    v = normal_bf16((T, num_kv_heads, head_dim), seed, _S_VNEW)
    s = torch.from_numpy(normal_f32(num_qo_heads, seed, _S_SINK)) if sinks else None
    sc = scale if scale is not None else 1.0 / math.sqrt(head_dim)
    prefix = None
    if prefix_lens is not None:
        maxp = max(1, max((P + PAGE_SIZE - 1) // PAGE_SIZE for P in prefix_lens)) + extra_pages_per_seq
        prefix = make_paged_cache(prefix_lens, num_kv_heads, head_dim, seed ^ 0x5EED, poison=poison,
                                  max_pages_per_seq=maxp, kv_dtype=prefix_kv_dtype,
                                  fp8_unit_scales=fp8_unit_scales)
    return PrefillInputs(q, k, v, cu, list(new_lens), prefix, s, sc, num_qo_heads, num_kv_heads,
                         head_dim, list(prefix_lens) if prefix_lens is not None else [])


@dataclass
class AppendInputs:
    """New K/V rows plus a page pool with room for them after each sequence's start position."""
    k: torch.Tensor  # [T, Hkv, D]
    v: torch.Tensor
    cu_seqlens: torch.Tensor
    start_pos: torch.Tensor  # [n] int32
    cache: PagedCache  # pool the rows are scattered into (block table covers start_pos + len)


def make_append(new_lens: list[int], start_pos: list[int], num_kv_heads: int, head_dim: int,
                seed: int = 0, kv_dtype: str = "bf16") -> AppendInputs:
    T = sum(new_lens)
    cu = torch.zeros(len(new_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(new_lens, dtype=torch.int64), 0).to(torch.int32)
    k = normal_bf16((T, num_kv_heads, head_dim), seed, _S_KNEW)
    v = normal_bf16((T, num_kv_heads, head_dim), seed, _S_VNEW)
    totals = [s + L for s, L in zip(start_pos, new_lens)]
    cache = make_paged_cache(totals, num_kv_heads, head_dim, seed, poison=True, kv_dtype=kv_dtype)
    return AppendInputs(k, v, cu, torch.tensor(start_pos, dtype=torch.int32), cache)


# Named workloads: the shapes the attention is used at (gpt-oss and Qwen3-235B
# attention layers) plus a tiny one for exhaustive checks.
WORKLOADS = {
    "tiny_decode": dict(kind="decode", batch=4, lens=[1, 17, 64, 129], num_qo_heads=8,
                        num_kv_heads=2, head_dim=64, sinks=True),
    "gptoss_decode": dict(kind="decode", batch=64, lens=("uniform", 512, 8192), num_qo_heads=64,
                          num_kv_heads=8, head_dim=64, sinks=True),
    "gptoss_prefill": dict(kind="prefill", lens=[4096, 2048, 1024, 512], num_qo_heads=64,
                           num_kv_heads=8, head_dim=64, sinks=True),
    "qwen3_decode": dict(kind="decode", batch=128, lens=("uniform", 1024, 32768), num_qo_heads=64,
                         num_kv_heads=4, head_dim=128, sinks=False),
    "longctx_decode": dict(kind="decode", batch=256, lens=("loguniform", 128, 131072),
                           num_qo_heads=64, num_kv_heads=8, head_dim=64, sinks=True),
    "longctx_chunked": dict(kind="chunked", lens=[512] * 8, prefix_lens=[16384] * 8,
                            num_qo_heads=64, num_kv_heads=8, head_dim=64, sinks=True),
    # the chunked prefill over an FP8 E4M3 prefix cache
    "longctx_chunked_fp8": dict(kind="chunked", lens=[512] * 8, prefix_lens=[16384] * 8,
                                num_qo_heads=64, num_kv_heads=8, head_dim=64, sinks=True,
                                prefix_kv_dtype="fp8"),
    # an embedding model's batch without a KV cache: documents of 4096, 512 and 128 tokens
    # (the lengths of the embedding benchmarks), attention heads of the Qwen3 family's small
    # models (16 query / 8 KV heads, head_dim 128), no sinks; non-causal attention
    "encoder_ragged": dict(kind="prefill", lens=[4096] * 2 + [512] * 12 + [128] * 32,
                           num_qo_heads=16, num_kv_heads=8, head_dim=128, sinks=False,
                           causal=False),
    # the decode shapes over an FP8 E4M3 cache
    "gptoss_decode_fp8": dict(kind="decode", batch=64, lens=("uniform", 512, 8192),
                              num_qo_heads=64, num_kv_heads=8, head_dim=64, sinks=True,
                              kv_dtype="fp8"),
    "qwen3_decode_fp8": dict(kind="decode", batch=128, lens=("uniform", 1024, 32768),
                             num_qo_heads=64, num_kv_heads=4, head_dim=128, sinks=False,
                             kv_dtype="fp8"),
    "longctx_decode_fp8": dict(kind="decode", batch=256, lens=("loguniform", 128, 131072),
                               num_qo_heads=64, num_kv_heads=8, head_dim=64, sinks=True,
                               kv_dtype="fp8"),
}


def make_workload(name: str, seed: int = 0):
    w = dict(WORKLOADS[name])
    kind = w.pop("kind")
    if kind == "decode":
        return make_decode(w["lens"], w["batch"], w["num_qo_heads"], w["num_kv_heads"],
                           w["head_dim"], seed=seed, sinks=w["sinks"],
                           kv_dtype=w.get("kv_dtype", "bf16"))
    if kind == "prefill":
        return make_prefill(w["lens"], w["num_qo_heads"], w["num_kv_heads"], w["head_dim"],
                            seed=seed, sinks=w["sinks"])
    if kind == "chunked":
        return make_prefill(w["lens"], w["num_qo_heads"], w["num_kv_heads"], w["head_dim"],
                            seed=seed, sinks=w["sinks"], prefix_lens=w["prefix_lens"],
                            prefix_kv_dtype=w.get("prefix_kv_dtype", "bf16"))
    raise ValueError(kind)
