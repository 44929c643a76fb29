"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each pin ties the oracle to something it does not share code with:
  * torch's scaled_dot_product_attention in float64 on the CPU, for the sink-free
    case (plain GQA softmax attention) and, through the virtual-token identity
    (a zero key/value row whose additive mask is the sink), for the sink case;
  * closed forms: one key, a hand-derived two-key example (tests/golden), a huge
    sink, an empty sequence;
  * brute force: every row of tiny decode and causal-prefill inputs (head_dim <= 4, at
    most 5 keys) enumerated in plain Python float64 as softmax over the keys plus one
    zero-valued virtual token carrying the sink;
  * invariances: permuting physical pages, splitting the keys and merging, the
    online (streaming) form seeded with the sink, decode == last causal row,
    chunked prefill == trailing rows of a full causal prefill;
  * the append scatter read back through the block table;
  * sliding window: SDPA on the last W keys sliced out explicitly (decode) or with
    a band mask built from the window's definition (prefill, chunked), a window of
    one key against the closed form, a window at least the length against no window;
  * FP8 E4M3 cache: the code table against torch's float8_e4m3fn and the format's
    closed forms; the rounding against torch's cast (in range), exact midpoints
    (ties to the even code) and saturation; decode with power-of-two scales equal,
    bit for bit, to the bf16 decode of the same values; decode with arbitrary
    per-head scales against SDPA on torch-dequantised keys and values; the
    quantising append against torch's cast, slot by slot;
  * rotary embedding with YaRN scaling: at factor 1 the textbook rotation written as a
    complex multiplication; position 0 and pair norms (the YaRN magnitude closed form);
    scores that depend on the position offset only; a hand-derived example
    (tests/golden/rope_yarn.json); bf16 rounding of every bf16 value, exact midpoints
    and torch's float32 cast; the decode step with rotation and append against the
    complex-form rotation, a contiguous copy of the keys and SDPA;
  * chunked prefill over an FP8 prefix: with power-of-two scales equal, bit for bit, to the
    bf16 prefill over the same values (also windowed); with arbitrary per-head scales
    against SDPA on torch-dequantised prefix pages and the bf16 new keys.

test_planted_mistakes_are_caught compiles copies of the oracle source with one
plausible mistake each (dropped sink term, wrong GQA head, off-by-one slot, sign
error, ...) and requires every copy to fail at least one pin.
"""
import json
import math
import os
import tempfile

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from paged_gqa_attention_head_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RTOL, ATOL = 1e-12, 1e-13


def _bf16(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16)


def contiguous_kv(cache: inputs.PagedCache, b: int):
    """Gather sequence b's K/V out of the pages: [Hkv, L, D] float64 (layout only)."""
    L = int(cache.lens[b])
    npg = (L + 15) // 16
    pages = cache.block_table[b, :npg].long()
    Hkv, D = cache.k_pages.shape[1], cache.k_pages.shape[3]
    k = cache.k_pages[pages].permute(1, 0, 2, 3).reshape(Hkv, npg * 16, D)[:, :L]
    v = cache.v_pages[pages].permute(1, 0, 2, 3).reshape(Hkv, npg * 16, D)[:, :L]
    return k.double(), v.double()


def sdpa_with_sink(q, k, v, scale, sinks, mask=None):
    """Library reference: SDPA in float64 over keys plus one zero key/value row whose
    additive mask column holds each head's sink.  q [Hq, M, D], k/v [Hkv, L, D];
    mask [M, L] additive or None.  Returns (out [Hq, M, D], lse [Hq, M])."""
    Hq, M, D = q.shape
    Hkv, L, _ = k.shape
    G = Hq // Hkv
    zero = torch.zeros(Hkv, 1, D, dtype=torch.float64)
    k1, v1 = torch.cat([k, zero], 1), torch.cat([v, zero], 1)
    base = torch.zeros(M, L, dtype=torch.float64) if mask is None else mask
    s = torch.full((Hq,), -math.inf, dtype=torch.float64) if sinks is None else sinks.double()
    full = torch.cat([base.expand(Hq, M, L), s.view(Hq, 1, 1).expand(Hq, M, 1)], 2)
    out = F.scaled_dot_product_attention(q[None], k1[None], v1[None], attn_mask=full[None],
                                         scale=scale, enable_gqa=True)[0]
    kr = k1.repeat_interleave(G, 0)
    logits = scale * torch.matmul(q, kr.transpose(1, 2)) + full
    return out, torch.logsumexp(logits, -1)


# ----------------------------------------------------------------------------- pins
# Each returns None on success and raises AssertionError otherwise, so the same
# checks serve the normal tests and the planted-mistake test.

def pin_decode_sdpa(o, sinks_on: bool):
    w = inputs.make_decode([1, 17, 64, 129, 40], 5, 8, 2, 64, seed=3, sinks=sinks_on)
    out, lse = o.decode(w.q, w.cache.k_pages, w.cache.v_pages, w.cache.block_table, w.seq_lens,
                        w.sinks, w.scale)
    for b in range(5):
        k, v = contiguous_kv(w.cache, b)
        ro, rl = sdpa_with_sink(w.q[b].double()[:, None, :], k, v, w.scale, w.sinks)
        np.testing.assert_allclose(out[b], ro[:, 0].numpy(), rtol=RTOL, atol=ATOL)
        np.testing.assert_allclose(lse[b], rl[:, 0].numpy(), rtol=RTOL, atol=ATOL)


def pin_prefill_sdpa(o, with_prefix: bool):
    new = [5, 33, 1, 20]
    pre = [0, 17, 40, 16] if with_prefix else None
    w = inputs.make_prefill(new, 8, 2, 64, seed=4, sinks=True, prefix_lens=pre)
    kw = {}
    if with_prefix:
        kw = dict(k_pages=w.prefix.k_pages, v_pages=w.prefix.v_pages,
                  prefix_block_table=w.prefix.block_table, prefix_lens=w.prefix.lens)
    out, lse = o.prefill(w.q, w.k, w.v, w.cu_seqlens, w.sinks, w.scale, **kw)
    cu = w.cu_seqlens.tolist()
    for i, L in enumerate(new):
        q = w.q[cu[i]:cu[i + 1]].double().permute(1, 0, 2)
        k = w.k[cu[i]:cu[i + 1]].double().permute(1, 0, 2)
        v = w.v[cu[i]:cu[i + 1]].double().permute(1, 0, 2)
        P = 0
        if with_prefix:
            pk, pv = contiguous_kv(w.prefix, i)
            P = pk.shape[1]
            k, v = torch.cat([pk, k], 1), torch.cat([pv, v], 1)
        t = torch.arange(L)[:, None]
        j = torch.arange(P + L)[None, :]
        mask = torch.where(j <= P + t, 0.0, -math.inf).double()
        ro, rl = sdpa_with_sink(q, k, v, w.scale, w.sinks, mask)
        np.testing.assert_allclose(out[cu[i]:cu[i + 1]], ro.permute(1, 0, 2).numpy(), rtol=RTOL, atol=ATOL)
        np.testing.assert_allclose(lse[cu[i]:cu[i + 1]], rl.T.numpy(), rtol=RTOL, atol=ATOL)


def pin_decode_window_sdpa(o):
    """Decode with window W == SDPA over the last W keys (sliced, not masked), incl.
    W < L, W == L, W > L, W == 1, W and L off the page grid."""
    lens = [1, 17, 64, 129, 40, 200]
    w = inputs.make_decode(lens, len(lens), 8, 2, 64, seed=11, sinks=True)
    for W in (1, 5, 40, 128, 300):
        out, lse = o.decode(w.q, w.cache.k_pages, w.cache.v_pages, w.cache.block_table, w.seq_lens,
                            w.sinks, w.scale, window=W)
        for b, L in enumerate(lens):
            k, v = contiguous_kv(w.cache, b)
            lo = max(0, L - W)
            ro, rl = sdpa_with_sink(w.q[b].double()[:, None, :], k[:, lo:], v[:, lo:], w.scale, w.sinks)
            np.testing.assert_allclose(out[b], ro[:, 0].numpy(), rtol=RTOL, atol=ATOL)
            np.testing.assert_allclose(lse[b], rl[:, 0].numpy(), rtol=RTOL, atol=ATOL)


def pin_prefill_window_sdpa(o):
    """Causal and chunked prefill with window W == SDPA with the band mask
    pos - W < j <= pos (pos = prefix length + t), built here from that definition."""
    new = [5, 33, 1, 20]
    for with_prefix in (False, True):
        pre = [0, 17, 40, 16] if with_prefix else None
        w = inputs.make_prefill(new, 8, 2, 64, seed=12, sinks=True, prefix_lens=pre)
        kw = {}
        if with_prefix:
            kw = dict(k_pages=w.prefix.k_pages, v_pages=w.prefix.v_pages,
                      prefix_block_table=w.prefix.block_table, prefix_lens=w.prefix.lens)
        for W in (1, 7, 24):
            out, lse = o.prefill(w.q, w.k, w.v, w.cu_seqlens, w.sinks, w.scale, window=W, **kw)
            cu = w.cu_seqlens.tolist()
            for i, L in enumerate(new):
                q = w.q[cu[i]:cu[i + 1]].double().permute(1, 0, 2)
                k = w.k[cu[i]:cu[i + 1]].double().permute(1, 0, 2)
                v = w.v[cu[i]:cu[i + 1]].double().permute(1, 0, 2)
                P = 0
                if with_prefix:
                    pk, pv = contiguous_kv(w.prefix, i)
                    P = pk.shape[1]
                    k, v = torch.cat([pk, k], 1), torch.cat([pv, v], 1)
                pos = P + torch.arange(L)[:, None]
                j = torch.arange(P + L)[None, :]
                mask = torch.where((j <= pos) & (j > pos - W), 0.0, -math.inf).double()
                ro, rl = sdpa_with_sink(q, k, v, w.scale, w.sinks, mask)
                np.testing.assert_allclose(out[cu[i]:cu[i + 1]], ro.permute(1, 0, 2).numpy(),
                                           rtol=RTOL, atol=ATOL)
                np.testing.assert_allclose(lse[cu[i]:cu[i + 1]], rl.T.numpy(), rtol=RTOL, atol=ATOL)


def pin_window_special_cases(o):
    """W = 1: only the query's own position, out = v * sigmoid(s - sink); W >= L (and
    W <= 0): identical to no window."""
    lens = [1, 16, 37]
    w = inputs.make_decode(lens, 3, 4, 4, 64, seed=13, sinks=True)
    args = (w.q, w.cache.k_pages, w.cache.v_pages, w.cache.block_table, w.seq_lens, w.sinks, w.scale)
    out1, _ = o.decode(*args, window=1)
    for b, L in enumerate(lens):
        k, v = contiguous_kv(w.cache, b)
        for h in range(4):
            s = w.scale * float(np.dot(w.q[b, h].double().numpy(), k[h, L - 1].numpy()))
            sig = 1.0 / (1.0 + math.exp(-(s - float(w.sinks[h]))))
            np.testing.assert_allclose(out1[b, h], v[h, L - 1].numpy() * sig, rtol=1e-12, atol=1e-14)
    full, full_lse = o.decode(*args)
    for W in (37, 1000, 0, -5):
        outw, lsew = o.decode(*args, window=W)
        assert np.array_equal(outw, full) and np.array_equal(lsew, full_lse)


def pin_single_key(o):
    w = inputs.make_decode([1, 1, 1], 3, 4, 4, 64, seed=5, sinks=True)
    out, lse = o.decode(w.q, w.cache.k_pages, w.cache.v_pages, w.cache.block_table, w.seq_lens,
                        w.sinks, w.scale)
    for b in range(3):
        k, v = contiguous_kv(w.cache, b)
        for h in range(4):
            s = w.scale * float(np.dot(w.q[b, h].double().numpy(), k[h, 0].numpy()))
            sk = float(w.sinks[h])
            sig = 1.0 / (1.0 + math.exp(-(s - sk)))
            np.testing.assert_allclose(out[b, h], v[h, 0].numpy() * sig, rtol=1e-12, atol=1e-14)
            assert abs(lse[b, h] - np.logaddexp(s, sk)) < 1e-12


def pin_two_keys_golden(o):
    g = json.load(open(os.path.join(GOLDEN, "two_keys.json")))
    e = math.e
    env = {"e": e, "log": math.log}
    want = np.array([eval(x, {}, env) for x in g["expected_out"]])
    want_lse = eval(g["expected_lse"], {}, env)
    # one sequence, one head, one page; the two keys sit in slots 0 and 1
    D = g["D"]
    kp = torch.zeros(1, 1, 16, D, dtype=torch.bfloat16)
    vp = torch.zeros(1, 1, 16, D, dtype=torch.bfloat16)
    kp[0, 0, :2] = _bf16(g["k"])
    vp[0, 0, :2] = _bf16(g["v"])
    q = _bf16([[g["q"]]])
    out, lse = o.decode(q, kp, vp, torch.zeros(1, 1, dtype=torch.int32), torch.tensor([2]),
                        torch.tensor([g["sink"]]), g["scale"])
    np.testing.assert_allclose(out[0, 0], want, rtol=1e-14)
    assert abs(lse[0, 0] - want_lse) < 1e-14


def pin_large_sink(o):
    w = inputs.make_decode([1, 17, 64], 3, 4, 2, 64, seed=6, sinks=True)
    for big in (1e4, 30.0):
        s = torch.full((4,), big)
        out, lse = o.decode(w.q, w.cache.k_pages, w.cache.v_pages, w.cache.block_table, w.seq_lens,
                            s, w.scale)
        # |s_j| < 10 here, so every key weighs at most e^(10 - big) relative to the sink
        bound = 64 * math.exp(10.0 - big) * 5.0
        assert np.all(np.abs(out) <= bound)
        assert np.all(np.abs(lse - big) <= 64 * math.exp(10.0 - big))
        if big == 1e4:
            assert np.all(out == 0.0) and np.all(lse == big)


def pin_empty(o):
    w = inputs.make_decode([0, 5], 2, 4, 2, 64, seed=7, sinks=True)
    out, lse = o.decode(w.q, w.cache.k_pages, w.cache.v_pages, w.cache.block_table, w.seq_lens,
                        w.sinks, w.scale)
    assert np.all(out[0] == 0.0)
    np.testing.assert_array_equal(lse[0], w.sinks.double().numpy())
    out2, lse2 = o.decode(w.q, w.cache.k_pages, w.cache.v_pages, w.cache.block_table, w.seq_lens,
                          None, w.scale)
    assert np.all(out2[0] == 0.0) and np.all(np.isneginf(lse2[0]))


def pin_page_permutation(o):
    w = inputs.make_decode([3, 50, 100, 16], 4, 8, 2, 64, seed=8, sinks=True, poison=True)
    c = w.cache
    out, lse = o.decode(w.q, c.k_pages, c.v_pages, c.block_table, w.seq_lens, w.sinks, w.scale)
    perm = torch.randperm(c.num_pages, generator=torch.Generator().manual_seed(1))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(c.num_pages)
    kp2, vp2 = c.k_pages[perm], c.v_pages[perm]  # new page i holds old page perm[i]
    bt2 = torch.where(c.block_table >= 0, inv[c.block_table.clamp(min=0).long()].int(), c.block_table)
    out2, lse2 = o.decode(w.q, kp2, vp2, bt2, w.seq_lens, w.sinks, w.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_decode_vs_prefill_row(o):
    L = 77
    w = inputs.make_prefill([L], 8, 2, 64, seed=9, sinks=True)
    pout, plse = o.prefill(w.q, w.k, w.v, w.cu_seqlens, w.sinks, w.scale)
    for t in (0, 15, 16, 76):
        npg = (t + 1 + 15) // 16
        kp = torch.zeros(npg, 2, 16, 64, dtype=torch.bfloat16)
        vp = torch.zeros(npg, 2, 16, 64, dtype=torch.bfloat16)
        for j in range(t + 1):
            kp[j // 16, :, j % 16] = w.k[j]
            vp[j // 16, :, j % 16] = w.v[j]
        bt = torch.arange(npg, dtype=torch.int32)[None]
        dout, dlse = o.decode(w.q[t:t + 1], kp, vp, bt, torch.tensor([t + 1]), w.sinks, w.scale)
        np.testing.assert_allclose(dout[0], pout[t], rtol=RTOL, atol=ATOL)
        np.testing.assert_allclose(dlse[0], plse[t], rtol=RTOL, atol=ATOL)


def pin_chunked_vs_full(o):
    new, pre = [9, 20], [35, 16]
    w = inputs.make_prefill(new, 8, 2, 64, seed=10, sinks=True, prefix_lens=pre)
    out, lse = o.prefill(w.q, w.k, w.v, w.cu_seqlens, w.sinks, w.scale, k_pages=w.prefix.k_pages,
                         v_pages=w.prefix.v_pages, prefix_block_table=w.prefix.block_table,
                         prefix_lens=w.prefix.lens)
    cu = w.cu_seqlens.tolist()
    for i in range(2):
        pk, pv = contiguous_kv(w.prefix, i)  # [Hkv, P, D]
        kf = torch.cat([pk.permute(1, 0, 2), w.k[cu[i]:cu[i + 1]].double()], 0).to(torch.bfloat16)
        vf = torch.cat([pv.permute(1, 0, 2), w.v[cu[i]:cu[i + 1]].double()], 0).to(torch.bfloat16)
        # full causal prefill over prefix + new; the prefix queries are arbitrary (zeros)
        qf = torch.cat([torch.zeros(pre[i], 8, 64, dtype=torch.bfloat16), w.q[cu[i]:cu[i + 1]]], 0)
        fo, fl = o.prefill(qf, kf, vf, torch.tensor([0, pre[i] + new[i]]), w.sinks, w.scale)
        np.testing.assert_allclose(out[cu[i]:cu[i + 1]], fo[pre[i]:], rtol=RTOL, atol=ATOL)
        np.testing.assert_allclose(lse[cu[i]:cu[i + 1]], fl[pre[i]:], rtol=RTOL, atol=ATOL)


def _one_query(seed=11, n=300):
    q = inputs.normal_bf16((64,), seed, 1)
    k = inputs.normal_bf16((n, 64), seed, 2)
    v = inputs.normal_bf16((n, 64), seed, 3)
    return q, k, v


def _plain(o, q, k, v, scale, sink):
    """The definition, through oracle_prefill's last causal row (one head, one sequence)."""
    n = k.shape[0]
    qq = torch.zeros(n, 1, 64, dtype=torch.bfloat16)
    qq[-1, 0] = q
    out, lse = o.prefill(qq, k[:, None], v[:, None], torch.tensor([0, n]),
                         None if sink == -math.inf else torch.tensor([sink]), 0.125)
    return out[-1, 0], lse[-1, 0]


def pin_split_merge(o):
    q, k, v = _one_query()
    for sink in (0.75, -math.inf, 4.0):  # fp32-exact: sinks are stored as fp32
        ref_out, ref_lse = _plain(o, q, k, v, 0.125, sink)
        for cuts in ([0, 300], [0, 1, 300], [0, 128, 129, 250, 300], [0, 0, 16, 300, 300]):
            parts = [o.partial(q, k, v, 0.125, a, b) for a, b in zip(cuts[:-1], cuts[1:])]
            out, lse = o.merge([p[0] for p in parts], [p[1] for p in parts], [p[2] for p in parts], sink)
            np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-14)
            assert abs(lse - ref_lse) < 1e-12


def pin_online(o):
    q, k, v = _one_query(seed=12)
    for sink in (0.3125, -math.inf, 6.0):  # fp32-exact
        ref_out, ref_lse = _plain(o, q, k, v, 0.125, sink)
        for block, split in ((16, 0), (128, 0), (7, 100), (300, 0), (64, 256)):
            out, lse = o.online(q, k, v, 0.125, sink, block, split)
            np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-14)
            assert abs(lse - ref_lse) < 1e-12


def pin_append_roundtrip(o):
    a = inputs.make_append([5, 16, 33, 0, 1], [0, 7, 16, 3, 31], 2, 64, seed=13)
    c = a.cache
    kp, vp = o.append_kv(a.k, a.v, a.cu_seqlens, c.block_table, a.start_pos, c.k_pages, c.v_pages)
    k_old = c.k_pages.view(torch.int16).numpy().view(np.uint16)
    touched = np.zeros(kp.shape[:1] + kp.shape[2:3], dtype=bool)  # [page, slot]
    cu = a.cu_seqlens.tolist()
    kb = a.k.view(torch.int16).numpy().view(np.uint16)
    vb = a.v.view(torch.int16).numpy().view(np.uint16)
    for i in range(5):
        for t in range(cu[i], cu[i + 1]):
            pos = int(a.start_pos[i]) + t - cu[i]
            pg = int(c.block_table[i, pos // 16])
            assert np.array_equal(kp[pg, :, pos % 16], kb[t]) and np.array_equal(vp[pg, :, pos % 16], vb[t])
            touched[pg, pos % 16] = True
    keep = ~touched
    assert np.array_equal(kp.transpose(0, 2, 1, 3)[keep], k_old.transpose(0, 2, 1, 3)[keep])


def _dequant_pages(pages_u8, scales):
    """torch (library) dequantisation of E4M3 pages [N, Hkv, 16, D] -> float64."""
    vals = pages_u8.view(torch.float8_e4m3fn).to(torch.float64)
    return vals * scales.to(torch.float64).view(1, -1, 1, 1)


def pin_e4m3_table(o):
    codes = np.arange(256, dtype=np.uint8)
    v = o.e4m3_values(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(v, ref)  # NaN positions must agree too
    closed = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
              0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0, 0xB8: -1.0,
              0xFE: -448.0}
    for c, x in closed.items():
        assert v[c] == x, (hex(c), v[c], x)
    assert math.copysign(1.0, v[0x80]) < 0 and v[0x80] == 0.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.all(np.diff(v[:0x7F]) > 0)  # positive codes increase strictly


def pin_e4m3_rounding(o):
    pos = np.arange(0x7F, dtype=np.uint8)  # every finite non-negative code
    vals = torch.from_numpy(pos).view(torch.float8_e4m3fn).float().numpy()
    np.testing.assert_array_equal(o.e4m3_codes(vals), pos)
    np.testing.assert_array_equal(o.e4m3_codes(-vals[1:]), pos[1:] | 0x80)
    # exact midpoints go to the even code; one float32 step either side goes to the nearer one
    mid = ((vals[:-1].astype(np.float64) + vals[1:]) / 2).astype(np.float32)
    lo_c, hi_c = pos[:-1], pos[1:]
    even = np.where(lo_c % 2 == 0, lo_c, hi_c)
    np.testing.assert_array_equal(o.e4m3_codes(mid), even)
    np.testing.assert_array_equal(o.e4m3_codes(np.nextafter(mid, np.float32(0))), lo_c)
    np.testing.assert_array_equal(o.e4m3_codes(np.nextafter(mid, np.float32(1e9))), hi_c)
    sat = np.array([448, 449, 463.9, 464, 480, 1e4, 3e38, np.inf], dtype=np.float32)
    assert np.all(o.e4m3_codes(sat) == 0x7E) and np.all(o.e4m3_codes(-sat) == 0xFE)
    assert np.all(o.e4m3_codes(np.array([np.nan], dtype=np.float32)) & 0x7F == 0x7F)
    assert o.e4m3_codes(np.array([-0.0], dtype=np.float32))[0] == 0x80
    y = np.random.default_rng(5).standard_normal(200_000).astype(np.float32) * np.float32(60)
    y = y[np.abs(y) < 448]
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(o.e4m3_codes(y), ref)


def _fp8_decode_case(seed=21):
    lens = [1, 17, 64, 129, 40, 200]
    return inputs.make_decode(lens, len(lens), 8, 2, 64, seed=seed, sinks=True, kv_dtype="fp8")


def pin_decode_fp8_pow2_is_bf16_decode(o):
    """With power-of-two scales every dequantised value is a bf16 number: the FP8 decode
    must equal the (pinned) bf16 decode of those values exactly."""
    w = _fp8_decode_case()
    c = w.cache
    ks = torch.tensor([2.0 ** -5, 2.0 ** -6], dtype=torch.float32)
    vs = torch.tensor([2.0 ** -4, 2.0 ** -7], dtype=torch.float32)
    kb = _dequant_pages(c.k_pages, ks).to(torch.bfloat16)
    vb = _dequant_pages(c.v_pages, vs).to(torch.bfloat16)
    for W in (0, 1, 40, 300):
        a_out, a_lse = o.decode_fp8(w.q, c.k_pages, c.v_pages, ks, vs, c.block_table, c.lens, w.sinks,
                                    w.scale, window=W)
        b_out, b_lse = o.decode(w.q, kb, vb, c.block_table, c.lens, w.sinks, w.scale, window=W)
        np.testing.assert_array_equal(a_out, b_out)
        np.testing.assert_array_equal(a_lse, b_lse)


def pin_decode_fp8_sdpa(o):
    """Arbitrary per-head scales: SDPA (float64) on keys/values dequantised by torch."""
    w = _fp8_decode_case(seed=22)
    c = w.cache
    deq = inputs.PagedCache(_dequant_pages(c.k_pages, c.k_scale), _dequant_pages(c.v_pages, c.v_scale),
                            c.block_table, c.lens, c.num_pages)
    for W in (0, 40):
        out, lse = o.decode_fp8(w.q, c.k_pages, c.v_pages, c.k_scale, c.v_scale, c.block_table, c.lens,
                                w.sinks, w.scale, window=W)
        for b, L in enumerate(c.lens.tolist()):
            k, v = contiguous_kv(deq, b)
            lo = max(0, L - W) if W else 0
            ro, rl = sdpa_with_sink(w.q[b].double()[:, None, :], k[:, lo:], v[:, lo:], w.scale, w.sinks)
            np.testing.assert_allclose(out[b], ro[:, 0].numpy(), rtol=RTOL, atol=ATOL)
            np.testing.assert_allclose(lse[b], rl[:, 0].numpy(), rtol=RTOL, atol=ATOL)


def pin_append_fp8(o):
    a = inputs.make_append([5, 16, 33, 0, 1], [0, 7, 16, 3, 31], 2, 64, seed=14, kv_dtype="fp8")
    c = a.cache
    kp, vp = o.append_kv_fp8(a.k, a.v, c.k_scale, c.v_scale, a.cu_seqlens, c.block_table, a.start_pos,
                             c.k_pages, c.v_pages)

    def torch_codes(x, s):  # [Hkv, D] bf16 -> codes, torch's cast after the float32 division
        y = x.float() / s.view(-1, 1)
        return y.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()

    touched = np.zeros(kp.shape[:1] + kp.shape[2:3], dtype=bool)
    cu = a.cu_seqlens.tolist()
    for i in range(5):
        for t in range(cu[i], cu[i + 1]):
            pos = int(a.start_pos[i]) + t - cu[i]
            pg = int(c.block_table[i, pos // 16])
            np.testing.assert_array_equal(kp[pg, :, pos % 16], torch_codes(a.k[t], c.k_scale))
            np.testing.assert_array_equal(vp[pg, :, pos % 16], torch_codes(a.v[t], c.v_scale))
            touched[pg, pos % 16] = True
    keep = ~touched
    old = c.k_pages.numpy()
    assert np.array_equal(kp.transpose(0, 2, 1, 3)[keep], old.transpose(0, 2, 1, 3)[keep])


# ---------------------------------------------------------------- rotary embedding (YaRN)
ROPE = dict(base=150000.0, factor=32.0, original_context=4096, beta_fast=32.0, beta_slow=1.0)


def _rope_complex(x, pos, theta, mscale):
    """Textbook form of the NeoX rotation: pair i is the complex number
    x[i] + j x[i + D/2], multiplied by mscale e^(j p theta_i).  x [n, H, D] float64."""
    half = x.shape[-1] // 2
    z = x[..., :half] + 1j * x[..., half:]
    z = z * (mscale * np.exp(1j * np.asarray(pos, dtype=np.float64)[:, None, None] * theta))
    return np.concatenate([z.real, z.imag], axis=-1)


def pin_rope_plain_is_textbook(o):
    # factor 1: no YaRN blend and mscale 1, plain NeoX rotary with w_i = base^(-2i/D)
    for D in (64, 128):
        x = inputs.normal_bf16((5, 3, D), seed=31, stream=1)
        pos = np.array([0, 1, 17, 4095, 131071])
        got = o.rope(x, pos, base=10000.0, factor=1.0)
        theta = 10000.0 ** (-2.0 * np.arange(D // 2) / D)
        want = _rope_complex(x.double().numpy(), pos, theta, 1.0)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-9)


def pin_rope_position_zero_and_norms(o):
    x = inputs.normal_bf16((4, 2, 64), seed=32, stream=1)
    xd = x.double().numpy()
    ms = 1.0 + 0.1 * math.log(ROPE["factor"])
    got0 = o.rope(x, np.zeros(4, dtype=np.int64), **ROPE)
    np.testing.assert_allclose(got0, ms * xd, rtol=1e-15, atol=0)
    got = o.rope(x, np.array([3, 900, 20000, 131000]), **ROPE)
    n_in = np.hypot(xd[..., :32], xd[..., 32:])
    n_out = np.hypot(got[..., :32], got[..., 32:])
    np.testing.assert_allclose(n_out, ms * n_in, rtol=1e-12, atol=1e-15)


def pin_rope_relative_position(o):
    # <R(m) q, R(n) k> = mscale <R(m - n) q, k>: the scores depend on the offset only
    q = inputs.normal_bf16((1, 1, 64), seed=33, stream=1)
    k = inputs.normal_bf16((1, 1, 64), seed=33, stream=2)
    kd = k.double().numpy().reshape(-1)
    ms = 1.0 + 0.1 * math.log(ROPE["factor"])
    for m, n in ((10, 3), (5000, 4990), (131071, 65536), (7, 7)):
        a = o.rope(q, [m], **ROPE).reshape(-1)
        b = o.rope(k, [n], **ROPE).reshape(-1)
        c = o.rope(q, [m - n], **ROPE).reshape(-1)
        assert abs(a @ b - ms * (c @ kd)) <= 1e-9 * (1 + abs(a @ b)), (m, n)


def pin_rope_golden(o):
    g = json.load(open(os.path.join(GOLDEN, "rope_yarn.json")))
    prm = g["params"]
    D = prm["head_dim"]
    env = {"log": math.log}
    ms = eval(g["mscale"], {}, env)
    kw = dict(base=prm["base"], factor=prm["factor"], original_context=prm["original_context"],
              beta_fast=prm["beta_fast"], beta_slow=prm["beta_slow"])
    theta, mscale = o.rope_freqs(D, **kw)
    assert abs(mscale - ms) < 1e-15
    for case in g["cases"]:
        i, p = case["i"], case["p"]
        th = eval(case["theta"], {}, env)
        assert abs(theta[i] - th) <= 1e-15 * th, case
        x = torch.zeros(2, 1, D, dtype=torch.bfloat16)
        x[0, 0, i] = 1.0
        x[1, 0, i + D // 2] = 1.0
        got = o.rope(x, [p, p], **kw)
        c, s = ms * math.cos(p * th), ms * math.sin(p * th)
        np.testing.assert_allclose([got[0, 0, i], got[0, 0, i + D // 2]], [c, s], atol=1e-12)
        np.testing.assert_allclose([got[1, 0, i], got[1, 0, i + D // 2]], [-s, c], atol=1e-12)
        others = np.delete(got[0, 0], [i, i + D // 2])
        assert np.all(others == 0.0)


def pin_bf16_round(o):
    # every bf16 value maps to itself
    bits = np.arange(65536, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    finite = np.isfinite(vals)
    got = o.bf16_round(vals[finite].astype(np.float64))
    want = bits[finite].astype(np.uint16)
    want[want == 0x8000] = 0x8000  # -0 stays -0
    assert np.array_equal(got, want)
    # exact midpoints between neighbours go to the even one; one double step off goes nearer
    lo = (np.arange(0x0001, 0x7F7F, 97, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    hi = ((np.arange(0x0001, 0x7F7F, 97, dtype=np.uint32) + 1) << 16).view(np.float32).astype(np.float64)
    mid = (lo + hi) / 2  # exact in double
    lob = (lo.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    hib = lob + 1
    even = np.where(lob % 2 == 0, lob, hib)
    assert np.array_equal(o.bf16_round(mid), even)
    assert np.array_equal(o.bf16_round(np.nextafter(mid, -np.inf)), lob)
    assert np.array_equal(o.bf16_round(np.nextafter(mid, np.inf)), hib)
    assert np.array_equal(o.bf16_round(-mid), even | 0x8000)
    # float32 inputs: torch's float32 -> bfloat16 cast (round to nearest even) agrees
    r = np.random.default_rng(3).standard_normal(200000).astype(np.float32) * 37.0
    want = torch.from_numpy(r).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(o.bf16_round(r.astype(np.float64)), want)
    assert o.bf16_round(np.array([3.4e38]))[0] == 0x7F80  # past the largest finite: inf


def pin_decode_append_rope(o):
    # the composed step against an independent path: the complex-number rotation with the
    # (golden-pinned) YaRN frequencies, the (pinned) bf16 rounding, the new rows put into a
    # contiguous copy of each sequence, and SDPA with the sink column
    B, Hq, Hkv, D = 4, 8, 2, 64
    w = inputs.make_decode([1, 17, 64, 300], B, Hq, Hkv, D, seed=34, sinks=True)
    c = w.cache
    kn, vn = inputs.new_rows(B, Hkv, D, seed=34)
    out, lse, kp, vp, q_rot, k_rot = o.decode_append_rope(
        w.q, kn, vn, c.k_pages, c.v_pages, c.block_table, c.lens, w.sinks, w.scale, **ROPE)
    theta, ms = o.rope_freqs(D, **ROPE)
    lens = c.lens.numpy()
    pos = lens - 1
    q_want = o.bf16_round(_rope_complex(w.q.double().numpy(), pos, theta, ms))
    k_want = o.bf16_round(_rope_complex(kn.double().numpy(), pos, theta, ms))
    assert np.array_equal(q_rot, q_want) and np.array_equal(k_rot, k_want)
    to_t = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    for b in range(B):
        k, v = contiguous_kv(c, b)
        k, v = k.clone(), v.clone()
        k[:, pos[b]] = to_t(k_want[b]).double()
        v[:, pos[b]] = vn[b].double()
        ref, ref_lse = sdpa_with_sink(to_t(q_want[b]).double()[:, None], k, v, w.scale, w.sinks)
        np.testing.assert_allclose(out[b], ref[:, 0].numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_lse[:, 0].numpy(), rtol=0, atol=1e-10)
        # the new slot holds the rotated key and the given value; nothing else changed
        pg = int(c.block_table[b, pos[b] // 16])
        assert np.array_equal(kp[pg, :, pos[b] % 16], k_want[b])
        assert np.array_equal(vp[pg, :, pos[b] % 16], vn[b].view(torch.int16).numpy().view(np.uint16))


# ---------------------------------------------------------------- chunked prefill, FP8 prefix
def _fp8_prefill_case(pow2: bool, seed: int):
    p = inputs.make_prefill([70, 1, 33], 8, 2, 64, seed=seed, sinks=True, prefix_lens=[100, 37, 0],
                            prefix_kv_dtype="fp8")
    c = p.prefix
    if pow2:
        c.k_scale = torch.tensor([0.25, 2.0], dtype=torch.float32)
        c.v_scale = torch.tensor([0.5, 0.125], dtype=torch.float32)
    return p, c


def _bf16_pages_from_fp8(pages_u8, scales):
    vals = pages_u8.view(torch.float8_e4m3fn).float() * scales.view(1, -1, 1, 1)
    return vals.to(torch.bfloat16)


def pin_prefill_fp8_pow2_is_bf16_prefill(o):
    # with power-of-two scales every prefix value is a bf16 number: the FP8 prefill must equal
    # the bf16 prefill over pages holding those values, bit for bit (also with a window)
    p, c = _fp8_prefill_case(True, 41)
    kb, vb = _bf16_pages_from_fp8(c.k_pages, c.k_scale), _bf16_pages_from_fp8(c.v_pages, c.v_scale)
    for window in (0, 50):
        got = o.prefill_fp8(p.q, p.k, p.v, p.cu_seqlens, p.sinks, p.scale, c.k_pages, c.v_pages,
                            c.k_scale, c.v_scale, c.block_table, c.lens, window=window)
        want = o.prefill(p.q, p.k, p.v, p.cu_seqlens, p.sinks, p.scale, kb, vb, c.block_table, c.lens,
                         window=window)
        assert np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1]), window


def pin_prefill_fp8_sdpa(o):
    # arbitrary per-head scales: SDPA over [torch-dequantised prefix ; new bf16 keys] with the
    # bottom-right causal mask and the sink column
    p, c = _fp8_prefill_case(False, 42)
    out, lse = o.prefill_fp8(p.q, p.k, p.v, p.cu_seqlens, p.sinks, p.scale, c.k_pages, c.v_pages,
                             c.k_scale, c.v_scale, c.block_table, c.lens)
    kd = c.k_pages.view(torch.float8_e4m3fn).double() * c.k_scale.double().view(1, -1, 1, 1)
    vd = c.v_pages.view(torch.float8_e4m3fn).double() * c.v_scale.double().view(1, -1, 1, 1)
    cu = p.cu_seqlens.tolist()
    for i in range(3):
        P, L = int(c.lens[i]), cu[i + 1] - cu[i]
        npg = (P + 15) // 16
        pages = c.block_table[i, :npg].long()
        kpre = kd[pages].permute(1, 0, 2, 3).reshape(2, npg * 16, 64)[:, :P]
        vpre = vd[pages].permute(1, 0, 2, 3).reshape(2, npg * 16, 64)[:, :P]
        kn = p.k[cu[i]:cu[i + 1]].double().permute(1, 0, 2)
        vn = p.v[cu[i]:cu[i + 1]].double().permute(1, 0, 2)
        k = torch.cat([kpre, kn], 1)
        v = torch.cat([vpre, vn], 1)
        q = p.q[cu[i]:cu[i + 1]].double().permute(1, 0, 2)
        pos = P + torch.arange(L)[:, None]
        mask = torch.where(torch.arange(P + L)[None, :] <= pos, 0.0, -math.inf).double()
        ref, ref_lse = sdpa_with_sink(q, k, v, p.scale, p.sinks, mask=mask)
        np.testing.assert_allclose(out[cu[i]:cu[i + 1]], ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(lse[cu[i]:cu[i + 1]], ref_lse.permute(1, 0).numpy(), rtol=0, atol=1e-10)


def pin_brute_force_tiny(o):
    # every decode, causal-prefill and non-causal-prefill row of tiny inputs (head_dim <= 4, at most 5 keys)
    # enumerated in plain Python float64 in the virtual-token form: the sink is one more
    # logit whose value row is zero; probabilities p_j = exp(x_j - logsumexp(x)) with the
    # sums taken by math.fsum (exactly rounded)
    def attend(q, keys, vals, scale, sink):
        xs = [scale * math.fsum(a * b for a, b in zip(q, k)) for k in keys] + [sink]
        D = len(q)
        if max(xs) == -math.inf:
            return [0.0] * D, -math.inf
        top = max(xs)
        lse = top + math.log(math.fsum(math.exp(x - top) for x in xs))
        ps = [math.exp(x - lse) for x in xs]
        out = [math.fsum(p * v[d] for p, v in zip(ps, vals + [[0.0] * D])) for d in range(D)]
        return out, lse

    rng = np.random.default_rng(17)
    for D in (1, 2, 4):
        for trial in range(3):
            # decode: 3 sequences of 0..5 keys, 4 q heads / 2 KV heads, one page each
            lens = [int(x) for x in rng.integers(0, 6, size=3)]
            q = torch.from_numpy(rng.standard_normal((3, 4, D)).astype(np.float32)).to(torch.bfloat16)
            kp = torch.from_numpy(rng.standard_normal((3, 2, 16, D)).astype(np.float32)).to(torch.bfloat16)
            vp = torch.from_numpy(rng.standard_normal((3, 2, 16, D)).astype(np.float32)).to(torch.bfloat16)
            bt = torch.tensor([[2], [0], [1]], dtype=torch.int32)
            sk = torch.from_numpy(rng.standard_normal(4).astype(np.float32)) if trial != 1 else None
            scale = 0.7
            out, lse = o.decode(q, kp, vp, bt, torch.tensor(lens, dtype=torch.int32), sk, scale)
            for b in range(3):
                for h in range(4):
                    g = h // 2
                    keys = [kp[bt[b, 0], g, j].double().tolist() for j in range(lens[b])]
                    vals = [vp[bt[b, 0], g, j].double().tolist() for j in range(lens[b])]
                    sink = -math.inf if sk is None else float(sk[h])
                    ro, rl = attend(q[b, h].double().tolist(), keys, vals, scale, sink)
                    np.testing.assert_allclose(out[b, h], ro, rtol=1e-12, atol=1e-14)
                    assert (rl == lse[b, h]) if rl == -math.inf else abs(rl - lse[b, h]) < 1e-12
            # causal prefill: one request of 5 tokens, 2 q heads / 1 KV head
            T = 5
            qq = torch.from_numpy(rng.standard_normal((T, 2, D)).astype(np.float32)).to(torch.bfloat16)
            kk = torch.from_numpy(rng.standard_normal((T, 1, D)).astype(np.float32)).to(torch.bfloat16)
            vv = torch.from_numpy(rng.standard_normal((T, 1, D)).astype(np.float32)).to(torch.bfloat16)
            sk2 = torch.from_numpy(rng.standard_normal(2).astype(np.float32))
            out, lse = o.prefill(qq, kk, vv, torch.tensor([0, T], dtype=torch.int32), sk2, scale)
            for t in range(T):
                for h in range(2):
                    keys = [kk[j, 0].double().tolist() for j in range(t + 1)]
                    vals = [vv[j, 0].double().tolist() for j in range(t + 1)]
                    ro, rl = attend(qq[t, h].double().tolist(), keys, vals, scale, float(sk2[h]))
                    np.testing.assert_allclose(out[t, h], ro, rtol=1e-12, atol=1e-14)
                    assert abs(rl - lse[t, h]) < 1e-12
            # non-causal prefill of the same request: every row sees all 5 keys
            out, lse = o.prefill_noncausal(qq, kk, vv, torch.tensor([0, T], dtype=torch.int32), sk2, scale)
            keys = [kk[j, 0].double().tolist() for j in range(T)]
            vals = [vv[j, 0].double().tolist() for j in range(T)]
            for t in range(T):
                for h in range(2):
                    ro, rl = attend(qq[t, h].double().tolist(), keys, vals, scale, float(sk2[h]))
                    np.testing.assert_allclose(out[t, h], ro, rtol=1e-12, atol=1e-14)
                    assert abs(rl - lse[t, h]) < 1e-12


def pin_noncausal_sdpa(o):
    # every query of a sequence sees all of its tokens: SDPA with no mask beyond the
    # sequence boundary, with sinks and without
    new = [5, 33, 1, 20]
    for sinks_on in (True, False):
        w = inputs.make_prefill(new, 8, 2, 64, seed=12, sinks=sinks_on)
        out, lse = o.prefill_noncausal(w.q, w.k, w.v, w.cu_seqlens, w.sinks, w.scale)
        cu = w.cu_seqlens.tolist()
        for i in range(len(new)):
            q = w.q[cu[i]:cu[i + 1]].double().permute(1, 0, 2)
            k = w.k[cu[i]:cu[i + 1]].double().permute(1, 0, 2)
            v = w.v[cu[i]:cu[i + 1]].double().permute(1, 0, 2)
            ro, rl = sdpa_with_sink(q, k, v, w.scale, w.sinks)
            np.testing.assert_allclose(out[cu[i]:cu[i + 1]], ro.permute(1, 0, 2).numpy(), rtol=RTOL, atol=ATOL)
            np.testing.assert_allclose(lse[cu[i]:cu[i + 1]], rl.T.numpy(), rtol=RTOL, atol=ATOL)


def pin_noncausal_vs_causal_and_permutation(o):
    # (a) the last query of a sequence sees the same keys either way, so its row equals the
    # causal prefill's; (b) permuting a sequence's key/value rows together leaves every
    # output unchanged (the key set is the whole sequence), while the queries' outputs
    # move with the queries
    new = [40, 17, 1]
    w = inputs.make_prefill(new, 8, 2, 64, seed=13, sinks=True)
    out, lse = o.prefill_noncausal(w.q, w.k, w.v, w.cu_seqlens, w.sinks, w.scale)
    cout, clse = o.prefill(w.q, w.k, w.v, w.cu_seqlens, w.sinks, w.scale)
    cu = w.cu_seqlens.tolist()
    for i in range(len(new)):
        t = cu[i + 1] - 1
        np.testing.assert_allclose(out[t], cout[t], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse[t], clse[t], rtol=1e-12, atol=1e-14)
    assert not np.allclose(out[cu[0]], cout[cu[0]], rtol=1e-3, atol=1e-3)  # first row differs
    perm = torch.arange(w.q.shape[0])
    perm[cu[0]:cu[1]] = cu[0] + torch.randperm(new[0], generator=torch.Generator().manual_seed(1))
    pout, plse = o.prefill_noncausal(w.q, w.k[perm], w.v[perm], w.cu_seqlens, w.sinks, w.scale)
    np.testing.assert_allclose(pout, out, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(plse, lse, rtol=1e-12, atol=1e-14)
    qout, qlse = o.prefill_noncausal(w.q[perm], w.k, w.v, w.cu_seqlens, w.sinks, w.scale)
    np.testing.assert_allclose(qout, out[perm.numpy()], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(qlse, lse[perm.numpy()], rtol=1e-12, atol=1e-14)


PINS = {
    "decode_sdpa_nosink": lambda o: pin_decode_sdpa(o, False),
    "decode_sdpa_sink": lambda o: pin_decode_sdpa(o, True),
    "prefill_sdpa": lambda o: pin_prefill_sdpa(o, False),
    "chunked_sdpa": lambda o: pin_prefill_sdpa(o, True),
    "single_key": pin_single_key,
    "two_keys_golden": pin_two_keys_golden,
    "large_sink": pin_large_sink,
    "empty": pin_empty,
    "page_permutation": pin_page_permutation,
    "decode_vs_prefill_row": pin_decode_vs_prefill_row,
    "chunked_vs_full": pin_chunked_vs_full,
    "split_merge": pin_split_merge,
    "online": pin_online,
    "append_roundtrip": pin_append_roundtrip,
    "decode_window_sdpa": pin_decode_window_sdpa,
    "prefill_window_sdpa": pin_prefill_window_sdpa,
    "window_special_cases": pin_window_special_cases,
    "e4m3_table": pin_e4m3_table,
    "e4m3_rounding": pin_e4m3_rounding,
    "decode_fp8_pow2_is_bf16_decode": pin_decode_fp8_pow2_is_bf16_decode,
    "decode_fp8_sdpa": pin_decode_fp8_sdpa,
    "append_fp8": pin_append_fp8,
    "rope_plain_is_textbook": pin_rope_plain_is_textbook,
    "rope_position_zero_and_norms": pin_rope_position_zero_and_norms,
    "rope_relative_position": pin_rope_relative_position,
    "rope_golden": pin_rope_golden,
    "bf16_round": pin_bf16_round,
    "decode_append_rope": pin_decode_append_rope,
    "prefill_fp8_pow2_is_bf16_prefill": pin_prefill_fp8_pow2_is_bf16_prefill,
    "prefill_fp8_sdpa": pin_prefill_fp8_sdpa,
    "brute_force_tiny": pin_brute_force_tiny,
    "noncausal_sdpa": pin_noncausal_sdpa,
    "noncausal_vs_causal_and_permutation": pin_noncausal_vs_causal_and_permutation,
}


@pytest.mark.parametrize("name", sorted(PINS))
def test_pin(oracle_mod, name):
    PINS[name](oracle_mod)


# (what the mistake is, text in the oracle source, its replacement)
MUTATIONS = [
    ("sink dropped from the denominator", "double den = exp(sink - m);", "double den = 0.0;"),
    ("sink left out of the running max", "    double m = sink;\n    for (int64_t j = 0; j < n; ++j) {",
     "    double m = -INFINITY;\n    for (int64_t j = 0; j < n; ++j) {"),
    ("sink multiplied by the scale (decode)", "attend(q + bh * D, D, scale, sink_of(sinks, h)",
     "attend(q + bh * D, D, scale, scale * sink_of(sinks, h)"),
    ("GQA head taken modulo (decode)", "h = (int)(bh % Hq), g = h / G;", "h = (int)(bh % Hq), g = h % Hkv;"),
    ("GQA head taken modulo (prefill)", "g = h / G, i = seq_of[t];", "g = h % Hkv, i = seq_of[t];"),
    ("slot off by one (decode keys)",
     "krow[j - lo] = page_row(k_pages, pg, Hkv, P, D, g, (int)(j % P));\n                vrow[j - lo] = page_row(v_pages, pg, Hkv, P, D, g, (int)(j % P));\n            }\n            attend(q + bh",
     "krow[j - lo] = page_row(k_pages, pg, Hkv, P, D, g, (int)((j + 1) % P));\n                vrow[j - lo] = page_row(v_pages, pg, Hkv, P, D, g, (int)(j % P));\n            }\n            attend(q + bh"),
    ("exponent sign flipped", "double w = exp(s[j] - m);", "double w = exp(m - s[j]);"),
    ("lse without the max", "*lse = m + log(den);\n}", "*lse = log(den);\n}"),
    ("keys used as values", "out[d] += w * bf16_to_double(vrow[j][d]);", "out[d] += w * bf16_to_double(krow[j][d]);"),
    ("causal window shifted by one", "krow[j - lo] = k + (row * Hkv + g) * D;",
     "krow[j - lo] = k + ((row > 0 ? row - 1 : row) * Hkv + g) * D;"),
    ("prefix page slot off by one",
     "krow[j - lo] = page_row(k_pages, pg, Hkv, P, D, g, (int)(j % P));\n                    vrow[j - lo] = page_row(v_pages, pg, Hkv, P, D, g, (int)(j % P));\n                } else {",
     "krow[j - lo] = page_row(k_pages, pg, Hkv, P, D, g, (int)((j + 1) % P));\n                    vrow[j - lo] = page_row(v_pages, pg, Hkv, P, D, g, (int)(j % P));\n                } else {"),
    ("decode window one key too short",
     "const int64_t lo = (window > 0 && L > window) ? L - window : 0;",
     "const int64_t lo = (window > 0 && L > window) ? L - window + 1 : 0;"),
    ("decode window ignored",
     "const int64_t lo = (window > 0 && L > window) ? L - window : 0;",
     "const int64_t lo = 0;"),
    ("prefill window one key too long",
     "const int64_t lo = (window > 0 && pos + 1 > window) ? pos + 1 - window : 0;",
     "const int64_t lo = (window > 0 && pos > window) ? pos - window : 0;"),
    ("prefill window measured from the new tokens only",
     "const int64_t lo = (window > 0 && pos + 1 > window) ? pos + 1 - window : 0;",
     "const int64_t lo = (window > 0 && tl + 1 > window) ? Pi + tl + 1 - window : 0;"),
    ("merge ignores the partial's max", "den += l[s] * w;", "den += l[s];"),
    ("online form skips the rescale", "den *= r;", "den *= 1.0;"),
    ("e4m3 subnormals decoded as normals", "mag = ldexp((double)m, -9);", "mag = ldexp(8.0 + m, -10);"),
    ("e4m3 exponent bias off by one", "mag = ldexp(8.0 + m, e - 10);", "mag = ldexp(8.0 + m, e - 9);"),
    ("e4m3 rounding ties away from zero", "double q = rint(ldexp(a, 3 - e));",
     "double q = round(ldexp(a, 3 - e));"),
    ("e4m3 subnormal rounding on the wrong grid", "double q = rint(ldexp(a, 9));",
     "double q = rint(ldexp(a, 8));"),
    ("e4m3 overflow saturates to NaN", "return (uint8_t)(sign | 0x7E); /* saturation",
     "return (uint8_t)(sign | 0x7F); /* saturation"),
    ("fp8 decode ignores the V scale", "out[d] += e * (vscale * oracle_e4m3_value(vrow[j][d]));",
     "out[d] += e * oracle_e4m3_value(vrow[j][d]);"),
    ("fp8 decode takes head 0's K scale", "k_scale ? (double)k_scale[g] : 1.0",
     "k_scale ? (double)k_scale[0] : 1.0"),
    ("fp8 decode drops the sink", "double z = exp(sink - top);", "double z = 0.0;"),
    ("fp8 decode ignores the window",
     "const int64_t first = (window > 0 && L > window) ? L - window : 0;", "const int64_t first = 0;"),
    ("fp8 append quantises V with the K scale", "v_pages[off + d] = oracle_e4m3_code(vx / vs);",
     "v_pages[off + d] = oracle_e4m3_code(vx / ks);"),
    ("rope pairs neighbours (GPT-J layout) instead of i, i + D/2",
     "const double x0 = bf16_to_double(xr[i]), x1 = bf16_to_double(xr[i + D / 2]);",
     "const double x0 = bf16_to_double(xr[(2 * i) % D]), x1 = bf16_to_double(xr[(2 * i + 1) % D]);"),
    ("rope rotates the other way", "o[i] = ms * (x0 * c - x1 * s);", "o[i] = ms * (x0 * c + x1 * s);"),
    ("rope frequency exponent i/D", "const double w = pow(base, -2.0 * i / D);",
     "const double w = pow(base, -1.0 * i / D);"),
    ("rope blend reversed", "theta[i] = (1.0 - y) * w + y * (w / factor);",
     "theta[i] = y * w + (1.0 - y) * (w / factor);"),
    ("rope correction dims not rounded",
     "double lo = floor(D * log(L0 / (two_pi * beta_fast)) / (2.0 * log(base)));",
     "double lo = (D * log(L0 / (two_pi * beta_fast)) / (2.0 * log(base)));"),
    ("rope slow correction dim taken from beta_fast",
     "double hi = ceil(D * log(L0 / (two_pi * beta_slow)) / (2.0 * log(base)));",
     "double hi = ceil(D * log(L0 / (two_pi * beta_fast)) / (2.0 * log(base)));"),
    ("rope without the YaRN magnitude", "*mscale = 1.0 + 0.1 * log(factor);", "*mscale = 1.0;"),
    ("rope position off by one", "const double a = (double)pos[r] * theta[i];",
     "const double a = (double)(pos[r] + 1) * theta[i];"),
    ("bf16 rounding ties away from zero", "double r = ldexp(rint(ldexp(x, -ulp)), ulp);",
     "double r = ldexp(round(ldexp(x, -ulp)), ulp);"),
    ("bf16 rounding keeps 9 bits", "int ulp = e - 8;", "int ulp = e - 9;"),
    ("fp8 prefill ignores the prefix V scale",
     "out[d] += wt * (vs * oracle_e4m3_value(vp[j][d]));", "out[d] += wt * oracle_e4m3_value(vp[j][d]);"),
    ("fp8 prefill takes the V scale for the prefix keys",
     "dot += bf16_to_double(q[d]) * (ks * oracle_e4m3_value(kp[j][d]));",
     "dot += bf16_to_double(q[d]) * (vs * oracle_e4m3_value(kp[j][d]));"),
    ("fp8 prefill drops the sink", "double z = exp(sink - m); /* the denominator",
     "double z = 0.0; /* the denominator"),
    ("fp8 prefill sees one new key too many", "const int64_t nn = tl + 1 - n0;",
     "const int64_t nn = (tl + 2 <= cu_seqlens[i + 1] - cu_seqlens[i] ? tl + 2 : tl + 1) - n0;"),
    ("fp8 prefill window ignored in the prefix", "const int64_t np = lo < Pi ? Pi - lo : 0;",
     "const int64_t np = Pi;"),
    ("non-causal prefill masks the keys after the query", "len, krow + (h / G) * len",
     "e / Hq + 1, krow + (h / G) * len"),
    ("non-causal prefill GQA head taken modulo", "krow + (h / G) * len", "krow + (h % Hkv) * len"),
    ("non-causal prefill drops the sink", "sink_of(sinks, h), len,", "-INFINITY, len,"),
    ("non-causal prefill reads keys one row late", "krow[g * len + j] = k + ((first + j) * Hkv + g) * D;",
     "krow[g * len + j] = k + ((first + j + 1 < cu_seqlens[n] ? first + j + 1 : first + j) * Hkv + g) * D;"),
    ("append writes the next slot",
     "uint16_t *kd = (uint16_t *)page_row(k_pages, pg, Hkv, P, D, g, (int)(pos % P));",
     "uint16_t *kd = (uint16_t *)page_row(k_pages, pg, Hkv, P, D, g, (int)((pos + 1) % P));"),
]


def test_planted_mistakes_are_caught(oracle_mod):
    src = open(oracle_mod.source_path()).read()
    with tempfile.TemporaryDirectory() as tmp:
        for idx, (what, old, new) in enumerate(MUTATIONS):
            assert src.count(old) == 1, f"mutation anchor not unique: {what}"
            so = oracle_mod.compile_source(src.replace(old, new), tmp, f"mutant{idx}")
            failed = []
            with oracle_mod.using_library(so):
                for name, pin in PINS.items():
                    try:
                        pin(oracle_mod)
                    except (AssertionError, ValueError, FloatingPointError):
                        failed.append(name)
            assert failed, f"no pin caught the planted mistake: {what}"
