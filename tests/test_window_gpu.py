"""Sliding-window attention on the GPU (desc.window = W: a query at position pos sees
the keys at positions pos - W < j <= pos), decode and prefill, against the fp64 oracle
with the same window.  A window at least as long as every query's history must give
exactly the unwindowed result."""
import numpy as np
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs
from tolerances import check_lse, check_out

pytestmark = pytest.mark.gpu


def _decode(sa, w, dev, window):
    c = w.cache
    out, lse = sa.decode(w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), c.block_table.to(dev),
                         c.lens.to(dev), None if w.sinks is None else w.sinks.to(dev), w.scale,
                         window=window)
    torch.cuda.synchronize()
    return out, lse


def _oracle_decode(o, w, window, select=None):
    c = w.cache
    return o.decode(w.q, c.k_pages, c.v_pages, c.block_table, c.lens, w.sinks, w.scale,
                    select=select, window=window)


def _prefill(sa, p, dev, window):
    kw = {}
    if p.prefix is not None:
        kw = dict(k_pages=p.prefix.k_pages.to(dev), v_pages=p.prefix.v_pages.to(dev),
                  prefix_block_table=p.prefix.block_table.to(dev), prefix_lens=p.prefix.lens.to(dev))
    out, lse = sa.prefill(p.q.to(dev), p.k.to(dev), p.v.to(dev), p.cu_seqlens.to(dev),
                          None if p.sinks is None else p.sinks.to(dev), p.scale, window=window, **kw)
    torch.cuda.synchronize()
    return out, lse


def _oracle_prefill(o, p, window, select=None):
    kw = {}
    if p.prefix is not None:
        kw = dict(k_pages=p.prefix.k_pages, v_pages=p.prefix.v_pages,
                  prefix_block_table=p.prefix.block_table, prefix_lens=p.prefix.lens)
    return o.prefill(p.q, p.k, p.v, p.cu_seqlens, p.sinks, p.scale, select=select, window=window,
                     **kw)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("window", [1, 16, 100, 128, 1000])
def test_decode_window(sa, oracle_mod, cuda_dev, D, window):
    lens = [0, 1, 15, 16, 17, 100, 128, 129, 300, 2049, 40000]
    w = inputs.make_decode(lens, len(lens), 4 * (2 if D == 64 else 4), 4, D, seed=60 + window,
                           sinks=D == 64)
    out, lse = _decode(sa, w, cuda_dev, window)
    ro, rl = _oracle_decode(oracle_mod, w, window)
    check_out(out, ro)
    check_lse(lse, rl)
    assert sa.get_status(sa.workspace(0, cuda_dev)) == 0


def test_decode_window_covering_everything_equals_no_window_bitwise(sa, cuda_dev):
    lens = [1, 17, 300, 2049]
    w = inputs.make_decode(lens, 4, 16, 2, 64, seed=61, sinks=True)
    a_out, a_lse = _decode(sa, w, cuda_dev, 0)
    b_out, b_lse = _decode(sa, w, cuda_dev, 2049)
    assert torch.equal(a_out.view(torch.int16), b_out.view(torch.int16))
    assert torch.equal(a_lse, b_lse)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("window", [1, 64, 128, 200])
def test_causal_prefill_window(sa, oracle_mod, cuda_dev, D, window):
    lens = [1, 5, 127, 128, 129, 300, 513]
    p = inputs.make_prefill(lens, 8, 2, D, seed=70 + window, sinks=True)
    out, lse = _prefill(sa, p, cuda_dev, window)
    ro, rl = _oracle_prefill(oracle_mod, p, window)
    check_out(out, ro)
    check_lse(lse, rl)
    assert sa.get_status(sa.workspace(0, cuda_dev, "prefill")) == 0


@pytest.mark.parametrize("window", [1, 100, 128, 1000])
def test_chunked_prefill_window(sa, oracle_mod, cuda_dev, window):
    """The window reaches back into the paged prefix for the first new tokens."""
    new = [1, 64, 130, 5, 256, 7]
    pre = [0, 1, 16, 300, 1000, 4096]
    p = inputs.make_prefill(new, 16, 2, 64, seed=80 + window, sinks=True, prefix_lens=pre)
    out, lse = _prefill(sa, p, cuda_dev, window)
    ro, rl = _oracle_prefill(oracle_mod, p, window)
    check_out(out, ro)
    check_lse(lse, rl)
    assert sa.get_status(sa.workspace(0, cuda_dev, "prefill")) == 0


def test_prefill_window_covering_everything_equals_no_window_bitwise(sa, cuda_dev):
    p = inputs.make_prefill([40, 300], 8, 2, 64, seed=90, sinks=True, prefix_lens=[100, 17])
    a_out, a_lse = _prefill(sa, p, cuda_dev, 0)
    b_out, b_lse = _prefill(sa, p, cuda_dev, 400)
    assert torch.equal(a_out.view(torch.int16), b_out.view(torch.int16))
    assert torch.equal(a_lse, b_lse)


def test_gptoss_decode_window_128_full_config_sampled(sa, oracle_mod, cuda_dev):
    """The gpt-oss decode batch on a sliding-window layer (W = 128): 16 sequences, all heads."""
    w = inputs.make_workload("gptoss_decode", seed=0)
    out, lse = _decode(sa, w, cuda_dev, 128)
    B, Hq = w.q.shape[:2]
    sel = np.zeros((B, Hq), dtype=bool)
    sel[np.random.default_rng(1).choice(B, 16, replace=False)] = True
    ro, rl = _oracle_decode(oracle_mod, w, 128, select=sel)
    check_out(out, ro, mask=sel)
    check_lse(lse, rl, mask=sel)


def test_gptoss_prefill_window_128_full_config_sampled(sa, oracle_mod, cuda_dev):
    """The gpt-oss prefill batch on a sliding-window layer (W = 128): 2000 random rows plus
    the first and last rows of each sequence."""
    p = inputs.make_workload("gptoss_prefill", seed=0)
    out, lse = _prefill(sa, p, cuda_dev, 128)
    T, Hq = p.q.shape[:2]
    rng = np.random.default_rng(2)
    sel = np.zeros((T, Hq), dtype=bool)
    sel[rng.integers(0, T, 2000), rng.integers(0, Hq, 2000)] = True
    cu = p.cu_seqlens.tolist()
    for i in range(len(cu) - 1):
        sel[cu[i]] = sel[cu[i + 1] - 1] = True
    ro, rl = _oracle_prefill(oracle_mod, p, 128, select=sel)
    check_out(out, ro, mask=sel)
    check_lse(lse, rl, mask=sel)


# ---- the one-launch plan of short sliding windows (W <= 2032: a CTA per (sequence, KV head),
# its four warps splitting the visible pages, merged in shared memory) against the two-stage
# split-KV plan (sinkattn_decode_splitkv + sinkattn_decode_merge) and the oracle
# (one 8-head tile for G <= 8, two for 16)
@pytest.mark.parametrize("D,window,G", [(64, 16, 8), (64, 128, 8), (128, 128, 16), (64, 2032, 8), (128, 1000, 16),
                                        (64, 128, 16), (128, 128, 1)])
def test_window_one_launch_matches_split_kv_plan(sa, oracle_mod, cuda_dev, D, window, G):
    lens = [0, 1, 15, 16, 17, 127, 128, 129, 2049, 5000]
    Hkv = 2
    w = inputs.make_decode(lens, len(lens), Hkv * G, Hkv, D, seed=90 + window + G, sinks=True)
    c = w.cache
    dev = cuda_dev
    q, kp, vp, bt, sl, sk = (w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), c.block_table.to(dev),
                             c.lens.to(dev), w.sinks.to(dev))
    out, lse = sa.decode(q, kp, vp, bt, sl, sk, w.scale, window=window)
    o2, l2, ws, desc = sa.decode_splitkv(q, kp, vp, bt, sl, sk, w.scale, window=window)
    sa.decode_merge(sl, sk, o2, l2, desc, ws)
    torch.cuda.synchronize()
    assert sa.get_status(sa.workspace(0, dev)) == 0
    ro, rl = _oracle_decode(oracle_mod, w, window)
    check_out(out, ro, what="one-launch window decode")
    check_lse(lse, rl, what="one-launch window lse")
    check_out(o2, ro, what="split-KV window decode")
    check_lse(l2, rl, what="split-KV window lse")


def test_window_one_launch_independent_of_the_grid(sa, cuda_dev):
    # each (sequence, KV head) is done by one CTA the same way whatever the grid: bitwise
    lens = [3, 128, 129, 500, 7000, 64, 1, 0] * 4
    w = inputs.make_decode(lens, len(lens), 16, 2, 64, seed=95, sinks=True)
    c = w.cache
    dev = cuda_dev
    args = (w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), c.block_table.to(dev), c.lens.to(dev),
            w.sinks.to(dev), w.scale)
    a_out, a_lse = sa.decode(*args, window=128)
    b_out, b_lse = sa.decode(*args, window=128, max_sms=3)
    torch.cuda.synchronize()
    assert torch.equal(a_out.view(torch.int16), b_out.view(torch.int16))
    assert torch.equal(a_lse.view(torch.int32), b_lse.view(torch.int32))


def test_window_one_launch_bad_page_and_length(sa, oracle_mod, cuda_dev):
    lens = [40, 300, 17, 1000]
    w = inputs.make_decode(lens, 4, 16, 2, 64, seed=96, sinks=True)
    c = w.cache
    dev = cuda_dev
    bt = c.block_table.clone()
    bt[1, 18] = c.num_pages + 3          # inside sequence 1's window of 128 keys
    sl = c.lens.clone()
    sl[3] = c.block_table.shape[1] * 16 + 5  # beyond the table
    ws = sa.workspace(0, dev)
    sa.get_status(ws)
    out, lse = sa.decode(w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), bt.to(dev), sl.to(dev),
                         w.sinks.to(dev), w.scale, window=128)
    torch.cuda.synchronize()
    st = sa.get_status(ws)
    assert st & sa.STATUS_BAD_PAGE and st & sa.STATUS_BAD_LENGTH
    # the untouched sequences stay exact
    ro, rl = _oracle_decode(oracle_mod, w, 128)
    keep = np.zeros((4, 16), dtype=bool)
    keep[[0, 2]] = True
    check_out(out, ro, mask=keep, what="sequences beside a bad page")
    check_lse(lse, rl, mask=keep)
