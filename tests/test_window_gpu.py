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
