"""Prefill parity on the GPU: the tcgen05 causal / chunked prefill kernel against
the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs
from tolerances import check_lse, check_out

pytestmark = pytest.mark.gpu


def run_prefill(sa, p, dev, sinks="same"):
    kw = {}
    if p.prefix is not None:
        kw = dict(k_pages=p.prefix.k_pages.to(dev), v_pages=p.prefix.v_pages.to(dev),
                  prefix_block_table=p.prefix.block_table.to(dev),
                  prefix_lens=p.prefix.lens.to(dev))
    s = p.sinks if sinks == "same" else sinks
    out, lse = sa.prefill(p.q.to(dev), p.k.to(dev), p.v.to(dev), p.cu_seqlens.to(dev),
                          None if s is None else s.to(dev), p.scale, **kw)
    torch.cuda.synchronize()
    return out, lse


def oracle_prefill(o, p, select=None, sinks="same"):
    kw = {}
    if p.prefix is not None:
        kw = dict(k_pages=p.prefix.k_pages, v_pages=p.prefix.v_pages,
                  prefix_block_table=p.prefix.block_table, prefix_lens=p.prefix.lens)
    s = p.sinks if sinks == "same" else sinks
    return o.prefill(p.q, p.k, p.v, p.cu_seqlens, s, p.scale, select=select, **kw)


def test_prefill_tiny_single_tile(sa, oracle_mod, cuda_dev):
    p = inputs.make_prefill([37], 8, 2, 64, seed=1, sinks=True)
    out, lse = run_prefill(sa, p, cuda_dev)
    ro, rl = oracle_prefill(oracle_mod, p)
    check_out(out, ro)
    check_lse(lse, rl)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 4, 8, 16])
@pytest.mark.parametrize("sinks_on", [True, False])
def test_prefill_causal_ragged(sa, oracle_mod, cuda_dev, D, G, sinks_on):
    lens = [1, 5, 127, 128, 129, 300, 513]
    p = inputs.make_prefill(lens, 2 * G, 2, D, seed=G + D, sinks=sinks_on)
    out, lse = run_prefill(sa, p, cuda_dev)
    ro, rl = oracle_prefill(oracle_mod, p)
    check_out(out, ro)
    check_lse(lse, rl)
    assert sa.get_status(sa.workspace(0, cuda_dev, "prefill")) == 0


@pytest.mark.parametrize("D", [64, 128])
def test_chunked_prefill_over_paged_prefix(sa, oracle_mod, cuda_dev, D):
    new = [1, 64, 130, 5, 256, 7, 1]
    pre = [0, 1, 16, 17, 300, 1000, 4096]
    p = inputs.make_prefill(new, 16, 2, D, seed=D + 3, sinks=True, prefix_lens=pre)
    out, lse = run_prefill(sa, p, cuda_dev)
    ro, rl = oracle_prefill(oracle_mod, p)
    check_out(out, ro)
    check_lse(lse, rl)
    assert sa.get_status(sa.workspace(0, cuda_dev, "prefill")) == 0


def _grow_keys(p, per_tile):
    """Scale every key by 1 + per_tile * position / 128, in the new tokens and in the prefix
    pages, so that each 128-key tile's scores reach higher than the tile before: the running
    max of every row grows through the row and the online softmax must rescale its output
    (the keys are rounded to bf16 again, so the oracle and the kernel see the same values)."""
    n = len(p.cu_seqlens) - 1
    cu = p.cu_seqlens.tolist()
    pre = p.prefix.lens.tolist() if p.prefix is not None else [0] * n
    k = p.k.float()
    for i in range(n):
        pos = torch.arange(cu[i + 1] - cu[i], dtype=torch.float32) + pre[i]
        k[cu[i]:cu[i + 1]] *= (1 + per_tile * pos / 128)[:, None, None]
    p.k = k.bfloat16()
    if p.prefix is not None:
        kp = p.prefix.k_pages.float()
        for i in range(n):
            for pg in range((pre[i] + 15) // 16):
                phys = int(p.prefix.block_table[i, pg])
                pos = torch.arange(16, dtype=torch.float32) + 16 * pg
                kp[phys] *= (1 + per_tile * pos / 128)[None, :, None]
        p.prefix.k_pages = kp.bfloat16()
    return p


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("per_tile", [3.0, 8.0])
def test_prefill_running_max_grows_across_tiles(sa, oracle_mod, cuda_dev, D, per_tile):
    """Scores that rise tile by tile (each tile's row max ~11 or ~30 log2 units above the
    last): the output is rescaled many times within a row, causal and chunked."""
    for prefix in (None, [300, 0, 700]):
        p = inputs.make_prefill([600, 129, 260], 8, 2, D, seed=int(per_tile) + D, sinks=True,
                                prefix_lens=prefix)
        p = _grow_keys(p, per_tile)
        out, lse = run_prefill(sa, p, cuda_dev)
        ro, rl = oracle_prefill(oracle_mod, p)
        check_out(out, ro)
        check_lse(lse, rl)
        assert sa.get_status(sa.workspace(0, cuda_dev, "prefill")) == 0


def test_prefill_null_sinks_equal_neg_inf_bitwise(sa, cuda_dev):
    p = inputs.make_prefill([300, 129], 16, 4, 128, seed=4, sinks=False, prefix_lens=[40, 0])
    o1, l1 = run_prefill(sa, p, cuda_dev, sinks=None)
    o2, l2 = run_prefill(sa, p, cuda_dev, sinks=torch.full((16,), -math.inf))
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_prefill_large_sink(sa, oracle_mod, cuda_dev):
    p = inputs.make_prefill([200], 8, 2, 64, seed=5, sinks=True)
    big = torch.full((8,), 1e4)
    out, lse = run_prefill(sa, p, cuda_dev, sinks=big)
    assert torch.count_nonzero(out.float()) == 0
    ro, rl = oracle_prefill(oracle_mod, p, sinks=big)
    check_lse(lse, rl)


def test_prefill_row_equals_decode(sa, cuda_dev):
    """Row t of a causal prefill equals a decode over the first t + 1 keys."""
    L = 300
    p = inputs.make_prefill([L], 16, 2, 64, seed=6, sinks=True)
    out, lse = run_prefill(sa, p, cuda_dev)
    npg = (L + 15) // 16
    kp = torch.zeros(npg, 2, 16, 64, dtype=torch.bfloat16)
    vp = torch.zeros(npg, 2, 16, 64, dtype=torch.bfloat16)
    for j in range(L):
        kp[j // 16, :, j % 16] = p.k[j]
        vp[j // 16, :, j % 16] = p.v[j]
    ts = [0, 15, 127, 128, 299]
    bt = torch.arange(npg, dtype=torch.int32).repeat(len(ts), 1)
    dout, dlse = sa.decode(p.q[ts].to(cuda_dev), kp.to(cuda_dev), vp.to(cuda_dev),
                           bt.to(cuda_dev), torch.tensor([t + 1 for t in ts], dtype=torch.int32,
                                                         device=cuda_dev),
                           p.sinks.to(cuda_dev), p.scale)
    check_out(dout, out[ts].double().cpu().numpy())
    check_lse(dlse, lse[ts].double().cpu().numpy())


def _large_rows(n, lo_exp, seed):
    """n x D-independent positive magnitudes in [2^lo_exp, 2^(lo_exp + 1)), still below
    2^(lo_exp + 1) once rounded to bf16."""
    g = torch.Generator().manual_seed(seed)
    return (2.0 ** lo_exp) * (1.0 + 0.99 * torch.rand(n, generator=g))


@pytest.mark.parametrize("D", [64, 128])
def test_prefill_v_quarters_with_different_scales(sa, oracle_mod, cuda_dev, D):
    """V rows at key positions 32..63 of each 128-key tile in [2^17, 2^18) and 96..127 in
    [2^20, 2^21): the kernel scales those 32-key quarters into fp16 range with different
    powers of two (k = 3 and 6) and the other quarters not at all.  No status is raised
    below 2^22."""
    p = inputs.make_prefill([300, 129, 64], 8, 2, D, seed=40 + D, sinks=True)
    cu = p.cu_seqlens.tolist()
    for i in range(len(cu) - 1):
        for t in range(cu[i], cu[i + 1]):
            pos = (t - cu[i]) % 128
            if 32 <= pos < 64:
                p.v[t] = _large_rows(D, 17, t).to(torch.bfloat16).expand(p.v.shape[1], D)
            elif pos >= 96:
                p.v[t] = _large_rows(D, 20, t).to(torch.bfloat16).expand(p.v.shape[1], D)
    ws = sa.workspace(0, cuda_dev, "prefill")
    sa.get_status(ws)
    out, lse = run_prefill(sa, p, cuda_dev)
    ro, rl = oracle_prefill(oracle_mod, p)
    check_out(out, ro)
    check_lse(lse, rl)
    assert sa.get_status(ws) == 0


def test_chunked_prefill_prefix_v_quarters_with_different_scales(sa, oracle_mod, cuda_dev):
    """The same scaling for prefix tiles read through the block table."""
    p = inputs.make_prefill([40, 3], 8, 2, 64, seed=52, sinks=True, prefix_lens=[300, 150])
    pre = p.prefix
    for i, P in enumerate(pre.lens.tolist()):
        for pos in range(P):
            page = int(pre.block_table[i, pos // 16])
            if 32 <= pos % 128 < 64:
                pre.v_pages[page, :, pos % 16] = _large_rows(64, 16, pos).to(torch.bfloat16)
    ws = sa.workspace(0, cuda_dev, "prefill")
    sa.get_status(ws)
    out, lse = run_prefill(sa, p, cuda_dev)
    ro, rl = oracle_prefill(oracle_mod, p)
    check_out(out, ro)
    check_lse(lse, rl)
    assert sa.get_status(ws) == 0


@pytest.mark.parametrize("D", [64, 128])
def test_prefill_v_at_the_top_of_the_supported_range(sa, oracle_mod, cuda_dev, D):
    """The edge of the documented range: a 32-key quarter of V in [2^21, 2^22) takes the
    largest power-of-two scale (k = 7) and must still match the oracle, with no status; one
    value at 2^22 is past it and sets SINKATTN_STATUS_VALUE_RANGE."""
    p = inputs.make_prefill([200, 130], 8, 2, D, seed=60 + D, sinks=True)
    cu = p.cu_seqlens.tolist()
    for i in range(len(cu) - 1):
        for t in range(cu[i], cu[i + 1]):
            if (t - cu[i]) % 128 < 32:
                row = _large_rows(D, 21, t) * torch.where(torch.arange(D) % 3 == 0, -1.0, 1.0)
                p.v[t] = row.to(torch.bfloat16).expand(p.v.shape[1], D)
    assert float(p.v.abs().max()) < 2.0 ** 22
    ws = sa.workspace(0, cuda_dev, "prefill")
    sa.get_status(ws)
    out, lse = run_prefill(sa, p, cuda_dev)
    assert sa.get_status(ws) == 0
    ro, rl = oracle_prefill(oracle_mod, p)
    check_out(out, ro)
    check_lse(lse, rl)
    p.v[5, 0, 3] = 2.0 ** 22
    run_prefill(sa, p, cuda_dev)
    assert sa.get_status(ws) & sa.STATUS_VALUE_RANGE


def test_prefill_v_beyond_fp16_range_sets_status(sa, cuda_dev):
    p = inputs.make_prefill([50], 8, 2, 64, seed=9, sinks=True)
    p.v[10, 1, 5] = 2.0 ** 23
    ws = sa.workspace(0, cuda_dev, "prefill")
    sa.get_status(ws)
    run_prefill(sa, p, cuda_dev)
    assert sa.get_status(ws) & sa.STATUS_VALUE_RANGE


def test_prefill_bad_prefix_page_sets_status(sa, cuda_dev):
    p = inputs.make_prefill([20, 20], 8, 2, 64, seed=7, sinks=True, prefix_lens=[64, 64])
    p.prefix.block_table[1, 1] = p.prefix.num_pages + 99
    ws = sa.workspace(0, cuda_dev, "prefill")
    sa.get_status(ws)
    run_prefill(sa, p, cuda_dev)
    assert sa.get_status(ws) & sa.STATUS_BAD_PAGE


def _sampled(sa, oracle_mod, cuda_dev, name, nrows):
    p = inputs.make_workload(name, seed=0)
    out, lse = run_prefill(sa, p, cuda_dev)
    T, Hq = p.q.shape[:2]
    rng = np.random.default_rng(0)
    sel = np.zeros((T, Hq), dtype=bool)
    sel[rng.integers(0, T, nrows), rng.integers(0, Hq, nrows)] = True
    cu = p.cu_seqlens.tolist()
    for i in range(len(cu) - 1):  # first and last row of every request, all heads
        sel[cu[i]] = True
        sel[cu[i + 1] - 1] = True
    ro, rl = oracle_prefill(oracle_mod, p, select=sel)
    check_out(out, ro, mask=sel)
    check_lse(lse, rl, mask=sel)


def test_gptoss_prefill_full_config_sampled(sa, oracle_mod, cuda_dev):
    """Lengths {4096, 2048, 1024, 512}, 64 q / 8 KV heads, D=64: 2000 random rows plus the
    first and last row of each sequence (all heads)."""
    _sampled(sa, oracle_mod, cuda_dev, "gptoss_prefill", 2000)


def test_longctx_chunked_full_config_sampled(sa, oracle_mod, cuda_dev):
    """8 requests x 512 new tokens over 16384-token paged prefixes: 300 random rows plus
    the first and last row of each request (all heads)."""
    _sampled(sa, oracle_mod, cuda_dev, "longctx_chunked", 300)
