"""Decode parity on the GPU: the split-KV kernel + LSE merge against the fp64 oracle,
through the C ABI, on seeded inputs (NaN-poisoned tail slots and distractor pages)."""
import math

import numpy as np
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs
from tolerances import check_lse, check_out

pytestmark = pytest.mark.gpu


def to_dev(w: inputs.DecodeInputs, dev):
    c = w.cache
    return dict(q=w.q.to(dev), k_pages=c.k_pages.to(dev), v_pages=c.v_pages.to(dev),
                block_table=c.block_table.to(dev), seq_lens=c.lens.to(dev),
                sinks=None if w.sinks is None else w.sinks.to(dev))


def run_decode(sa, w, dev, sinks="same", **kw):
    d = to_dev(w, dev)
    if sinks != "same":
        d["sinks"] = sinks
    out, lse = sa.decode(d["q"], d["k_pages"], d["v_pages"], d["block_table"], d["seq_lens"],
                         d["sinks"], w.scale, **kw)
    torch.cuda.synchronize()
    return out, lse


def oracle_decode(o, w, select=None, sinks="same"):
    c = w.cache
    s = w.sinks if sinks == "same" else sinks
    return o.decode(w.q, c.k_pages, c.v_pages, c.block_table, c.lens, s, w.scale, select=select)


def test_tiny_decode_config(sa, oracle_mod, cuda_dev):
    """B=4, L={1,17,64,129}, 8 q / 2 KV heads, D=64, shuffled pages, sinks ~N(0,1), seed 0."""
    w = inputs.make_workload("tiny_decode", seed=0)
    out, lse = run_decode(sa, w, cuda_dev)
    ro, rl = oracle_decode(oracle_mod, w)
    check_out(out, ro)
    check_lse(lse, rl)
    assert sa.get_status(sa.workspace(0, cuda_dev)) == 0


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("sinks_on", [True, False])
def test_decode_shapes(sa, oracle_mod, cuda_dev, D, G, sinks_on):
    Hkv = 2
    lens = [0, 1, 15, 16, 17, 33, 300, 1000, 2049]
    w = inputs.make_decode(lens, len(lens), Hkv * G, Hkv, D, seed=G * 7 + D, sinks=sinks_on)
    out, lse = run_decode(sa, w, cuda_dev)
    ro, rl = oracle_decode(oracle_mod, w)
    check_out(out, ro)
    check_lse(lse, rl)
    assert sa.get_status(sa.workspace(0, cuda_dev)) == 0


@pytest.mark.parametrize("seed", [1, 2])
def test_decode_long_sequences_split_across_warps(sa, oracle_mod, cuda_dev, seed):
    """Few long sequences: every (sequence, KV head) is cut across many warps and merged."""
    lens = [40000, 70001, 131072, 5]
    w = inputs.make_decode(lens, 4, 16, 2, 64, seed=seed, sinks=True)
    out, lse = run_decode(sa, w, cuda_dev)
    ro, rl = oracle_decode(oracle_mod, w)
    check_out(out, ro)
    check_lse(lse, rl)


def test_decode_null_sinks_equal_neg_inf_sinks_bitwise(sa, cuda_dev):
    w = inputs.make_decode(("uniform", 1, 3000), 16, 32, 4, 128, seed=5, sinks=False)
    o1, l1 = run_decode(sa, w, cuda_dev, sinks=None)
    ninf = torch.full((32,), -math.inf, device=cuda_dev)
    o2, l2 = run_decode(sa, w, cuda_dev, sinks=ninf)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_decode_large_sink_drives_output_to_zero(sa, oracle_mod, cuda_dev):
    w = inputs.make_decode([1, 200, 5000], 3, 16, 2, 64, seed=6, sinks=True)
    big = torch.full((16,), 1e4)
    out, lse = run_decode(sa, w, cuda_dev, sinks=big.to(cuda_dev))
    assert torch.count_nonzero(out.float()) == 0
    ro, rl = oracle_decode(oracle_mod, w, sinks=big)
    check_lse(lse, rl)


def test_decode_page_permutation_is_bitwise_invariant(sa, cuda_dev):
    w = inputs.make_decode(("uniform", 1, 4000), 24, 64, 8, 64, seed=7, sinks=True)
    o1, l1 = run_decode(sa, w, cuda_dev)
    c = w.cache
    perm = torch.randperm(c.num_pages, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(c.num_pages)
    c.k_pages, c.v_pages = c.k_pages[perm].contiguous(), c.v_pages[perm].contiguous()
    c.block_table = torch.where(c.block_table >= 0, inv[c.block_table.clamp(min=0).long()].int(),
                                c.block_table)
    o2, l2 = run_decode(sa, w, cuda_dev)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_decode_two_half_batches_match_one_call(sa, cuda_dev):
    """Sharding the batch (one half per replica) gives the same results within tolerance
    (the per-warp split plan differs, so the summation order may differ)."""
    w = inputs.make_decode(("uniform", 512, 8192), 32, 64, 8, 64, seed=8, sinks=True)
    d = to_dev(w, cuda_dev)
    full, full_lse = sa.decode(d["q"], d["k_pages"], d["v_pages"], d["block_table"], d["seq_lens"],
                               d["sinks"], w.scale)
    parts = [sa.decode(d["q"][s].contiguous(), d["k_pages"], d["v_pages"],
                       d["block_table"][s].contiguous(), d["seq_lens"][s].contiguous(), d["sinks"],
                       w.scale) for s in (slice(0, 16), slice(16, 32))]
    torch.cuda.synchronize()
    half = torch.cat([p[0] for p in parts]).double().cpu().numpy()
    half_lse = torch.cat([p[1] for p in parts]).double().cpu().numpy()
    check_out(full, half)
    check_lse(full_lse, half_lse)


def test_decode_bad_block_table_entry_sets_status(sa, oracle_mod, cuda_dev):
    """An out-of-range page index is skipped (never dereferenced) and reported."""
    w = inputs.make_decode([100, 100, 100], 3, 8, 2, 64, seed=9, sinks=True)
    bt = w.cache.block_table.clone()
    bt[1, 2] = w.cache.num_pages + 1000
    d = to_dev(w, cuda_dev)
    d["block_table"] = bt.to(cuda_dev)
    ws = sa.workspace(0, cuda_dev)
    sa.get_status(ws)  # clear
    out, lse = sa.decode(d["q"], d["k_pages"], d["v_pages"], d["block_table"], d["seq_lens"],
                         d["sinks"], w.scale)
    assert sa.get_status(ws) & sa.STATUS_BAD_PAGE
    ro, rl = oracle_decode(oracle_mod, w)
    keep = np.array([True, False, True])
    check_out(out, ro, mask=keep)


def test_decode_length_beyond_block_table_sets_status(sa, cuda_dev):
    w = inputs.make_decode([20, 20], 2, 8, 2, 64, seed=10, sinks=True)
    d = to_dev(w, cuda_dev)
    d["seq_lens"] = torch.tensor([20, 10_000], dtype=torch.int32, device=cuda_dev)
    ws = sa.workspace(0, cuda_dev)
    sa.get_status(ws)
    sa.decode(d["q"], d["k_pages"], d["v_pages"], d["block_table"], d["seq_lens"], d["sinks"],
              w.scale)
    assert sa.get_status(ws) & sa.STATUS_BAD_LENGTH


def _sampled_parity(sa, oracle_mod, cuda_dev, name, nseq):
    w = inputs.make_workload(name, seed=0)
    out, lse = run_decode(sa, w, cuda_dev)
    B, Hq = w.q.shape[:2]
    rng = np.random.default_rng(0)
    sel = np.zeros((B, Hq), dtype=bool)
    seqs = rng.choice(B, size=min(nseq, B), replace=False)
    sel[seqs] = True
    # always include the longest and the shortest sequence
    lens = w.seq_lens.numpy()
    sel[lens.argmax()] = sel[lens.argmin()] = True
    ro, rl = oracle_decode(oracle_mod, w, select=sel)
    check_out(out, ro, mask=sel)
    check_lse(lse, rl, mask=sel)
    assert sa.get_status(sa.workspace(0, cuda_dev)) == 0


def test_gptoss_decode_full_config(sa, oracle_mod, cuda_dev):
    """B=64, 64/8 heads, D=64, L ~ U[512, 8192]: every row against the oracle."""
    _sampled_parity(sa, oracle_mod, cuda_dev, "gptoss_decode", 64)


def test_qwen3_decode_full_config_sampled(sa, oracle_mod, cuda_dev):
    """B=128, 64/4 heads, D=128, L ~ U[1024, 32768], no sink: 24 sequences x all heads."""
    _sampled_parity(sa, oracle_mod, cuda_dev, "qwen3_decode", 24)


def test_longctx_decode_full_config_sampled(sa, oracle_mod, cuda_dev):
    """B=256, L log-uniform [128, 131072]: 24 sequences x all heads (incl. longest/shortest)."""
    _sampled_parity(sa, oracle_mod, cuda_dev, "longctx_decode", 24)
