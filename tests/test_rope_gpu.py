"""Decode step with rotary embedding and K/V append (sinkattn_decode_append_rope) against
the fp64 oracle's rotate -> append -> decode (TensorSharp gptoss.md, section 3 "Forward
graph": RoPE_NeoX with YaRN scaling on Q and K, K/V appended to the cache, attention).

Checked per case: out and lse within the parity bar; every page byte other than the new
slots unchanged; the new V rows bit for bit; the new K rows within one bf16 step of the
exact rotation (the kernel rotates in float arithmetic, the oracle in double, and the two
roundings to bf16 may fall on either side of a boundary the exact value sits next to).
"""
import numpy as np
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs
from tolerances import check_lse, check_out

pytestmark = pytest.mark.gpu

GPTOSS = dict(base=150000.0, factor=32.0, original_context=4096, beta_fast=32.0, beta_slow=1.0)
PLAIN = dict(base=10000.0, factor=1.0, original_context=4096, beta_fast=32.0, beta_slow=1.0)


def _run(sa, oracle_mod, dev, w, rope, window=0, sample=None):
    c = w.cache
    B, Hq, D = w.q.shape
    Hkv = c.k_pages.shape[1]
    kn, vn = inputs.new_rows(B, Hkv, D, seed=B + D)
    kp, vp = c.k_pages.to(dev), c.v_pages.to(dev)
    out, lse = sa.decode_append_rope(w.q.to(dev), kn.to(dev), vn.to(dev), kp, vp, c.block_table.to(dev),
                                     c.lens.to(dev), None if w.sinks is None else w.sinks.to(dev),
                                     w.scale, sa.rope_desc(**rope), window=window)
    torch.cuda.synchronize()
    assert sa.get_status(sa.workspace(0, dev)) == 0
    sel = None
    if sample is not None:
        sel = np.zeros((B, Hq), dtype=bool)
        sel[::sample] = True
    ro, rl, rkp, rvp, _, _ = oracle_mod.decode_append_rope(
        w.q, kn, vn, c.k_pages, c.v_pages, c.block_table, c.lens, w.sinks, w.scale, select=sel,
        window=window, **rope)
    check_out(out, ro, mask=sel, what="rope decode out")
    check_lse(lse, rl, mask=sel, what="rope decode lse")
    # pages: only the new slots changed; V there bit for bit, K within one bf16 step
    gk = kp.cpu().view(torch.int16).numpy().view(np.uint16)
    gv = vp.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gv, rvp), "V pages differ from the oracle's append"
    lens = c.lens.numpy()
    new = np.zeros(gk.shape[:1] + gk.shape[2:3], dtype=bool)  # [page, slot]
    for b in range(B):
        if lens[b] > 0:
            new[int(c.block_table[b, (lens[b] - 1) // 16]), (lens[b] - 1) % 16] = True
    keep = ~new
    assert np.array_equal(gk.transpose(0, 2, 1, 3)[keep], rkp.transpose(0, 2, 1, 3)[keep])
    pos = np.maximum(lens.astype(np.int64) - 1, 0)
    exact = oracle_mod.rope(kn, pos, **rope)  # [B, Hkv, D] float64, not rounded
    for b in range(B):
        if lens[b] == 0:
            continue
        pg, slot = int(c.block_table[b, (lens[b] - 1) // 16]), (lens[b] - 1) % 16
        got = torch.from_numpy(gk[pg, :, slot].view(np.int16)).view(torch.bfloat16).double().numpy()
        step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(exact[b]), 1e-30))) - 7)
        assert np.all(np.abs(got - exact[b]) <= step + 1e-30), f"rotated key of sequence {b}"


@pytest.mark.parametrize("D,G", [(64, 8), (64, 1), (128, 16), (128, 4), (64, 16)])
@pytest.mark.parametrize("rope", ["gptoss", "plain"])
def test_rope_decode_shapes(sa, oracle_mod, cuda_dev, D, G, rope):
    Hkv = 2 if G < 16 else 4
    lens = [0, 1, 16, 17, 100, 2049]
    w = inputs.make_decode(lens, len(lens), G * Hkv, Hkv, D, seed=40 + D + G, sinks=G != 4)
    _run(sa, oracle_mod, cuda_dev, w, GPTOSS if rope == "gptoss" else PLAIN)


def test_rope_decode_long_positions(sa, oracle_mod, cuda_dev):
    # positions up to 131071: the angle reduction must stay accurate where p * theta ~ 1e5
    lens = [131072, 100000, 65537, 4097]
    w = inputs.make_decode(lens, len(lens), 16, 2, 64, seed=44, sinks=True)
    _run(sa, oracle_mod, cuda_dev, w, GPTOSS, sample=1)


@pytest.mark.parametrize("G", [8, 16])
def test_rope_decode_window(sa, oracle_mod, cuda_dev, G):
    # the one-launch window kernel, one and two 8-head tiles
    w = inputs.make_decode([5, 128, 129, 3000], 4, 2 * G, 2, 64, seed=45 + G, sinks=True)
    _run(sa, oracle_mod, cuda_dev, w, GPTOSS, window=128)


def test_rope_decode_gptoss_batch(sa, oracle_mod, cuda_dev):
    # the gpt-oss decode batch (64 sequences, 64 / 8 heads, lengths U[512, 8192]), sampled rows
    w = inputs.make_workload("gptoss_decode", seed=0)
    _run(sa, oracle_mod, cuda_dev, w, GPTOSS, sample=7)


def test_rope_rejects_bad_parameters(sa, cuda_dev):
    w = inputs.make_decode([5, 9], 2, 8, 2, 64, seed=46, sinks=True)
    c = w.cache
    kn, vn = (t.to(cuda_dev) for t in inputs.new_rows(2, 2, 64, seed=46))
    args = (w.q.to(cuda_dev), kn, vn, c.k_pages.to(cuda_dev), c.v_pages.to(cuda_dev),
            c.block_table.to(cuda_dev), c.lens.to(cuda_dev), w.sinks.to(cuda_dev), w.scale)
    for bad in (dict(GPTOSS, factor=0.5), dict(GPTOSS, base=1.0), dict(GPTOSS, beta_fast=0.5),
                dict(GPTOSS, original_context=0)):
        with pytest.raises(sa.SinkAttnError) as e:
            sa.decode_append_rope(*args, rope=sa.rope_desc(**bad))
        assert e.value.code == sa.ERR_INVALID_ARG
