"""Chunked prefill over an FP8 E4M3 paged prefix (sinkattn_prefill_fp8) against the fp64
oracle (oracle.prefill_fp8: value = scale[g] * e4m3(code) for the prefix, bf16 new tokens).

With power-of-two scales every prefix value is a bf16 number and the kernel's arithmetic is
the bf16 prefill's step for step (the K scale multiplies the score by an exact power of two,
the V values round to the same fp16 numbers), so the result must equal sinkattn_prefill over
bf16 pages holding those values bit for bit.
"""
import numpy as np
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs
from tolerances import check_lse, check_out

pytestmark = pytest.mark.gpu


def _dev_prefill(p, dev):
    c = p.prefix
    return dict(q=p.q.to(dev), k=p.k.to(dev), v=p.v.to(dev), cu=p.cu_seqlens.to(dev),
                sk=None if p.sinks is None else p.sinks.to(dev), kp=c.k_pages.to(dev),
                vp=c.v_pages.to(dev), ks=c.k_scale.to(dev), vs=c.v_scale.to(dev),
                bt=c.block_table.to(dev), pl=c.lens.to(dev))


def _run(sa, p, d, window=0):
    out, lse = sa.prefill_fp8(d["q"], d["k"], d["v"], d["cu"], d["sk"], p.scale, d["kp"], d["vp"],
                              d["ks"], d["vs"], d["bt"], d["pl"], window=window)
    torch.cuda.synchronize()
    return out, lse


def _oracle(o, p, window=0, select=None):
    c = p.prefix
    return o.prefill_fp8(p.q, p.k, p.v, p.cu_seqlens, p.sinks, p.scale, c.k_pages, c.v_pages,
                         c.k_scale, c.v_scale, c.block_table, c.lens, select=select, window=window)


@pytest.mark.parametrize("D,G,Hkv", [(64, 8, 2), (64, 1, 4), (128, 16, 1), (128, 4, 2)])
def test_prefill_fp8_prefix_shapes(sa, oracle_mod, cuda_dev, D, G, Hkv):
    new, pre = [300, 1, 129, 40], [1000, 37, 0, 129]
    p = inputs.make_prefill(new, G * Hkv, Hkv, D, seed=100 + D + G, sinks=G != 4, prefix_lens=pre,
                            prefix_kv_dtype="fp8")
    d = _dev_prefill(p, cuda_dev)
    ws = sa.workspace(256, cuda_dev, "prefill")
    sa.get_status(ws)
    out, lse = _run(sa, p, d)
    assert sa.get_status(ws) == 0
    ro, rl = _oracle(oracle_mod, p)
    check_out(out, ro, what="fp8-prefix prefill out")
    check_lse(lse, rl, what="fp8-prefix prefill lse")


@pytest.mark.parametrize("D", [64, 128])
def test_prefill_fp8_pow2_scales_equal_bf16_prefill_bitwise(sa, cuda_dev, D):
    new, pre = [257, 3, 128], [2048, 17, 300]
    p = inputs.make_prefill(new, 16, 2, D, seed=110 + D, sinks=True, prefix_lens=pre,
                            prefix_kv_dtype="fp8")
    c = p.prefix
    c.k_scale = torch.tensor([0.25, 0.0625], dtype=torch.float32)
    c.v_scale = torch.tensor([2.0, 0.5], dtype=torch.float32)
    d = _dev_prefill(p, cuda_dev)
    out8, lse8 = _run(sa, p, d)
    # bf16 pages holding the same values (exact: E4M3 values times powers of two)
    kb = (c.k_pages.view(torch.float8_e4m3fn).float() * c.k_scale.view(1, -1, 1, 1)).to(torch.bfloat16)
    vb = (c.v_pages.view(torch.float8_e4m3fn).float() * c.v_scale.view(1, -1, 1, 1)).to(torch.bfloat16)
    out, lse = sa.prefill(d["q"], d["k"], d["v"], d["cu"], d["sk"], p.scale, kb.to(cuda_dev),
                          vb.to(cuda_dev), d["bt"], d["pl"])
    torch.cuda.synchronize()
    # rows of keys past a prefix end hold NaN codes / NaN bf16 values in both pools; both
    # kernels skip them, so the results must agree everywhere
    assert torch.equal(out8.view(torch.int16), out.view(torch.int16))
    assert torch.equal(lse8.view(torch.int32), lse.view(torch.int32))


@pytest.mark.parametrize("window", [1, 100, 128, 1000])
def test_prefill_fp8_window(sa, oracle_mod, cuda_dev, window):
    new, pre = [200, 64, 1], [900, 128, 50]
    p = inputs.make_prefill(new, 16, 2, 64, seed=120 + window, sinks=True, prefix_lens=pre,
                            prefix_kv_dtype="fp8")
    d = _dev_prefill(p, cuda_dev)
    out, lse = _run(sa, p, d, window=window)
    ro, rl = _oracle(oracle_mod, p, window=window)
    check_out(out, ro, what=f"fp8-prefix prefill, window {window}")
    check_lse(lse, rl, what=f"fp8-prefix lse, window {window}")


def test_prefill_fp8_longctx_chunked_sampled(sa, oracle_mod, cuda_dev):
    # the long-context chunked workload (8 x 512 new tokens over 16384-token prefixes) over an
    # FP8 prefix cache; every 97th query row, all heads
    p = inputs.make_workload("longctx_chunked_fp8", seed=0)
    d = _dev_prefill(p, cuda_dev)
    ws = sa.workspace(256, cuda_dev, "prefill")
    sa.get_status(ws)
    out, lse = _run(sa, p, d)
    assert sa.get_status(ws) == 0
    T, Hq = p.q.shape[:2]
    sel = np.zeros((T, Hq), dtype=bool)
    sel[::97] = True
    ro, rl = _oracle(oracle_mod, p, select=sel)
    check_out(out, ro, mask=sel, what="long-context fp8-prefix prefill")
    check_lse(lse, rl, mask=sel, what="long-context fp8-prefix lse")


def test_prefill_fp8_bad_prefix_page(sa, oracle_mod, cuda_dev):
    new, pre = [64, 64], [500, 500]
    p = inputs.make_prefill(new, 8, 2, 64, seed=130, sinks=True, prefix_lens=pre, prefix_kv_dtype="fp8")
    d = _dev_prefill(p, cuda_dev)
    d["bt"] = d["bt"].clone()
    d["bt"][0, 5] = p.prefix.num_pages + 9
    ws = sa.workspace(256, cuda_dev, "prefill")
    sa.get_status(ws)
    out, lse = _run(sa, p, d)
    assert sa.get_status(ws) & sa.STATUS_BAD_PAGE
    ro, rl = _oracle(oracle_mod, p)
    keep = np.zeros(p.q.shape[:2], dtype=bool)
    keep[64:] = True  # request 1 is untouched
    check_out(out, ro, mask=keep, what="request beside a bad prefix page")
    check_lse(lse, rl, mask=keep)


def test_prefill_fp8_large_v_scale(sa, oracle_mod, cuda_dev):
    """V scales large enough that 448 * scale passes 2^15: the converted V takes a power-of-two
    exponent k > 0 (k = 4 and 7 here) and must still match the oracle; a scale past k = 7 sets
    SINKATTN_STATUS_VALUE_RANGE.  The prefix values are the N(0,1) data times c = the new
    scale over the old one, so the absolute part of the bar is taken c times larger."""
    p = inputs.make_prefill([100, 30], 8, 2, 64, seed=140, sinks=True, prefix_lens=[300, 129],
                            prefix_kv_dtype="fp8")
    c = p.prefix
    old = c.v_scale.clone()
    c.v_scale = torch.tensor([700.0, 9000.0], dtype=torch.float32)
    mag = (c.v_scale / old).double().repeat_interleave(4).numpy()[None, :, None]  # [1, Hq, 1]
    d = _dev_prefill(p, cuda_dev)
    ws = sa.workspace(256, cuda_dev, "prefill")
    sa.get_status(ws)
    out, lse = _run(sa, p, d)
    assert sa.get_status(ws) == 0
    ro, rl = _oracle(oracle_mod, p)
    check_out(out, ro, what="fp8-prefix prefill, large V scales", v_mag=mag)
    check_lse(lse, rl, what="fp8-prefix lse, large V scales")
    d["vs"] = torch.tensor([700.0, 20000.0], dtype=torch.float32, device=cuda_dev)
    _run(sa, p, d)
    assert sa.get_status(ws) & sa.STATUS_VALUE_RANGE


@pytest.mark.parametrize("vs", [100.0, 1.5 * 2.0 ** -12, 127.9, 2.0 ** -12])
def test_prefill_fp8_v_scale_at_the_power_of_two_form_edges(sa, oracle_mod, cuda_dev, vs):
    """V scales m * 2^e with e from -12 to 6 take the form in which the converters write
    code * 2^e (exact in fp16) and the softmax multiplies those keys' P by m; these sit at both
    ends of that range (the values are the N(0,1) data scaled by vs / the old scale)."""
    p = inputs.make_prefill([150, 40], 8, 2, 64, seed=141, sinks=True, prefix_lens=[260, 129],
                            prefix_kv_dtype="fp8")
    c = p.prefix
    old = c.v_scale.clone()
    c.v_scale = torch.full_like(c.v_scale, vs)
    mag = np.maximum(1.0, (c.v_scale / old).double().repeat_interleave(4).numpy())[None, :, None]
    d = _dev_prefill(p, cuda_dev)
    ws = sa.workspace(256, cuda_dev, "prefill")
    sa.get_status(ws)
    out, lse = _run(sa, p, d)
    assert sa.get_status(ws) == 0
    ro, rl = _oracle(oracle_mod, p)
    check_out(out, ro, what=f"fp8-prefix prefill, V scale {vs}", v_mag=mag)
    check_lse(lse, rl, what=f"fp8-prefix lse, V scale {vs}")
