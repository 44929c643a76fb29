"""Degenerate inputs through the C ABI: an empty batch, a batch whose sequences are all
empty (out = 0, lse = the sink, or -inf without sinks: the virtual token alone), a packed
prefill with an empty request between two others, and a prefill with no tokens."""
import numpy as np
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs
from tolerances import check_lse, check_out

pytestmark = pytest.mark.gpu


def test_decode_empty_batch(sa, cuda_dev):
    dev = cuda_dev
    q = torch.empty(0, 8, 64, dtype=torch.bfloat16, device=dev)
    kp = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(0, 2, dtype=torch.int32, device=dev)
    sl = torch.zeros(0, dtype=torch.int32, device=dev)
    out, lse = sa.decode(q, kp, kp.clone(), bt, sl, None, 0.125)
    torch.cuda.synchronize()
    assert out.shape == (0, 8, 64) and lse.shape == (0, 8)


@pytest.mark.parametrize("sinks_on", [True, False])
def test_decode_all_sequences_empty(sa, oracle_mod, cuda_dev, sinks_on):
    w = inputs.make_decode([0, 0, 0], 3, 16, 2, 64, seed=31, sinks=sinks_on)
    c = w.cache
    dev = cuda_dev
    out, lse = sa.decode(w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), c.block_table.to(dev),
                         c.lens.to(dev), None if w.sinks is None else w.sinks.to(dev), w.scale)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    expect = (np.broadcast_to(w.sinks.double().numpy(), (3, 16)) if sinks_on
              else np.full((3, 16), -np.inf))
    check_lse(lse, expect)
    ro, rl = oracle_mod.decode(w.q, c.k_pages, c.v_pages, c.block_table, c.lens, w.sinks, w.scale)
    check_out(out, ro)
    check_lse(lse, rl)


@pytest.mark.parametrize("prefix", [None, [40, 17, 0]])
def test_prefill_with_an_empty_request_between_others(sa, oracle_mod, cuda_dev, prefix):
    p = inputs.make_prefill([100, 0, 130], 8, 2, 64, seed=32, sinks=True, prefix_lens=prefix)
    dev = cuda_dev
    kw = {}
    if p.prefix is not None:
        pre = p.prefix
        kw = dict(k_pages=pre.k_pages.to(dev), v_pages=pre.v_pages.to(dev),
                  prefix_block_table=pre.block_table.to(dev), prefix_lens=pre.lens.to(dev))
    out, lse = sa.prefill(p.q.to(dev), p.k.to(dev), p.v.to(dev), p.cu_seqlens.to(dev),
                          p.sinks.to(dev), p.scale, **kw)
    torch.cuda.synchronize()
    oargs = ()
    if p.prefix is not None:
        oargs = (p.prefix.k_pages, p.prefix.v_pages, p.prefix.block_table, p.prefix.lens)
    ro, rl = oracle_mod.prefill(p.q, p.k, p.v, p.cu_seqlens, p.sinks, p.scale, *oargs)
    check_out(out, ro)
    check_lse(lse, rl)


def test_prefill_without_tokens(sa, cuda_dev):
    p = inputs.make_prefill([0, 0], 8, 2, 64, seed=33, sinks=True)
    dev = cuda_dev
    out, lse = sa.prefill(p.q.to(dev), p.k.to(dev), p.v.to(dev), p.cu_seqlens.to(dev),
                          p.sinks.to(dev), p.scale)
    torch.cuda.synchronize()
    assert out.shape == (0, 8, 64) and lse.shape == (0, 8)
