"""Non-causal ragged prefill without a KV cache (sinkattn_prefill_noncausal) against the fp64
oracle (oracle.prefill_noncausal): query t of request i attends every token of request i, the
attention of an embedding model served through ragged kernels with no KV cache ("Fast
embeddings on GPUs", section on attention kernels).
"""
import numpy as np
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs
from tolerances import check_lse, check_out

pytestmark = pytest.mark.gpu


def _run(sa, p, dev, **kw):
    out, lse = sa.prefill_noncausal(p.q.to(dev), p.k.to(dev), p.v.to(dev), p.cu_seqlens.to(dev),
                                    None if p.sinks is None else p.sinks.to(dev), p.scale, **kw)
    torch.cuda.synchronize()
    return out, lse


def _oracle(o, p, select=None):
    return o.prefill_noncausal(p.q, p.k, p.v, p.cu_seqlens, p.sinks, p.scale, select=select)


@pytest.mark.parametrize("D,G,Hkv", [(64, 8, 2), (64, 1, 4), (128, 16, 1), (128, 2, 4)])
@pytest.mark.parametrize("sinks", [True, False])
def test_noncausal_shapes(sa, oracle_mod, cuda_dev, D, G, Hkv, sinks):
    # ragged lengths around the 128-key tile: one token, a tile and one, an empty request,
    # an exact tile, several tiles with a ragged end
    lens = [300, 1, 129, 0, 128, 40, 513]
    p = inputs.make_prefill(lens, G * Hkv, Hkv, D, seed=200 + D + G, sinks=sinks)
    ws = sa.workspace(0, cuda_dev, "prefill")
    sa.get_status(ws)
    out, lse = _run(sa, p, cuda_dev)
    assert sa.get_status(ws) == 0
    ro, rl = _oracle(oracle_mod, p)
    check_out(out, ro, what="non-causal prefill out")
    check_lse(lse, rl, what="non-causal prefill lse")


def test_noncausal_is_not_the_causal_result(sa, cuda_dev):
    # guard against the causal kernel being run: the first row of a request differs, the
    # last row sees the same keys in both
    p = inputs.make_prefill([300, 77], 8, 2, 64, seed=210, sinks=True)
    out, _ = _run(sa, p, cuda_dev)
    cout, _ = sa.prefill(p.q.to(cuda_dev), p.k.to(cuda_dev), p.v.to(cuda_dev), p.cu_seqlens.to(cuda_dev),
                         p.sinks.to(cuda_dev), p.scale)
    torch.cuda.synchronize()
    first = (out[0].float() - cout[0].float()).abs().max()
    last = (out[299].float() - cout[299].float()).abs().max()
    assert first > 1e-2 and last < 1e-2


def test_noncausal_long_requests_last(sa, oracle_mod, cuda_dev):
    # the long requests at the end of the batch and many one-tile requests before them: the
    # work list puts the heaviest blocks first whatever the order of the requests
    lens = [128] * 40 + [64] * 30 + [1000, 2500, 4096]
    p = inputs.make_prefill(lens, 16, 8, 128, seed=220, sinks=False)
    out, lse = _run(sa, p, cuda_dev)
    T, Hq = p.q.shape[:2]
    sel = np.zeros((T, Hq), dtype=bool)
    sel[::13] = True
    sel[-1] = True
    ro, rl = _oracle(oracle_mod, p, select=sel)
    check_out(out, ro, mask=sel, what="non-causal prefill, long requests last")
    check_lse(lse, rl, mask=sel, what="non-causal lse, long requests last")


def test_noncausal_encoder_batch_sampled(sa, oracle_mod, cuda_dev):
    # the embedding batch (2 x 4096 + 12 x 512 + 32 x 128 tokens, 16 / 8 heads, head_dim
    # 128) in the launch configuration the benchmark times; every 41st query row, all heads
    p = inputs.make_workload("encoder_ragged", seed=0)
    ws = sa.workspace(0, cuda_dev, "prefill")
    sa.get_status(ws)
    out, lse = _run(sa, p, cuda_dev)
    assert sa.get_status(ws) == 0
    T, Hq = p.q.shape[:2]
    sel = np.zeros((T, Hq), dtype=bool)
    sel[::41] = True
    ro, rl = _oracle(oracle_mod, p, select=sel)
    check_out(out, ro, mask=sel, what="encoder batch out")
    check_lse(lse, rl, mask=sel, what="encoder batch lse")


def test_noncausal_grid_size_does_not_change_the_result(sa, cuda_dev):
    # every item is computed the same way whichever CTA takes it: bit-equal on 8, 37 SMs
    # and all of them
    p = inputs.make_prefill([700, 129, 3, 256], 16, 2, 64, seed=230, sinks=True)
    ref, rlse = _run(sa, p, cuda_dev)
    for sms in (8, 37):
        out, lse = _run(sa, p, cuda_dev, max_sms=sms)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), rlse.view(torch.int32))


def test_noncausal_many_requests_slow_lookup(sa, oracle_mod, cuda_dev):
    # more than 1024 requests: the work list falls back to walking cu_seqlens in global memory
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(0, 200, size=1100)]
    p = inputs.make_prefill(lens, 8, 2, 64, seed=240, sinks=True)
    out, lse = _run(sa, p, cuda_dev)
    T, Hq = p.q.shape[:2]
    sel = np.zeros((T, Hq), dtype=bool)
    sel[::29] = True
    ro, rl = _oracle(oracle_mod, p, select=sel)
    check_out(out, ro, mask=sel, what="non-causal prefill, 1100 requests")
    check_lse(lse, rl, mask=sel, what="non-causal lse, 1100 requests")
