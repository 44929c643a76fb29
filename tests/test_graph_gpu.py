"""The boundary calls are capturable in CUDA graphs (they allocate nothing and never
synchronise inside a call): a captured decode, prefill and append, replayed on new
inputs copied into the captured buffers, give exactly the results of direct calls."""
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs

pytestmark = pytest.mark.gpu


def _decode_args(w, dev):
    c = w.cache
    return [w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), c.block_table.to(dev), c.lens.to(dev),
            w.sinks.to(dev)]


@pytest.mark.parametrize("window", [0, 128])
def test_decode_graph_replay_matches_direct_calls(sa, cuda_dev, window):
    """Capture once; replay with the captured batch, then with new queries and shorter
    lengths copied into the same buffers (the graph's launch shapes depend only on the
    buffer shapes, the work plan is made on the device every call)."""
    w = inputs.make_decode(("uniform", 100, 3000), 16, 32, 4, 64, seed=101, sinks=True)
    bufs = _decode_args(w, cuda_dev)
    out = torch.empty_like(bufs[0])
    lse = torch.empty(bufs[0].shape[:2], dtype=torch.float32, device=cuda_dev)
    call = lambda: sa.decode(*bufs, w.scale, out=out, lse=lse, window=window)  # noqa: E731
    call()  # allocates the workspace and sets kernel attributes before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    q2 = inputs.normal_bf16(tuple(bufs[0].shape), 105, 1).to(cuda_dev)
    for q_new, lens_new in ((bufs[0].clone(), bufs[4].clone()), (q2, bufs[4] // 2)):
        bufs[0].copy_(q_new)
        bufs[4].copy_(lens_new)
        g.replay()
        torch.cuda.synchronize()
        ref_out, ref_lse = sa.decode(*bufs, w.scale, window=window)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse, ref_lse)


def test_prefill_and_append_graph_replay_match_direct_calls(sa, cuda_dev):
    p = inputs.make_prefill([300, 129, 64], 16, 2, 64, seed=103, sinks=True, prefix_lens=[40, 0, 500])
    dev = cuda_dev
    kw = dict(k_pages=p.prefix.k_pages.to(dev), v_pages=p.prefix.v_pages.to(dev),
              prefix_block_table=p.prefix.block_table.to(dev), prefix_lens=p.prefix.lens.to(dev))
    args = (p.q.to(dev), p.k.to(dev), p.v.to(dev), p.cu_seqlens.to(dev), p.sinks.to(dev), p.scale)
    out = torch.empty_like(args[0])
    lse = torch.empty(args[0].shape[:2], dtype=torch.float32, device=dev)
    a = inputs.make_append([300, 129, 64], [0, 17, 3], 2, 64, seed=104)
    ac = a.cache
    kp, vp = ac.k_pages.to(dev), ac.v_pages.to(dev)
    aargs = (a.k.to(dev), a.v.to(dev), a.cu_seqlens.to(dev), ac.block_table.to(dev), a.start_pos.to(dev))

    def step():
        sa.prefill(*args, out=out, lse=lse, **kw)
        sa.append_kv(*aargs, kp, vp)

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    kp.copy_(ac.k_pages.to(dev))
    vp.copy_(ac.v_pages.to(dev))
    g.replay()
    torch.cuda.synchronize()
    ref_out, ref_lse = sa.prefill(*args, **kw)
    ref_kp, ref_vp = ac.k_pages.to(dev), ac.v_pages.to(dev)
    sa.append_kv(*aargs, ref_kp, ref_vp)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse, ref_lse)
    assert torch.equal(kp.view(torch.int16), ref_kp.view(torch.int16))
    assert torch.equal(vp.view(torch.int16), ref_vp.view(torch.int16))
