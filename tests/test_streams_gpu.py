"""Calls on different streams run concurrently and independently: a decode and a chunked
prefill issued at the same time on two streams (each with its own workspace, as a
serving loop mixing decode and prefill requests would do) give bit for bit the results
of the same calls issued one after the other.  With desc.max_sms the persistent grids
leave SMs free for such concurrent work; capped calls keep their results."""
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs
from tolerances import check_lse, check_out

pytestmark = pytest.mark.gpu


def test_decode_and_chunked_prefill_on_two_streams_match_sequential(sa, cuda_dev):
    dev = cuda_dev
    w = inputs.make_decode(("uniform", 200, 20000), 96, 64, 8, 64, seed=211, sinks=True)
    c = w.cache
    dargs = (w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), c.block_table.to(dev),
             c.lens.to(dev), w.sinks.to(dev), w.scale)
    p = inputs.make_prefill([700, 129, 512], 64, 8, 64, seed=212, sinks=True,
                            prefix_lens=[3000, 0, 1200])
    pre = p.prefix
    pargs = (p.q.to(dev), p.k.to(dev), p.v.to(dev), p.cu_seqlens.to(dev), p.sinks.to(dev), p.scale)
    pkw = dict(k_pages=pre.k_pages.to(dev), v_pages=pre.v_pages.to(dev),
               prefix_block_table=pre.block_table.to(dev), prefix_lens=pre.lens.to(dev))

    ref_d = sa.decode(*dargs)
    ref_p = sa.prefill(*pargs, **pkw)
    torch.cuda.synchronize()
    ref_d = tuple(t.clone() for t in ref_d)
    ref_p = tuple(t.clone() for t in ref_p)

    dws = torch.zeros(sa.decode_workspace_size(sa.paged_desc(
        w.q.shape[0], 64, 8, 64, c.k_pages.shape[0], c.block_table.shape[1])), dtype=torch.uint8,
        device=dev)
    pws = torch.zeros(max(256, sa.prefill_workspace_size(sa.paged_desc(
        3, 64, 8, 64, pre.k_pages.shape[0], pre.block_table.shape[1]))), dtype=torch.uint8,
        device=dev)
    d_out, d_lse = torch.empty_like(ref_d[0]), torch.empty_like(ref_d[1])
    p_out, p_lse = torch.empty_like(ref_p[0]), torch.empty_like(ref_p[1])
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    for _ in range(4):
        d_out.fill_(0)
        p_out.fill_(0)
        ev = torch.cuda.Event()
        ev.record()
        s1.wait_event(ev)
        s2.wait_event(ev)
        with torch.cuda.stream(s1):
            sa.decode(*dargs, out=d_out, lse=d_lse, workspace_buf=dws)
        with torch.cuda.stream(s2):
            sa.prefill(*pargs, **pkw, out=p_out, lse=p_lse, workspace_buf=pws)
        torch.cuda.synchronize()
        assert torch.equal(d_out, ref_d[0]) and torch.equal(d_lse, ref_d[1])
        assert torch.equal(p_out, ref_p[0]) and torch.equal(p_lse, ref_p[1])
    assert sa.get_status(dws) == 0 and sa.get_status(pws) == 0


@pytest.mark.parametrize("max_sms", [1, 37])
def test_prefill_on_fewer_sms_is_bit_identical(sa, cuda_dev, max_sms):
    """desc.max_sms caps the persistent prefill grid; every item is computed the same way
    whichever CTA takes it, so the results do not change."""
    dev = cuda_dev
    p = inputs.make_prefill([700, 129, 512], 64, 8, 64, seed=213, sinks=True,
                            prefix_lens=[3000, 0, 1200])
    pre = p.prefix
    args = (p.q.to(dev), p.k.to(dev), p.v.to(dev), p.cu_seqlens.to(dev), p.sinks.to(dev), p.scale)
    kw = dict(k_pages=pre.k_pages.to(dev), v_pages=pre.v_pages.to(dev),
              prefix_block_table=pre.block_table.to(dev), prefix_lens=pre.lens.to(dev))
    ref = [t.clone() for t in sa.prefill(*args, **kw)]
    got = sa.prefill(*args, **kw, max_sms=max_sms)
    torch.cuda.synchronize()
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])


@pytest.mark.parametrize("max_sms", [1, 20])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_decode_on_fewer_sms_matches_the_oracle(sa, oracle_mod, cuda_dev, max_sms, kv):
    """desc.max_sms caps the persistent split-KV grid (fewer warps, longer shares, other
    split points): the results stay within the parity bar of the oracle."""
    dev = cuda_dev
    w = inputs.make_decode(("uniform", 1, 5000), 24, 32, 4, 64, seed=214, sinks=True, kv_dtype=kv)
    c = w.cache
    common = (c.block_table.to(dev), c.lens.to(dev), w.sinks.to(dev), w.scale)
    if kv == "fp8":
        out, lse = sa.decode_fp8(w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev),
                                 c.k_scale.to(dev), c.v_scale.to(dev), *common, max_sms=max_sms)
        ro, rl = oracle_mod.decode_fp8(w.q, c.k_pages, c.v_pages, c.k_scale, c.v_scale,
                                       c.block_table, c.lens, w.sinks, w.scale)
    else:
        out, lse = sa.decode(w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), *common,
                             max_sms=max_sms)
        ro, rl = oracle_mod.decode(w.q, c.k_pages, c.v_pages, c.block_table, c.lens, w.sinks,
                                   w.scale)
    torch.cuda.synchronize()
    check_out(out, ro)
    check_lse(lse, rl)


@pytest.mark.parametrize("split", [40, 100])
def test_prefill_then_decode_started_early_on_one_stream(sa, cuda_dev, split):
    """A chunked prefill that lets the next kernel start early (SINKATTN_FLAG_LAUNCH_NEXT_EARLY,
    on `split` SMs) and a decode started early after it (SINKATTN_FLAG_START_EARLY, on the
    other SMs), on one stream, in a captured graph and called directly: each result is bit for
    bit that of the same call made alone, and the decode's merge waits for its split-KV pass."""
    dev = cuda_dev
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    w = inputs.make_decode(("uniform", 200, 20000), 96, 64, 8, 64, seed=213, sinks=True)
    c = w.cache
    dargs = (w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), c.block_table.to(dev),
             c.lens.to(dev), w.sinks.to(dev), w.scale)
    p = inputs.make_prefill([700, 129, 512], 64, 8, 64, seed=214, sinks=True,
                            prefix_lens=[3000, 0, 1200])
    pre = p.prefix
    pargs = (p.q.to(dev), p.k.to(dev), p.v.to(dev), p.cu_seqlens.to(dev), p.sinks.to(dev), p.scale)
    pkw = dict(k_pages=pre.k_pages.to(dev), v_pages=pre.v_pages.to(dev),
               prefix_block_table=pre.block_table.to(dev), prefix_lens=pre.lens.to(dev))
    dcap = n_sms - split
    ref_d = tuple(t.clone() for t in sa.decode(*dargs, max_sms=dcap))
    ref_p = tuple(t.clone() for t in sa.prefill(*pargs, **pkw, max_sms=split))
    torch.cuda.synchronize()
    dws = torch.zeros(sa.decode_workspace_size(sa.paged_desc(
        w.q.shape[0], 64, 8, 64, c.k_pages.shape[0], c.block_table.shape[1], max_sms=dcap)),
        dtype=torch.uint8, device=dev)
    pws = torch.zeros(256, dtype=torch.uint8, device=dev)
    d_out, d_lse = torch.empty_like(ref_d[0]), torch.empty_like(ref_d[1])
    p_out, p_lse = torch.empty_like(ref_p[0]), torch.empty_like(ref_p[1])

    def step():
        sa.prefill(*pargs, **pkw, out=p_out, lse=p_lse, workspace_buf=pws, max_sms=split,
                   flags=sa.FLAG_LAUNCH_NEXT_EARLY)
        sa.decode(*dargs, out=d_out, lse=d_lse, workspace_buf=dws, max_sms=dcap,
                  flags=sa.FLAG_START_EARLY)

    for _ in range(3):
        d_out.fill_(0)
        p_out.fill_(0)
        step()
        torch.cuda.synchronize()
        assert torch.equal(d_out, ref_d[0]) and torch.equal(d_lse, ref_d[1])
        assert torch.equal(p_out, ref_p[0]) and torch.equal(p_lse, ref_p[1])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        d_out.fill_(0)
        p_out.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(d_out, ref_d[0]) and torch.equal(d_lse, ref_d[1])
        assert torch.equal(p_out, ref_p[0]) and torch.equal(p_lse, ref_p[1])
    assert sa.get_status(dws) == 0 and sa.get_status(pws) == 0


@pytest.mark.parametrize("D", [64, 128])
def test_decode_grid_stops_at_its_cap(sa, cuda_dev, D):
    """The split-KV grid stops at 18 MB of page copies in flight (576 CTAs of 32 KB rings at
    head_dim 64, 288 of 64 KB at 128; 115 and 96 of GB300's 152 SMs' worth): an SM cap that
    leaves more CTAs than that gives the same grid and bits as none."""
    dev = cuda_dev
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    keep = (n_sms * 130) // 152  # five CTAs an SM at 64 (three at 128): above the budget
    w = inputs.make_decode(("uniform", 100, 6000), 40, 16, 2, D, seed=215 + D, sinks=True)
    c = w.cache
    args = (w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), c.block_table.to(dev), c.lens.to(dev),
            w.sinks.to(dev), w.scale)
    shape = (w.q.shape[0], 16, 2, D, c.k_pages.shape[0], c.block_table.shape[1])
    assert sa.decode_workspace_size(sa.paged_desc(*shape, max_sms=n_sms)) == \
        sa.decode_workspace_size(sa.paged_desc(*shape))
    ref = sa.decode(*args)
    torch.cuda.synchronize()
    ref = tuple(t.clone() for t in ref)
    for m in (keep, n_sms):
        out, lse = sa.decode(*args, max_sms=m)
        torch.cuda.synchronize()
        assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])


@pytest.mark.slow
def test_long_context_step_with_early_start_matches_the_calls_alone(sa, cuda_dev):
    """The long-context mixed step in the launch configuration the benchmark picks on GB300
    (chunked prefill on 88 of 152 SMs starting the decode early, the decode on the others): bit
    for bit the results of the two calls made alone with the same SM caps."""
    dev = cuda_dev
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    S = (n_sms * 88) // 152
    w = inputs.make_workload("longctx_decode", seed=0)
    c = w.cache
    dargs = (w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), c.block_table.to(dev), c.lens.to(dev),
             w.sinks.to(dev), w.scale)
    p = inputs.make_workload("longctx_chunked", seed=0)
    pre = p.prefix
    pargs = (p.q.to(dev), p.k.to(dev), p.v.to(dev), p.cu_seqlens.to(dev), p.sinks.to(dev), p.scale)
    pkw = dict(k_pages=pre.k_pages.to(dev), v_pages=pre.v_pages.to(dev),
               prefix_block_table=pre.block_table.to(dev), prefix_lens=pre.lens.to(dev))
    ref_d = tuple(t.clone() for t in sa.decode(*dargs, max_sms=n_sms - S))
    ref_p = tuple(t.clone() for t in sa.prefill(*pargs, **pkw, max_sms=S))
    torch.cuda.synchronize()
    d_out, d_lse = torch.empty_like(ref_d[0]), torch.empty_like(ref_d[1])
    p_out, p_lse = torch.empty_like(ref_p[0]), torch.empty_like(ref_p[1])
    dws = torch.zeros(sa.decode_workspace_size(sa.paged_desc(
        w.q.shape[0], 64, 8, 64, c.k_pages.shape[0], c.block_table.shape[1], max_sms=n_sms - S)),
        dtype=torch.uint8, device=dev)
    pws = torch.zeros(256, dtype=torch.uint8, device=dev)
    for _ in range(2):
        sa.prefill(*pargs, **pkw, out=p_out, lse=p_lse, workspace_buf=pws, max_sms=S,
                   flags=sa.FLAG_LAUNCH_NEXT_EARLY)
        sa.decode(*dargs, out=d_out, lse=d_lse, workspace_buf=dws, max_sms=n_sms - S,
                  flags=sa.FLAG_START_EARLY)
        torch.cuda.synchronize()
        assert torch.equal(d_out, ref_d[0]) and torch.equal(d_lse, ref_d[1])
        assert torch.equal(p_out, ref_p[0]) and torch.equal(p_lse, ref_p[1])
    assert sa.get_status(dws) == 0 and sa.get_status(pws) == 0
