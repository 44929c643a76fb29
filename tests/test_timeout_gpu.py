"""The kernels' watchdog: every pipeline wait gives up after the call's wait limit
(sinkattn_paged_desc.wait_limit_us), the kernel records SINKATTN_STATUS_WAIT_TIMEOUT, lets
the copies and MMAs it issued finish, and returns.

A limit of 1 us is the testing setting: a wait gives up unless its barrier has completed
when first tested, and the first wait of every kernel finds its copy from HBM still in
flight, so the call gives up while copies (and, in prefill, possibly MMAs) are in flight -
the path that must let them finish before the CTA leaves.  Every call must end - the stream
synchronises without a CUDA error - with no status bit but the timeout, and a normal call
right after, on the same workspace and device, must match the oracle again.
"""
import numpy as np
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs
from tolerances import check_lse, check_out

pytestmark = pytest.mark.gpu


def _until_timeout(sa, call, ws, tries=20):
    for _ in range(tries):
        call()
        torch.cuda.synchronize()  # the call ended: no hang, no CUDA error
        st = sa.get_status(ws)
        assert st & ~sa.STATUS_WAIT_TIMEOUT == 0, f"unexpected status bits {st:#x}"
        if st & sa.STATUS_WAIT_TIMEOUT:
            return True
    return False


def _decode_ws(sa, w, dev):
    c = w.cache
    desc = sa.paged_desc(w.q.shape[0], w.q.shape[1], c.k_pages.shape[1], w.q.shape[2],
                         c.k_pages.shape[0], c.block_table.shape[1])
    return torch.zeros(sa.decode_workspace_size(desc), dtype=torch.uint8, device=dev)


def _sel(B, Hq, every):
    sel = np.zeros((B, Hq), dtype=bool)
    sel[::every] = True
    return sel


@pytest.mark.parametrize("fp8,window", [(False, 0), (True, 0), (False, 128)])
def test_decode_wait_timeout_then_clean_call(sa, oracle_mod, cuda_dev, fp8, window):
    # window 128: the one-launch sliding-window kernel, whose warps meet at CTA barriers
    name = "gptoss_decode_fp8" if fp8 else "gptoss_decode"
    w = inputs.make_workload(name, seed=0)
    c = w.cache
    dev = cuda_dev
    ws = _decode_ws(sa, w, dev)
    q, sk = w.q.to(dev), w.sinks.to(dev)
    kp, vp, bt, sl = c.k_pages.to(dev), c.v_pages.to(dev), c.block_table.to(dev), c.lens.to(dev)
    if fp8:
        ks, vs = c.k_scale.to(dev), c.v_scale.to(dev)
        call = lambda lim: sa.decode_fp8(q, kp, vp, ks, vs, bt, sl, sk, w.scale,  # noqa: E731
                                         workspace_buf=ws, wait_limit_us=lim, window=window)
    else:
        call = lambda lim: sa.decode(q, kp, vp, bt, sl, sk, w.scale, workspace_buf=ws,  # noqa: E731
                                     wait_limit_us=lim, window=window)
    assert _until_timeout(sa, lambda: call(1), ws), "no wait ran out with a 1 us limit"
    out, lse = call(0)
    torch.cuda.synchronize()
    assert sa.get_status(ws) == 0
    sel = _sel(*w.q.shape[:2], 9)
    if fp8:
        ro, rl = oracle_mod.decode_fp8(w.q, c.k_pages, c.v_pages, c.k_scale, c.v_scale, c.block_table,
                                       c.lens, w.sinks, w.scale, select=sel, window=window)
    else:
        ro, rl = oracle_mod.decode(w.q, c.k_pages, c.v_pages, c.block_table, c.lens, w.sinks, w.scale,
                                   select=sel, window=window)
    check_out(out, ro, mask=sel, what="decode after a timed-out call")
    check_lse(lse, rl, mask=sel, what="decode lse after a timed-out call")


def test_decode_append_wait_timeout_then_clean_call(sa, oracle_mod, cuda_dev):
    w = inputs.make_workload("gptoss_decode", seed=0)
    c = w.cache
    dev = cuda_dev
    ws = _decode_ws(sa, w, dev)
    B, Hq, D = w.q.shape
    kn, vn = (t.to(dev) for t in inputs.new_rows(B, c.k_pages.shape[1], D, seed=0))
    q, sk, bt, sl = w.q.to(dev), w.sinks.to(dev), c.block_table.to(dev), c.lens.to(dev)
    kp, vp = c.k_pages.to(dev), c.v_pages.to(dev)
    assert _until_timeout(sa, lambda: sa.decode_append(q, kn, vn, kp, vp, bt, sl, sk, w.scale,
                                                        workspace_buf=ws, wait_limit_us=1), ws)
    # a clean step on a fresh copy of the cache
    kp, vp = c.k_pages.to(dev), c.v_pages.to(dev)
    out, lse = sa.decode_append(q, kn, vn, kp, vp, bt, sl, sk, w.scale, workspace_buf=ws)
    torch.cuda.synchronize()
    assert sa.get_status(ws) == 0
    cu1 = torch.arange(B + 1, dtype=torch.int32)
    ek, ev = oracle_mod.append_kv(kn.cpu(), vn.cpu(), cu1, c.block_table, (c.lens - 1).clamp(min=0),
                                  c.k_pages, c.v_pages)
    assert np.array_equal(kp.cpu().view(torch.int16).numpy().view(np.uint16), ek)
    assert np.array_equal(vp.cpu().view(torch.int16).numpy().view(np.uint16), ev)
    sel = _sel(B, Hq, 9)
    ro, rl = oracle_mod.decode(w.q, ek, ev, c.block_table, c.lens, w.sinks, w.scale, select=sel)
    check_out(out, ro, mask=sel, what="decode with append after a timed-out call")
    check_lse(lse, rl, mask=sel, what="lse after a timed-out call")


@pytest.mark.parametrize("prefix", [False, True])
def test_prefill_wait_timeout_then_clean_call(sa, oracle_mod, cuda_dev, prefix):
    dev = cuda_dev
    if prefix:
        p = inputs.make_prefill([512, 300, 129], 16, 2, 64, seed=51, sinks=True,
                                prefix_lens=[1000, 0, 37])
    else:
        p = inputs.make_prefill([2048, 700, 129, 1], 64, 8, 64, seed=52, sinks=True)
    kw = {}
    if p.prefix is not None:
        kw = dict(k_pages=p.prefix.k_pages.to(dev), v_pages=p.prefix.v_pages.to(dev),
                  prefix_block_table=p.prefix.block_table.to(dev), prefix_lens=p.prefix.lens.to(dev))
    args = (p.q.to(dev), p.k.to(dev), p.v.to(dev), p.cu_seqlens.to(dev), p.sinks.to(dev), p.scale)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    assert _until_timeout(sa, lambda: sa.prefill(*args, **kw, workspace_buf=ws, wait_limit_us=1), ws)
    out, lse = sa.prefill(*args, **kw, workspace_buf=ws)
    torch.cuda.synchronize()
    assert sa.get_status(ws) == 0
    T, Hq = p.q.shape[:2]
    sel = _sel(T, Hq, 5)
    pre = p.prefix
    ro, rl = oracle_mod.prefill(p.q, p.k, p.v, p.cu_seqlens, p.sinks, p.scale,
                                None if pre is None else pre.k_pages, None if pre is None else pre.v_pages,
                                None if pre is None else pre.block_table, None if pre is None else pre.lens,
                                select=sel)
    check_out(out, ro, mask=sel, what="prefill after a timed-out call")
    check_lse(lse, rl, mask=sel, what="prefill lse after a timed-out call")
