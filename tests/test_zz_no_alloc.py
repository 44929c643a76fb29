"""sinkattn_decode_noalloc: decode for callers that cannot allocate device memory
(their memory belongs to another allocator, or their path must not call cudaMalloc),
using the library's fixed scratch array instead of a workspace.

Called through the C ABI directly (ctypes), several times in a row with different
batches.  It runs the same kernels, grid and split plan as sinkattn_decode, so its
results must equal that call's bit for bit; they are also checked against the fp64
oracle.  The status output is this call's bits only: a planted bad block-table entry
must show up in the call that read it and be gone in the next clean call.  This file
sorts last so a run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs
from tolerances import check_lse, check_out

pytestmark = pytest.mark.gpu


def _noalloc(sa, d, scale, status):
    q = d["q"]
    B, Hq, D = q.shape
    num_pages, Hkv = d["kp"].shape[:2]
    out = torch.empty_like(q)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=q.device)
    desc = sa.paged_desc(B, Hq, Hkv, D, num_pages, d["bt"].shape[1])
    stream = torch.cuda.current_stream(q.device).cuda_stream
    sk = d["sk"]
    rc = sa.load().sinkattn_decode_noalloc(
        q.data_ptr(), d["kp"].data_ptr(), d["vp"].data_ptr(), d["bt"].data_ptr(),
        d["sl"].data_ptr(), None if sk is None else sk.data_ptr(), ctypes.c_float(scale),
        out.data_ptr(), lse.data_ptr(), ctypes.byref(desc), status.data_ptr(), stream)
    assert rc == 0, f"{sa.error_string(rc)} [{sa.load().sinkattn_last_cuda_error().decode()}]"
    return out, lse


def _dev(w, dev):
    c = w.cache
    return dict(q=w.q.to(dev), kp=c.k_pages.to(dev), vp=c.v_pages.to(dev),
                bt=c.block_table.to(dev), sl=c.lens.to(dev),
                sk=None if w.sinks is None else w.sinks.to(dev))


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row(sa, cuda_dev, oracle_mod):
    batches = [
        inputs.make_decode(("uniform", 512, 8192), 64, 64, 8, 64, seed=21, sinks=True),
        inputs.make_decode([0, 1, 17, 40000, 300, 5], 6, 64, 4, 128, seed=22, sinks=False),
    ]
    status = torch.full((1,), 0x7FFFFFFF, dtype=torch.int32, device=cuda_dev)
    for w in batches:
        d = _dev(w, cuda_dev)
        got, got_lse = _noalloc(sa, d, w.scale, status)
        ref, ref_lse = sa.decode(d["q"], d["kp"], d["vp"], d["bt"], d["sl"], d["sk"], w.scale)
        torch.cuda.synchronize()
        # same kernels, grid and plan as the workspace decode: bit for bit
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), "out differs from sinkattn_decode"
        assert torch.equal(got_lse.view(torch.int32), ref_lse.view(torch.int32)), "lse differs"
        assert int(status.item()) == 0
        # and within the parity bar of the fp64 oracle (a sample of rows on the big batch)
        c = w.cache
        B, Hq = w.q.shape[:2]
        sel = np.zeros((B, Hq), dtype=bool)
        sel[:: max(1, B // 8)] = True
        ro, rl = oracle_mod.decode(w.q, c.k_pages, c.v_pages, c.block_table, c.lens, w.sinks, w.scale,
                                   select=sel)
        check_out(got, ro, mask=sel, what="noalloc out vs oracle")
        check_lse(got_lse, rl, mask=sel, what="noalloc lse vs oracle")


def test_noalloc_status_is_per_call(sa, cuda_dev, oracle_mod):
    w = inputs.make_decode([40, 300, 17, 1000], 4, 16, 4, 64, seed=23, sinks=True)
    d = _dev(w, cuda_dev)
    status = torch.zeros((1,), dtype=torch.int32, device=cuda_dev)
    # one out-of-range block-table entry in sequence 1: that call reports it
    bad = dict(d)
    bad["bt"] = d["bt"].clone()
    bad["bt"][1, 3] = w.cache.num_pages + 5
    _noalloc(sa, bad, w.scale, status)
    torch.cuda.synchronize()
    assert int(status.item()) & sa.STATUS_BAD_PAGE
    # the next clean call overwrites the word (not an OR): 0, and its results are right
    got, got_lse = _noalloc(sa, d, w.scale, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    c = w.cache
    ro, rl = oracle_mod.decode(w.q, c.k_pages, c.v_pages, c.block_table, c.lens, w.sinks, w.scale)
    check_out(got, ro, what="noalloc out after a bad call")
    check_lse(got_lse, rl, what="noalloc lse after a bad call")
    # an empty batch clears the word as well; a rejected call (q NULL) leaves it alone
    status.fill_(0x55)
    desc = sa.paged_desc(0, 16, 4, 64, 8, 4)
    stream = torch.cuda.current_stream(cuda_dev).cuda_stream
    rc = sa.load().sinkattn_decode_noalloc(None, None, None, None, None, None, ctypes.c_float(1.0),
                                           None, None, ctypes.byref(desc), status.data_ptr(), stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    status.fill_(0x55)
    desc = sa.paged_desc(4, 16, 4, 64, w.cache.num_pages, d["bt"].shape[1])
    rc = sa.load().sinkattn_decode_noalloc(None, d["kp"].data_ptr(), d["vp"].data_ptr(), d["bt"].data_ptr(),
                                           d["sl"].data_ptr(), None, ctypes.c_float(1.0),
                                           d["q"].data_ptr(), None, ctypes.byref(desc), status.data_ptr(),
                                           stream)
    assert rc == sa.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(status.item()) == 0x55


def test_noalloc_rejects_shapes_beyond_its_scratch(sa, cuda_dev):
    # 4096 sequences x 16 KV heads x G=16 x D=128 needs far more than 32 MiB of partials
    desc = sa.paged_desc(4096, 256, 16, 128, 1000, 8)
    need = sa.decode_workspace_size(desc)
    assert need > 32 * 1024 * 1024
    rc = sa.load().sinkattn_decode_noalloc(16, 16, 16, 16, 16, None, ctypes.c_float(1.0), 16,
                                           None, ctypes.byref(desc), None, None)
    assert rc == sa.ERR_WORKSPACE_TOO_SMALL
