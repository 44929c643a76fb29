"""sinkattn_decode_noalloc: decode for callers that cannot allocate device memory
(their memory belongs to another allocator, or their path must not call cudaMalloc),
using the library's fixed scratch array instead of a workspace.

Called through the C ABI directly (ctypes), twice in a row with different batches,
and compared with sinkattn_decode on the same inputs.  This file sorts last so a
run that stops at the first failure has already run every other test.
"""
import ctypes

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


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row(sa, cuda_dev):
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
        check_out(got, ref.double().cpu().numpy(), what="noalloc out")
        check_lse(got_lse, ref_lse.double().cpu().numpy(), what="noalloc lse")
        assert int(status.item()) == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(sa, cuda_dev):
    # 4096 sequences x 16 KV heads x G=16 x D=128 needs far more than 32 MiB of partials
    desc = sa.paged_desc(4096, 256, 16, 128, 1000, 8)
    need = sa.decode_workspace_size(desc)
    assert need > 32 * 1024 * 1024
    rc = sa.load().sinkattn_decode_noalloc(16, 16, 16, 16, 16, None, ctypes.c_float(1.0), 16,
                                           None, ctypes.byref(desc), None, None)
    assert rc == sa.ERR_WORKSPACE_TOO_SMALL
