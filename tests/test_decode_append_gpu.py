"""Decode with append on the GPU (sinkattn_decode_append): the new K/V rows written into
the cache and attended in one pass.  Checked bit for bit against the two-call path
(sinkattn_append_kv at start positions seq_lens - 1, then sinkattn_decode) for the
outputs, the lse and every byte of the pages, and against the oracle's append and
decode within the parity tolerance."""
import numpy as np
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs
from tolerances import check_lse, check_out

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16)


def _dev(w, dev):
    c = w.cache
    return dict(q=w.q.to(dev), kp=c.k_pages.to(dev), vp=c.v_pages.to(dev), bt=c.block_table.to(dev),
                sl=c.lens.to(dev), sk=None if w.sinks is None else w.sinks.to(dev))


def _append_args(w, k_new, v_new):
    """The same rows as a packed append: one token per sequence with seq_lens >= 1."""
    lens = w.cache.lens.tolist()
    has = [L >= 1 for L in lens]
    cu = np.concatenate([[0], np.cumsum(has)]).astype(np.int32)
    rows = [b for b, h in enumerate(has) if h]
    start = torch.tensor([max(L - 1, 0) for L in lens], dtype=torch.int32)
    return k_new[rows].contiguous(), v_new[rows].contiguous(), torch.from_numpy(cu), start


def _two_calls(sa, w, d, k_new, v_new, dev, window):
    kp, vp = d["kp"].clone(), d["vp"].clone()
    ka, va, cu, start = _append_args(w, k_new, v_new)
    if ka.shape[0]:
        sa.append_kv(ka.to(dev), va.to(dev), cu.to(dev), d["bt"], start.to(dev), kp, vp)
    out, lse = sa.decode(d["q"], kp, vp, d["bt"], d["sl"], d["sk"], w.scale, window=window)
    torch.cuda.synchronize()
    return out, lse, kp, vp


CASES = [
    # lengths, Hq, Hkv, D, window
    ([1, 16, 17, 64, 129, 0, 300, 2049], 8, 2, 64, 0),
    ([1, 16, 17, 64, 129, 0, 300, 2049], 32, 2, 128, 0),
    ([5, 15, 32, 33, 700, 1000, 128, 129], 16, 4, 64, 128),
    ([2, 31, 48, 4000], 4, 4, 128, 100),
    # two 8-head tiles at head_dim 64: split-KV, and the one-launch window kernel
    ([1, 16, 17, 129, 0, 300, 2049], 32, 2, 64, 0),
    ([5, 15, 33, 700, 129, 0], 32, 2, 64, 128),
]


@pytest.mark.parametrize("lens,Hq,Hkv,D,window", CASES)
def test_decode_append_equals_append_then_decode_bitwise(sa, cuda_dev, lens, Hq, Hkv, D, window):
    w = inputs.make_decode(lens, len(lens), Hq, Hkv, D, seed=D + Hq + window, sinks=True)
    k_new, v_new = inputs.new_rows(len(lens), Hkv, D, seed=D + Hq)
    d = _dev(w, cuda_dev)
    ref_out, ref_lse, ref_kp, ref_vp = _two_calls(sa, w, d, k_new, v_new, cuda_dev, window)
    kp, vp = d["kp"].clone(), d["vp"].clone()
    ws = sa.workspace(0, cuda_dev)
    sa.get_status(ws)
    out, lse = sa.decode_append(d["q"], k_new.to(cuda_dev), v_new.to(cuda_dev), kp, vp, d["bt"],
                                d["sl"], d["sk"], w.scale, window=window)
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(ref_out))
    assert torch.equal(lse.cpu().view(torch.int32), ref_lse.cpu().view(torch.int32))
    assert torch.equal(_bits(kp), _bits(ref_kp)) and torch.equal(_bits(vp), _bits(ref_vp))
    assert sa.get_status(ws) == 0


def test_decode_append_matches_oracle(sa, oracle_mod, cuda_dev):
    lens = [1, 16, 17, 130, 0, 555]
    w = inputs.make_decode(lens, len(lens), 16, 2, 64, seed=5, sinks=True)
    k_new, v_new = inputs.new_rows(len(lens), 2, 64, seed=5)
    c = w.cache
    ka, va, cu, start = _append_args(w, k_new, v_new)
    ek, ev = oracle_mod.append_kv(ka, va, cu, c.block_table, start, c.k_pages, c.v_pages)
    kp_ref = torch.from_numpy(ek.view(np.int16)).view(torch.bfloat16)
    vp_ref = torch.from_numpy(ev.view(np.int16)).view(torch.bfloat16)
    ro, rl = oracle_mod.decode(w.q, kp_ref, vp_ref, c.block_table, c.lens, w.sinks, w.scale)
    d = _dev(w, cuda_dev)
    out, lse = sa.decode_append(d["q"], k_new.to(cuda_dev), v_new.to(cuda_dev), d["kp"], d["vp"],
                                d["bt"], d["sl"], d["sk"], w.scale)
    torch.cuda.synchronize()
    check_out(out, ro)
    check_lse(lse, rl)
    assert np.array_equal(_bits(d["kp"]).numpy().view(np.uint16), ek)
    assert np.array_equal(_bits(d["vp"]).numpy().view(np.uint16), ev)


def test_decode_append_gptoss_decode_config(sa, cuda_dev):
    """The gpt-oss-shape decode batch (64 sequences, lengths U[512, 8192], 64 q / 8 KV heads)."""
    w = inputs.make_workload("gptoss_decode", seed=0)
    k_new, v_new = inputs.new_rows(64, 8, 64, seed=0)
    d = _dev(w, cuda_dev)
    ref_out, ref_lse, ref_kp, ref_vp = _two_calls(sa, w, d, k_new, v_new, cuda_dev, 0)
    kp, vp = d["kp"].clone(), d["vp"].clone()
    out, lse = sa.decode_append(d["q"], k_new.to(cuda_dev), v_new.to(cuda_dev), kp, vp, d["bt"],
                                d["sl"], d["sk"], w.scale)
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(ref_out))
    assert torch.equal(lse.cpu().view(torch.int32), ref_lse.cpu().view(torch.int32))
    assert torch.equal(_bits(kp), _bits(ref_kp)) and torch.equal(_bits(vp), _bits(ref_vp))


def test_decode_append_length_beyond_block_table_writes_nothing(sa, cuda_dev):
    """A length past the block table sets the status bit; that sequence's new row goes nowhere
    (the other sequences' rows are written as usual)."""
    lens = [20, 40, 33]
    w = inputs.make_decode(lens, 3, 8, 2, 64, seed=9, sinks=True)
    k_new, v_new = inputs.new_rows(3, 2, 64, seed=9)
    d = _dev(w, cuda_dev)
    cap = d["bt"].shape[1] * 16
    bad = d["sl"].clone()
    bad[1] = cap + 5
    ok_kp, ok_vp = d["kp"].clone(), d["vp"].clone()
    sa.decode_append(d["q"], k_new.to(cuda_dev), v_new.to(cuda_dev), ok_kp, ok_vp, d["bt"], d["sl"],
                     d["sk"], w.scale)
    kp, vp = d["kp"].clone(), d["vp"].clone()
    ws = sa.workspace(0, cuda_dev)
    sa.get_status(ws)
    sa.decode_append(d["q"], k_new.to(cuda_dev), v_new.to(cuda_dev), kp, vp, d["bt"], bad, d["sk"],
                     w.scale)
    torch.cuda.synchronize()
    assert sa.get_status(ws) & sa.STATUS_BAD_LENGTH
    # the pages of sequence 1 keep their old contents, the others take the new rows
    bt = w.cache.block_table
    own1 = [int(p) for p in bt[1].tolist() if p >= 0]
    others = [int(p) for r in (0, 2) for p in bt[r].tolist() if p >= 0]
    assert torch.equal(_bits(kp[own1]), _bits(d["kp"][own1]))
    assert torch.equal(_bits(vp[own1]), _bits(d["vp"][own1]))
    assert torch.equal(_bits(kp[others]), _bits(ok_kp[others]))
    assert torch.equal(_bits(vp[others]), _bits(ok_vp[others]))
