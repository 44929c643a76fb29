"""Paged KV append on the GPU: bit-exact against the oracle scatter."""
import numpy as np
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("D", [64, 128])
def test_append_matches_oracle_bitwise(sa, oracle_mod, cuda_dev, D):
    a = inputs.make_append([5, 16, 33, 0, 1, 300], [0, 7, 16, 3, 31, 1000], 4, D, seed=D)
    c = a.cache
    ek, ev = oracle_mod.append_kv(a.k, a.v, a.cu_seqlens, c.block_table, a.start_pos, c.k_pages,
                                  c.v_pages)
    kp, vp = c.k_pages.to(cuda_dev), c.v_pages.to(cuda_dev)
    ws = sa.workspace(256, cuda_dev, "append")
    sa.get_status(ws)
    sa.append_kv(a.k.to(cuda_dev), a.v.to(cuda_dev), a.cu_seqlens.to(cuda_dev),
                 c.block_table.to(cuda_dev), a.start_pos.to(cuda_dev), kp, vp)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kp), ek) and np.array_equal(_bits(vp), ev)
    assert sa.get_status(ws) == 0


def test_append_gptoss_prefill_config(sa, oracle_mod, cuda_dev):
    """The prefill workload's K/V (T = 7680, 8 KV heads, D = 64) written into pages."""
    a = inputs.make_append([4096, 2048, 1024, 512], [0, 0, 0, 0], 8, 64, seed=0)
    c = a.cache
    ek, ev = oracle_mod.append_kv(a.k, a.v, a.cu_seqlens, c.block_table, a.start_pos, c.k_pages,
                                  c.v_pages)
    kp, vp = c.k_pages.to(cuda_dev), c.v_pages.to(cuda_dev)
    sa.append_kv(a.k.to(cuda_dev), a.v.to(cuda_dev), a.cu_seqlens.to(cuda_dev),
                 c.block_table.to(cuda_dev), a.start_pos.to(cuda_dev), kp, vp)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(kp), ek) and np.array_equal(_bits(vp), ev)


def test_append_out_of_range_destination_is_skipped_and_reported(sa, cuda_dev):
    a = inputs.make_append([4, 4], [0, 0], 2, 64, seed=3)
    c = a.cache
    bt = c.block_table.clone()
    bt[1, 0] = c.num_pages + 7
    kp, vp = c.k_pages.to(cuda_dev), c.v_pages.to(cuda_dev)
    before = _bits(kp)
    ws = sa.workspace(256, cuda_dev, "append")
    sa.get_status(ws)
    sa.append_kv(a.k.to(cuda_dev), a.v.to(cuda_dev), a.cu_seqlens.to(cuda_dev), bt.to(cuda_dev),
                 a.start_pos.to(cuda_dev), kp, vp)
    assert sa.get_status(ws) & sa.STATUS_BAD_PAGE
    after = _bits(kp)
    # sequence 0 landed, nothing else changed
    pg0 = int(c.block_table[0, 0])
    assert np.array_equal(after[pg0, :, :4], _bits(a.k[:4]).transpose(1, 0, 2))
    changed = np.any(after != before, axis=(1, 2, 3))
    assert set(np.nonzero(changed)[0].tolist()) <= {pg0}
