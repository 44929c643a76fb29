"""FP8 E4M3 KV cache on the GPU: the quantising append bit for bit, and the decode over
FP8 pages within the output/lse tolerances, against the fp64 oracle through the C ABI.

Element value = scale[g] * e4m3(code), one fp32 scale per KV head for K and for V; the
append stores the code nearest to x / scale[g] (single-precision division, ties to
even, saturating at +-448).  Inputs: seeded synthetic caches (codes of N(0,1) / scale,
NaN codes in the unused slots and distractor pages)."""
import numpy as np
import pytest
import torch

from paged_gqa_attention_head_gb300 import inputs
from tolerances import check_lse, check_out

pytestmark = pytest.mark.gpu


def _scales(c, dev):
    return c.k_scale.to(dev), c.v_scale.to(dev)


def _decode(sa, w, dev, window=0, split_only=False):
    c = w.cache
    ks, vs = _scales(c, dev)
    args = (w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), ks, vs, c.block_table.to(dev),
            c.lens.to(dev), None if w.sinks is None else w.sinks.to(dev), w.scale)
    out, lse = sa.decode_fp8(*args, window=window)
    torch.cuda.synchronize()
    return out, lse


def _oracle(o, w, window=0, select=None):
    c = w.cache
    return o.decode_fp8(w.q, c.k_pages, c.v_pages, c.k_scale, c.v_scale, c.block_table, c.lens,
                        w.sinks, w.scale, select=select, window=window)


def _special_bf16_values() -> torch.Tensor:
    """Values that exercise the rounding: every E4M3 value, the midpoints between
    neighbours (ties) and one bf16 step either side, saturation, infinities, zeros."""
    codes = torch.arange(0x7F, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).double()
    mids = (vals[:-1] + vals[1:]) / 2
    near = torch.cat([mids.to(torch.bfloat16).double(),
                      torch.nextafter(mids.float(), torch.zeros(1)).to(torch.bfloat16).double()])
    extra = torch.tensor([448.0, 449.0, 464.0, 480.0, 1e4, 3e38, float("inf"), 0.0, 2.0 ** -10,
                          3 * 2.0 ** -11, 2.0 ** -12, 1e-30])
    allv = torch.cat([vals, mids, near, extra])
    return torch.cat([allv, -allv, torch.tensor([-0.0])]).to(torch.bfloat16)


@pytest.mark.parametrize("D", [64, 128])
def test_append_fp8_codes_bit_exact(sa, oracle_mod, cuda_dev, D):
    new, start = [5, 16, 33, 0, 1, 70], [0, 7, 16, 3, 31, 100]
    a = inputs.make_append(new, start, 4, D, seed=30 + D, kv_dtype="fp8")
    c = a.cache
    # with scale 1 on head 0 the special values reach the rounding unchanged
    k = a.k.clone()
    sp = _special_bf16_values()
    flat = k[:, 0].reshape(-1)
    flat[: min(sp.numel(), flat.numel())] = sp[: flat.numel()]
    k[:, 0] = flat.view(k.shape[0], D)
    ks = c.k_scale.clone()
    ks[0] = 1.0
    dev = cuda_dev
    kp, vp = c.k_pages.to(dev), c.v_pages.to(dev)
    sa.append_kv_fp8(k.to(dev), a.v.to(dev), ks.to(dev), c.v_scale.to(dev), a.cu_seqlens.to(dev),
                     c.block_table.to(dev), a.start_pos.to(dev), kp, vp)
    torch.cuda.synchronize()
    rk, rv = oracle_mod.append_kv_fp8(k, a.v, ks, c.v_scale, a.cu_seqlens, c.block_table, a.start_pos,
                                      c.k_pages, c.v_pages)
    assert np.array_equal(kp.cpu().numpy(), rk)
    assert np.array_equal(vp.cpu().numpy(), rv)


def test_append_fp8_nan_stays_nan(sa, cuda_dev):
    a = inputs.make_append([3], [0], 2, 64, seed=33, kv_dtype="fp8")
    c = a.cache
    k = a.k.clone()
    k[1, 1, 5] = float("nan")
    dev = cuda_dev
    kp, vp = c.k_pages.to(dev), c.v_pages.to(dev)
    sa.append_kv_fp8(k.to(dev), a.v.to(dev), c.k_scale.to(dev), c.v_scale.to(dev),
                     a.cu_seqlens.to(dev), c.block_table.to(dev), a.start_pos.to(dev), kp, vp)
    code = int(kp[int(c.block_table[0, 0]), 1, 1, 5])
    assert code & 0x7F == 0x7F


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("sinks_on", [True, False])
def test_decode_fp8_shapes(sa, oracle_mod, cuda_dev, D, G, sinks_on):
    Hkv = 2
    lens = [0, 1, 15, 16, 17, 33, 300, 1000, 2049]
    w = inputs.make_decode(lens, len(lens), Hkv * G, Hkv, D, seed=G * 7 + D + 500, sinks=sinks_on,
                           kv_dtype="fp8")
    out, lse = _decode(sa, w, cuda_dev)
    ro, rl = _oracle(oracle_mod, w)
    check_out(out, ro)
    check_lse(lse, rl)
    assert sa.get_status(sa.workspace(0, cuda_dev)) == 0


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("window", [1, 16, 100, 1000])
def test_decode_fp8_window(sa, oracle_mod, cuda_dev, D, window):
    lens = [0, 1, 15, 16, 17, 100, 128, 129, 300, 2049, 40000]
    w = inputs.make_decode(lens, len(lens), 4 * (2 if D == 64 else 4), 4, D, seed=600 + window,
                           sinks=True, kv_dtype="fp8")
    out, lse = _decode(sa, w, cuda_dev, window=window)
    ro, rl = _oracle(oracle_mod, w, window=window)
    check_out(out, ro)
    check_lse(lse, rl)


@pytest.mark.parametrize("seed", [1, 2])
def test_decode_fp8_long_sequences_split_across_warps(sa, oracle_mod, cuda_dev, seed):
    lens = [40000, 70001, 131072, 5]
    w = inputs.make_decode(lens, 4, 16, 2, 64, seed=700 + seed, sinks=True, kv_dtype="fp8")
    out, lse = _decode(sa, w, cuda_dev)
    ro, rl = _oracle(oracle_mod, w)
    check_out(out, ro)
    check_lse(lse, rl)


def test_decode_fp8_null_scales_mean_one(sa, oracle_mod, cuda_dev):
    """NULL scale arrays act as scale 1 (codes generated at scale 1, so the values keep
    the N(0,1) magnitude the tolerance is stated for)."""
    w = inputs.make_decode([1, 40, 300, 4000], 4, 16, 2, 64, seed=710, sinks=True, kv_dtype="fp8",
                           fp8_unit_scales=True)
    c, dev = w.cache, cuda_dev
    out, lse = sa.decode_fp8(w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), None, None,
                             c.block_table.to(dev), c.lens.to(dev), w.sinks.to(dev), w.scale)
    torch.cuda.synchronize()
    ro, rl = oracle_mod.decode_fp8(w.q, c.k_pages, c.v_pages, None, None, c.block_table, c.lens,
                                   w.sinks, w.scale)
    check_out(out, ro)
    check_lse(lse, rl)


def test_decode_fp8_split_then_merge_equals_decode_bitwise(sa, cuda_dev):
    w = inputs.make_decode(("uniform", 1, 9000), 24, 64, 8, 64, seed=720, sinks=True, kv_dtype="fp8")
    c, dev = w.cache, cuda_dev
    ks, vs = _scales(c, dev)
    args = (w.q.to(dev), c.k_pages.to(dev), c.v_pages.to(dev), ks, vs, c.block_table.to(dev),
            c.lens.to(dev), w.sinks.to(dev), w.scale)
    o1, l1 = sa.decode_fp8(*args)
    o2, l2, ws, desc = sa.decode_fp8_splitkv(*args)
    sa.decode_merge(args[6], args[7], o2, l2, desc, ws)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_append_then_decode_fp8(sa, oracle_mod, cuda_dev):
    """A decode step as served: quantise-append the new token, then attend over the cache."""
    lens_before = [0, 15, 16, 100, 2047]
    a = inputs.make_append([1] * 5, lens_before, 8, 64, seed=730, kv_dtype="fp8")
    c, dev = a.cache, cuda_dev
    kp, vp = c.k_pages.to(dev), c.v_pages.to(dev)
    ks, vs = _scales(c, dev)
    sa.append_kv_fp8(a.k.to(dev), a.v.to(dev), ks, vs, a.cu_seqlens.to(dev), c.block_table.to(dev),
                     a.start_pos.to(dev), kp, vp)
    q = inputs.normal_bf16((5, 64, 64), 731, 1)
    sinks = torch.from_numpy(inputs.normal_f32(64, 731, 2))
    lens = torch.tensor([L + 1 for L in lens_before], dtype=torch.int32)
    out, lse = sa.decode_fp8(q.to(dev), kp, vp, ks, vs, c.block_table.to(dev), lens.to(dev),
                             sinks.to(dev), 0.125)
    torch.cuda.synchronize()
    rk, rv = oracle_mod.append_kv_fp8(a.k, a.v, c.k_scale, c.v_scale, a.cu_seqlens, c.block_table,
                                      a.start_pos, c.k_pages, c.v_pages)
    assert np.array_equal(kp.cpu().numpy(), rk) and np.array_equal(vp.cpu().numpy(), rv)
    ro, rl = oracle_mod.decode_fp8(q, rk, rv, c.k_scale, c.v_scale, c.block_table, lens, sinks, 0.125)
    check_out(out, ro)
    check_lse(lse, rl)


@pytest.mark.parametrize("name", ["gptoss_decode_fp8", "qwen3_decode_fp8", "longctx_decode_fp8"])
def test_fp8_full_configs_sampled(sa, oracle_mod, cuda_dev, name):
    """The decode shapes over an FP8 cache at full size: all heads of 12 random sequences
    (plus the longest and the shortest) against the oracle."""
    w = inputs.make_workload(name, seed=0)
    out, lse = _decode(sa, w, cuda_dev)
    B, Hq = w.q.shape[:2]
    lens = w.cache.lens.numpy()
    rows = set(np.random.default_rng(3).choice(B, 12, replace=False).tolist())
    rows |= {int(lens.argmax()), int(lens.argmin())}
    sel = np.zeros((B, Hq), dtype=bool)
    sel[sorted(rows)] = True
    ro, rl = _oracle(oracle_mod, w, select=sel)
    check_out(out, ro, mask=sel)
    check_lse(lse, rl, mask=sel)
    assert sa.get_status(sa.workspace(0, cuda_dev)) == 0


@pytest.mark.parametrize("D", [64, 128])
def test_decode_fp8_q_at_the_edge_of_fp16(sa, oracle_mod, cuda_dev, D):
    """The FP8 decode forms q.k with q in fp16: exact for |q| in [2^-14, 65504].  Rows whose
    entries reach 60000 and rows of tiny entries (2^-13) must still match the oracle."""
    lens = [17, 300, 2000, 1]
    w = inputs.make_decode(lens, len(lens), 16, 2, D, seed=70 + D, sinks=True, kv_dtype="fp8")
    q = w.q.float()
    q[0, :, ::7] = 60000.0
    q[1, 3] = 2.0 ** -13 * torch.sign(q[1, 3])
    q[2, :, 1] = -65000.0
    w.q = q.to(torch.bfloat16)
    assert float(w.q.float().abs().max()) < 65504
    # a small K scale keeps the logits moderate (an lse near 1e5 would be beyond fp32's 1e-3)
    w.cache.k_scale = torch.full_like(w.cache.k_scale, 2e-6)
    out, lse = _decode(sa, w, cuda_dev)
    ro, rl = _oracle(oracle_mod, w)
    check_out(out, ro, what="fp8 decode, q at the edge of fp16")
    check_lse(lse, rl, what="fp8 decode lse, q at the edge of fp16")
