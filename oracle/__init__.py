"""fp64 CPU oracle for paged GQA attention with sinks (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg, never by the library.  The arithmetic lives in
sinkattn_oracle.c (plain C, double precision, OpenMP over query rows); this file
only builds it with gcc, marshals numpy arrays and reshapes results.

bf16 tensors are handed over as their raw 16-bit patterns, so the oracle reads
exactly the values the GPU reads.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sinkattn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libsinkattn_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math: IEEE double semantics kept)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC,
                        "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_decode.argtypes = [P, P, P, P, P, P, D, I, I, I, I, I, I64, I, I, P, P, P]
        lib.oracle_decode.restype = I
        lib.oracle_prefill.argtypes = [P, P, P, P, I, P, P, P, P, I64, I, P, D, I, I, I, I, I, P, P, P]
        lib.oracle_prefill.restype = I
        lib.oracle_prefill_noncausal.argtypes = [P, P, P, P, I, P, D, I, I, I, P, P, P]
        lib.oracle_prefill_noncausal.restype = I
        lib.oracle_append_kv.argtypes = [P, P, P, I, P, P, I, I64, I, I, I, P, P]
        lib.oracle_append_kv.restype = I
        lib.oracle_partial.argtypes = [P, P, P, I, D, I64, I64, P, P, P]
        lib.oracle_partial.restype = None
        lib.oracle_merge.argtypes = [I, P, P, P, I, D, P, P]
        lib.oracle_merge.restype = None
        lib.oracle_online.argtypes = [P, P, P, I, D, D, I64, I, I64, P, P]
        lib.oracle_online.restype = None
        lib.oracle_decode_fp8.argtypes = [P, P, P, P, P, P, P, P, D, I, I, I, I, I, I64, I, I, P, P, P]
        lib.oracle_decode_fp8.restype = I
        lib.oracle_append_kv_fp8.argtypes = [P, P, P, P, P, I, P, P, I, I64, I, I, I, P, P]
        lib.oracle_append_kv_fp8.restype = I
        lib.oracle_e4m3_codes.argtypes = [P, I64, P]
        lib.oracle_e4m3_codes.restype = None
        lib.oracle_e4m3_values.argtypes = [P, I64, P]
        lib.oracle_e4m3_values.restype = None
        lib.oracle_prefill_fp8.argtypes = [P, P, P, P, I, P, P, P, P, P, P, I64, I, P, D, I, I, I, I, I,
                                           P, P, P]
        lib.oracle_prefill_fp8.restype = I
        lib.oracle_rope_freqs.argtypes = [I, D, D, I, D, D, P, P]
        lib.oracle_rope_freqs.restype = None
        lib.oracle_rope.argtypes = [P, I64, I, I, P, D, D, I, D, D, P]
        lib.oracle_rope.restype = None
        lib.oracle_bf16_round_array.argtypes = [P, I64, P]
        lib.oracle_bf16_round_array.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = I
        _lib = lib
    return _lib


def _bits(t) -> np.ndarray:
    """bf16 torch tensor or uint16 array -> contiguous uint16 numpy array of its bits."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16, t.dtype
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _i32(t) -> np.ndarray:
    if t is None:
        return None
    a = t if isinstance(t, np.ndarray) else t.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _f32(t) -> Optional[np.ndarray]:
    if t is None:
        return None
    a = t if isinstance(t, np.ndarray) else t.detach().cpu().float().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def _u8(t) -> np.ndarray:
    """uint8 / float8_e4m3fn torch tensor or uint8 array -> contiguous uint8 numpy array."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint8
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype in (torch.uint8, torch.float8_e4m3fn), t.dtype
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.uint8).numpy())


def _ptr(a) -> Optional[int]:
    return None if a is None else a.ctypes.data


def max_threads() -> int:
    return _load().oracle_max_threads()


def decode(q, k_pages, v_pages, block_table, seq_lens, sinks, scale: float,
           select: Optional[np.ndarray] = None, window: int = 0):
    """Decode attention.  q [B,Hq,D]; pages [num_pages,Hkv,P,D]; returns (out [B,Hq,D], lse [B,Hq])
    in float64.  select: bool [B,Hq] restricting which rows are computed (others NaN).
    window > 0: only the last `window` cached tokens are seen (sliding window)."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k_pages), _bits(v_pages)
    B, Hq, D = qb.shape
    num_pages, Hkv, P, D2 = kb.shape
    assert D == D2
    bt, sl, sk = _i32(block_table), _i32(seq_lens), _f32(sinks)
    out = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    sel = None if select is None else np.ascontiguousarray(select, dtype=np.uint8)
    rc = lib.oracle_decode(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(bt), _ptr(sl), _ptr(sk), float(scale),
                           B, Hq, Hkv, D, P, num_pages, bt.shape[1], int(window), _ptr(sel), _ptr(out),
                           _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_decode rejected its inputs ({rc})")
    return out, lse


def prefill(q, k, v, cu_seqlens, sinks, scale: float, k_pages=None, v_pages=None,
            prefix_block_table=None, prefix_lens=None, select: Optional[np.ndarray] = None,
            page_size: int = 16, window: int = 0):
    """Causal ragged prefill, optionally over a paged prefix.  Returns (out [T,Hq,D], lse [T,Hq]).
    window > 0: each query sees only the keys at its last `window` absolute positions."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    T, Hq, D = qb.shape
    Hkv = kb.shape[1]
    cu = _i32(cu_seqlens)
    n = cu.shape[0] - 1
    if k_pages is not None:
        kp, vp = _bits(k_pages), _bits(v_pages)
        num_pages, _, page_size, _ = kp.shape
        pbt, pl = _i32(prefix_block_table), _i32(prefix_lens)
        maxp = pbt.shape[1]
    else:
        kp = vp = pbt = pl = None
        num_pages, maxp = 0, 0
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    sel = None if select is None else np.ascontiguousarray(select, dtype=np.uint8)
    rc = lib.oracle_prefill(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cu), n, _ptr(kp), _ptr(vp), _ptr(pbt),
                            _ptr(pl), num_pages, maxp, _ptr(_f32(sinks)), float(scale), Hq, Hkv, D,
                            page_size, int(window), _ptr(sel), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_prefill rejected its inputs ({rc})")
    return out, lse


def prefill_noncausal(q, k, v, cu_seqlens, sinks, scale: float, select: Optional[np.ndarray] = None):
    """Non-causal ragged prefill without a KV cache: query t of sequence i sees every token
    of sequence i.  Returns (out [T,Hq,D], lse [T,Hq])."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    T, Hq, D = qb.shape
    Hkv = kb.shape[1]
    cu = _i32(cu_seqlens)
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    sel = None if select is None else np.ascontiguousarray(select, dtype=np.uint8)
    rc = lib.oracle_prefill_noncausal(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cu), cu.shape[0] - 1,
                                      _ptr(_f32(sinks)), float(scale), Hq, Hkv, D, _ptr(sel),
                                      _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_prefill_noncausal rejected its inputs ({rc})")
    return out, lse


def append_kv(k, v, cu_seqlens, block_table, start_pos, k_pages, v_pages):
    """Scatter new rows into copies of the pages; returns (k_pages, v_pages) as uint16 arrays."""
    lib = _load()
    kb, vb = _bits(k), _bits(v)
    kp, vp = _bits(k_pages).copy(), _bits(v_pages).copy()
    num_pages, Hkv, P, D = kp.shape
    cu, bt, sp = _i32(cu_seqlens), _i32(block_table), _i32(start_pos)
    rc = lib.oracle_append_kv(_ptr(kb), _ptr(vb), _ptr(cu), cu.shape[0] - 1, _ptr(bt), _ptr(sp),
                              bt.shape[1], num_pages, Hkv, D, P, _ptr(kp), _ptr(vp))
    if rc != 0:
        raise ValueError("oracle_append_kv rejected its inputs")
    return kp, vp


def e4m3_values(codes) -> np.ndarray:
    """Value of each E4M3 code (float64; NaN for the NaN codes)."""
    c = _u8(codes)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e4m3_values(_ptr(c), c.size, _ptr(out))
    return out


def e4m3_codes(y) -> np.ndarray:
    """Nearest E4M3 code of each float32 (ties to even, saturating to +-448, NaN kept)."""
    a = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint8)
    _load().oracle_e4m3_codes(_ptr(a), a.size, _ptr(out))
    return out


def decode_fp8(q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, sinks, scale: float,
               select: Optional[np.ndarray] = None, window: int = 0):
    """Decode over an FP8 E4M3 cache: pages uint8 [num_pages,Hkv,P,D] of codes, element
    value scale[g] * e4m3(code) with fp32 k_scale / v_scale [Hkv] (None: 1).  Otherwise as
    decode(); returns (out [B,Hq,D], lse [B,Hq]) in float64."""
    lib = _load()
    qb, kb, vb = _bits(q), _u8(k_pages), _u8(v_pages)
    B, Hq, D = qb.shape
    num_pages, Hkv, P, D2 = kb.shape
    assert D == D2
    bt, sl, sk = _i32(block_table), _i32(seq_lens), _f32(sinks)
    ks, vs = _f32(k_scale), _f32(v_scale)
    out = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    sel = None if select is None else np.ascontiguousarray(select, dtype=np.uint8)
    rc = lib.oracle_decode_fp8(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl),
                               _ptr(sk), float(scale), B, Hq, Hkv, D, P, num_pages, bt.shape[1],
                               int(window), _ptr(sel), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_decode_fp8 rejected its inputs ({rc})")
    return out, lse


def prefill_fp8(q, k, v, cu_seqlens, sinks, scale: float, k_pages, v_pages, k_scale, v_scale,
                prefix_block_table, prefix_lens, select: Optional[np.ndarray] = None, window: int = 0):
    """Chunked prefill over an FP8 E4M3 paged prefix: pages uint8 [num_pages, Hkv, P, D] of
    codes (value scale[g] * e4m3(code), k_scale / v_scale fp32 [Hkv] or None for 1); the
    new tokens' q, k, v bf16.  Returns (out [T, Hq, D], lse [T, Hq]) in float64."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    T, Hq, D = qb.shape
    Hkv = kb.shape[1]
    cu = _i32(cu_seqlens)
    n = cu.shape[0] - 1
    kp, vp = _u8(k_pages), _u8(v_pages)
    num_pages, _, page_size, _ = kp.shape
    pbt, pl = _i32(prefix_block_table), _i32(prefix_lens)
    out = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    sel = None if select is None else np.ascontiguousarray(select, dtype=np.uint8)
    rc = lib.oracle_prefill_fp8(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(cu), n, _ptr(kp), _ptr(vp),
                                _ptr(_f32(k_scale)), _ptr(_f32(v_scale)), _ptr(pbt), _ptr(pl), num_pages,
                                pbt.shape[1], _ptr(_f32(sinks)), float(scale), Hq, Hkv, D, page_size,
                                int(window), _ptr(sel), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_prefill_fp8 rejected its inputs ({rc})")
    return out, lse


def append_kv_fp8(k, v, k_scale, v_scale, cu_seqlens, block_table, start_pos, k_pages, v_pages):
    """Quantise new bf16 rows to E4M3 codes (x / scale[g], nearest, saturating) and scatter
    them into copies of the uint8 pages; returns (k_pages, v_pages) as uint8 arrays."""
    lib = _load()
    kb, vb = _bits(k), _bits(v)
    kp, vp = _u8(k_pages).copy(), _u8(v_pages).copy()
    num_pages, Hkv, P, D = kp.shape
    cu, bt, sp = _i32(cu_seqlens), _i32(block_table), _i32(start_pos)
    ks, vs = _f32(k_scale), _f32(v_scale)
    rc = lib.oracle_append_kv_fp8(_ptr(kb), _ptr(vb), _ptr(ks), _ptr(vs), _ptr(cu), cu.shape[0] - 1,
                                  _ptr(bt), _ptr(sp), bt.shape[1], num_pages, Hkv, D, P, _ptr(kp),
                                  _ptr(vp))
    if rc != 0:
        raise ValueError("oracle_append_kv_fp8 rejected its inputs")
    return kp, vp


def partial(q, k, v, scale: float, j0: int, j1: int):
    """Sink-free state (m, l, acc[D]) of contiguous keys [j0, j1); q [D], k/v [n, D] bf16."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    D = qb.shape[-1]
    m, l = ctypes.c_double(), ctypes.c_double()
    acc = np.zeros(D)
    lib.oracle_partial(_ptr(qb), _ptr(kb), _ptr(vb), D, float(scale), j0, j1, ctypes.byref(m),
                       ctypes.byref(l), _ptr(acc))
    return m.value, l.value, acc


def merge(ms, ls, accs, sink: float):
    """Log-sum-exp merge of partial states plus the sink; returns (out [D], lse)."""
    lib = _load()
    m = np.ascontiguousarray(ms, dtype=np.float64)
    l = np.ascontiguousarray(ls, dtype=np.float64)
    a = np.ascontiguousarray(accs, dtype=np.float64)
    S, D = a.shape
    out = np.zeros(D)
    lse = ctypes.c_double()
    lib.oracle_merge(S, _ptr(m), _ptr(l), _ptr(a), D, float(sink), _ptr(out), ctypes.byref(lse))
    return out, lse.value


def online(q, k, v, scale: float, sink: float, block: int, split_at: int = 0):
    """Streaming softmax seeded with the sink (see sinkattn_oracle.c); returns (out [D], lse)."""
    lib = _load()
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    n, D = kb.shape
    out = np.zeros(D)
    lse = ctypes.c_double()
    lib.oracle_online(_ptr(qb), _ptr(kb), _ptr(vb), D, float(scale), float(sink), n, block, split_at,
                      _ptr(out), ctypes.byref(lse))
    return out, lse.value


# gpt-oss's YaRN settings as TensorSharp gptoss.md section 3 gives them (original context
# 4096, beta_fast 32, beta_slow 1); base and factor are the model's own (not on the pages)
# and are arguments everywhere.
ROPE_DEFAULTS = dict(original_context=4096, beta_fast=32.0, beta_slow=1.0)


def rope_freqs(head_dim: int, base: float, factor: float, original_context: int = 4096,
               beta_fast: float = 32.0, beta_slow: float = 1.0):
    """YaRN-scaled rotation frequency of every pair (float64 [D/2]) and the magnitude
    factor mscale (see sinkattn_oracle.c)."""
    th = np.empty(head_dim // 2)
    ms = ctypes.c_double()
    _load().oracle_rope_freqs(head_dim, float(base), float(factor), int(original_context),
                              float(beta_fast), float(beta_slow), _ptr(th), ctypes.byref(ms))
    return th, ms.value


def rope(x, positions, base: float, factor: float, original_context: int = 4096,
         beta_fast: float = 32.0, beta_slow: float = 1.0) -> np.ndarray:
    """NeoX rotary embedding with YaRN scaling of bf16 rows x [n, H, D], row r at
    positions[r]; float64 [n, H, D], not rounded."""
    xb = _bits(x)
    n, H, D = xb.shape
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int64).reshape(n))
    out = np.empty((n, H, D))
    _load().oracle_rope(_ptr(xb), n, H, D, _ptr(pos), float(base), float(factor),
                        int(original_context), float(beta_fast), float(beta_slow), _ptr(out))
    return out


def bf16_round(x) -> np.ndarray:
    """Nearest bf16 (ties to even) of each float64 value, as uint16 bit patterns."""
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_bf16_round_array(_ptr(a), a.size, _ptr(out))
    return out


def decode_append_rope(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, sinks,
                       scale: float, base: float, factor: float, original_context: int = 4096,
                       beta_fast: float = 32.0, beta_slow: float = 1.0,
                       select: Optional[np.ndarray] = None, window: int = 0):
    """A decode step with rotary embedding and K/V append, in the pages' order
    (TensorSharp gptoss.md section 3: RoPE on Q and K, append K and V to the cache, then
    attention): q [B, Hq, D] and k_new [B, Hkv, D] (bf16, not yet rotated) are rotated at
    the new token's position seq_lens[b] - 1 and rounded to bf16; the rotated key and
    v_new are written to copies of the pages at that position (sequences with length 0
    have no new token); then the rotated query attends the seq_lens[b] cached tokens.
    Returns (out, lse, k_pages, v_pages, q_rot, k_rot) with the pages and the rotated rows
    as uint16 bf16 bit arrays."""
    lens = _i32(seq_lens)
    B = lens.shape[0]
    pos = np.maximum(lens.astype(np.int64) - 1, 0)
    kw = dict(base=base, factor=factor, original_context=original_context, beta_fast=beta_fast,
              beta_slow=beta_slow)
    q_rot = bf16_round(rope(q, pos, **kw))
    k_rot = bf16_round(rope(k_new, pos, **kw))
    has = (lens > 0).astype(np.int64)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(has)
    idx = np.nonzero(has)[0]
    vb = _bits(v_new)
    kp, vp = append_kv(np.ascontiguousarray(k_rot[idx]), np.ascontiguousarray(vb[idx]), cu,
                       block_table, pos.astype(np.int32), k_pages, v_pages)
    out, lse = decode(q_rot, kp, vp, block_table, lens, sinks, scale, select=select, window=window)
    return out, lse, kp, vp, q_rot, k_rot


class using_library:
    """Context manager: route this module's functions through another build of the
    oracle (used by the tests that plant a mistake in a copy of the oracle source)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self._saved = _lib
        lib = ctypes.CDLL(self.path)
        for name in ("oracle_decode", "oracle_prefill", "oracle_append_kv", "oracle_partial",
                     "oracle_merge", "oracle_online", "oracle_max_threads", "oracle_decode_fp8",
                     "oracle_append_kv_fp8", "oracle_e4m3_codes", "oracle_e4m3_values",
                     "oracle_rope_freqs", "oracle_rope", "oracle_bf16_round_array",
                     "oracle_prefill_fp8", "oracle_prefill_noncausal"):
            f, g = getattr(lib, name), getattr(self._saved, name)
            f.argtypes, f.restype = g.argtypes, g.restype
        _lib = lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def source_path() -> str:
    return _SRC


def compile_source(src_text: str, out_dir: str, name: str) -> str:
    """Compile an oracle source text (e.g. a mutated copy) into out_dir/name.so."""
    c = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, name + ".so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", so, c, "-lm"],
                   check=True)
    return so
