"""Thin ctypes binding of libsinkattn (include/sinkattn.h).

Argument marshalling only: tensors are checked (device, dtype, contiguity,
shape), their device pointers and the current CUDA stream are passed to the C
ABI, and error codes become exceptions.  Every step of the attention runs in
the library's CUDA kernels; there is no fallback.  Workspaces are torch
allocations owned by this module (one per device and size, zero-initialised).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsinkattn.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE_TOO_SMALL, ERR_CUDA = range(5)
STATUS_BAD_PAGE, STATUS_BAD_LENGTH, STATUS_BAD_CU_SEQLENS, STATUS_WAIT_TIMEOUT = 1, 2, 4, 8
STATUS_VALUE_RANGE = 16
FLAG_LAUNCH_NEXT_EARLY, FLAG_START_EARLY = 1, 2
PAGE_SIZE = 16

# every symbol the header declares, with (restype, argtypes)
_P, _I32, _F, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t


class PagedDesc(ctypes.Structure):
    _fields_ = [("num_seqs", _I32), ("num_qo_heads", _I32), ("num_kv_heads", _I32),
                ("head_dim", _I32), ("page_size", _I32), ("num_pages", _I32),
                ("max_pages_per_seq", _I32), ("window", _I32), ("max_sms", _I32),
                ("wait_limit_us", _I32), ("flags", _I32)]


class RopeDesc(ctypes.Structure):
    _fields_ = [("base", ctypes.c_double), ("factor", ctypes.c_double),
                ("original_context", _I32), ("beta_fast", ctypes.c_double),
                ("beta_slow", ctypes.c_double)]


_DP = ctypes.POINTER(PagedDesc)
SIGNATURES = {
    "sinkattn_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "sinkattn_version": (ctypes.c_int, []),
    "sinkattn_last_cuda_error": (ctypes.c_char_p, []),
    "sinkattn_decode_workspace_size": (ctypes.c_int, [_DP, ctypes.POINTER(_SZ)]),
    "sinkattn_workspace_init": (ctypes.c_int, [_P, _SZ, _P]),
    "sinkattn_decode": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _F, _P, _P, _DP, _P, _SZ, _P]),
    "sinkattn_decode_splitkv": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _F, _P, _P, _DP, _P, _SZ, _P]),
    "sinkattn_decode_merge": (ctypes.c_int, [_P, _P, _P, _P, _DP, _P, _SZ, _P]),
    "sinkattn_decode_append": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _F, _P, _P, _DP, _P, _SZ,
                                              _P]),
    "sinkattn_decode_append_rope": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _F,
                                                   ctypes.POINTER(RopeDesc), _P, _P, _DP, _P, _SZ, _P]),
    "sinkattn_decode_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _F, _P, _P, _DP, _P, _P]),
    "sinkattn_prefill_workspace_size": (ctypes.c_int, [_DP, ctypes.POINTER(_SZ)]),
    "sinkattn_prefill": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _F, _P, _P, _DP,
                                        _P, _SZ, _P]),
    "sinkattn_prefill_noncausal": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _F, _P, _P, _DP, _P, _SZ,
                                                  _P]),
    "sinkattn_prefill_fp8": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _F, _P,
                                            _P, _DP, _P, _SZ, _P]),
    "sinkattn_append_kv": (ctypes.c_int, [_P, _P, _P, _I32, _P, _P, _P, _P, _DP, _P, _SZ, _P]),
    "sinkattn_decode_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _F, _P, _P, _DP, _P, _SZ,
                                           _P]),
    "sinkattn_decode_fp8_splitkv": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _F, _P, _P, _DP,
                                                   _P, _SZ, _P]),
    "sinkattn_append_kv_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _P, _P, _P, _P, _DP, _P, _SZ,
                                              _P]),
    "sinkattn_get_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32), _P]),
}

_lib = None


class SinkAttnError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        detail = ""
        if code == ERR_CUDA:
            detail = f" [{load().sinkattn_last_cuda_error().decode()}]"
        super().__init__(f"{what}: {error_string(code)} ({code}){detail}")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libsinkattn.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -m "
                               "paged_gqa_attention_head_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def error_string(code: int) -> str:
    return load().sinkattn_error_string(code).decode()


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise SinkAttnError(rc, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, device: torch.device, ndim: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_workspaces: dict = {}


def workspace(nbytes: int, device: torch.device, tag: str = "default") -> torch.Tensor:
    """A zero-initialised uint8 device buffer of at least nbytes, cached per (device, tag)."""
    key = (device, tag)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def paged_desc(num_seqs, num_qo_heads, num_kv_heads, head_dim, num_pages, max_pages_per_seq,
               page_size=PAGE_SIZE, window=0, max_sms=0, wait_limit_us=0, flags=0) -> PagedDesc:
    """window > 0: sliding window (each query sees the keys at its last `window`
    positions); 0: full attention.  max_sms > 0: the persistent decode and prefill grids
    use at most that many SMs (the rest stay free for concurrent work on other streams);
    0: all SMs.  wait_limit_us > 0: give-up time of the kernels' pipeline waits (0: 2 s).
    flags: FLAG_LAUNCH_NEXT_EARLY (prefill) / FLAG_START_EARLY (split-KV decode), the
    overlap of a prefill and the decode after it on one stream."""
    return PagedDesc(num_seqs, num_qo_heads, num_kv_heads, head_dim, page_size, num_pages,
                     max_pages_per_seq, int(window), int(max_sms), int(wait_limit_us), int(flags))


_ws_sizes: dict = {}


def decode_workspace_size(desc: PagedDesc) -> int:
    """Bytes of decode workspace for desc on the current device (memoised)."""
    key = (torch.cuda.current_device() if torch.cuda.is_available() else -1,
           tuple(getattr(desc, f) for f, _ in desc._fields_))
    n = _ws_sizes.get(key)
    if n is None:
        c = _SZ()
        _check(load().sinkattn_decode_workspace_size(ctypes.byref(desc), ctypes.byref(c)),
               "decode_workspace_size")
        n = _ws_sizes[key] = c.value
    return n


def prefill_workspace_size(desc: PagedDesc) -> int:
    n = _SZ()
    _check(load().sinkattn_prefill_workspace_size(ctypes.byref(desc), ctypes.byref(n)),
           "prefill_workspace_size")
    return n.value


def get_status(ws: torch.Tensor) -> int:
    """Read and clear the device status word of a workspace (synchronous)."""
    v = ctypes.c_uint32()
    _check(load().sinkattn_get_status(_ptr(ws), ctypes.byref(v), _stream(ws.device)), "get_status")
    return v.value


def _codes(t: torch.Tensor) -> torch.Tensor:
    """An FP8 E4M3 cache tensor as its uint8 codes (float8_e4m3fn tensors are viewed)."""
    return t.view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t


def _decode_prep(q, k_pages, v_pages, block_table, seq_lens, sinks, scale, out, lse, ws,
                 want_lse, window=0, kv_dtype=torch.bfloat16, max_sms=0, wait_limit_us=0, flags=0):
    dev = q.device
    _need(q, "q", torch.bfloat16, dev, 3)
    _need(k_pages, "k_pages", kv_dtype, dev, 4)
    _need(v_pages, "v_pages", kv_dtype, dev, 4)
    _need(block_table, "block_table", torch.int32, dev, 2)
    _need(seq_lens, "seq_lens", torch.int32, dev, 1)
    B, Hq, D = q.shape
    num_pages, Hkv, P, D2 = k_pages.shape
    if D2 != D or tuple(v_pages.shape) != tuple(k_pages.shape) or P != PAGE_SIZE:
        raise ValueError("k_pages / v_pages must be [num_pages, Hkv, 16, D] matching q")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_table / seq_lens rows must equal the batch")
    if sinks is not None:
        _need(sinks, "sinks", torch.float32, dev, 1)
        if sinks.shape[0] != Hq:
            raise ValueError("sinks must have one entry per query head")
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.bfloat16, dev, 3)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    elif lse is not None:
        _need(lse, "lse", torch.float32, dev, 2)
    desc = paged_desc(B, Hq, Hkv, D, num_pages, block_table.shape[1], window=window,
                      max_sms=max_sms, wait_limit_us=wait_limit_us, flags=flags)
    nbytes = decode_workspace_size(desc)
    if ws is None:
        ws = workspace(nbytes, dev)
    elif ws.numel() < nbytes:
        raise ValueError(f"workspace needs {nbytes} bytes")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    return desc, out, lse, ws, scale


def decode(q, k_pages, v_pages, block_table, seq_lens, sinks=None, scale=None, out=None, lse=None,
           workspace_buf=None, return_lse=True, window=0, max_sms=0, wait_limit_us=0, flags=0):
    """Split-KV paged decode with sinks (sinkattn_decode).  window > 0: sliding window;
    max_sms > 0: the split-KV grid on at most that many SMs.  Returns (out, lse)."""
    desc, out, lse, ws, scale = _decode_prep(q, k_pages, v_pages, block_table, seq_lens, sinks,
                                             scale, out, lse, workspace_buf, return_lse, window,
                                             max_sms=max_sms, wait_limit_us=wait_limit_us, flags=flags)
    _check(load().sinkattn_decode(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                  _ptr(seq_lens), _ptr(sinks), scale, _ptr(out), _ptr(lse),
                                  ctypes.byref(desc), _ptr(ws), ws.numel(), _stream(q.device)),
           "sinkattn_decode")
    return out, lse


def decode_splitkv(q, k_pages, v_pages, block_table, seq_lens, sinks=None, scale=None, out=None,
                   lse=None, workspace_buf=None, return_lse=True, window=0, max_sms=0, wait_limit_us=0):
    """First decode kernel only (sinkattn_decode_splitkv); follow with decode_merge."""
    desc, out, lse, ws, scale = _decode_prep(q, k_pages, v_pages, block_table, seq_lens, sinks,
                                             scale, out, lse, workspace_buf, return_lse, window,
                                             max_sms=max_sms, wait_limit_us=wait_limit_us)
    _check(load().sinkattn_decode_splitkv(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                          _ptr(seq_lens), _ptr(sinks), scale, _ptr(out), _ptr(lse),
                                          ctypes.byref(desc), _ptr(ws), ws.numel(),
                                          _stream(q.device)), "sinkattn_decode_splitkv")
    return out, lse, ws, desc


def decode_merge(seq_lens, sinks, out, lse, desc, ws):
    """Second decode kernel (sinkattn_decode_merge) on the split-KV kernel's workspace."""
    _check(load().sinkattn_decode_merge(_ptr(seq_lens), _ptr(sinks), _ptr(out), _ptr(lse),
                                        ctypes.byref(desc), _ptr(ws), ws.numel(),
                                        _stream(out.device)), "sinkattn_decode_merge")
    return out, lse


def prefill(q, k, v, cu_seqlens, sinks=None, scale=None, k_pages=None, v_pages=None,
            prefix_block_table=None, prefix_lens=None, out=None, lse=None, workspace_buf=None,
            return_lse=True, window=0, max_sms=0, wait_limit_us=0, flags=0):
    """Causal ragged prefill, optionally over a paged prefix (sinkattn_prefill).  window > 0:
    sliding window; max_sms > 0: the persistent grid on at most that many SMs.  Returns
    (out, lse)."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev, 3)
    _need(k, "k", torch.bfloat16, dev, 3)
    _need(v, "v", torch.bfloat16, dev, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev, 1)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (T, Hkv, D) or tuple(v.shape) != (T, Hkv, D):
        raise ValueError("k / v must be [T, Hkv, D] matching q")
    n = cu_seqlens.shape[0] - 1
    if sinks is not None:
        _need(sinks, "sinks", torch.float32, dev, 1)
    num_pages = maxp = 0
    if k_pages is not None:
        _need(k_pages, "k_pages", torch.bfloat16, dev, 4)
        _need(v_pages, "v_pages", torch.bfloat16, dev, 4)
        _need(prefix_block_table, "prefix_block_table", torch.int32, dev, 2)
        _need(prefix_lens, "prefix_lens", torch.int32, dev, 1)
        num_pages, maxp = k_pages.shape[0], prefix_block_table.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(T, Hq, dtype=torch.float32, device=dev)
    desc = paged_desc(n, Hq, Hkv, D, num_pages, maxp, window=window, max_sms=max_sms,
                      wait_limit_us=wait_limit_us, flags=flags)
    nbytes = prefill_workspace_size(desc)
    ws = workspace_buf if workspace_buf is not None else workspace(nbytes, dev, "prefill")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(load().sinkattn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), T, _ptr(k_pages),
                                   _ptr(v_pages), _ptr(prefix_block_table), _ptr(prefix_lens),
                                   _ptr(sinks), scale, _ptr(out), _ptr(lse), ctypes.byref(desc),
                                   _ptr(ws), ws.numel(), _stream(dev)), "sinkattn_prefill")
    return out, lse


def prefill_noncausal(q, k, v, cu_seqlens, sinks=None, scale=None, out=None, lse=None,
                      workspace_buf=None, return_lse=True, max_sms=0, wait_limit_us=0):
    """Non-causal ragged prefill without a KV cache (sinkattn_prefill_noncausal): query t of
    request i attends every token of request i.  Returns (out, lse)."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev, 3)
    _need(k, "k", torch.bfloat16, dev, 3)
    _need(v, "v", torch.bfloat16, dev, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev, 1)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (T, Hkv, D) or tuple(v.shape) != (T, Hkv, D):
        raise ValueError("k / v must be [T, Hkv, D] matching q")
    n = cu_seqlens.shape[0] - 1
    if sinks is not None:
        _need(sinks, "sinks", torch.float32, dev, 1)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(T, Hq, dtype=torch.float32, device=dev)
    desc = paged_desc(n, Hq, Hkv, D, 0, 0, max_sms=max_sms, wait_limit_us=wait_limit_us)
    nbytes = prefill_workspace_size(desc)
    ws = workspace_buf if workspace_buf is not None else workspace(nbytes, dev, "prefill")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(load().sinkattn_prefill_noncausal(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), T, _ptr(sinks),
                                             scale, _ptr(out), _ptr(lse), ctypes.byref(desc), _ptr(ws),
                                             ws.numel(), _stream(dev)), "sinkattn_prefill_noncausal")
    return out, lse


def prefill_fp8(q, k, v, cu_seqlens, sinks=None, scale=None, k_pages=None, v_pages=None,
                k_scale=None, v_scale=None, prefix_block_table=None, prefix_lens=None, out=None,
                lse=None, workspace_buf=None, return_lse=True, window=0, max_sms=0, wait_limit_us=0):
    """Chunked prefill over an FP8 E4M3 paged prefix (sinkattn_prefill_fp8): k_pages / v_pages
    uint8 (or float8_e4m3fn) [num_pages, Hkv, 16, D] codes, k_scale / v_scale float32 [Hkv] or
    None (1); the new tokens' q, k, v bf16.  Returns (out, lse)."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev, 3)
    _need(k, "k", torch.bfloat16, dev, 3)
    _need(v, "v", torch.bfloat16, dev, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev, 1)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (T, Hkv, D) or tuple(v.shape) != (T, Hkv, D):
        raise ValueError("k / v must be [T, Hkv, D] matching q")
    if k_pages is None or v_pages is None or prefix_block_table is None or prefix_lens is None:
        raise ValueError("prefill_fp8 needs the FP8 prefix pages, block table and lengths")
    k_pages, v_pages = _codes(k_pages), _codes(v_pages)
    _need(k_pages, "k_pages", torch.uint8, dev, 4)
    _need(v_pages, "v_pages", torch.uint8, dev, 4)
    _need(prefix_block_table, "prefix_block_table", torch.int32, dev, 2)
    _need(prefix_lens, "prefix_lens", torch.int32, dev, 1)
    _scales(k_scale, v_scale, Hkv, dev)
    if sinks is not None:
        _need(sinks, "sinks", torch.float32, dev, 1)
    n = cu_seqlens.shape[0] - 1
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty(T, Hq, dtype=torch.float32, device=dev)
    desc = paged_desc(n, Hq, Hkv, D, k_pages.shape[0], prefix_block_table.shape[1], window=window,
                      max_sms=max_sms, wait_limit_us=wait_limit_us)
    ws = workspace_buf if workspace_buf is not None else workspace(prefill_workspace_size(desc), dev,
                                                                   "prefill")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(load().sinkattn_prefill_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), T, _ptr(k_pages),
                                       _ptr(v_pages), _ptr(k_scale), _ptr(v_scale),
                                       _ptr(prefix_block_table), _ptr(prefix_lens), _ptr(sinks), scale,
                                       _ptr(out), _ptr(lse), ctypes.byref(desc), _ptr(ws), ws.numel(),
                                       _stream(dev)), "sinkattn_prefill_fp8")
    return out, lse


def append_kv(k, v, cu_seqlens, block_table, start_pos, k_pages, v_pages, workspace_buf=None):
    """Scatter new K/V rows into the paged cache in place (sinkattn_append_kv)."""
    dev = k.device
    _need(k, "k", torch.bfloat16, dev, 3)
    _need(v, "v", torch.bfloat16, dev, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev, 1)
    _need(block_table, "block_table", torch.int32, dev, 2)
    _need(start_pos, "start_pos", torch.int32, dev, 1)
    _need(k_pages, "k_pages", torch.bfloat16, dev, 4)
    _need(v_pages, "v_pages", torch.bfloat16, dev, 4)
    T, Hkv, D = k.shape
    n = cu_seqlens.shape[0] - 1
    desc = paged_desc(n, Hkv, Hkv, D, k_pages.shape[0], block_table.shape[1])
    ws = workspace_buf if workspace_buf is not None else workspace(256, dev, "append")
    _check(load().sinkattn_append_kv(_ptr(k), _ptr(v), _ptr(cu_seqlens), T, _ptr(block_table),
                                     _ptr(start_pos), _ptr(k_pages), _ptr(v_pages),
                                     ctypes.byref(desc), _ptr(ws), ws.numel(), _stream(dev)),
           "sinkattn_append_kv")
    return k_pages, v_pages


def _scales(k_scale, v_scale, Hkv, dev):
    for name, t in (("k_scale", k_scale), ("v_scale", v_scale)):
        if t is not None:
            _need(t, name, torch.float32, dev, 1)
            if t.shape[0] != Hkv:
                raise ValueError(f"{name} must have one entry per KV head")


def decode_append(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, sinks=None, scale=None,
                  out=None, lse=None, workspace_buf=None, return_lse=True, window=0, max_sms=0,
                  wait_limit_us=0):
    """Decode step with its K/V append (sinkattn_decode_append): the new rows k_new / v_new
    [B, Hkv, D] go into the cache at position seq_lens - 1 (seq_lens counts them) and are
    attended in the same pass.  k_pages / v_pages are written in place.  Returns (out, lse)."""
    desc, out, lse, ws, scale = _decode_prep(q, k_pages, v_pages, block_table, seq_lens, sinks,
                                             scale, out, lse, workspace_buf, return_lse, window,
                                             max_sms=max_sms, wait_limit_us=wait_limit_us)
    B, Hkv, D = q.shape[0], k_pages.shape[1], q.shape[2]
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _need(t, name, torch.bfloat16, q.device, 3)
        if tuple(t.shape) != (B, Hkv, D):
            raise ValueError(f"{name} must be [B, Hkv, D] = {(B, Hkv, D)}")
    _check(load().sinkattn_decode_append(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pages),
                                         _ptr(v_pages), _ptr(block_table), _ptr(seq_lens),
                                         _ptr(sinks), scale, _ptr(out), _ptr(lse), ctypes.byref(desc),
                                         _ptr(ws), ws.numel(), _stream(q.device)),
           "sinkattn_decode_append")
    return out, lse


def rope_desc(base: float, factor: float = 1.0, original_context: int = 4096,
              beta_fast: float = 32.0, beta_slow: float = 1.0) -> RopeDesc:
    """Rotary-embedding parameters (NeoX layout, YaRN scaling; factor 1 = plain RoPE)."""
    return RopeDesc(float(base), float(factor), int(original_context), float(beta_fast),
                    float(beta_slow))


def decode_append_rope(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, sinks=None,
                       scale=None, rope: Optional[RopeDesc] = None, out=None, lse=None,
                       workspace_buf=None, return_lse=True, window=0, max_sms=0,
                       wait_limit_us=0):
    """Decode step with rotary embedding and K/V append (sinkattn_decode_append_rope): q and
    k_new (not yet rotated) are rotated at position seq_lens - 1, the rotated key and v_new go
    into the cache there, and the rotated query attends.  rope: a RopeDesc (rope_desc(...)).
    k_pages / v_pages are written in place.  Returns (out, lse)."""
    if not isinstance(rope, RopeDesc):
        raise TypeError("rope must be a RopeDesc (see rope_desc)")
    desc, out, lse, ws, scale = _decode_prep(q, k_pages, v_pages, block_table, seq_lens, sinks,
                                             scale, out, lse, workspace_buf, return_lse, window,
                                             max_sms=max_sms, wait_limit_us=wait_limit_us)
    B, Hkv, D = q.shape[0], k_pages.shape[1], q.shape[2]
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        _need(t, name, torch.bfloat16, q.device, 3)
        if tuple(t.shape) != (B, Hkv, D):
            raise ValueError(f"{name} must be [B, Hkv, D] = {(B, Hkv, D)}")
    _check(load().sinkattn_decode_append_rope(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pages),
                                              _ptr(v_pages), _ptr(block_table), _ptr(seq_lens),
                                              _ptr(sinks), scale, ctypes.byref(rope), _ptr(out),
                                              _ptr(lse), ctypes.byref(desc), _ptr(ws), ws.numel(),
                                              _stream(q.device)), "sinkattn_decode_append_rope")
    return out, lse


def decode_fp8(q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, sinks=None, scale=None,
               out=None, lse=None, workspace_buf=None, return_lse=True, window=0, max_sms=0,
               wait_limit_us=0):
    """Split-KV paged decode over an FP8 E4M3 cache (sinkattn_decode_fp8).  k_pages / v_pages:
    uint8 (or float8_e4m3fn) [num_pages, Hkv, 16, D] codes; k_scale / v_scale: float32 [Hkv]
    per-KV-head scales or None (1).  Returns (out, lse)."""
    k_pages, v_pages = _codes(k_pages), _codes(v_pages)
    desc, out, lse, ws, scale = _decode_prep(q, k_pages, v_pages, block_table, seq_lens, sinks,
                                             scale, out, lse, workspace_buf, return_lse, window,
                                             kv_dtype=torch.uint8, max_sms=max_sms,
                                             wait_limit_us=wait_limit_us)
    _scales(k_scale, v_scale, k_pages.shape[1], q.device)
    _check(load().sinkattn_decode_fp8(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(k_scale),
                                      _ptr(v_scale), _ptr(block_table), _ptr(seq_lens), _ptr(sinks),
                                      scale, _ptr(out), _ptr(lse), ctypes.byref(desc), _ptr(ws),
                                      ws.numel(), _stream(q.device)), "sinkattn_decode_fp8")
    return out, lse


def decode_fp8_splitkv(q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, sinks=None,
                       scale=None, out=None, lse=None, workspace_buf=None, return_lse=True, window=0,
                       max_sms=0, wait_limit_us=0):
    """First kernel of decode_fp8 only (sinkattn_decode_fp8_splitkv); follow with decode_merge."""
    k_pages, v_pages = _codes(k_pages), _codes(v_pages)
    desc, out, lse, ws, scale = _decode_prep(q, k_pages, v_pages, block_table, seq_lens, sinks,
                                             scale, out, lse, workspace_buf, return_lse, window,
                                             kv_dtype=torch.uint8, max_sms=max_sms,
                                             wait_limit_us=wait_limit_us)
    _scales(k_scale, v_scale, k_pages.shape[1], q.device)
    _check(load().sinkattn_decode_fp8_splitkv(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(k_scale),
                                              _ptr(v_scale), _ptr(block_table), _ptr(seq_lens),
                                              _ptr(sinks), scale, _ptr(out), _ptr(lse),
                                              ctypes.byref(desc), _ptr(ws), ws.numel(),
                                              _stream(q.device)), "sinkattn_decode_fp8_splitkv")
    return out, lse, ws, desc


def append_kv_fp8(k, v, k_scale, v_scale, cu_seqlens, block_table, start_pos, k_pages, v_pages,
                  workspace_buf=None):
    """Quantise new bf16 K/V rows to E4M3 codes (x / scale[g], nearest, saturating) and scatter
    them into an FP8 cache in place (sinkattn_append_kv_fp8)."""
    dev = k.device
    k_pages, v_pages = _codes(k_pages), _codes(v_pages)
    _need(k, "k", torch.bfloat16, dev, 3)
    _need(v, "v", torch.bfloat16, dev, 3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev, 1)
    _need(block_table, "block_table", torch.int32, dev, 2)
    _need(start_pos, "start_pos", torch.int32, dev, 1)
    _need(k_pages, "k_pages", torch.uint8, dev, 4)
    _need(v_pages, "v_pages", torch.uint8, dev, 4)
    T, Hkv, D = k.shape
    _scales(k_scale, v_scale, Hkv, dev)
    n = cu_seqlens.shape[0] - 1
    desc = paged_desc(n, Hkv, Hkv, D, k_pages.shape[0], block_table.shape[1])
    ws = workspace_buf if workspace_buf is not None else workspace(256, dev, "append")
    _check(load().sinkattn_append_kv_fp8(_ptr(k), _ptr(v), _ptr(k_scale), _ptr(v_scale),
                                         _ptr(cu_seqlens), T, _ptr(block_table), _ptr(start_pos),
                                         _ptr(k_pages), _ptr(v_pages), ctypes.byref(desc), _ptr(ws),
                                         ws.numel(), _stream(dev)), "sinkattn_append_kv_fp8")
    return k_pages, v_pages


def decode_noalloc(q, k_pages, v_pages, block_table, seq_lens, sinks=None, scale=None, out=None,
                   lse=None, status=None, window=0):
    """sinkattn_decode_noalloc: the same decode with the library's fixed scratch array
    instead of a workspace, for callers that cannot allocate device memory.  Calls on
    one device must not overlap on the GPU.  status: optional int32/uint32 device
    tensor of one element receiving this call's status bits."""
    dev = q.device
    _need(q, "q", torch.bfloat16, dev, 3)
    _need(k_pages, "k_pages", torch.bfloat16, dev, 4)
    B, Hq, D = q.shape
    num_pages, Hkv = k_pages.shape[:2]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, dtype=torch.float32, device=dev)
    desc = paged_desc(B, Hq, Hkv, D, num_pages, block_table.shape[1], window=window)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    _check(load().sinkattn_decode_noalloc(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                          _ptr(seq_lens), _ptr(sinks), scale, _ptr(out), _ptr(lse),
                                          ctypes.byref(desc), _ptr(status), _stream(dev)),
           "sinkattn_decode_noalloc")
    return out, lse
