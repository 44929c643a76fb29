"""The C-ABI library builds, loads and exports every declared symbol; host-side
argument checks reject bad calls before any CUDA work (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sinkattn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sinkattn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("sinkattn_decode", "sinkattn_prefill", "sinkattn_decode_merge",
              "sinkattn_decode_splitkv", "sinkattn_append_kv", "sinkattn_get_status"):
        assert n in names


def test_library_exports_every_declared_symbol(built_lib):
    out = subprocess.run(["nm", "-D", "--defined-only", built_lib], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (sinkattn_[a-z0-9_]+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(sa):
    assert sorted(sa.SIGNATURES) == declared_functions()
    lib = sa.load()
    for n in declared_functions():
        assert hasattr(lib, n)


def test_error_strings_and_version(sa):
    assert sa.error_string(0) == "ok"
    assert "workspace" in sa.error_string(3)
    assert sa.load().sinkattn_version() >= 10000


def _desc(sa, **kw):
    d = dict(num_seqs=4, num_qo_heads=8, num_kv_heads=2, head_dim=64, num_pages=10,
             max_pages_per_seq=4)
    d.update(kw)
    return sa.paged_desc(**d)


@pytest.mark.parametrize("bad,code", [
    (dict(head_dim=96), 2), (dict(num_qo_heads=12, num_kv_heads=4), 2),   # G = 3
    (dict(num_qo_heads=9), 1), (dict(num_pages=0), 1), (dict(max_pages_per_seq=0), 1),
    (dict(num_kv_heads=0), 1), (dict(num_qo_heads=64, num_kv_heads=2), 2),  # G = 32
    (dict(max_sms=-1), 1), (dict(wait_limit_us=-1), 1),
])
def test_decode_workspace_size_rejects(sa, bad, code):
    n = ctypes.c_size_t()
    d = _desc(sa, **bad)
    assert sa.load().sinkattn_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == code


def test_page_size_must_be_16(sa):
    n = ctypes.c_size_t()
    d = _desc(sa)
    d.page_size = 32
    assert sa.load().sinkattn_decode_workspace_size(ctypes.byref(d), ctypes.byref(n)) == 2


def test_null_pointers_rejected_before_cuda(sa):
    lib = sa.load()
    d = _desc(sa)
    assert lib.sinkattn_decode(None, None, None, None, None, None, 0.125, None, None,
                               ctypes.byref(d), None, 0, None) == 1
    assert lib.sinkattn_prefill(None, None, None, None, 8, None, None, None, None, None, 0.125,
                                None, None, ctypes.byref(d), None, 0, None) == 1
    assert lib.sinkattn_append_kv(None, None, None, 8, None, None, None, None, ctypes.byref(d),
                                  None, 0, None) == 1
    assert lib.sinkattn_get_status(None, None, None) == 1
    assert lib.sinkattn_decode_append(None, None, None, None, None, None, None, None, 0.125, None,
                                      None, ctypes.byref(d), None, 0, None) == 1
    # every other pointer in place, the new rows missing or misaligned
    buf = (ctypes.c_uint8 * 4096)()
    p16 = (ctypes.addressof(buf) + 15) // 16 * 16
    ws = (ctypes.addressof(buf) + 255) // 256 * 256
    for k_new, v_new in ((None, p16), (p16, None), (p16 + 4, p16)):
        assert lib.sinkattn_decode_append(p16, k_new, v_new, p16, p16, p16, p16, None, 0.125, p16,
                                          None, ctypes.byref(d), ws, 256, None) == 1


def test_empty_work_is_a_no_op_before_cuda(sa):
    """No sequences (decode) or no tokens (prefill, append): OK at once, NULL data allowed;
    the descriptor is still checked."""
    lib = sa.load()
    d = _desc(sa, num_seqs=0)
    assert lib.sinkattn_decode(None, None, None, None, None, None, 0.125, None, None,
                               ctypes.byref(d), None, 0, None) == 0
    d = _desc(sa)
    assert lib.sinkattn_prefill(None, None, None, None, 0, None, None, None, None, None, 0.125,
                                None, None, ctypes.byref(d), None, 0, None) == 0
    assert lib.sinkattn_append_kv(None, None, None, 0, None, None, None, None, ctypes.byref(d),
                                  None, 0, None) == 0
    d0 = _desc(sa, num_seqs=0)
    assert lib.sinkattn_decode_append(None, None, None, None, None, None, None, None, 0.125, None,
                                      None, ctypes.byref(d0), None, 0, None) == 0
    bad = _desc(sa, num_seqs=0, head_dim=96)
    assert lib.sinkattn_decode(None, None, None, None, None, None, 0.125, None, None,
                               ctypes.byref(bad), None, 0, None) == 2


def test_misaligned_pointers_rejected(sa):
    lib = sa.load()
    d = _desc(sa)
    buf = (ctypes.c_uint8 * 4096)()
    base = ctypes.addressof(buf)
    p16 = (base + 15) // 16 * 16
    # a prefill whose q is 2 bytes off a 16-byte boundary
    rc = lib.sinkattn_prefill(p16 + 2, p16, p16, p16, 8, None, None, None, None, None, 0.125,
                              p16, None, ctypes.byref(d), (base + 255) // 256 * 256, 256, None)
    assert rc == 1
    # a prefill whose out is 16-byte but not 32-byte aligned
    p32 = (base + 31) // 32 * 32
    rc = lib.sinkattn_prefill(p16, p16, p16, p16, 8, None, None, None, None, None, 0.125,
                              p32 + 16, None, ctypes.byref(d), (base + 255) // 256 * 256, 256, None)
    assert rc == 1


def test_prefix_arguments_all_or_nothing(sa):
    lib = sa.load()
    d = _desc(sa)
    buf = (ctypes.c_uint8 * 8192)()
    p = (ctypes.addressof(buf) + 255) // 256 * 256
    # k_pages given without the other prefix arguments
    rc = lib.sinkattn_prefill(p, p, p, p, 8, p, None, None, None, None, 0.125, p, None,
                              ctypes.byref(d), p, 256, None)
    assert rc == 1


def test_noncausal_prefill_rejects_before_cuda(sa):
    """No tokens: OK at once; NULL data or a sliding window: SINKATTN_ERR_INVALID_ARG, all
    before any CUDA call (a window has no meaning without the causal order)."""
    lib = sa.load()
    d = _desc(sa)
    assert lib.sinkattn_prefill_noncausal(None, None, None, None, 0, None, 0.125, None, None,
                                          ctypes.byref(d), None, 0, None) == 0
    assert lib.sinkattn_prefill_noncausal(None, None, None, None, 8, None, 0.125, None, None,
                                          ctypes.byref(d), None, 0, None) == 1
    buf = (ctypes.c_uint8 * 4096)()
    p = (ctypes.addressof(buf) + 255) // 256 * 256
    dw = _desc(sa, window=128)
    assert lib.sinkattn_prefill_noncausal(p, p, p, p, 8, None, 0.125, p, None, ctypes.byref(dw), p,
                                          256, None) == 1


def test_flags_match_the_header_and_unknown_bits_are_rejected(sa):
    text = open(HEADER).read()
    for name in ("LAUNCH_NEXT_EARLY", "START_EARLY"):
        m = re.search(r"#define SINKATTN_FLAG_%s (0x[0-9a-fA-F]+|\d+)" % name, text)
        assert m, name
        assert int(m.group(1), 0) == getattr(sa, "FLAG_" + name)
    lib = sa.load()
    size = ctypes.c_size_t(0)
    ok = _desc(sa, flags=sa.FLAG_LAUNCH_NEXT_EARLY | sa.FLAG_START_EARLY)
    assert lib.sinkattn_prefill_workspace_size(ctypes.byref(ok), ctypes.byref(size)) == 0
    bad = _desc(sa, flags=4)
    assert lib.sinkattn_prefill_workspace_size(ctypes.byref(bad), ctypes.byref(size)) == 1
    assert lib.sinkattn_decode_workspace_size(ctypes.byref(bad), ctypes.byref(size)) == 1


def test_desc_layout_matches_the_header(sa):
    """The binding's struct has the header's fields, in order, all int32."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct sinkattn_paged_desc \{(.*?)\} sinkattn_paged_desc;", text,
                     flags=re.S).group(1)
    fields = re.findall(r"int32_t\s+(\w+)\s*;", body)
    assert [f for f, _ in sa.PagedDesc._fields_] == fields
    assert ctypes.sizeof(sa.PagedDesc) == 4 * len(fields)


def test_rope_desc_layout_matches_the_header(sa):
    """The binding's rotary-parameter struct has the header's fields, in order and type."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    body = re.search(r"typedef struct sinkattn_rope_desc \{(.*?)\} sinkattn_rope_desc;", text,
                     flags=re.S).group(1)
    fields = re.findall(r"(double|int32_t)\s+(\w+)\s*;", body)
    ctype = {"double": ctypes.c_double, "int32_t": ctypes.c_int32}
    assert [(f, t) for f, t in sa.RopeDesc._fields_] == [(n, ctype[t]) for t, n in fields]


def test_rope_decode_rejects_bad_parameters_before_cuda(sa):
    """Parameter checks of the rotary decode come before anything touches the device."""
    d = _desc(sa)
    good = sa.rope_desc(150000.0, 32.0)
    lib = sa.load()
    for rope in (sa.rope_desc(150000.0, 0.5), sa.rope_desc(1.0, 32.0), sa.rope_desc(150000.0, 32.0, 0),
                 sa.rope_desc(150000.0, 32.0, 4096, 1.0, 1.0), None):
        rc = lib.sinkattn_decode_append_rope(16, 16, 16, 16, 16, 16, 16, None, ctypes.c_float(1.0),
                                             None if rope is None else ctypes.byref(rope), 16, None,
                                             ctypes.byref(d), 256, 1 << 20, None)
        assert rc == sa.ERR_INVALID_ARG, rc
    assert good.factor == 32.0


def test_header_compiles_as_c99_and_cpp17(tmp_path):
    """The boundary is a C ABI: its header stands alone in C99 and in C++17, warning-free."""
    import shutil
    for cc, std, lang in (("gcc", "c99", "c"), ("g++", "c++17", "c++")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not installed")
        r = subprocess.run([cc, "-fsyntax-only", f"-std={std}", "-Wall", "-Wextra", "-Werror",
                            "-x", lang, HEADER], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
