"""The C ABI without a GPU: the library builds and loads, exports every function
include/pa_decode.h declares, and rejects bad arguments on the host (no CUDA
call happens before these checks)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa_decode.h")


@pytest.fixture(scope="module")
def pa():
    import importlib.util
    spec = importlib.util.spec_from_file_location("pa_build", os.path.join(ROOT, "paged_kv_attention_19_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import paged_kv_attention_19_gb300 as pkg
    return pkg


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for required in ("pa_workspace_size", "pa_decode_gqa", "pa_decode_mla_absorbed", "pa_status_string",
                     "pa_read_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(pa):
    out = subprocess.run(["nm", "-D", "--defined-only", pa.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (pa_[a-z0-9_]+)\b", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    # and the binding declares a signature for each of them
    assert set(declared_functions()) <= set(pa.SIGNATURES)


def test_status_strings(pa):
    assert pa.pa_status_string(0) == "ok"
    for code in (-1, -2, -3, -4, -5):
        assert pa.pa_status_string(code) not in ("ok", "unknown status")
    assert pa.pa_status_string(42) == "unknown status"


def test_workspace_size(pa):
    ws = lambda *a: pa.pa_workspace_size(pa.PA_KIND_GQA, *a)
    g = ws(32, 64, 8, 128, 16384, 32, 0)
    assert g > 0
    # two partial slots of 32 rows (two 16-row tiles) per share, growing with head_dim and with an
    # explicit share count (automatic mode: 256 shares), plus two int32 tables with one entry per
    # (row, KV head, tile) for up to 64 query positions; independent of the context
    assert abs(ws(64, 64, 8, 128, 16384, 32, 0) - g - 32 * 8 * 64 * 2 * 4) <= 256
    assert ws(32, 64, 8, 128, 131072, 32, 0) == g
    assert ws(32, 64, 8, 128, 16384, 32, 256) == g
    tables = 32 * 8 * 64 * 2 * 4
    assert 256 * 2 * 32 * 128 * 4 + tables <= g < 256 * 2 * 32 * 128 * 4 + tables + (1 << 17)  # + descriptors, LSEs
    assert ws(32, 64, 8, 128, 16384, 32, 4) < g
    assert ws(32, 64, 8, 128, 16384, 32, 512) > g
    assert ws(32, 64, 8, 256, 16384, 32, 0) > g
    # rejected shapes report 0
    assert ws(32, 64, 7, 128, 16384, 32, 0) == 0     # Hq % Hkv
    assert ws(32, 64, 8, 96, 16384, 32, 0) == 0      # head_dim
    assert ws(32, 64, 8, 128, 16384, 48, 0) == 0     # page size
    assert ws(32, 64, 8, 128, 16384, 32, 4097) == 0  # num_splits
    assert pa.pa_workspace_size(pa.PA_KIND_MLA_ABSORBED, 16, 128, 0, 0, 8192, 64, 0) > 0
    assert pa.pa_workspace_size(pa.PA_KIND_MLA_ABSORBED, 16, 0, 0, 0, 8192, 64, 0) == 0
    assert pa.pa_workspace_size(7, 16, 128, 1, 128, 8192, 64, 0) == 0


def test_mla_workspace_layout(pa):
    """The MLA workspace as the header describes it: per share two fp32 partial slots of
    min(H, 128) heads x 256 columns (plus a 16-byte descriptor and the slots' LSEs), per
    (row, head) q_abs, q_lo and o_lat in bf16 (576 + 512 + 512 values), and per (row, tile of 128
    heads) two int32 entries for each of its two column-half sequences; each region rounded up to
    256 bytes."""
    ws = lambda B, H, n: pa.pa_workspace_size(pa.PA_KIND_MLA_ABSORBED, B, H, 0, 0, 8192, 64, n)
    per_row_head = (576 + 512 + 512) * 2
    for H in (1, 16, 128, 200, 256):
        rs = min(H, 128)
        per_share = 16 + 2 * rs * 4 + 2 * rs * 256 * 4
        per_row_tables = 2 * 2 * ((H + 127) // 128) * 4
        # shares: an explicit count n grows the workspace by per_share bytes each (up to rounding)
        d = ws(16, H, 512) - ws(16, H, 256)
        assert abs(d - 256 * per_share) <= 3 * 256, (H, d)
        # rows: each adds H * per_row_head bytes plus its table entries (up to rounding)
        d = ws(32, H, 256) - ws(16, H, 256)
        assert abs(d - 16 * (H * per_row_head + per_row_tables)) <= 4 * 256, (H, d)
        # automatic mode sizes for 256 shares
        assert ws(16, H, 0) == ws(16, H, 256)
        # the context length and page size do not enter
        assert pa.pa_workspace_size(pa.PA_KIND_MLA_ABSORBED, 16, H, 0, 0, 1024, 16, 0) == ws(16, H, 0)


def _gqa(pa, **kw):
    a = dict(q=0x10000, k=0x20000, v=0x30000, bt=0x40000, lens=0x50000, out=0x60000, lse=None, batch=2, hq=8,
             hkv=2, d=128, p=16, pages=10, maxp=5, maxctx=80, scale=0.1, window=0, splits=0, ws=0x70000,
             wsb=1 << 30)
    a.update(kw)
    return pa.lib.pa_decode_gqa(a["q"], a["k"], a["v"], a["bt"], a["lens"], a["out"], a["lse"], a["batch"],
                                a["hq"], a["hkv"], a["d"], a["p"], a["pages"], a["maxp"], a["maxctx"], a["scale"],
                                a["window"], a["splits"], a["ws"], a["wsb"], None)


def test_gqa_host_validation(pa):
    assert _gqa(pa, batch=0) == pa.PA_OK                       # empty batch: no-op
    assert _gqa(pa, batch=-1) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa(pa, hkv=3) == pa.PA_ERR_INVALID_ARGUMENT        # 8 % 3 != 0
    assert _gqa(pa, hq=0) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa(pa, d=96) == pa.PA_ERR_UNSUPPORTED
    assert _gqa(pa, p=4) == pa.PA_ERR_UNSUPPORTED
    assert _gqa(pa, p=24) == pa.PA_ERR_UNSUPPORTED
    assert _gqa(pa, splits=4097) == pa.PA_ERR_UNSUPPORTED
    assert _gqa(pa, splits=-1) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa(pa, q=None) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa(pa, ws=None) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa(pa, pages=0) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa(pa, maxp=4) == pa.PA_ERR_INVALID_ARGUMENT      # 4 pages of 16 < 80 tokens
    assert _gqa(pa, scale=float("nan")) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa(pa, q=0x10002) == pa.PA_ERR_MISALIGNED
    assert _gqa(pa, k=0x20008) == pa.PA_ERR_MISALIGNED
    assert _gqa(pa, bt=0x40002) == pa.PA_ERR_MISALIGNED
    assert _gqa(pa, lse=0x80001) == pa.PA_ERR_MISALIGNED
    assert _gqa(pa, wsb=1024) == pa.PA_ERR_WORKSPACE_TOO_SMALL


def _mla(pa, **kw):
    a = dict(q=0x10000, c=0x20000, wk=0x30000, wv=0x40000, bt=0x50000, lens=0x60000, out=0x70000, lse=None,
             batch=2, h=16, p=64, pages=10, maxp=5, maxctx=300, scale=0.07, splits=0, ws=0x80000, wsb=1 << 30)
    a.update(kw)
    return pa.lib.pa_decode_mla_absorbed(a["q"], a["c"], a["wk"], a["wv"], a["bt"], a["lens"], a["out"], a["lse"],
                                         a["batch"], a["h"], a["p"], a["pages"], a["maxp"], a["maxctx"], a["scale"],
                                         a["splits"], a["ws"], a["wsb"], None)


def test_mla_host_validation(pa):
    assert _mla(pa, batch=0) == pa.PA_OK
    assert _mla(pa, h=0) == pa.PA_ERR_INVALID_ARGUMENT
    assert _mla(pa, p=48) == pa.PA_ERR_UNSUPPORTED
    assert _mla(pa, p=4) == pa.PA_ERR_UNSUPPORTED
    assert _mla(pa, wk=None) == pa.PA_ERR_INVALID_ARGUMENT
    assert _mla(pa, maxp=4) == pa.PA_ERR_INVALID_ARGUMENT
    assert _mla(pa, c=0x20004) == pa.PA_ERR_MISALIGNED
    assert _mla(pa, wsb=16) == pa.PA_ERR_WORKSPACE_TOO_SMALL


def test_profile_hook_arguments(pa):
    assert pa.lib.pa_set_profile_events(None, None) == pa.PA_OK
    assert pa.lib.pa_set_profile_events(ctypes.c_void_p(0x1234), None) == pa.PA_ERR_INVALID_ARGUMENT
    assert pa.lib.pa_read_device_status(None, None, None) == pa.PA_ERR_INVALID_ARGUMENT


def test_kv_write_host_validation(pa):
    kw = lambda **a: pa.lib.pa_kv_write(a.get("k", 0x10000), a.get("v", 0x20000), a.get("s", 0x30000),
                                        a.get("kp", 0x40000), a.get("vp", 0x50000), a.get("T", 4),
                                        a.get("H", 2), a.get("D", 64), a.get("P", 16), a.get("pages", 4),
                                        a.get("st", None), None)
    assert kw(T=0) == pa.PA_OK
    assert kw(T=-1) == pa.PA_ERR_INVALID_ARGUMENT
    assert kw(H=0) == pa.PA_ERR_INVALID_ARGUMENT
    assert kw(D=60) == pa.PA_ERR_UNSUPPORTED
    assert kw(k=None) == pa.PA_ERR_INVALID_ARGUMENT
    assert kw(k=0x10008) == pa.PA_ERR_MISALIGNED
    assert kw(s=0x30004) == pa.PA_ERR_MISALIGNED
    assert kw(st=0x60002) == pa.PA_ERR_MISALIGNED
    mw = lambda **a: pa.lib.pa_mla_cache_write(a.get("c", 0x10000), a.get("r", 0x20000), a.get("s", 0x30000),
                                               a.get("cache", 0x40000), a.get("T", 4), a.get("P", 16),
                                               a.get("pages", 4), None, None)
    assert mw(T=0) == pa.PA_OK
    assert mw(P=0) == pa.PA_ERR_INVALID_ARGUMENT
    assert mw(cache=None) == pa.PA_ERR_INVALID_ARGUMENT
    assert mw(r=0x20008) == pa.PA_ERR_MISALIGNED


def _gqa_fp8(pa, **kw):
    a = dict(q=0x10000, k=0x20000, v=0x30000, bt=0x40000, lens=0x50000, out=0x60000, lse=None, batch=2, nq=1,
             hq=8, hkv=2, d=128, p=16, pages=10, maxp=5, maxctx=80, scale=0.1, ks=0.02, vs=0.03, window=0,
             splits=0, ws=0x70000, wsb=1 << 30)
    a.update(kw)
    return pa.lib.pa_decode_gqa_fp8(a["q"], a["k"], a["v"], a["bt"], a["lens"], a["out"], a["lse"], a["batch"],
                                    a["nq"], a["hq"], a["hkv"], a["d"], a["p"], a["pages"], a["maxp"], a["maxctx"],
                                    a["scale"], a["ks"], a["vs"], a["window"], a["splits"], a["ws"], a["wsb"], None)


def test_gqa_fp8_host_validation(pa):
    assert _gqa_fp8(pa, batch=0) == pa.PA_OK
    assert _gqa_fp8(pa, ks=0.0) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa_fp8(pa, vs=-1.0) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa_fp8(pa, ks=float("inf")) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa_fp8(pa, vs=float("nan"), batch=0) == pa.PA_ERR_INVALID_ARGUMENT  # scales checked first
    assert _gqa_fp8(pa, d=64) == pa.PA_ERR_UNSUPPORTED                          # bf16 pools only
    assert _gqa_fp8(pa, d=96) == pa.PA_ERR_UNSUPPORTED
    assert _gqa_fp8(pa, nq=0) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa_fp8(pa, nq=65) == pa.PA_ERR_UNSUPPORTED
    assert _gqa_fp8(pa, k=None) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa_fp8(pa, v=0x30008) == pa.PA_ERR_MISALIGNED
    assert _gqa_fp8(pa, wsb=1024) == pa.PA_ERR_WORKSPACE_TOO_SMALL


def test_kv_write_fp8_host_validation(pa):
    kw = lambda **a: pa.lib.pa_kv_write_fp8(a.get("k", 0x10000), a.get("v", 0x20000), a.get("s", 0x30000),
                                            a.get("kp", 0x40000), a.get("vp", 0x50000), a.get("T", 4),
                                            a.get("H", 2), a.get("D", 64), a.get("P", 16), a.get("pages", 4),
                                            a.get("ks", 0.5), a.get("vs", 0.5), a.get("st", None), None)
    assert kw(T=0) == pa.PA_OK
    assert kw(T=-1) == pa.PA_ERR_INVALID_ARGUMENT
    assert kw(ks=0.0) == pa.PA_ERR_INVALID_ARGUMENT
    assert kw(vs=float("nan")) == pa.PA_ERR_INVALID_ARGUMENT
    assert kw(D=40) == pa.PA_ERR_UNSUPPORTED          # rows of whole 16-byte code vectors
    assert kw(kp=None) == pa.PA_ERR_INVALID_ARGUMENT
    assert kw(vp=0x50008) == pa.PA_ERR_MISALIGNED
    assert kw(s=0x30004) == pa.PA_ERR_MISALIGNED


def test_last_cuda_error_starts_clean(pa):
    # no call on this thread has returned PA_ERR_CUDA: no error recorded
    assert pa.pa_last_cuda_error() == 0
    assert isinstance(pa.pa_last_cuda_error_string(), str)


def _gqa_nvfp4(pa, **kw):
    a = dict(q=0x10000, k=0x20000, v=0x30000, bt=0x40000, lens=0x50000, out=0x60000, lse=None, batch=2, nq=1,
             hq=8, hkv=2, d=128, p=16, pages=10, maxp=5, maxctx=80, scale=0.1, ks=0.25, vs=0.5, window=0,
             splits=0, ws=0x70000, wsb=1 << 30)
    a.update(kw)
    return pa.lib.pa_decode_gqa_nvfp4(a["q"], a["k"], a["v"], a["bt"], a["lens"], a["out"], a["lse"], a["batch"],
                                      a["nq"], a["hq"], a["hkv"], a["d"], a["p"], a["pages"], a["maxp"],
                                      a["maxctx"], a["scale"], a["ks"], a["vs"], a["window"], a["splits"], a["ws"],
                                      a["wsb"], None)


def test_gqa_nvfp4_host_validation(pa):
    """Every rejection happens on the host, before any CUDA call (this machine has no GPU)."""
    assert _gqa_nvfp4(pa, batch=0) == pa.PA_OK
    assert _gqa_nvfp4(pa, ks=0.0) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa_nvfp4(pa, vs=-1.0) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa_nvfp4(pa, ks=float("inf")) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa_nvfp4(pa, vs=float("nan"), batch=0) == pa.PA_ERR_INVALID_ARGUMENT  # scales checked first
    assert _gqa_nvfp4(pa, d=96) == pa.PA_ERR_UNSUPPORTED
    assert _gqa_nvfp4(pa, p=12) == pa.PA_ERR_UNSUPPORTED
    assert _gqa_nvfp4(pa, nq=0) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa_nvfp4(pa, nq=65) == pa.PA_ERR_UNSUPPORTED
    assert _gqa_nvfp4(pa, k=None) == pa.PA_ERR_INVALID_ARGUMENT
    assert _gqa_nvfp4(pa, v=0x30008) == pa.PA_ERR_MISALIGNED
    assert _gqa_nvfp4(pa, wsb=1024) == pa.PA_ERR_WORKSPACE_TOO_SMALL


def test_kv_write_nvfp4_host_validation(pa):
    kw = lambda **a: pa.lib.pa_kv_write_nvfp4(a.get("k", 0x10000), a.get("v", 0x20000), a.get("s", 0x30000),
                                              a.get("kp", 0x40000), a.get("vp", 0x50000), a.get("T", 4),
                                              a.get("H", 2), a.get("D", 64), a.get("P", 16), a.get("pages", 4),
                                              a.get("ks", 0.5), a.get("vs", 0.5), a.get("st", None), None)
    assert kw(T=0) == pa.PA_OK
    assert kw(T=-1) == pa.PA_ERR_INVALID_ARGUMENT
    assert kw(ks=0.0) == pa.PA_ERR_INVALID_ARGUMENT
    assert kw(vs=float("nan")) == pa.PA_ERR_INVALID_ARGUMENT
    assert kw(D=96) == pa.PA_ERR_UNSUPPORTED           # head_dim 64, 128 or 256
    assert kw(D=32) == pa.PA_ERR_UNSUPPORTED
    assert kw(kp=None) == pa.PA_ERR_INVALID_ARGUMENT
    assert kw(vp=0x50008) == pa.PA_ERR_MISALIGNED
    assert kw(s=0x30004) == pa.PA_ERR_MISALIGNED
    assert kw(st=0x60002) == pa.PA_ERR_MISALIGNED
