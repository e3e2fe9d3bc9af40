"""Paged decode attention for GB300 (sm_103a): Python binding of the C ABI.

The binding only marshals arguments: every step of the decode runs in the CUDA
kernels of ``_lib/libpa_decode.so`` (declared in ``include/pa_decode.h``).
There is no CPU fallback: importing this package fails with ImportError if the
library has not been built (``python paged_kv_attention_19_gb300/build.py``).

Names follow the C ABI: ``pa_workspace_size``, ``pa_decode_gqa``,
``pa_decode_mla_absorbed``, ``pa_verify_gqa``, ``pa_decode_gqa_fp8``, ``pa_decode_gqa_nvfp4``,
``pa_decode_gqa_noalloc``, ``pa_kv_write``, ``pa_kv_write_fp8``, ``pa_kv_write_nvfp4``, ``pa_mla_cache_write``, ``pa_status_string``, ``pa_read_device_status``,
``pa_set_profile_events``, ``pa_last_launch_count``, ``pa_set_wait_limit_ns``, ``pa_last_cuda_error``,
``pa_last_cuda_error_string``.  The tensor-taking
functions accept torch tensors (device memory, the layouts of the header) and
infer every size from their shapes.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpa_decode.so")

PA_OK = 0
PA_ERR_INVALID_ARGUMENT = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_MISALIGNED = -3
PA_ERR_WORKSPACE_TOO_SMALL = -4
PA_ERR_CUDA = -5
PA_KIND_GQA = 0
PA_KIND_MLA_ABSORBED = 1
PA_DEV_BAD_PAGE = 0x1
PA_DEV_BAD_LEN = 0x2
PA_DEV_TIMEOUT = 0x4
PA_DEV_BAD_SLOT = 0x8
PA_DEFAULT_WAIT_LIMIT_NS = 1_000_000_000

# Every symbol include/pa_decode.h declares, with its ctypes signature.
_P, _I, _F, _Z, _U32P = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.POINTER(ctypes.c_uint32)
SIGNATURES = {
    "pa_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "pa_decode_gqa": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _Z, _P]),
    "pa_decode_mla_absorbed": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _Z, _P]),
    "pa_decode_gqa_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "pa_verify_gqa": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _Z,
                           _P]),
    "pa_decode_gqa_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _F, _F, _I,
                               _I, _P, _Z, _P]),
    "pa_decode_gqa_nvfp4": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _F, _F, _I,
                                 _I, _P, _Z, _P]),
    "pa_kv_write_nvfp4": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _P, _P]),
    "pa_kv_write": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "pa_kv_write_fp8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _P, _P]),
    "pa_mla_cache_write": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "pa_status_string": (ctypes.c_char_p, [_I]),
    "pa_read_device_status": (_I, [_P, _P, _U32P]),
    "pa_set_profile_events": (_I, [_P, _P]),
    "pa_last_launch_count": (_I, []),
    "pa_set_wait_limit_ns": (_I, [ctypes.c_ulonglong]),
    "pa_last_cuda_error": (_I, []),
    "pa_last_cuda_error_string": (ctypes.c_char_p, []),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python paged_kv_attention_19_gb300/build.py` "
                          "(the decode has no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class PaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = f"; {lib.pa_last_cuda_error_string().decode()}" if status == PA_ERR_CUDA else ""
        super().__init__(f"{what}: {pa_status_string(status)} ({status}){detail}")


def pa_status_string(status: int) -> str:
    return lib.pa_status_string(int(status)).decode()


def _check(rc: int, what: str):
    if rc != PA_OK:
        raise PaError(rc, what)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def pa_workspace_size(kind: int, batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                      max_context_len: int, page_size: int, num_splits: int = 0) -> int:
    return int(lib.pa_workspace_size(kind, batch, num_q_heads, num_kv_heads, head_dim, max_context_len,
                                     page_size, num_splits))


def pa_decode_gqa(q, k_pool, v_pool, block_table, context_lens, out, lse=None, *, scale: float,
                  workspace, window: int = 0, num_splits: int = 0, max_context_len=None, stream=None) -> None:
    """GQA paged decode.  q [B, Hq, D], pools [pages, P, Hkv, D] bf16; block_table [B, max_pages]
    int32; context_lens [B] int32; out [B, Hq, D] bf16; lse [B, Hq] fp32 or None; workspace: a
    device tensor of at least pa_workspace_size(...) bytes.  max_context_len defaults to
    max_pages * page_size (an upper bound that needs no device read)."""
    B, Hq, D = q.shape
    num_pages, P, Hkv, _ = k_pool.shape
    max_pages = block_table.shape[1]
    if max_context_len is None:
        max_context_len = max_pages * P
    rc = lib.pa_decode_gqa(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), _ptr(context_lens),
                           _ptr(out), _ptr(lse), B, Hq, Hkv, D, P, num_pages, max_pages, int(max_context_len),
                           float(scale), int(window), int(num_splits), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "pa_decode_gqa")


def pa_verify_gqa(q, k_pool, v_pool, block_table, context_lens, out, lse=None, *, scale: float,
                  workspace, window: int = 0, num_splits: int = 0, max_context_len=None, stream=None) -> None:
    """GQA multi-query verify.  q [B, Q, Hq, D]; out [B, Q, Hq, D]; lse [B, Q, Hq] or None;
    context_lens count the Q new tokens; the rest as for pa_decode_gqa."""
    B, Q, Hq, D = q.shape
    num_pages, P, Hkv, _ = k_pool.shape
    max_pages = block_table.shape[1]
    if max_context_len is None:
        max_context_len = max_pages * P
    rc = lib.pa_verify_gqa(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), _ptr(context_lens),
                           _ptr(out), _ptr(lse), B, Q, Hq, Hkv, D, P, num_pages, max_pages, int(max_context_len),
                           float(scale), int(window), int(num_splits), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "pa_verify_gqa")


def pa_decode_gqa_fp8(q, k_pool, v_pool, block_table, context_lens, out, lse=None, *, scale: float,
                      k_scale: float, v_scale: float, workspace, window: int = 0, num_splits: int = 0,
                      max_context_len=None, stream=None) -> None:
    """GQA decode (q [B, Hq, D]) or multi-query verify (q [B, Q, Hq, D]) over FP8 E4M3 pools
    [pages, P, Hkv, D] uint8 whose values are code * k_scale (keys) and code * v_scale (values);
    out and lse shaped like q without / with its last dim; the rest as for pa_verify_gqa."""
    if q.dim() == 3:
        B, Hq, D = q.shape
        Q = 1
    else:
        B, Q, Hq, D = q.shape
    num_pages, P, Hkv, _ = k_pool.shape
    max_pages = block_table.shape[1]
    if max_context_len is None:
        max_context_len = max_pages * P
    rc = lib.pa_decode_gqa_fp8(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), _ptr(context_lens),
                               _ptr(out), _ptr(lse), B, Q, Hq, Hkv, D, P, num_pages, max_pages,
                               int(max_context_len), float(scale), float(k_scale), float(v_scale), int(window),
                               int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               _stream(stream))
    _check(rc, "pa_decode_gqa_fp8")


def pa_decode_gqa_nvfp4(q, k_pool, v_pool, block_table, context_lens, out, lse=None, *, scale: float,
                        k_scale: float, v_scale: float, workspace, window: int = 0, num_splits: int = 0,
                        max_context_len=None, stream=None) -> None:
    """GQA decode (q [B, Hq, D]) or multi-query verify (q [B, Q, Hq, D]) over NVFP4 pools
    [pages, P, Hkv, R] uint8 (R = nvfp4_row_bytes(D): code pairs, block scales, padding) whose
    values are e2m1(code) * e4m3(block scale) * k_scale (keys; v_scale for values); out and lse
    shaped like q without / with its last dim; the rest as for pa_verify_gqa."""
    if q.dim() == 3:
        B, Hq, D = q.shape
        Q = 1
    else:
        B, Q, Hq, D = q.shape
    num_pages, P, Hkv, _ = k_pool.shape
    max_pages = block_table.shape[1]
    if max_context_len is None:
        max_context_len = max_pages * P
    rc = lib.pa_decode_gqa_nvfp4(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), _ptr(context_lens),
                                 _ptr(out), _ptr(lse), B, Q, Hq, Hkv, D, P, num_pages, max_pages,
                                 int(max_context_len), float(scale), float(k_scale), float(v_scale), int(window),
                                 int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream))
    _check(rc, "pa_decode_gqa_nvfp4")


def nvfp4_row_bytes(head_dim: int) -> int:
    """Bytes of one NVFP4 pool row: head_dim / 2 code bytes and head_dim / 16 scale codes,
    padded to a multiple of 16."""
    return (head_dim // 2 + head_dim // 16 + 15) // 16 * 16


def pa_decode_mla_absorbed(q, cache, w_uk, w_uv, block_table, context_lens, out, lse=None, *, scale: float,
                           workspace, num_splits: int = 0, max_context_len=None, stream=None) -> None:
    """MLA absorbed decode.  q [B, H, 192], cache [pages, P, 576], w_uk / w_uv [H, 128, 512] bf16;
    out [B, H, 128] bf16; lse [B, H] fp32 or None."""
    B, H, _ = q.shape
    num_pages, P, _ = cache.shape
    max_pages = block_table.shape[1]
    if max_context_len is None:
        max_context_len = max_pages * P
    rc = lib.pa_decode_mla_absorbed(_ptr(q), _ptr(cache), _ptr(w_uk), _ptr(w_uv), _ptr(block_table),
                                    _ptr(context_lens), _ptr(out), _ptr(lse), B, H, P, num_pages, max_pages,
                                    int(max_context_len), float(scale), int(num_splits), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "pa_decode_mla_absorbed")


def pa_kv_write(k, v, slot_mapping, k_pool, v_pool, *, status=None, stream=None) -> None:
    """Paged KV write.  k, v [T, Hkv, D] bf16; slot_mapping [T] int64 (negative: padding, skipped);
    pools [pages, P, Hkv, D] bf16 (written at the named slots); status: optional uint32 device
    word that gets PA_DEV_BAD_SLOT for a slot past the pool."""
    T, Hkv, D = k.shape
    num_pages, P, _, _ = k_pool.shape
    _check(lib.pa_kv_write(_ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(k_pool), _ptr(v_pool), T, Hkv, D, P,
                           num_pages, _ptr(status), _stream(stream)), "pa_kv_write")


def pa_kv_write_fp8(k, v, slot_mapping, k_pool, v_pool, *, k_scale: float, v_scale: float, status=None,
                    stream=None) -> None:
    """FP8 paged KV write.  k, v [T, Hkv, D] bf16; pools [pages, P, Hkv, D] uint8 E4M3 codes of
    value / scale (nearest, ties to even, saturated at 448); the rest as for pa_kv_write."""
    T, Hkv, D = k.shape
    num_pages, P, _, _ = k_pool.shape
    _check(lib.pa_kv_write_fp8(_ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(k_pool), _ptr(v_pool), T, Hkv, D, P,
                               num_pages, float(k_scale), float(v_scale), _ptr(status), _stream(stream)),
           "pa_kv_write_fp8")


def pa_kv_write_nvfp4(k, v, slot_mapping, k_pool, v_pool, *, k_scale: float, v_scale: float, status=None,
                      stream=None) -> None:
    """NVFP4 paged KV write.  k, v [T, Hkv, D] bf16; pools [pages, P, Hkv, nvfp4_row_bytes(D)] uint8
    rows (E2M1 code pairs and E4M3 block scales of value / pool scale); the rest as for
    pa_kv_write."""
    T, Hkv, D = k.shape
    num_pages, P, _, _ = k_pool.shape
    _check(lib.pa_kv_write_nvfp4(_ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(k_pool), _ptr(v_pool), T, Hkv, D,
                                 P, num_pages, float(k_scale), float(v_scale), _ptr(status), _stream(stream)),
           "pa_kv_write_nvfp4")


def pa_mla_cache_write(c_lat, k_rope, slot_mapping, cache, *, status=None, stream=None) -> None:
    """MLA cache write.  c_lat [T, 512], k_rope [T, 64] bf16; cache [pages, P, 576] bf16."""
    T = c_lat.shape[0]
    num_pages, P, _ = cache.shape
    _check(lib.pa_mla_cache_write(_ptr(c_lat), _ptr(k_rope), _ptr(slot_mapping), _ptr(cache), T, P, num_pages,
                                  _ptr(status), _stream(stream)), "pa_mla_cache_write")


def pa_read_device_status(workspace, stream=None) -> int:
    bits = ctypes.c_uint32(0)
    _check(lib.pa_read_device_status(_ptr(workspace), _stream(stream), ctypes.byref(bits)),
           "pa_read_device_status")
    return int(bits.value)


def pa_set_profile_events(before=None, after=None) -> None:
    """Record torch.cuda.Event pair around the dominant kernel of later calls (None, None: off)."""
    def handle(ev):
        if ev is None:
            return None
        if ev.cuda_event == 0:  # torch creates the event lazily
            ev.record()
        return ev.cuda_event
    _check(lib.pa_set_profile_events(handle(before), handle(after)), "pa_set_profile_events")


def pa_last_launch_count() -> int:
    return int(lib.pa_last_launch_count())


def pa_set_wait_limit_ns(limit_ns: int = PA_DEFAULT_WAIT_LIMIT_NS) -> None:
    """Limit (global-timer ns) of the GQA split kernels' ring waits for later calls from this thread."""
    _check(lib.pa_set_wait_limit_ns(int(limit_ns)), "pa_set_wait_limit_ns")


def pa_last_cuda_error() -> int:
    return int(lib.pa_last_cuda_error())


def pa_last_cuda_error_string() -> str:
    return lib.pa_last_cuda_error_string().decode()


def workspace_for_gqa(q, k_pool, block_table, num_splits: int = 0, max_context_len=None, device=None):
    """Allocate a uint8 device workspace sized for a pa_decode_gqa call with these tensors."""
    import torch
    B, Hq, D = q.shape[0], q.shape[-2], q.shape[-1]
    _, P, Hkv, _ = k_pool.shape
    mcl = block_table.shape[1] * P if max_context_len is None else max_context_len
    n = pa_workspace_size(PA_KIND_GQA, B, Hq, Hkv, D, mcl, P, num_splits)
    if n == 0:
        raise PaError(PA_ERR_INVALID_ARGUMENT, "pa_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device or q.device)


def workspace_for_mla(q, cache, block_table, num_splits: int = 0, max_context_len=None, device=None):
    import torch
    B, H, _ = q.shape
    _, P, _ = cache.shape
    mcl = block_table.shape[1] * P if max_context_len is None else max_context_len
    n = pa_workspace_size(PA_KIND_MLA_ABSORBED, B, H, 1, 576, mcl, P, num_splits)
    if n == 0:
        raise PaError(PA_ERR_INVALID_ARGUMENT, "pa_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device or q.device)
