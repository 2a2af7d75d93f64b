"""Paged KV-cache attention for GB300 (sm_103a): Python binding.

A thin ctypes layer over the C ABI of ``include/pd_attn.h``: it checks tensor
dtypes, devices and contiguity, marshals ``data_ptr()`` values and the current
CUDA stream, and raises on a non-OK status.  Every step of the computation
runs in the library's CUDA kernels; there is no other code path.  The library
must have been built (``paged_kv_attention_26_gb300.build.build()``); loading
fails loudly otherwise.

Functions carry the C names: ``pd_reshape_and_cache``,
``pd_paged_attention_decode`` (+ ``pd_decode_workspace_bytes``),
``pd_decode_step`` (store + decode), ``pd_paged_attention_verify`` (several
query tokens per sequence), the ``_fp8`` variants, ``pd_copy_blocks``,
``pd_kv_pack``/``pd_kv_unpack``, ``pd_paged_prefill_chunk``; ``BlockManager``
and ``PrefixCache`` wrap the host-side ``pd_bm_*`` and ``pd_pc_*`` calls;
``DecodeStep`` runs one host-to-host decode step (one copy in, the fused
step, one copy out), optionally replayed from a CUDA graph.
"""
from __future__ import annotations

import collections
import ctypes
import os
import threading

from . import build as _build

LIB_PATH = _build.LIB

PD_OK = 0
PD_F16, PD_BF16, PD_FP8_E4M3 = 0, 1, 2
PD_DEVERR_SLOT_RANGE = 0x1
PD_DEVERR_BLOCK_RANGE = 0x2
PD_DEVERR_CTX_RANGE = 0x4
PD_DEVERR_TIMEOUT = 0x8
PD_DEVERR_SHARED_PREFIX = 0x10
PD_DEVERR_STEP_SLOT = 0x20

STATUS_NAMES = {0: "PD_OK", 1: "PD_ERR_INVALID_ARG", 2: "PD_ERR_UNSUPPORTED", 3: "PD_ERR_CUDA",
                4: "PD_ERR_NO_FREE_BLOCK", 5: "PD_ERR_WORKSPACE_TOO_SMALL",
                6: "PD_ERR_NOT_FOUND"}

# Every symbol include/pd_attn.h exports: name -> (restype, argtypes)
_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t
SIGNATURES = {
    "pd_status_string": (ctypes.c_char_p, [_I]),
    "pd_last_cuda_error": (_I, []),
    "pd_launch_count": (ctypes.c_uint64, []),
    "pd_reshape_and_cache": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I64, _I64, _I, _P, _P]),
    "pd_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "pd_decode_partition_tokens": (_I, [_I]),
    "pd_paged_attention_decode": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I,
                                       _F, _P, _SZ, _I, _P, _P]),
    "pd_paged_attention_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I,
                                               _I, _I, _F, _I, _P, _P]),
    "pd_decode_shared_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "pd_paged_attention_decode_shared": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I,
                                              _I, _I, _F, _P, _P, _I, _I, _P, _SZ, _I, _P, _P]),
    "pd_decode_step_shared": (_I, [_P, _I, _P, _P, _P, _I, _I64, _I64, _P, _P, _P, _P, _P, _I,
                                   _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _I, _I, _P, _SZ,
                                   _I, _P, _P]),
    "pd_find_shared_prefixes": (_I, [ctypes.POINTER(ctypes.c_int32), _I,
                                     ctypes.POINTER(ctypes.c_int32), _I, _I, _I, _I,
                                     ctypes.POINTER(ctypes.c_int32),
                                     ctypes.POINTER(ctypes.c_int32),
                                     ctypes.POINTER(ctypes.c_int)]),
    "pd_copy_blocks": (_I, [_P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "pd_reshape_and_cache_fp8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I64, _I64,
                                      _P, _P, _I, _P, _P]),
    "pd_paged_attention_decode_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I,
                                           _I, _I, _I, _F, _P, _SZ, _I, _P, _P]),
    "pd_paged_attention_verify": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _I,
                                       _I, _F, _P, _SZ, _I, _P, _P]),
    "pd_decode_step": (_I, [_P, _P, _P, _I, _I64, _I64, _P, _P, _P, _P, _P, _I, _P, _I, _I,
                            _I, _I, _I, _I, _I, _F, _P, _SZ, _I, _P, _P]),
    "pd_decode_step_fused": (_I, [_P, _P, _P, _I, _I64, _I64, _P, _P, _P, _P, _P, _I, _P, _I, _I,
                                  _I, _I, _I, _I, _I, _F, _P, _SZ, _I, _P, _P]),
    "pd_decode_step_fp8": (_I, [_P, _P, _P, _I, _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _I,
                                _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _SZ, _I, _P, _P]),
    "pd_selftest_bounded_wait": (_I, [_P, ctypes.c_uint64, _P]),
    "pd_copy_bytes": (_I, [_P, _P, _SZ, _P]),
    "pd_verify_step": (_I, [_P, _P, _P, _I, _I64, _I64, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I,
                            _I, _I, _I, _I, _I, _F, _P, _SZ, _I, _P, _P]),
    "pd_kv_pack": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "pd_kv_unpack": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "pd_paged_prefill_chunk": (_I, [_P, _P, _I, _P, _I, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I,
                                    _I, _F, _I, _P, _P]),
    "pd_bm_create": (_P, [_I, _I]),
    "pd_bm_destroy": (None, [_P]),
    "pd_bm_add_seq": (_I, [_P, _I]),
    "pd_bm_append_slot": (_I, [_P, _I, ctypes.POINTER(ctypes.c_int64),
                               ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]),
    "pd_bm_fork": (_I, [_P, _I, _I]),
    "pd_bm_release": (_I, [_P, _I]),
    "pd_bm_block_table": (_I, [_P, _I, ctypes.POINTER(ctypes.c_int32), _I,
                               ctypes.POINTER(ctypes.c_int)]),
    "pd_bm_seq_len": (_I64, [_P, _I]),
    "pd_bm_usage": (ctypes.c_double, [_P]),
    "pd_bm_ref_count": (_I, [_P, _I]),
    "pd_bm_num_free": (_I, [_P]),
    "pd_bm_add_seq_shared": (_I, [_P, _I, ctypes.POINTER(ctypes.c_int32), _I, _I64]),
    "pd_bm_retain": (_I, [_P, _I]),
    "pd_bm_drop": (_I, [_P, _I]),
    "pd_pc_create": (_P, [_I, _I]),
    "pd_pc_destroy": (None, [_P]),
    "pd_pc_lookup": (_I, [_P, ctypes.POINTER(ctypes.c_int32), _I, ctypes.c_char_p,
                          ctypes.POINTER(ctypes.c_int), ctypes.c_char_p,
                          ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int)]),
    "pd_pc_insert": (_I, [_P, ctypes.c_char_p, _I, ctypes.POINTER(ctypes.c_int32),
                          ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int)]),
    "pd_pc_size": (_I, [_P]),
    "pd_pc_hits": (_I64, [_P]),
    "pd_pc_misses": (_I64, [_P]),
}

_lock = threading.Lock()
_lib = None


class PDError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        extra = ""
        if status == 3 and _lib is not None:
            extra = f" (cudaError {_lib.pd_last_cuda_error()})"
        super().__init__(f"{fn}: {name}{extra}")


def load():
    """Load the built library (raises FileNotFoundError if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise FileNotFoundError(
                f"{LIB_PATH} is missing: build it with paged_kv_attention_26_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != PD_OK:
        raise PDError(fn, status)


def launch_count() -> int:
    return int(load().pd_launch_count())


# ---- tensor helpers ---------------------------------------------------------------

def _torch():
    import torch
    return torch


def _dt(t) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return PD_F16
    if t.dtype == torch.bfloat16:
        return PD_BF16
    if t.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        return PD_FP8_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _is_fp8(t) -> bool:
    return _dt(t) == PD_FP8_E4M3


def _dev(t, name, dtype=None, contiguous=True, host_ok=False):
    # host_ok: pinned host memory is accepted too (with unified addressing its
    # host address is the address the kernels use, over the host link)
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor" +
                         (" or pinned host memory" if host_ok else ""))
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _opt(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ---- ops -------------------------------------------------------------------------------

def pd_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, dev_err=None,
                         stream=None):
    """Store key/value [T, Hk, D] (token-strided, heads contiguous) into the
    paged caches [NB, Hk, S, D] at ``slot_mapping`` (int64 [T])."""
    torch = _torch()
    T, Hk, D = key.shape
    NB, Hk2, S, D2 = key_cache.shape
    if (Hk2, D2) != (Hk, D) or value.shape != key.shape or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch")
    for t, n in ((key, "key"), (value, "value")):
        if t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError(f"{n} must have contiguous heads and dims")
    dt = _dt(key_cache)
    if key.dtype != key_cache.dtype or value.dtype != key_cache.dtype:
        raise TypeError("dtype mismatch")
    st = load().pd_reshape_and_cache(
        _dev(key, "key", contiguous=False), _dev(value, "value", contiguous=False),
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
        _dev(slot_mapping, "slot_mapping", torch.int64), T, Hk, D, S, NB,
        key.stride(0), value.stride(0), dt, _opt(dev_err), _stream(stream))
    _check("pd_reshape_and_cache", st)


def pd_reshape_and_cache_fp8(key, value, key_cache, value_cache, slot_mapping, k_scale, v_scale,
                             dev_err=None, stream=None):
    """Quantise key/value [T, Hk, D] (fp16/bf16) to E4M3 and store them into the
    one-byte pools [NB, Hk, S, D] at ``slot_mapping``; ``k_scale``/``v_scale``
    are float32 CUDA [Hk] (a code c stands for e4m3(c) * scale)."""
    torch = _torch()
    T, Hk, D = key.shape
    NB, Hk2, S, D2 = key_cache.shape
    if (Hk2, D2) != (Hk, D) or value.shape != key.shape or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch")
    if not (_is_fp8(key_cache) and _is_fp8(value_cache)):
        raise TypeError("the pools must be one-byte (uint8 or float8_e4m3fn)")
    for t, n in ((key, "key"), (value, "value")):
        if t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError(f"{n} must have contiguous heads and dims")
    if value.dtype != key.dtype:
        raise TypeError("dtype mismatch")
    for sc in (k_scale, v_scale):
        if sc.shape != (Hk,):
            raise ValueError("scales must be [Hk]")
    st = load().pd_reshape_and_cache_fp8(
        _dev(key, "key", contiguous=False), _dev(value, "value", contiguous=False),
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
        _dev(slot_mapping, "slot_mapping", torch.int64), T, Hk, D, S, NB,
        key.stride(0), value.stride(0), _dev(k_scale, "k_scale", torch.float32),
        _dev(v_scale, "v_scale", torch.float32), _dt(key), _opt(dev_err), _stream(stream))
    _check("pd_reshape_and_cache_fp8", st)


def pd_paged_attention_decode_fp8(out, q, key_cache, value_cache, k_scale, v_scale, block_tables,
                                  context_lens, max_context_len: int, scale: float,
                                  workspace=None, dev_err=None, stream=None):
    """Decode over E4M3 pools [NB, Hk, S, D] (uint8 or float8_e4m3fn) with float32
    scales [Hk]; out, q [B, H, D] fp16/bf16."""
    torch = _torch()
    B, H, D = q.shape
    NB, Hk, S, D2 = key_cache.shape
    if out.shape != q.shape or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables / context_lens shape")
    if not (_is_fp8(key_cache) and _is_fp8(value_cache)):
        raise TypeError("the pools must be one-byte (uint8 or float8_e4m3fn)")
    if out.dtype != q.dtype:
        raise TypeError("dtype mismatch")
    for sc in (k_scale, v_scale):
        if sc.shape != (Hk,):
            raise ValueError("scales must be [Hk]")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    st = load().pd_paged_attention_decode_fp8(
        _dev(out, "out"), _dev(q, "q"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(k_scale, "k_scale", torch.float32),
        _dev(v_scale, "v_scale", torch.float32),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), B, H, Hk, D, S, NB,
        int(max_context_len), float(scale), ws_ptr, ws_bytes, _dt(q), _opt(dev_err),
        _stream(stream))
    _check("pd_paged_attention_decode_fp8", st)


def pd_decode_workspace_bytes(B: int, H: int, D: int, max_context_len: int) -> int:
    return int(load().pd_decode_workspace_bytes(B, H, D, max_context_len))


def pd_decode_partition_tokens(max_context_len: int) -> int:
    return int(load().pd_decode_partition_tokens(max_context_len))


def decode_workspace(B, H, D, max_context_len, device="cuda"):
    """Allocate a workspace of the required size (uint8, 256-byte aligned)."""
    torch = _torch()
    n = pd_decode_workspace_bytes(B, H, D, max_context_len)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def pd_paged_attention_decode(out, q, key_cache, value_cache, block_tables, context_lens,
                              max_context_len: int, scale: float, workspace=None,
                              dev_err=None, stream=None):
    """out, q [B, H, D]; caches [NB, Hk, S, D]; block_tables int32 [B, max_blocks];
    context_lens int32 [B].  ``workspace`` (uint8 CUDA tensor) must hold
    ``pd_decode_workspace_bytes`` bytes when that is non-zero."""
    torch = _torch()
    B, H, D = q.shape
    NB, Hk, S, D2 = key_cache.shape
    if out.shape != q.shape or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables / context_lens shape")
    dt = _dt(key_cache)
    for t in (q, out, value_cache):
        if t.dtype != key_cache.dtype:
            raise TypeError("dtype mismatch")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    st = load().pd_paged_attention_decode(
        _dev(out, "out"), _dev(q, "q"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), B, H, Hk, D, S,
        NB, int(max_context_len), float(scale), ws_ptr, ws_bytes, dt, _opt(dev_err),
        _stream(stream))
    _check("pd_paged_attention_decode", st)


def pd_decode_shared_workspace_bytes(n_groups: int, max_group: int, H: int, Hk: int,
                                     D: int) -> int:
    return int(load().pd_decode_shared_workspace_bytes(n_groups, max_group, H, Hk, D))


def decode_shared_workspace(n_groups, max_group, H, Hk, D, device="cuda"):
    """Allocate the workspace of ``pd_paged_attention_decode_shared``."""
    torch = _torch()
    n = pd_decode_shared_workspace_bytes(n_groups, max_group, H, Hk, D)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def find_shared_prefixes(block_tables, context_lens, S: int, max_group: int = 8,
                         min_shared_tokens: int = 0):
    """Groups of consecutive sequences sharing leading blocks (host tensors in,
    ``pd_find_shared_prefixes``): returns (group_starts int32 [n_groups + 1],
    shared_lens int32 [n_groups]) as CPU tensors."""
    torch = _torch()
    bt = block_tables.detach().to("cpu", torch.int32).contiguous()
    cl = context_lens.detach().to("cpu", torch.int32).contiguous()
    B, mb = bt.shape
    if cl.shape != (B,):
        raise ValueError("context_lens shape")
    gs = torch.zeros(B + 1, dtype=torch.int32)
    sl = torch.zeros(max(B, 1), dtype=torch.int32)
    n = ctypes.c_int(0)
    i32p = ctypes.POINTER(ctypes.c_int32)
    st = load().pd_find_shared_prefixes(
        ctypes.cast(bt.data_ptr(), i32p), mb, ctypes.cast(cl.data_ptr(), i32p), B, int(S),
        int(max_group), int(min_shared_tokens), ctypes.cast(gs.data_ptr(), i32p),
        ctypes.cast(sl.data_ptr(), i32p), ctypes.byref(n))
    _check("pd_find_shared_prefixes", st)
    return gs[:n.value + 1].clone(), sl[:n.value].clone()


def pd_paged_attention_decode_shared(out, q, key_cache, value_cache, block_tables,
                                     context_lens, max_context_len: int, scale: float,
                                     group_starts, shared_lens, max_group: int,
                                     workspace=None, dev_err=None, stream=None):
    """Decode for groups of forks that share leading blocks: the result of
    ``pd_paged_attention_decode``, each shared block read once per group.
    group_starts int32 CUDA [n_groups + 1], shared_lens int32 CUDA [n_groups]
    (from ``find_shared_prefixes``); ``workspace`` from
    ``decode_shared_workspace``."""
    torch = _torch()
    B, H, D = q.shape
    NB, Hk, S, D2 = key_cache.shape
    if out.shape != q.shape or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables / context_lens shape")
    n_groups = shared_lens.numel()
    if group_starts.shape != (n_groups + 1,):
        raise ValueError("group_starts must have n_groups + 1 entries")
    dt = _dt(key_cache)
    for t in (q, out, value_cache):
        if t.dtype != key_cache.dtype:
            raise TypeError("dtype mismatch")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    st = load().pd_paged_attention_decode_shared(
        _dev(out, "out"), _dev(q, "q"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), B, H, Hk, D, S,
        NB, int(max_context_len), float(scale), _dev(group_starts, "group_starts", torch.int32),
        _dev(shared_lens, "shared_lens", torch.int32), n_groups, int(max_group), ws_ptr,
        ws_bytes, dt, _opt(dev_err), _stream(stream))
    _check("pd_paged_attention_decode_shared", st)


def pd_decode_step_shared(out, q, key_cache, value_cache, block_tables, context_lens,
                          max_context_len: int, scale: float, group_starts, shared_lens,
                          max_group: int, key=None, value=None, slot_mapping=None,
                          block_mapping=None, workspace=None, dev_err=None, stream=None):
    """One copy-on-write decode step of one layer over forks sharing blocks:
    ``block_mapping`` (int64 CUDA [npairs, 2], or None) block copies in these
    pools, then the store of ``key``/``value`` [T, Hk, D] at ``slot_mapping``
    (or None), then ``pd_paged_attention_decode_shared``; each grid a
    programmatic dependent of the one before it."""
    torch = _torch()
    B, H, D = q.shape
    NB, Hk, S, D2 = key_cache.shape
    if out.shape != q.shape or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables / context_lens shape")
    n_groups = shared_lens.numel()
    if group_starts.shape != (n_groups + 1,):
        raise ValueError("group_starts must have n_groups + 1 entries")
    dt = _dt(key_cache)
    for t in (q, out, value_cache):
        if t.dtype != key_cache.dtype:
            raise TypeError("dtype mismatch")
    npairs, bm = 0, None
    if block_mapping is not None and block_mapping.numel():
        if block_mapping.dim() != 2 or block_mapping.shape[1] != 2:
            raise ValueError("block_mapping must be [npairs, 2]")
        npairs, bm = block_mapping.shape[0], _dev(block_mapping, "block_mapping", torch.int64)
    T, kp, vp, sp, ks, vs = 0, None, None, None, 0, 0
    if key is not None and key.shape[0]:
        T = key.shape[0]
        if key.shape != (T, Hk, D) or value.shape != key.shape or slot_mapping.shape != (T,):
            raise ValueError("key / value / slot_mapping shape")
        for t, n in ((key, "key"), (value, "value")):
            if t.stride(2) != 1 or t.stride(1) != D:
                raise ValueError(f"{n} must have contiguous heads and dims")
            if t.dtype != key_cache.dtype:
                raise TypeError("dtype mismatch")
        kp, vp = _dev(key, "key", contiguous=False), _dev(value, "value", contiguous=False)
        sp = _dev(slot_mapping, "slot_mapping", torch.int64)
        ks, vs = key.stride(0), value.stride(0)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    st = load().pd_decode_step_shared(
        bm, npairs, kp, vp, sp, T, ks, vs, _dev(out, "out"), _dev(q, "q"),
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), B, H, Hk, D, S, NB,
        int(max_context_len), float(scale), _dev(group_starts, "group_starts", torch.int32),
        _dev(shared_lens, "shared_lens", torch.int32), n_groups, int(max_group), ws_ptr,
        ws_bytes, dt, _opt(dev_err), _stream(stream))
    _check("pd_decode_step_shared", st)


def pd_paged_attention_verify(out, q, key_cache, value_cache, block_tables, context_lens,
                              max_context_len: int, scale: float, workspace=None,
                              dev_err=None, stream=None):
    """Speculative verification: q, out [B, nq, H, D] (nq = 1..8), the last nq
    positions of each context, causal among themselves; caches [NB, Hk, S, D]
    (16-bit); ``workspace`` holds ``pd_decode_workspace_bytes(B * nq, ...)``
    bytes (``verify_workspace``)."""
    torch = _torch()
    B, nq, H, D = q.shape
    NB, Hk, S, D2 = key_cache.shape
    if out.shape != q.shape or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables / context_lens shape")
    dt = _dt(key_cache)
    for t in (q, out, value_cache):
        if t.dtype != key_cache.dtype:
            raise TypeError("dtype mismatch")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    st = load().pd_paged_attention_verify(
        _dev(out, "out"), _dev(q, "q"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), B, nq, H, Hk, D,
        S, NB, int(max_context_len), float(scale), ws_ptr, ws_bytes, dt, _opt(dev_err),
        _stream(stream))
    _check("pd_paged_attention_verify", st)


def pd_verify_step(out, q, key_cache, value_cache, block_tables, context_lens,
                   max_context_len: int, scale: float, key, value, slot_mapping,
                   workspace=None, dev_err=None, stream=None):
    """Store the drafted tokens ``key``/``value`` [T, Hk, D] at ``slot_mapping``,
    then verify ``q`` [B, nq, H, D] into ``out``: ``pd_reshape_and_cache``
    followed by ``pd_paged_attention_verify``, the verify grid launched as a
    dependent of the store grid."""
    torch = _torch()
    B, nq, H, D = q.shape
    NB, Hk, S, D2 = key_cache.shape
    T = key.shape[0]
    if out.shape != q.shape or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch")
    if key.shape != (T, Hk, D) or value.shape != key.shape or slot_mapping.shape != (T,):
        raise ValueError("key / value / slot_mapping shape")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables / context_lens shape")
    for t, n in ((key, "key"), (value, "value")):
        if t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError(f"{n} must have contiguous heads and dims")
    for t in (q, out, key, value, value_cache):
        if t.dtype != key_cache.dtype:
            raise TypeError("dtype mismatch")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    st = load().pd_verify_step(
        _dev(key, "key", contiguous=False), _dev(value, "value", contiguous=False),
        _dev(slot_mapping, "slot_mapping", torch.int64), T, key.stride(0), value.stride(0),
        _dev(out, "out"), _dev(q, "q"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), B, nq, H, Hk, D,
        S, NB, int(max_context_len), float(scale), ws_ptr, ws_bytes, _dt(key_cache),
        _opt(dev_err), _stream(stream))
    _check("pd_verify_step", st)


def verify_workspace(B, nq, H, D, max_context_len, device="cuda"):
    """Workspace for ``pd_paged_attention_verify`` (B sequences of nq queries)."""
    return decode_workspace(B * nq, H, D, max_context_len, device=device)


def pd_copy_bytes(dst, src, stream=None):
    """Copy ``src`` into ``dst`` (same byte size, contiguous, 16-byte aligned,
    a multiple of 16 bytes) with an SM kernel; either side may be a CUDA
    tensor or a pinned host tensor."""
    nb = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nb:
        raise ValueError("size mismatch")
    if not (dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("tensors must be contiguous")
    for t in (dst, src):
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError("host tensors must be pinned")
    st = load().pd_copy_bytes(dst.data_ptr(), src.data_ptr(), nb, _stream(stream))
    _check("pd_copy_bytes", st)


def pd_selftest_bounded_wait(dev_err, limit_ns: int = 1_000_000, stream=None):
    """One CTA waits on a barrier nothing completes; after ``limit_ns`` the
    wait gives up and PD_DEVERR_TIMEOUT is OR-ed into ``dev_err`` (int32 CUDA
    [1]), as in every kernel of the library.  A failure-detection test aid."""
    torch = _torch()
    st = load().pd_selftest_bounded_wait(_dev(dev_err, "dev_err", torch.int32), int(limit_ns),
                                         _stream(stream))
    _check("pd_selftest_bounded_wait", st)


def pd_decode_step_fused(out, q, key_cache, value_cache, block_tables, context_lens,
                         max_context_len: int, scale: float, key, value, slot_mapping,
                         workspace=None, dev_err=None, stream=None):
    """``pd_decode_step`` in one kernel, for a step whose row i of
    ``key``/``value`` [B, Hk, D] is the last token of sequence i (its slot in
    ``slot_mapping``, or < 0 for none): the decode stores each row right
    before it copies the row's block.  16-bit pools, G <= 8; a slot that is
    not the last token's flags ``PD_DEVERR_STEP_SLOT`` and is not stored."""
    pd_decode_step(out, q, key_cache, value_cache, block_tables, context_lens, max_context_len,
                   scale, key, value, slot_mapping, workspace=workspace, dev_err=dev_err,
                   stream=stream, _fused=True)


def pd_decode_step(out, q, key_cache, value_cache, block_tables, context_lens,
                   max_context_len: int, scale: float, key, value, slot_mapping,
                   workspace=None, k_scale=None, v_scale=None, dev_err=None, stream=None,
                   _fused=False):
    """One decode step of one layer: store ``key``/``value`` [T, Hk, D] at
    ``slot_mapping``, then decode ``q`` [B, H, D] over the paged caches into
    ``out``.  The same result as ``pd_reshape_and_cache`` (``_fp8`` with
    scales) followed by ``pd_paged_attention_decode`` (``_fp8``); the decode
    grid's prologue overlaps the store.  One-byte pools need ``k_scale`` and
    ``v_scale`` (float32 [Hk]).  ``q``, ``key``, ``value``, ``slot_mapping``,
    ``block_tables``, ``context_lens`` and ``out`` may be pinned host tensors:
    the kernels then read and write them over the host link, with no separate
    copy."""
    torch = _torch()
    B, H, D = q.shape
    NB, Hk, S, D2 = key_cache.shape
    T = key.shape[0]
    if out.shape != q.shape or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch")
    if key.shape != (T, Hk, D) or value.shape != key.shape or slot_mapping.shape != (T,):
        raise ValueError("key / value / slot_mapping shape")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables / context_lens shape")
    for t, n in ((key, "key"), (value, "value")):
        if t.stride(2) != 1 or t.stride(1) != D:
            raise ValueError(f"{n} must have contiguous heads and dims")
    fp8 = _is_fp8(key_cache)
    if fp8 != _is_fp8(value_cache):
        raise TypeError("dtype mismatch")
    for t in (q, key, value):
        if t.dtype != out.dtype or (not fp8 and t.dtype != key_cache.dtype):
            raise TypeError("dtype mismatch")
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    head = (_dev(key, "key", contiguous=False, host_ok=True),
            _dev(value, "value", contiguous=False, host_ok=True),
            _dev(slot_mapping, "slot_mapping", torch.int64, host_ok=True), T, key.stride(0),
            value.stride(0), _dev(out, "out", host_ok=True), _dev(q, "q", host_ok=True),
            _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"))
    tail = (_dev(block_tables, "block_tables", torch.int32, host_ok=True), block_tables.shape[1],
            _dev(context_lens, "context_lens", torch.int32, host_ok=True), B, H, Hk, D, S, NB,
            int(max_context_len), float(scale), ws_ptr, ws_bytes, _dt(q), _opt(dev_err),
            _stream(stream))
    if fp8 and _fused:
        raise TypeError("the fused step takes 16-bit pools")
    if fp8:
        if k_scale is None or v_scale is None:
            raise ValueError("one-byte pools need k_scale and v_scale")
        for sc in (k_scale, v_scale):
            if sc.shape != (Hk,):
                raise ValueError("scales must be [Hk]")
        st = load().pd_decode_step_fp8(*head, _dev(k_scale, "k_scale", torch.float32),
                                       _dev(v_scale, "v_scale", torch.float32), *tail)
        _check("pd_decode_step_fp8", st)
    elif _fused:
        st = load().pd_decode_step_fused(*head, *tail)
        _check("pd_decode_step_fused", st)
    else:
        st = load().pd_decode_step(*head, *tail)
        _check("pd_decode_step", st)


class DecodeStep:
    """One layer's decode step from host memory to host memory.

    The step's inputs live in one pinned host buffer, exposed as views in
    ``host`` (``q`` [B, H, D], ``key``/``value`` [T, Hk, D], ``slot_mapping``
    int64 [T], ``block_tables`` int32 [B, max_blocks_per_seq],
    ``context_lens`` int32 [B]); the result lands in the pinned ``host_out``.
    A call runs ``pd_decode_step`` (store, then decode as a dependent grid)
    with every input and ``out`` passed as the pinned host buffers themselves:
    the store and the decode read them and write the result over the host
    link, so there is no copy at all (copying the block tables and context
    lengths to the device first measured the same, ~71 us per Qwen3-8B batch-64
    step).  With ``graph=True`` the step is captured once in a CUDA graph and
    each call replays it;
    ``max_context_len`` and ``scale`` are fixed at construction (contexts may
    vary per call up to that bound).  ``fused=True`` runs
    ``pd_decode_step_fused`` instead (T == B, row i the last token of
    sequence i; 16-bit pools).  One-byte pools take
    ``k_scale``/``v_scale`` (float32 CUDA [Hk]).  The device error word of the
    last call is ``dev_err``."""

    def __init__(self, key_cache, value_cache, B: int, H: int, T: int, max_blocks_per_seq: int,
                 max_context_len: int, scale: float, dtype, k_scale=None, v_scale=None,
                 graph: bool = True, fused: bool = False):
        torch = _torch()
        dev = key_cache.device
        NB, Hk, S, D = key_cache.shape
        # every field is read by the kernels in place
        fields = (("q", (B, H, D), dtype), ("key", (T, Hk, D), dtype),
                  ("value", (T, Hk, D), dtype), ("slot_mapping", (T,), torch.int64),
                  ("block_tables", (B, max_blocks_per_seq), torch.int32),
                  ("context_lens", (B,), torch.int32))
        spans, off = [], 0
        for name, shape, dt in fields:
            n = torch.empty(shape, dtype=dt, device="meta").numel() * \
                torch.empty((), dtype=dt, device="meta").element_size()
            spans.append((name, shape, dt, off, n))
            off += (n + 255) // 256 * 256
        self.host_buf = torch.zeros(max(off, 256), dtype=torch.uint8).pin_memory()
        self.host = {n: self.host_buf[o:o + b].view(dt).view(shape) for n, shape, dt, o, b in spans}
        self.host["slot_mapping"].fill_(-1)      # until the caller writes it: store nothing
        self.host_out = torch.zeros((B, H, D), dtype=dtype).pin_memory()
        self.workspace = decode_workspace(B, H, D, max_context_len, device=dev)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.key_cache, self.value_cache = key_cache, value_cache
        self.k_scale, self.v_scale = k_scale, v_scale
        self.max_context_len, self.scale = int(max_context_len), float(scale)
        self.fused = bool(fused)
        self.device = dev
        self.graph = None
        # one eager run on the harmless initial inputs (no slot stored, empty
        # contexts) sets up the launch attributes before any capture
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            self._body()
        torch.cuda.current_stream(dev).wait_stream(side)
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._body()
            self.graph = g

    def _body(self):
        h = self.host
        if self.fused:
            pd_decode_step_fused(self.host_out, h["q"], self.key_cache, self.value_cache,
                                 h["block_tables"], h["context_lens"], self.max_context_len,
                                 self.scale, h["key"], h["value"], h["slot_mapping"],
                                 workspace=self.workspace, dev_err=self.dev_err)
            return
        pd_decode_step(self.host_out, h["q"], self.key_cache, self.value_cache,
                       h["block_tables"], h["context_lens"], self.max_context_len, self.scale,
                       h["key"], h["value"], h["slot_mapping"], workspace=self.workspace,
                       k_scale=self.k_scale, v_scale=self.v_scale, dev_err=self.dev_err)

    def __call__(self):
        torch = _torch()
        if self.graph is not None:
            self.graph.replay()
        else:
            self._body()
        torch.cuda.current_stream(self.device).synchronize()
        return self.host_out

    @property
    def h2d_bytes(self) -> int:
        """Input bytes that cross the host link per call: q, the new K/V, the
        slots, the block tables and the context lengths, all read in place."""
        return self.host_buf.numel()

    @property
    def d2h_bytes(self) -> int:
        return self.host_out.numel() * self.host_out.element_size()


def pd_paged_attention_decode_noalloc(out, q, key_cache, value_cache, block_tables,
                                      context_lens, max_context_len: int, scale: float,
                                      dev_err=None, stream=None):
    """Decode attention that needs no workspace from the caller: the library
    keeps a fixed 32 MiB scratch array per GPU for the partition results.
    For callers that cannot allocate device memory on the call path.  Batches
    whose workspace would exceed 32 MiB raise (PD_ERR_WORKSPACE_TOO_SMALL);
    calls that overlap on the GPU share the scratch and race."""
    torch = _torch()
    B, H, D = q.shape
    NB, Hk, S, D2 = key_cache.shape
    if out.shape != q.shape or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables / context_lens shape")
    dt = _dt(key_cache)
    for t in (q, out, value_cache):
        if t.dtype != key_cache.dtype:
            raise TypeError("dtype mismatch")
    st = load().pd_paged_attention_decode_noalloc(
        _dev(out, "out"), _dev(q, "q"), _dev(key_cache, "key_cache"),
        _dev(value_cache, "value_cache"), _dev(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _dev(context_lens, "context_lens", torch.int32), B, H, Hk, D, S,
        NB, int(max_context_len), float(scale), dt, _opt(dev_err), _stream(stream))
    _check("pd_paged_attention_decode_noalloc", st)


_ptr_arrays: "collections.OrderedDict" = collections.OrderedDict()
_PTR_ARRAYS_MAX = 64


def pointer_array(tensors, device=None):
    """Device int64 array of the tensors' data pointers, cached per (device,
    pointer tuple); the cache keeps the _PTR_ARRAYS_MAX most recently used
    arrays, so callers that reallocate their pools do not grow it without
    bound.  An evicted array is freed through torch's stream-ordered caching
    allocator, so a launch already enqueued with it still reads it."""
    torch = _torch()
    dev = torch.device(device) if device is not None else tensors[0].device
    key = (str(dev),) + tuple(t.data_ptr() for t in tensors)
    arr = _ptr_arrays.get(key)
    if arr is None:
        arr = torch.tensor(key[1:], dtype=torch.int64).to(dev)
        _ptr_arrays[key] = arr
        while len(_ptr_arrays) > _PTR_ARRAYS_MAX:
            _ptr_arrays.popitem(last=False)
    else:
        _ptr_arrays.move_to_end(key)
    return arr


def pd_copy_blocks(key_caches, value_caches, block_mapping, dev_err=None, stream=None):
    """Copy whole blocks src -> dst for every (src, dst) row of ``block_mapping``
    (int64 CUDA [npairs, 2]) in every layer's K and V pool (lists of [NB, Hk, S, D])."""
    torch = _torch()
    L = len(key_caches)
    if L == 0 or L != len(value_caches):
        raise ValueError("need the same number (> 0) of key and value pools")
    NB, Hk, S, D = key_caches[0].shape
    for t in list(key_caches) + list(value_caches):
        if t.shape != key_caches[0].shape or t.dtype != key_caches[0].dtype:
            raise ValueError("all pools must share shape and dtype")
        if _dev(t, "cache") % 16:
            raise ValueError("cache pools must be 16-byte aligned")
    if block_mapping.dim() != 2 or block_mapping.shape[1] != 2:
        raise ValueError("block_mapping must be [npairs, 2]")
    kp = pointer_array(key_caches)
    vp = pointer_array(value_caches)
    st = load().pd_copy_blocks(kp.data_ptr(), vp.data_ptr(), L,
                               _dev(block_mapping, "block_mapping", torch.int64),
                               block_mapping.shape[0], Hk, D, S, NB, _dt(key_caches[0]),
                               _opt(dev_err), _stream(stream))
    _check("pd_copy_blocks", st)


def _pools_check(key_caches, value_caches):
    L = len(key_caches)
    if L == 0 or L != len(value_caches):
        raise ValueError("need the same number (> 0) of key and value pools")
    for t in list(key_caches) + list(value_caches):
        if t.shape != key_caches[0].shape or t.dtype != key_caches[0].dtype:
            raise ValueError("all pools must share shape and dtype")
        if _dev(t, "cache") % 16:
            raise ValueError("cache pools must be 16-byte aligned")
    return L


def kv_staging(L: int, nblk: int, key_cache, device=None):
    """Allocate a staging buffer [L, 2, nblk, Hk, S, D] for ``pd_kv_pack``."""
    torch = _torch()
    NB, Hk, S, D = key_cache.shape
    return torch.empty((L, 2, nblk, Hk, S, D), dtype=key_cache.dtype,
                       device=device or key_cache.device)


def pd_kv_pack(staging, key_caches, value_caches, block_ids, dev_err=None, stream=None):
    """Gather blocks ``block_ids`` (int32 CUDA [nblk]) of every layer's K and V pool
    into ``staging`` ([L, 2, nblk, Hk, S, D], layer-major)."""
    torch = _torch()
    L = _pools_check(key_caches, value_caches)
    NB, Hk, S, D = key_caches[0].shape
    nblk = block_ids.shape[0]
    if tuple(staging.shape) != (L, 2, nblk, Hk, S, D) or staging.dtype != key_caches[0].dtype:
        raise ValueError("staging must be [L, 2, nblk, Hk, S, D] of the pools' dtype")
    st = load().pd_kv_pack(_dev(staging, "staging"), pointer_array(key_caches).data_ptr(),
                           pointer_array(value_caches).data_ptr(), L,
                           _dev(block_ids, "block_ids", torch.int32), nblk, Hk, D, S, NB,
                           _dt(key_caches[0]), _opt(dev_err), _stream(stream))
    _check("pd_kv_pack", st)


def pd_kv_unpack(staging, key_caches, value_caches, block_ids, dev_err=None, stream=None):
    """Scatter ``staging`` ([L, 2, nblk, Hk, S, D]) into blocks ``block_ids`` of the
    pools (the receiver's ids)."""
    torch = _torch()
    L = _pools_check(key_caches, value_caches)
    NB, Hk, S, D = key_caches[0].shape
    nblk = block_ids.shape[0]
    if tuple(staging.shape) != (L, 2, nblk, Hk, S, D) or staging.dtype != key_caches[0].dtype:
        raise ValueError("staging must be [L, 2, nblk, Hk, S, D] of the pools' dtype")
    st = load().pd_kv_unpack(_dev(staging, "staging"), pointer_array(key_caches).data_ptr(),
                             pointer_array(value_caches).data_ptr(), L,
                             _dev(block_ids, "block_ids", torch.int32), nblk, Hk, D, S, NB,
                             _dt(key_caches[0]), _opt(dev_err), _stream(stream))
    _check("pd_kv_unpack", st)


def pd_paged_prefill_chunk(out, q, cu_q_lens, max_q_len: int, key_cache, value_cache,
                           block_tables, context_lens, scale: float, dev_err=None, stream=None):
    """out, q packed [sumC, H, D]; cu_q_lens int32 [B+1]; context_lens int32 [B]
    (= prior + chunk length); caches [NB, Hk, S, D]; block_tables int32 [B, max_blocks]."""
    torch = _torch()
    NT, H, D = q.shape
    NB, Hk, S, D2 = key_cache.shape
    B = cu_q_lens.shape[0] - 1
    if out.shape != q.shape or D2 != D or value_cache.shape != key_cache.shape:
        raise ValueError("shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables / context_lens shape")
    for t in (q, out, value_cache):
        if t.dtype != key_cache.dtype:
            raise TypeError("dtype mismatch")
    st = load().pd_paged_prefill_chunk(
        _dev(out, "out"), _dev(q, "q"), NT, _dev(cu_q_lens, "cu_q_lens", torch.int32),
        int(max_q_len), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
        _dev(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _dev(context_lens, "context_lens", torch.int32), B, H, Hk, D, S, NB, float(scale),
        _dt(key_cache), _opt(dev_err), _stream(stream))
    _check("pd_paged_prefill_chunk", st)


class BlockManager:
    """Host block manager (pd_bm_*): ref-counted blocks, copy-on-write, fork."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = load()
        self._h = self._lib.pd_bm_create(num_blocks, block_size)
        if not self._h:
            raise ValueError("pd_bm_create failed")
        self.num_blocks = num_blocks
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.pd_bm_destroy(h)
            self._h = None

    def add_seq(self, seq_id: int):
        _check("pd_bm_add_seq", self._lib.pd_bm_add_seq(self._h, seq_id))

    def append_slot(self, seq_id: int):
        """Returns (slot, (src, dst) copy or None)."""
        slot = ctypes.c_int64()
        src = ctypes.c_int32()
        dst = ctypes.c_int32()
        _check("pd_bm_append_slot", self._lib.pd_bm_append_slot(
            self._h, seq_id, ctypes.byref(slot), ctypes.byref(src), ctypes.byref(dst)))
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def fork(self, parent_id: int, child_id: int):
        _check("pd_bm_fork", self._lib.pd_bm_fork(self._h, parent_id, child_id))

    def release(self, seq_id: int):
        _check("pd_bm_release", self._lib.pd_bm_release(self._h, seq_id))

    def block_table(self, seq_id: int) -> list:
        n = ctypes.c_int()
        st = self._lib.pd_bm_block_table(self._h, seq_id, None, 0, ctypes.byref(n))
        if st not in (PD_OK, 1):
            _check("pd_bm_block_table", st)
        buf = (ctypes.c_int32 * max(1, n.value))()
        _check("pd_bm_block_table", self._lib.pd_bm_block_table(self._h, seq_id, buf, n.value,
                                                                ctypes.byref(n)))
        return list(buf[: n.value])

    def seq_len(self, seq_id: int) -> int:
        return int(self._lib.pd_bm_seq_len(self._h, seq_id))

    @property
    def usage(self) -> float:
        return float(self._lib.pd_bm_usage(self._h))

    def ref_count(self, block_id: int) -> int:
        return int(self._lib.pd_bm_ref_count(self._h, block_id))

    @property
    def num_free(self) -> int:
        return int(self._lib.pd_bm_num_free(self._h))

    def add_seq_shared(self, seq_id: int, blocks, length: int):
        """New sequence starting on existing blocks (a cached prefix)."""
        arr = (ctypes.c_int32 * max(1, len(blocks)))(*blocks)
        _check("pd_bm_add_seq_shared", self._lib.pd_bm_add_seq_shared(
            self._h, seq_id, arr, len(blocks), int(length)))

    def retain(self, block_id: int):
        _check("pd_bm_retain", self._lib.pd_bm_retain(self._h, block_id))

    def drop(self, block_id: int):
        _check("pd_bm_drop", self._lib.pd_bm_drop(self._h, block_id))


class PrefixCache:
    """Host prefix cache (pd_pc_*): block hash chain -> physical block, LRU."""

    KEY = 32

    def __init__(self, capacity_blocks: int, block_size: int):
        self._lib = load()
        self._h = self._lib.pd_pc_create(capacity_blocks, block_size)
        if not self._h:
            raise ValueError("pd_pc_create failed")
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.pd_pc_destroy(h)
            self._h = None

    def lookup(self, token_ids, extra: str = ""):
        """Returns (hit tokens, chain of block keys walked, block ids of the hits)."""
        n = len(token_ids)
        nfull = n // self.block_size
        toks = (ctypes.c_int32 * max(1, n))(*token_ids)
        chain = ctypes.create_string_buffer(max(1, nfull) * (self.KEY + 1))
        hits = (ctypes.c_int32 * max(1, nfull))()
        hit = ctypes.c_int()
        nc = ctypes.c_int()
        _check("pd_pc_lookup", self._lib.pd_pc_lookup(self._h, toks, n, extra.encode(),
                                                      ctypes.byref(hit), chain, hits,
                                                      ctypes.byref(nc)))
        raw = chain.raw
        keys = [raw[i * (self.KEY + 1): i * (self.KEY + 1) + self.KEY].decode()
                for i in range(nc.value)]
        return hit.value, keys, list(hits[: hit.value // self.block_size])

    def insert(self, chain, block_ids):
        """Returns the block ids of the entries evicted to make room."""
        n = len(chain)
        if len(block_ids) < n:
            raise ValueError("need a block id per chain key")
        buf = b"".join(k.encode()[: self.KEY].ljust(self.KEY + 1, b"\0") for k in chain)
        ids = (ctypes.c_int32 * max(1, n))(*block_ids[:n])
        ev = (ctypes.c_int32 * max(1, n))()
        ne = ctypes.c_int()
        _check("pd_pc_insert", self._lib.pd_pc_insert(self._h, buf if n else None, n, ids, ev,
                                                      ctypes.byref(ne)))
        return list(ev[: ne.value])

    def __len__(self):
        return int(self._lib.pd_pc_size(self._h))

    @property
    def hits(self) -> int:
        return int(self._lib.pd_pc_hits(self._h))

    @property
    def misses(self) -> int:
        return int(self._lib.pd_pc_misses(self._h))

    @property
    def hit_rate(self) -> float:
        tot = self.hits + self.misses
        return self.hits / tot if tot else 0.0
