"""Float64 CPU oracle for paged KV-cache attention.

TEST INFRASTRUCTURE ONLY: the product package never imports this.  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA path.

Contents
- ``oracle.c`` (loaded here through ctypes): store, copy-on-write block copy,
  decode attention (plain and split-context), chunked-prefill attention, all
  the plain definitions in float64.
- ``block_manager.py``: the ref-counted block manager with copy-on-write fork,
  following the tutorial page "LLM 推理服务引擎深度拆解", section 2.3.
- ``kv_bytes.py``: the KV-cache size formula of the same page, section 1.3.
- ``prefix_cache.py``: the block hash chain prefix cache of the same page,
  sections 4.2 and 4.3.
- ``oracle.c`` also holds the KV pack/unpack staging layout for the
  prefill -> decode hand-over.

Parity pins for every function here live in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .block_manager import BlockManager, Sequence  # noqa: F401
from .prefix_cache import PrefixCache, block_key  # noqa: F401
from .kv_bytes import concurrency_limit, kv_cache_bytes, pd_transfer_bytes  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F16, BF16 = 0, 1
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc (plain C, float64)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                    "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp,
                    "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def swap_library(path: str | None):
    """Point the wrappers at another build of oracle.c (the mutation tests plant
    mistakes in a copy); ``None`` restores the normal build.  Returns the
    previous library object."""
    global _lib
    with _lock:
        prev = _lib
        _lib = _bind(ctypes.CDLL(path)) if path else None
        return prev


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.orc_to_double.restype = dbl
    lib.orc_to_double.argtypes = [ctypes.c_uint16, i32]
    lib.orc_to_double_array.restype = None
    lib.orc_to_double_array.argtypes = [P, P, i64, i32]
    lib.orc_slot_of.restype = i64
    lib.orc_slot_of.argtypes = [P, i64, i32]
    lib.orc_reshape_and_cache.restype = i32
    lib.orc_reshape_and_cache.argtypes = [P, P, P, P, P, i32, i32, i32, i32,
                                          i32, i64, i64]
    lib.orc_copy_blocks.restype = i32
    lib.orc_copy_blocks.argtypes = [P, P, i32, P, i32, i32, i32, i32, i32]
    lib.orc_kv_pack.restype = i32
    lib.orc_kv_pack.argtypes = [i32, P, P, P, i32, P, i32, i32, i32, i32, i32]
    lib.orc_e4m3_to_double.restype = dbl
    lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_encode.restype = ctypes.c_uint8
    lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
    lib.orc_reshape_and_cache_fp8.restype = i32
    lib.orc_reshape_and_cache_fp8.argtypes = [P, P, i32, P, P, P, i32, i32, i32, i32, i32, P, P]
    lib.orc_decode_fp8.restype = i32
    lib.orc_decode_fp8.argtypes = [P, P, i32, P, P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                   dbl, i64, i64]
    lib.orc_decode.restype = i32
    lib.orc_decode.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32,
                               i32, i32, dbl, i32, i64, i64]
    lib.orc_decode_split.restype = i32
    lib.orc_decode_split.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32,
                                     i32, i32, i32, dbl, i32, i32, i64, i64]
    lib.orc_prefill.restype = i32
    lib.orc_prefill.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32,
                                i32, i32, i32, dbl, i32, P, i64]
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    """A C-contiguous uint16 view of fp16/bf16 data (numpy array or CPU torch tensor)."""
    if hasattr(a, "detach"):  # torch tensor: reinterpret the 16-bit payload
        import torch
        a = a.detach().contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(a)
    assert a.itemsize == 2, "expected 16-bit float payload"
    return a.view(np.uint16)


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().contiguous().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _i64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().contiguous().numpy()
    return np.ascontiguousarray(a, dtype=np.int64)


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def to_double(a, dtype: int) -> np.ndarray:
    """Exact fp16/bf16 -> float64 conversion, decoded from the bit fields."""
    src = _u16(a)
    out = np.empty(src.shape, dtype=np.float64)
    _load().orc_to_double_array(_ptr(src), _ptr(out), src.size, dtype)
    return out


def slot_of(block_table_row, t: int, S: int) -> int:
    row = _i32(block_table_row)
    return int(_load().orc_slot_of(_ptr(row), t, S))


def reshape_and_cache(key, value, key_cache: np.ndarray, value_cache: np.ndarray,
                      slot_mapping, S: int) -> int:
    """In place on the uint16 cache arrays [NB, Hk, S, D].  key/value are [T, Hk, D]
    (token stride Hk*D).  Returns the count of out-of-range slots skipped."""
    k, v = _u16(key), _u16(value)
    sm = _i64(slot_mapping)
    assert key_cache.dtype == np.uint16 and key_cache.flags.c_contiguous
    assert value_cache.dtype == np.uint16 and value_cache.flags.c_contiguous
    NB, Hk, S2, D = key_cache.shape
    assert S2 == S
    T = sm.shape[0]
    return _load().orc_reshape_and_cache(_ptr(k), _ptr(v), _ptr(key_cache),
                                         _ptr(value_cache), _ptr(sm), T, Hk, D,
                                         S, NB, Hk * D, Hk * D)


def copy_blocks(key_caches: list, value_caches: list, block_mapping) -> int:
    """In place on lists of uint16 cache arrays (one per layer)."""
    bm = _i64(block_mapping).reshape(-1, 2)
    L = len(key_caches)
    NB, Hk, S, D = key_caches[0].shape
    kp = (ctypes.c_void_p * L)(*[_ptr(c) for c in key_caches])
    vp = (ctypes.c_void_p * L)(*[_ptr(c) for c in value_caches])
    return _load().orc_copy_blocks(kp, vp, L, _ptr(bm), bm.shape[0], Hk, D, S, NB)


def kv_pack(key_caches: list, value_caches: list, block_ids) -> tuple[np.ndarray, int]:
    """Staging buffer [L][2][nblk][Hk][S][D] (uint16) gathered from the pools, and
    the number of skipped (out-of-range) ids."""
    ids = np.ascontiguousarray(np.asarray(block_ids, dtype=np.int32))
    L = len(key_caches)
    NB, Hk, S, D = key_caches[0].shape
    st = np.zeros((L, 2, ids.shape[0], Hk, S, D), dtype=np.uint16)
    kp = (ctypes.c_void_p * L)(*[_ptr(c) for c in key_caches])
    vp = (ctypes.c_void_p * L)(*[_ptr(c) for c in value_caches])
    bad = _load().orc_kv_pack(0, _ptr(st), kp, vp, L, _ptr(ids), ids.shape[0], Hk, D, S, NB)
    return st, bad


def kv_unpack(staging: np.ndarray, key_caches: list, value_caches: list, block_ids) -> int:
    """In place: scatter a staging buffer into the pools' blocks ``block_ids``."""
    ids = np.ascontiguousarray(np.asarray(block_ids, dtype=np.int32))
    st = np.ascontiguousarray(staging, dtype=np.uint16)
    L = len(key_caches)
    NB, Hk, S, D = key_caches[0].shape
    kp = (ctypes.c_void_p * L)(*[_ptr(c) for c in key_caches])
    vp = (ctypes.c_void_p * L)(*[_ptr(c) for c in value_caches])
    return _load().orc_kv_pack(1, _ptr(st), kp, vp, L, _ptr(ids), ids.shape[0], Hk, D, S, NB)


def e4m3_to_double(code: int) -> float:
    return float(_load().orc_e4m3_to_double(int(code) & 0xFF))


def e4m3_encode(y: float) -> int:
    """Nearest E4M3 code of a float32 value (ties to even, saturating at 448)."""
    return int(_load().orc_e4m3_encode(float(np.float32(y))))


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _u8(a) -> np.ndarray:
    if hasattr(a, "detach"):
        import torch
        a = a.detach().contiguous().view(torch.uint8).numpy()
    return np.ascontiguousarray(a, dtype=np.uint8)


def reshape_and_cache_fp8(key, value, dtype: int, key_cache: np.ndarray,
                          value_cache: np.ndarray, slot_mapping, k_scale, v_scale,
                          S: int) -> int:
    """In place on uint8 pools [NB, Hk, S, D]; key/value are fp16/bf16 [T, Hk, D]."""
    k, v = _u16(key), _u16(value)
    T, Hk, D = k.shape
    sm = _i64(slot_mapping)
    ks, vs = _f32(k_scale), _f32(v_scale)
    NB = key_cache.shape[0]
    return _load().orc_reshape_and_cache_fp8(_ptr(k), _ptr(v), dtype, _ptr(key_cache),
                                             _ptr(value_cache), _ptr(sm), T, Hk, D, S, NB,
                                             _ptr(ks), _ptr(vs))


def decode_fp8(q, qdtype: int, key_cache, value_cache, k_scale, v_scale, block_tables,
               context_lens, scale: float, threads: int | None = None,
               rows: tuple[int, int] | None = None) -> np.ndarray:
    """Decode attention over FP8 pools in float64 -> [B, H, D] (or the row range)."""
    qa = _u16(q)
    B, H, D = qa.shape
    kc, vc = _u8(key_cache), _u8(value_cache)
    NB, Hk, S, _ = kc.shape
    bt, cl = _i32(block_tables), _i32(context_lens)
    ks, vs = _f32(k_scale), _f32(v_scale)
    r0, r1 = rows if rows is not None else (0, B * H)
    out = np.zeros((B * H, D), dtype=np.float64)
    lib = _load()

    def work(a, b):
        return lib.orc_decode_fp8(_ptr(out), _ptr(qa), qdtype, _ptr(kc), _ptr(vc), _ptr(ks),
                                  _ptr(vs), _ptr(bt), bt.shape[1], _ptr(cl), H, Hk, D, S, NB,
                                  float(scale), a, b)
    bad = _run_rows(lambda a, b: work(r0 + a, r0 + b), r1 - r0, threads or os.cpu_count() or 1)
    if bad:
        raise ValueError(f"{bad} rows named a block outside the pool")
    res = out[r0:r1]
    return res.reshape(B, H, D) if rows is None else res


def _run_rows(fn, nrows: int, threads: int):
    threads = max(1, min(threads, nrows))
    if threads == 1:
        return fn(0, nrows)
    bounds = np.linspace(0, nrows, threads + 1).astype(np.int64)
    with ThreadPoolExecutor(threads) as ex:  # ctypes drops the GIL in C
        futs = [ex.submit(fn, int(bounds[t]), int(bounds[t + 1]))
                for t in range(threads) if bounds[t + 1] > bounds[t]]
        return sum(f.result() for f in futs)


def decode(q, key_cache, value_cache, block_tables, context_lens, scale: float,
           dtype: int, threads: int | None = None, split_part: int | None = None,
           rows: tuple[int, int] | None = None) -> np.ndarray:
    """Decode attention in float64 -> [B, H, D].  With ``split_part`` the split
    partition + merge formulation is used instead of the plain softmax.
    ``rows`` = (begin, end) restricts the flattened (seq, head) rows computed
    (others stay zero)."""
    qa = _u16(q)
    B, H, D = qa.shape
    kc, vc = _u16(key_cache), _u16(value_cache)
    NB, Hk, S, D2 = kc.shape
    assert D2 == D and H % Hk == 0
    bt, cl = _i32(block_tables), _i32(context_lens)
    out = np.zeros((B, H, D), dtype=np.float64)
    lib = _load()
    r0, r1 = rows if rows is not None else (0, B * H)

    def fn(a, b):
        a, b = a + r0, b + r0
        if split_part is None:
            return lib.orc_decode(_ptr(out), _ptr(qa), _ptr(kc), _ptr(vc), _ptr(bt),
                                  bt.shape[1], _ptr(cl), B, H, Hk, D, S, NB, scale,
                                  dtype, a, b)
        return lib.orc_decode_split(_ptr(out), _ptr(qa), _ptr(kc), _ptr(vc),
                                    _ptr(bt), bt.shape[1], _ptr(cl), B, H, Hk, D,
                                    S, NB, scale, dtype, split_part, a, b)

    bad = _run_rows(fn, r1 - r0, threads or default_threads())
    if bad:
        raise ValueError(f"oracle decode: {bad} rows reference blocks outside the pool")
    return out


def prefill(q, cu_q_lens, key_cache, value_cache, block_tables, context_lens,
            scale: float, dtype: int, rows=None, threads: int | None = None) -> np.ndarray:
    """Chunked-prefill attention in float64.  q is packed [sumC, H, D].  With
    ``rows`` (flattened tok*H + h indices) only those rows are computed and the
    result is [len(rows), D]; otherwise the full [sumC, H, D]."""
    qa = _u16(q)
    NT, H, D = qa.shape
    kc, vc = _u16(key_cache), _u16(value_cache)
    NB, Hk, S, _ = kc.shape
    cu, bt, cl = _i32(cu_q_lens), _i32(block_tables), _i32(context_lens)
    B = cu.shape[0] - 1
    full = rows is None
    r = np.arange(NT * H, dtype=np.int64) if full else _i64(rows)
    out = np.zeros((r.shape[0], D), dtype=np.float64)
    lib = _load()

    def fn(a, b):
        return lib.orc_prefill(_ptr(out) + a * D * 8, _ptr(qa), _ptr(cu), _ptr(kc),
                               _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cl), B, H, Hk,
                               D, S, NB, scale, dtype, _ptr(r) + a * 8, b - a)

    bad = _run_rows(fn, r.shape[0], threads or default_threads())
    if bad:
        raise ValueError(f"oracle prefill: {bad} bad rows")
    return out.reshape(NT, H, D) if full else out
