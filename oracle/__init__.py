"""fp64 CPU oracle for fp8 paged decode attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package. The CUDA
product path never imports, links or calls it, and this package never imports
the product package: the two share no code.

The arithmetic lives in ``pda_oracle.cpp`` (plain C++, binary64, one OpenMP
loop over (sequence, head) rows). This module only compiles that file with
``g++`` and marshals numpy arrays of raw bit patterns into it.

Inputs are raw bit patterns so that nothing here depends on how any other
library decodes fp8 or bf16:

* ``q``            uint16 ``[S, H, D]``      bfloat16 bits
* ``k_cache``      uint8  ``[NB, Hk, D/16, bs, 16]`` OCP e4m3 bytes
* ``v_cache``      uint8  ``[NB, Hk, D, bs]``        OCP e4m3 bytes
* ``block_tables`` int32  ``[S, MB]``
* ``seq_lens``     int32  ``[S]``
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pda_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "libpda_oracle.so")
_lock = threading.Lock()
_lib = None

STATUS = {
    0: "ok",
    -1: "bad shape",
    -2: "bad seq_len",
    -3: "bad block id",
    -4: "bad seq id",
}


class OracleError(RuntimeError):
    pass


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with g++ (OpenMP) into a shared library; returns its path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-shared", "-fPIC", src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) and return the ctypes library handle."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
        return _lib


def _bind(lib):
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_longlong, ctypes.c_double
    lib.pda_oracle_decode.restype = i32
    lib.pda_oracle_decode.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i64,
                                      f64, f64, f64, P, P, P, i32, P, i32, i32]
    lib.pda_oracle_quantize_e4m3.restype = None
    lib.pda_oracle_quantize_e4m3.argtypes = [P, P, i64, f64]
    lib.pda_oracle_e4m3_value.restype = f64
    lib.pda_oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.pda_oracle_bf16_value.restype = f64
    lib.pda_oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.pda_oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.pda_oracle_e4m3_encode.argtypes = [f64]
    lib.pda_oracle_reshape_and_cache.restype = i32
    lib.pda_oracle_reshape_and_cache.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i64, ctypes.c_float,
                                                 ctypes.c_float, i32]
    lib.pda_oracle_max_threads.restype = i32
    lib.pda_oracle_max_threads.argtypes = []
    return lib


def e4m3_value(code: int) -> float:
    return load().pda_oracle_e4m3_value(int(code) & 0xFF)


def bf16_value(bits: int) -> float:
    return load().pda_oracle_bf16_value(int(bits) & 0xFFFF)


def max_threads() -> int:
    return load().pda_oracle_max_threads()


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError("expected %s array, got %s" % (np.dtype(dtype), a.dtype))
    return a


def decode(q, k_cache, v_cache, block_tables, seq_lens, *, scale: float, k_scale: float = 1.0,
           v_scale: float = 1.0, k_scales=None, v_scales=None, sinks=None, v_shuffled: bool = False,
           num_blocks: int | None = None, seq_ids=None, num_threads: int = 0, lib=None) -> np.ndarray:
    """Exact (binary64) decode attention; returns float64 ``[n, H, D]``.

    ``seq_ids`` selects a subset of sequences (rows of the result follow its
    order); ``None`` computes every sequence. ``k_scales`` / ``v_scales``
    (float32 ``[NB, Hk, bs]``) replace the per-tensor scales slot by slot.
    ``sinks`` (float32 ``[H]``) adds one value-less logit per head to the
    softmax normaliser. ``v_shuffled``: ``v_cache`` is ``[NB, Hk, bs/16, D, 16]``.
    """
    q = _c(q, np.uint16)
    k_cache = _c(k_cache, np.uint8)
    v_cache = _c(v_cache, np.uint8)
    block_tables = _c(block_tables, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    S, H, D = q.shape
    NB, Hk, D16, bs, sixteen = k_cache.shape
    v_want = (NB, Hk, bs // 16, D, 16) if v_shuffled else (NB, Hk, D, bs)
    if sixteen != 16 or D16 * 16 != D or v_cache.shape != v_want:
        raise OracleError("cache shapes do not match q: k %s v %s q %s" % (k_cache.shape, v_cache.shape, q.shape))
    if block_tables.ndim != 2 or block_tables.shape[0] != S or seq_lens.shape != (S,):
        raise OracleError("table shapes do not match q")
    MB = block_tables.shape[1]
    if num_blocks is None:
        num_blocks = NB
    ids_p = None
    n = S
    if seq_ids is not None:
        seq_ids = _c(np.asarray(seq_ids, dtype=np.int32), np.int32)
        ids_p = seq_ids.ctypes.data
        n = int(seq_ids.shape[0])
    ks_p = vs_p = None
    if k_scales is not None or v_scales is not None:
        k_scales = _c(k_scales, np.float32)
        v_scales = _c(v_scales, np.float32)
        if k_scales.shape != (NB, Hk, bs) or v_scales.shape != (NB, Hk, bs):
            raise OracleError("scale tables must be [num_blocks, num_kv_heads, block_size]")
        ks_p, vs_p = k_scales.ctypes.data, v_scales.ctypes.data
    sk_p = None
    if sinks is not None:
        sinks = _c(np.asarray(sinks, dtype=np.float32), np.float32)
        if sinks.shape != (H,):
            raise OracleError("sinks must be float32 [num_heads]")
        sk_p = sinks.ctypes.data
    out = np.zeros((n, H, D), dtype=np.float64)
    L = lib if lib is not None else load()
    rc = L.pda_oracle_decode(out.ctypes.data, q.ctypes.data, k_cache.ctypes.data, v_cache.ctypes.data,
                             block_tables.ctypes.data, seq_lens.ctypes.data, S, H, Hk, D, bs, MB,
                             int(num_blocks), float(scale), float(k_scale), float(v_scale), ks_p, vs_p, sk_p,
                             1 if v_shuffled else 0, ids_p, n, int(num_threads))
    if rc != 0:
        raise OracleError("oracle rejected the inputs: %s (%d)" % (STATUS.get(rc, "?"), rc))
    return out


def e4m3_encode(x: float, lib=None) -> int:
    return (lib or load()).pda_oracle_e4m3_encode(float(x))


def reshape_and_cache(k_cache, v_cache, key, value, slot_mapping, *, k_scale: float, v_scale: float,
                      v_shuffled: bool = False, lib=None) -> None:
    """Quantise and scatter new tokens into the paged caches, in place.

    key / value: uint16 bf16 bits ``[T, Hk, D]``; slot_mapping: int64 ``[T]``
    (negative = skip); caches: uint8 arrays as for ``decode`` (modified).
    """
    for a, dt in ((k_cache, np.uint8), (v_cache, np.uint8)):
        if a.dtype != dt or not a.flags["C_CONTIGUOUS"]:
            raise TypeError("caches must be C-contiguous uint8 arrays")
    key = _c(key, np.uint16)
    value = _c(value, np.uint16)
    slot_mapping = _c(slot_mapping, np.int64)
    T, Hk, D = key.shape
    NB, Hk2, D16, bs, sixteen = k_cache.shape
    v_want = (NB, Hk, bs // 16, D, 16) if v_shuffled else (NB, Hk, D, bs)
    if value.shape != key.shape or Hk2 != Hk or D16 * 16 != D or v_cache.shape != v_want:
        raise OracleError("shapes do not match")
    L = lib if lib is not None else load()
    rc = L.pda_oracle_reshape_and_cache(k_cache.ctypes.data, v_cache.ctypes.data, key.ctypes.data,
                                        value.ctypes.data, slot_mapping.ctypes.data, T, Hk, D, bs, NB,
                                        float(k_scale), float(v_scale), 1 if v_shuffled else 0)
    if rc != 0:
        raise OracleError("oracle rejected the inputs: %s (%d)" % (STATUS.get(rc, "?"), rc))


def quantize_e4m3(x, output_scale: float, lib=None) -> np.ndarray:
    """Static per-tensor fp8 output quantisation: E4M3(x / output_scale) codes (uint8)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    codes = np.zeros(x.shape, dtype=np.uint8)
    (lib or load()).pda_oracle_quantize_e4m3(x.ctypes.data, codes.ctypes.data, x.size, float(output_scale))
    return codes
