"""ctypes binding of the C ABI declared in ``include/pda.h``.

Argument marshalling only: tensors become device pointers and sizes, and
every step of the computation runs in the library's CUDA kernels. The shared
library ``libpda.so`` is built in-tree (``paged_kv_decode_pda_gb300.build``);
if it is missing the first call raises ``PdaError`` -- there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpda.so")

PDA_OK = 0
PDA_ERR_INVALID_ARG = 1
PDA_ERR_UNSUPPORTED = 2
PDA_ERR_WORKSPACE = 3
PDA_ERR_CUDA = 4
PDA_ERR_DEVICE_TIMEOUT = 5
PDA_ERR_NOALLOC_CAPACITY = 6

# Functions (name -> (restype, argtypes)) the header declares.
_P, _I, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
SIGNATURES = {
    "pda_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _F, _P]),
    "pda_status_string": (ctypes.c_char_p, [_I]),
    "pda_choose_splits": (_I, [_I, _I, _I, _I, _I, _I]),
    "pda_plan_splits": (_I, [_I, _I, _I, _I, _I]),
    "pda_plan_kernel": (_I, [_I, _I, _I, _I, _I]),
    "pda_plan_launches": (_I, [_I, _I, _I, _I, _I]),
    "pda_plan_slot_scales": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "pda_tail_pieces": (_I, [_I, _I, _I, _I, ctypes.POINTER(_I), _I]),
    "pda_choose_kernel": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "pda_set_split_override": (None, [_I]),
    "pda_set_tail_split": (None, [_I]),
    "pda_set_tma_gather": (None, [_I]),
    "pda_set_block_check": (None, [ctypes.c_longlong]),
    "pda_reserve": (_I, [_I, _I, _I, _I, _I, _P]),
    "pda_release": (_I, []),
    "pda_workspace_info": (_I, [_P, ctypes.POINTER(ctypes.c_longlong), ctypes.POINTER(_I)]),
    "pda_query_device_status": (_I, [_P, ctypes.POINTER(ctypes.c_int)]),
    "pda_set_profile_events": (None, [_P, _P]),
    "pda_test_bounded_wait": (_I, [_I, _P]),
    "pda_reshape_and_cache": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_longlong, _F, _F, _I, _P]),
    "pda_decode_slot_scales": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "pda_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _F, _P]),
    "pda_decode_host": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_longlong, _F, _F, _F, _P]),
    "pda_decode_ex": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _F, _F, _I, _P, _I, _F, _P]),
    "pda_decode_strided": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I] + [ctypes.c_longlong] * 7
                           + [_F, _F, _F, _P]),
}

PDA_OUT_BF16 = 0
PDA_OUT_E4M3 = 1
PDA_KV_NATIVE = 0
PDA_KV_SHUFFLED_V = 1

_lock = threading.RLock()
_lib = None


class PdaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what or "pda", status_string(status), status))


def load(path: str | None = None):
    """Load libpda.so (once) and bind every declared entry point."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise PdaError(PDA_ERR_CUDA, "libpda.so not built at %s (run paged_kv_decode_pda_gb300.build.build())" % p)
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    if _lib is None:
        return _STATUS_TEXT.get(int(status), "unknown status")
    return _lib.pda_status_string(int(status)).decode()


_STATUS_TEXT = {PDA_OK: "ok", PDA_ERR_INVALID_ARG: "invalid argument", PDA_ERR_UNSUPPORTED: "unsupported configuration",
                PDA_ERR_WORKSPACE: "workspace must grow during stream capture", PDA_ERR_CUDA: "CUDA runtime error",
                PDA_ERR_DEVICE_TIMEOUT: "a kernel gave up on a bounded wait",
                PDA_ERR_NOALLOC_CAPACITY: "the call needs more split scratch than the static buffer holds"}


def _check(status: int, what: str):
    if status != PDA_OK:
        raise PdaError(status, what)


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return int(stream.cuda_stream)
    return int(stream)


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
           seq_lens: torch.Tensor, scale: float, k_scale: float, v_scale: float, *,
           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Decode attention over a paged fp8 cache (``pda_decode``).

    q ``[S, H, 128]`` bf16; k_cache ``[NB, Hk, 8, bs, 16]`` and v_cache
    ``[NB, Hk, 128, bs]`` float8_e4m3fn (or uint8 bytes); block_tables
    ``[S, MB]`` int32; seq_lens ``[S]`` int32; all contiguous on one CUDA
    device. Returns ``out`` (allocated like q when not given).
    """
    lib = load()
    _check_decode_args(q, k_cache, v_cache, block_tables, seq_lens)
    out = _out_like(q, out)
    S, H, D = q.shape
    NB, Hk, D16, bs, sixteen = k_cache.shape
    st = lib.pda_decode(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                        block_tables.data_ptr(), seq_lens.data_ptr(), S, H, Hk, D, bs,
                        int(block_tables.shape[1]), float(scale), float(k_scale), float(v_scale),
                        _stream_ptr(stream))
    _check(st, "pda_decode")
    return out


def _out_like(q, out):
    if out is None:
        return torch.empty_like(q)
    if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous() or not out.is_cuda:
        raise PdaError(PDA_ERR_INVALID_ARG, "decode: out")
    return out


def _check_decode_args(q, k_cache, v_cache, block_tables, seq_lens, v_shuffled=False):
    if (q.dim() != 3 or k_cache.dim() != 5 or v_cache.dim() != (5 if v_shuffled else 4) or block_tables.dim() != 2
            or seq_lens.dim() != 1):
        raise PdaError(PDA_ERR_INVALID_ARG, "decode: tensor ranks")
    if q.dtype != torch.bfloat16 or block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise PdaError(PDA_ERR_INVALID_ARG, "decode: dtypes (q bf16, tables/seq_lens int32)")
    for t in (k_cache, v_cache):
        if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise PdaError(PDA_ERR_INVALID_ARG, "decode: cache dtype must be float8_e4m3fn")
    ts = [q, k_cache, v_cache, block_tables, seq_lens]
    if not all(t.is_cuda and t.is_contiguous() for t in ts):
        raise PdaError(PDA_ERR_INVALID_ARG, "decode: tensors must be contiguous CUDA tensors")
    S, H, D = q.shape
    NB, Hk, D16, bs, sixteen = k_cache.shape
    v_want = (NB, Hk, bs // 16, D, 16) if v_shuffled else (NB, Hk, D, bs)
    if (sixteen != 16 or D16 * 16 != D or tuple(v_cache.shape) != v_want
            or block_tables.shape[0] != S or seq_lens.shape[0] != S):
        raise PdaError(PDA_ERR_INVALID_ARG, "decode: shapes")


def decode_slot_scales(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, k_scales: torch.Tensor,
                       v_scales: torch.Tensor, block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float, *,
                       out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """``pda_decode_slot_scales``: decode with per-slot fp32 scale tables ``[NB, Hk, bs]``."""
    lib = load()
    _check_decode_args(q, k_cache, v_cache, block_tables, seq_lens)
    NB, Hk, _, bs, _ = k_cache.shape
    for t in (k_scales, v_scales):
        if t.dtype != torch.float32 or tuple(t.shape) != (NB, Hk, bs) or not t.is_cuda or not t.is_contiguous():
            raise PdaError(PDA_ERR_INVALID_ARG, "decode_slot_scales: scale tables must be fp32 [NB, Hk, bs]")
    out = _out_like(q, out)
    S, H, D = q.shape
    st = lib.pda_decode_slot_scales(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                    k_scales.data_ptr(), v_scales.data_ptr(), block_tables.data_ptr(),
                                    seq_lens.data_ptr(), S, H, Hk, D, bs, int(block_tables.shape[1]), float(scale),
                                    _stream_ptr(stream))
    _check(st, "pda_decode_slot_scales")
    return out


def decode_ex(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
              seq_lens: torch.Tensor, scale: float, k_scale: float, v_scale: float, *, sinks=None,
              output_scale: float | None = None, v_shuffled: bool = False, out: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """``pda_decode_ex``: decode with optional per-head sinks (fp32 ``[H]``),
    e4m3 output ``E4M3(o / output_scale)`` when ``output_scale`` is given, and
    the shuffled V layout ``[NB, Hk, bs/16, 128, 16]`` when ``v_shuffled``."""
    lib = load()
    _check_decode_args(q, k_cache, v_cache, block_tables, seq_lens, v_shuffled)
    S, H, D = q.shape
    NB, Hk, _, bs, _ = k_cache.shape
    if sinks is not None and (sinks.dtype != torch.float32 or tuple(sinks.shape) != (H,) or not sinks.is_cuda):
        raise PdaError(PDA_ERR_INVALID_ARG, "decode_ex: sinks must be a CUDA float32 [num_heads] tensor")
    fp8 = output_scale is not None
    want = torch.float8_e4m3fn if fp8 else torch.bfloat16
    if out is None:
        out = torch.empty(q.shape, dtype=want, device=q.device)
    elif out.shape != q.shape or out.dtype not in ((want, torch.uint8) if fp8 else (want,)) or not out.is_contiguous():
        raise PdaError(PDA_ERR_INVALID_ARG, "decode_ex: out")
    st = lib.pda_decode_ex(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                           block_tables.data_ptr(), seq_lens.data_ptr(), S, H, Hk, D, bs, int(block_tables.shape[1]),
                           float(scale), float(k_scale), float(v_scale),
                           PDA_KV_SHUFFLED_V if v_shuffled else PDA_KV_NATIVE,
                           sinks.data_ptr() if sinks is not None else None,
                           PDA_OUT_E4M3 if fp8 else PDA_OUT_BF16, float(output_scale) if fp8 else 1.0,
                           _stream_ptr(stream))
    _check(st, "pda_decode_ex")
    return out


def decode_strided(q: torch.Tensor, k_rows_base: int, v_rows_base: int, block_tables: torch.Tensor,
                   seq_lens: torch.Tensor, scale: float, k_scale: float, v_scale: float, *, num_kv_heads: int,
                   block_size: int, num_blocks: int, k_strides, v_strides, out: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """``pda_decode_strided``: decode on a token-major fp8 cache.

    ``k_rows_base`` / ``v_rows_base`` are device addresses of the (block 0,
    token 0, head 0) rows; ``k_strides`` / ``v_strides`` are byte strides
    (block, token, kv head); every row holds 128 contiguous e4m3 bytes.
    """
    lib = load()
    if q.dim() != 3 or q.dtype != torch.bfloat16 or not q.is_cuda or not q.is_contiguous():
        raise PdaError(PDA_ERR_INVALID_ARG, "decode_strided: q")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise PdaError(PDA_ERR_INVALID_ARG, "decode_strided: tables / seq_lens dtype")
    out = _out_like(q, out)
    S, H, D = q.shape
    kb, kt, kh = (int(x) for x in k_strides)
    vb, vt, vh = (int(x) for x in v_strides)
    st = lib.pda_decode_strided(out.data_ptr(), q.data_ptr(), int(k_rows_base), int(v_rows_base),
                                block_tables.data_ptr(), seq_lens.data_ptr(), S, H, int(num_kv_heads), D,
                                int(block_size), int(block_tables.shape[1]), int(num_blocks), kb, kt, kh, vb, vt, vh,
                                float(scale), float(k_scale), float(v_scale), _stream_ptr(stream))
    _check(st, "pda_decode_strided")
    return out


def decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                   seq_lens: torch.Tensor, scale: float, k_scale: float, v_scale: float, *, out: torch.Tensor,
                   stream=None) -> torch.Tensor:
    """``pda_decode_noalloc``: ``decode`` without any device allocation.

    The output buffer must be given (nothing is allocated here either); the
    library keeps split partials in its fixed 16 MiB device array.
    """
    lib = load()
    _check_decode_args(q, k_cache, v_cache, block_tables, seq_lens)
    if out is None:
        raise PdaError(PDA_ERR_INVALID_ARG, "decode_noalloc: out must be given")
    out = _out_like(q, out)
    S, H, D = q.shape
    NB, Hk, _, bs, _ = k_cache.shape
    st = lib.pda_decode_noalloc(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                block_tables.data_ptr(), seq_lens.data_ptr(), S, H, Hk, D, bs,
                                int(block_tables.shape[1]), float(scale), float(k_scale), float(v_scale),
                                _stream_ptr(stream))
    _check(st, "pda_decode_noalloc")
    return out


def decode_host(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                seq_lens: torch.Tensor, scale: float, k_scale: float, v_scale: float, *, out: torch.Tensor,
                stream=None) -> torch.Tensor:
    """``pda_decode_host``: ``decode`` on CPU tensors (pinned for asynchronous copies).

    Shapes and dtypes as ``decode``; every tensor, ``out`` included, is a
    contiguous CPU tensor. The call enqueues the copies in, the decode and
    the copy out on ``stream`` and returns: synchronise the stream before
    reading ``out``, and keep the inputs unchanged until then.
    """
    lib = load()
    if (q.dim() != 3 or k_cache.dim() != 5 or v_cache.dim() != 4 or block_tables.dim() != 2
            or seq_lens.dim() != 1):
        raise PdaError(PDA_ERR_INVALID_ARG, "decode_host: tensor ranks")
    if q.dtype != torch.bfloat16 or block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise PdaError(PDA_ERR_INVALID_ARG, "decode_host: dtypes (q bf16, tables/seq_lens int32)")
    if any(t.dtype not in (torch.float8_e4m3fn, torch.uint8) for t in (k_cache, v_cache)):
        raise PdaError(PDA_ERR_INVALID_ARG, "decode_host: cache dtype must be float8_e4m3fn")
    if out is None or out.shape != q.shape or out.dtype != torch.bfloat16:
        raise PdaError(PDA_ERR_INVALID_ARG, "decode_host: out must be given, shaped and typed like q")
    ts = [out, q, k_cache, v_cache, block_tables, seq_lens]
    if any(t.is_cuda or not t.is_contiguous() for t in ts):
        raise PdaError(PDA_ERR_INVALID_ARG, "decode_host: tensors must be contiguous CPU tensors")
    S, H, D = q.shape
    NB, Hk, D16, bs, sixteen = k_cache.shape
    if (sixteen != 16 or D16 * 16 != D or tuple(v_cache.shape) != (NB, Hk, D, bs) or block_tables.shape[0] != S
            or seq_lens.shape[0] != S):
        raise PdaError(PDA_ERR_INVALID_ARG, "decode_host: shapes")
    st = lib.pda_decode_host(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                             block_tables.data_ptr(), seq_lens.data_ptr(), S, H, Hk, D, bs,
                             int(block_tables.shape[1]), NB, float(scale), float(k_scale), float(v_scale),
                             _stream_ptr(stream))
    _check(st, "pda_decode_host")
    return out


def decode_raw(out_ptr: int, q_ptr: int, k_ptr: int, v_ptr: int, tables_ptr: int, lens_ptr: int, num_seqs: int,
               num_heads: int, num_kv_heads: int, head_size: int, block_size: int, max_num_blocks_per_seq: int,
               scale: float, k_scale: float, v_scale: float, stream_ptr: int = 0) -> int:
    """``pda_decode`` on raw device addresses; returns the status code."""
    return load().pda_decode(out_ptr, q_ptr, k_ptr, v_ptr, tables_ptr, lens_ptr, num_seqs, num_heads,
                             num_kv_heads, head_size, block_size, max_num_blocks_per_seq, float(scale),
                             float(k_scale), float(v_scale), stream_ptr)


def choose_splits(num_seqs, num_kv_heads, max_num_blocks_per_seq, block_size, sm_count, ctas_per_sm) -> int:
    return load().pda_choose_splits(num_seqs, num_kv_heads, max_num_blocks_per_seq, block_size, sm_count,
                                    ctas_per_sm)


def plan_splits(num_seqs, num_heads, num_kv_heads, max_num_blocks_per_seq, block_size) -> int:
    n = load().pda_plan_splits(num_seqs, num_heads, num_kv_heads, max_num_blocks_per_seq, block_size)
    if n < 1:
        raise PdaError(PDA_ERR_CUDA, "pda_plan_splits")
    return n


PDA_KERNEL_PER_UNIT, PDA_KERNEL_PER_UNIT_DENSE, PDA_KERNEL_PERSISTENT = 0, 1, 2
KERNEL_NAMES = {PDA_KERNEL_PER_UNIT: "per-unit (3 CTAs/SM)", PDA_KERNEL_PER_UNIT_DENSE: "per-unit dense (4 CTAs/SM)",
                PDA_KERNEL_PERSISTENT: "persistent"}


def plan_kernel(num_seqs, num_heads, num_kv_heads, max_num_blocks_per_seq, block_size) -> int:
    """The decode kernel instance (PDA_KERNEL_*) pda_decode would launch for these sizes."""
    k = load().pda_plan_kernel(num_seqs, num_heads, num_kv_heads, max_num_blocks_per_seq, block_size)
    if k < 0:
        raise PdaError(PDA_ERR_CUDA, "pda_plan_kernel")
    return k


def choose_kernel(num_seqs, num_kv_heads, max_num_blocks_per_seq, block_size, sm_count, ctas_per_sm,
                  ctas_per_sm_dense) -> tuple[int, int, int]:
    """The planner's pure choice: (PDA_KERNEL_* instance, split count, launches per call)."""
    ns, nl = ctypes.c_int(0), ctypes.c_int(0)
    k = load().pda_choose_kernel(num_seqs, num_kv_heads, max_num_blocks_per_seq, block_size, sm_count, ctas_per_sm,
                                 ctas_per_sm_dense, ctypes.byref(ns), ctypes.byref(nl))
    if k < 0:
        raise PdaError(PDA_ERR_INVALID_ARG, "pda_choose_kernel")
    return k, ns.value, nl.value


def plan_launches(num_seqs, num_heads, num_kv_heads, max_num_blocks_per_seq, block_size) -> int:
    """Kernels one pda_decode call launches for these sizes."""
    n = load().pda_plan_launches(num_seqs, num_heads, num_kv_heads, max_num_blocks_per_seq, block_size)
    if n < 0:
        raise PdaError(PDA_ERR_CUDA, "pda_plan_launches")
    return n


def plan_slot_scales(num_seqs, num_heads, num_kv_heads, max_num_blocks_per_seq, block_size) -> tuple[int, int, int]:
    """The plan of a pda_decode_slot_scales call: (PDA_KERNEL_* instance, split count, launches per call)."""
    k, ns, nl = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    if load().pda_plan_slot_scales(num_seqs, num_heads, num_kv_heads, max_num_blocks_per_seq, block_size,
                                   ctypes.byref(k), ctypes.byref(ns), ctypes.byref(nl)) != 0:
        raise PdaError(PDA_ERR_CUDA, "pda_plan_slot_scales")
    return k.value, ns.value, nl.value


def tail_pieces(pages: int, tail_units: int, ctas: int, block_size: int) -> list[int]:
    """``pda_tail_pieces``: the piece sizes (pages) a tail unit of ``pages`` pages is cut into."""
    buf = (_I * 8)()
    n = load().pda_tail_pieces(pages, tail_units, ctas, block_size, buf, 8)
    if n < 0:
        raise PdaError(PDA_ERR_INVALID_ARG, "pda_tail_pieces")
    return [buf[i] for i in range(n)]


def set_split_override(n: int) -> None:
    load().pda_set_split_override(int(n))


def set_tail_split(enable: bool) -> None:
    """``pda_set_tail_split``: tail pieces of the persistent kernel on (default) or off."""
    load().pda_set_tail_split(1 if enable else 0)


def set_tma_gather(enable: bool) -> None:
    """``pda_set_tma_gather``: four-row TMA gathers of pages and scale rows on (default) or off."""
    load().pda_set_tma_gather(1 if enable else 0)


def set_block_check(num_blocks: int) -> None:
    """``pda_set_block_check``: check decode block ids against [0, num_blocks) on the device (0 = off)."""
    load().pda_set_block_check(int(num_blocks))


def reserve(num_seqs, num_heads, num_kv_heads, max_num_blocks_per_seq, block_size, stream=None) -> None:
    _check(load().pda_reserve(num_seqs, num_heads, num_kv_heads, max_num_blocks_per_seq, block_size,
                              _stream_ptr(stream)), "pda_reserve")


def release() -> None:
    _check(load().pda_release(), "pda_release")


def workspace_info(stream=None) -> tuple[int, int]:
    """``pda_workspace_info``: (current bytes, retired buffers kept alive) of
    the current device's workspace for ``stream``."""
    lib = load()
    nbytes, retired = ctypes.c_longlong(0), _I(0)
    _check(lib.pda_workspace_info(_stream_ptr(stream), ctypes.byref(nbytes), ctypes.byref(retired)),
           "pda_workspace_info")
    return int(nbytes.value), int(retired.value)


def query_device_status(stream=None) -> int:
    code = ctypes.c_int(0)
    st = load().pda_query_device_status(_stream_ptr(stream), ctypes.byref(code))
    if st not in (PDA_OK, PDA_ERR_DEVICE_TIMEOUT):
        raise PdaError(st, "pda_query_device_status")
    return int(code.value)


def set_profile_events(before, after) -> None:
    """Record two torch.cuda.Event around the decode kernel (None, None: off)."""
    if before is None or after is None:
        load().pda_set_profile_events(None, None)
    else:
        for e in (before, after):
            if int(e.cuda_event) == 0:   # torch creates the event on its first record
                e.record()
        load().pda_set_profile_events(int(before.cuda_event), int(after.cuda_event))


def bounded_wait_check(timeout_us: int, stream=None) -> None:
    _check(load().pda_test_bounded_wait(int(timeout_us), _stream_ptr(stream)), "pda_test_bounded_wait")


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      slot_mapping: torch.Tensor, k_scale: float, v_scale: float, *, v_shuffled: bool = False,
                      stream=None) -> None:
    """Quantise and scatter new tokens into the paged fp8 cache (``pda_reshape_and_cache``).

    key / value ``[T, Hk, 128]`` bf16; slot_mapping ``[T]`` int64 (negative =
    skip); caches as for ``decode`` (written in place).
    """
    lib = load()
    if key.dim() != 3 or value.shape != key.shape or key.dtype != torch.bfloat16 or value.dtype != torch.bfloat16:
        raise PdaError(PDA_ERR_INVALID_ARG, "reshape_and_cache: key/value")
    if slot_mapping.dtype != torch.int64 or slot_mapping.shape != (key.shape[0],):
        raise PdaError(PDA_ERR_INVALID_ARG, "reshape_and_cache: slot_mapping")
    for t in (k_cache, v_cache):
        if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise PdaError(PDA_ERR_INVALID_ARG, "reshape_and_cache: cache dtype")
    ts = [key, value, k_cache, v_cache, slot_mapping]
    if not all(t.is_cuda and t.is_contiguous() for t in ts):
        raise PdaError(PDA_ERR_INVALID_ARG, "reshape_and_cache: tensors must be contiguous CUDA tensors")
    T, Hk, D = key.shape
    NB, Hk2, D16, bs, sixteen = k_cache.shape
    v_want = (NB, Hk, bs // 16, D, 16) if v_shuffled else (NB, Hk, D, bs)
    if Hk2 != Hk or D16 * 16 != D or sixteen != 16 or tuple(v_cache.shape) != v_want:
        raise PdaError(PDA_ERR_INVALID_ARG, "reshape_and_cache: shapes")
    _check(lib.pda_reshape_and_cache(key.data_ptr(), value.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                     slot_mapping.data_ptr(), T, Hk, D, bs, NB, float(k_scale), float(v_scale),
                                     PDA_KV_SHUFFLED_V if v_shuffled else PDA_KV_NATIVE, _stream_ptr(stream)),
           "pda_reshape_and_cache")
