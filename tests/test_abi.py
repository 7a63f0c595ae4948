"""C-ABI surface on the CPU: symbols, status strings, heuristic, host validation.

No test here launches a kernel or needs a GPU: every pda_decode call below is
rejected by host-side validation before any CUDA call.
"""

import ctypes
import os
import re

import pytest

import paged_kv_decode_pda_gb300 as pda
from paged_kv_decode_pda_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pda.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pda.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pda_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("pda_decode", "pda_status_string", "pda_choose_splits", "pda_reserve", "pda_release",
                 "pda_query_device_status"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(_binding.SIGNATURES), "binding and header disagree"


def test_status_strings(lib):
    for code in range(7):
        s = lib.pda_status_string(code)
        assert s and s != b"unknown status"
    assert lib.pda_status_string(99) == b"unknown status"


# --------------------------------------------------------------- heuristic

SM, OCC = 152, 3


@pytest.mark.parametrize("S,Hk,MB,bs,expect", [
    (16, 8, 64, 16, 3),       # 128 units < 456 slots: split to fill one wave (3 x 128 <= 456)
    (64, 8, 64, 16, 1),       # 512 units already fill a wave; 256 KiB per unit
    (256, 8, 256, 16, 1),     # 1 MiB per unit, 2048 units
    (256, 8, 250, 16, 1),
    (128, 8, 128, 64, 2),     # 64-token blocks: 2 MiB per unit -> two 1 MiB splits
    (1, 8, 256, 16, 16),      # a single long sequence splits to the 256-token cap
    (1, 1, 2, 16, 1),         # too short to split
    (4, 8, 2048, 16, 14),     # 32 units of 8 MiB: one wave needs 14 splits (cap 128)
])
def test_choose_splits_table(lib, S, Hk, MB, bs, expect):
    assert lib.pda_choose_splits(S, Hk, MB, bs, SM, OCC) == expect


def test_choose_splits_bounds_and_monotonicity(lib):
    for bs in (16, 32, 64, 128):
        for MB in (1, 2, 7, 64, 255, 1000):
            prev = None
            for S in (1, 2, 3, 8, 16, 64, 256, 1024):
                n = lib.pda_choose_splits(S, 8, MB, bs, SM, OCC)
                assert 1 <= n <= max(1, MB)
                # enough tokens per split
                if n > 1:
                    assert MB * bs // n >= 256
                if prev is not None:
                    assert n <= prev, "more sequences must never mean more splits"
                prev = n
                if S * 8 >= SM * OCC and MB * bs * 256 <= (1 << 20):
                    assert n == 1, "a full wave of small units needs no split"


# GB300: 152 SMs, 3 per-unit / persistent CTAs or 4 dense per-unit CTAs per SM
@pytest.mark.parametrize("S,Hk,MB,bs,kind,splits,launches", [
    (16, 8, 64, 16, pda.PDA_KERNEL_PER_UNIT_DENSE, 4, 1),   # 16 x 1024: one wave of 4/SM, 4 splits merged in clusters
    (64, 8, 64, 16, pda.PDA_KERNEL_PER_UNIT_DENSE, 1, 1),   # 64 x 1024: 512 CTAs fit 608 slots
    (256, 8, 256, 16, pda.PDA_KERNEL_PERSISTENT, 1, 3),     # headline: order kernel + persistent + tail merge
    (256, 8, 250, 16, pda.PDA_KERNEL_PERSISTENT, 1, 3),     # ragged up to 4000 tokens
    (128, 8, 128, 64, pda.PDA_KERNEL_PERSISTENT, 2, 4),     # 64-token blocks: + tail merge + merge
    (2200, 8, 8, 16, pda.PDA_KERNEL_PERSISTENT, 1, 1),      # 17,600 units: ticket order, no order kernel
    (76, 8, 8, 16, pda.PDA_KERNEL_PER_UNIT_DENSE, 1, 1),    # 608 units: exactly one dense wave
    (77, 8, 8, 16, pda.PDA_KERNEL_PERSISTENT, 1, 3),        # 616 units: one more than a dense wave
    (65535, 65535, 2, 16, pda.PDA_KERNEL_PER_UNIT, 1, 1),   # past 2^31 units: per-unit kernel
    # long contexts: a few sequences split into page ranges up to a dense wave
    (1, 8, 8192, 16, pda.PDA_KERNEL_PER_UNIT_DENSE, 76, 2),   # 1 x 128K tokens: 608 CTAs + wide merge
    (4, 8, 2048, 16, pda.PDA_KERNEL_PER_UNIT_DENSE, 19, 2),   # 4 x 32K: 19 splits (> 16 for a cluster), wide merge
    (8, 8, 512, 16, pda.PDA_KERNEL_PER_UNIT_DENSE, 9, 1),     # 8 x 8K: 9 splits merged in clusters
    (8, 8, 256, 16, pda.PDA_KERNEL_PER_UNIT_DENSE, 9, 1),     # 8 x 4K: the same split count
    (19, 4, 256, 16, pda.PDA_KERNEL_PER_UNIT_DENSE, 8, 1),    # 76 units x 8 splits fill one wave: clusters of 8
    (1, 1, 64, 16, pda.PDA_KERNEL_PER_UNIT_DENSE, 4, 1),      # 1 x 1K, one kv head: 4 splits (256 tokens each)
    (16, 8, 640, 64, pda.PDA_KERNEL_PERSISTENT, 10, 4),       # 16 x 40,960, 64-token blocks
    (8, 8, 8192, 16, pda.PDA_KERNEL_PERSISTENT, 32, 4),       # 8 x 128K
    (64, 8, 2048, 16, pda.PDA_KERNEL_PERSISTENT, 8, 4),       # 64 x 32K: 1 MiB split units
])
def test_choose_kernel_table(lib, S, Hk, MB, bs, kind, splits, launches):
    assert pda.choose_kernel(S, Hk, MB, bs, 152, 3, 4) == (kind, splits, launches)


# ----------------------------------------------------------- tail pieces

@pytest.mark.parametrize("pages,K,C,bs,want", [
    (256, 224, 456, 16, [126, 64, 32, 17, 17]),   # 256 x 4096 tokens: 224 tail units shrink
    (64, 224, 456, 64, [31, 16, 8, 4, 5]),        # 128 x 8192, 64-token blocks, 2 splits
    (11, 56, 456, 128, [2, 2, 2, 2, 3]),          # a short tail: equal pieces, none empty
    (69, 48, 456, 16, [17, 17, 17, 18]),          # equal pieces of a 69-page unit
    (128, 128, 456, 16, [16] * 8),                # equal pieces at the cap of 8
    (63, 224, 456, 16, [63]),                     # under 1024 tokens: whole
    (0, 224, 456, 16, [0]),                       # an empty split stays whole
])
def test_tail_piece_table(lib, pages, K, C, bs, want):
    assert pda.tail_pieces(pages, K, C, bs) == want


def test_tail_piece_invariants(lib):
    # every cut covers the unit, pieces are never empty, hold at least 256
    # tokens (the last shrinking piece may hold fewer only when the rest is
    # smaller than that), stay within the cap, and shrinking pieces never grow
    # by more than the minimum piece
    for bs in (16, 32, 48, 64, 128):
        m = -(-256 // bs)
        for C in (152, 456, 608):
            for K in (1, 7, C // 4, C // 3, C // 3 + 1, C // 2, C - 1):
                for pages in range(0, 300, 7):
                    sizes = pda.tail_pieces(pages, K, C, bs)
                    assert sum(sizes) == pages, (bs, C, K, pages, sizes)
                    assert 1 <= len(sizes) <= 8
                    if len(sizes) == 1:
                        continue
                    assert pages >= 4 * m
                    assert min(sizes) >= m, (bs, C, K, pages, sizes)
                    if 3 * K < C:
                        assert max(sizes) - min(sizes) <= 1
                        assert len(sizes) <= -(-2 * C // K)
                    else:
                        assert all(b <= a + m for a, b in zip(sizes, sizes[1:])), (bs, C, K, pages, sizes)


def test_tail_pieces_rejects_bad_arguments(lib):
    for args in [(-1, 10, 456, 16), (10, 0, 456, 16), (10, 456, 456, 16), (10, 10, 456, 24), (10, 10, 0, 16)]:
        with pytest.raises(pda.PdaError):
            pda.tail_pieces(*args)


def test_choose_kernel_rejects_bad_sizes(lib):
    for args in [(0, 8, 64, 16, 152, 3, 4), (16, 0, 64, 16, 152, 3, 4), (16, 8, 0, 16, 152, 3, 4),
                 (16, 8, 64, 16, 0, 3, 4), (16, 8, 64, 16, 152, 0, 4), (16, 8, 64, 16, 152, 3, 0)]:
        with pytest.raises(pda.PdaError):
            pda.choose_kernel(*args)


def test_choose_splits_invalid_inputs_return_one(lib):
    for args in [(0, 8, 64, 16, SM, OCC), (16, 0, 64, 16, SM, OCC), (16, 8, 0, 16, SM, OCC),
                 (16, 8, 64, 0, SM, OCC), (16, 8, 64, 16, 0, OCC), (16, 8, 64, 16, SM, 0), (-1, 8, 64, 16, SM, OCC)]:
        assert lib.pda_choose_splits(*args) == 1


# -------------------------------------------------------- host validation

A = 1 << 20  # a 16-byte-aligned fake address (never dereferenced: validation fails first)


def call(lib, **kw):
    a = dict(out=A, q=A, k=A, v=A, tables=A, lens=A, S=2, H=8, Hk=2, D=128, bs=16, MB=4, scale=0.1, ks=0.05,
             vs=0.05, stream=None)
    a.update(kw)
    return lib.pda_decode(a["out"], a["q"], a["k"], a["v"], a["tables"], a["lens"], a["S"], a["H"], a["Hk"],
                          a["D"], a["bs"], a["MB"], a["scale"], a["ks"], a["vs"], a["stream"])


@pytest.mark.parametrize("kw,status", [
    (dict(D=64), pda.PDA_ERR_UNSUPPORTED),
    (dict(D=256), pda.PDA_ERR_UNSUPPORTED),
    (dict(bs=8), pda.PDA_ERR_UNSUPPORTED),
    (dict(bs=24), pda.PDA_ERR_UNSUPPORTED),
    (dict(bs=144), pda.PDA_ERR_UNSUPPORTED),
    (dict(H=18, Hk=2), pda.PDA_ERR_UNSUPPORTED),   # GQA 9 > 8
    (dict(H=7, Hk=2), pda.PDA_ERR_INVALID_ARG),     # not a multiple
    (dict(S=-1), pda.PDA_ERR_INVALID_ARG),
    (dict(H=0), pda.PDA_ERR_INVALID_ARG),
    (dict(Hk=0), pda.PDA_ERR_INVALID_ARG),
    (dict(MB=-1), pda.PDA_ERR_INVALID_ARG),
    (dict(out=None), pda.PDA_ERR_INVALID_ARG),
    (dict(q=None), pda.PDA_ERR_INVALID_ARG),
    (dict(k=None), pda.PDA_ERR_INVALID_ARG),
    (dict(v=None), pda.PDA_ERR_INVALID_ARG),
    (dict(tables=None), pda.PDA_ERR_INVALID_ARG),
    (dict(lens=None), pda.PDA_ERR_INVALID_ARG),
    (dict(q=A + 8), pda.PDA_ERR_INVALID_ARG),       # misaligned
    (dict(k=A + 4), pda.PDA_ERR_INVALID_ARG),
    (dict(out=A + 2), pda.PDA_ERR_INVALID_ARG),
    (dict(tables=A + 2), pda.PDA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), pda.PDA_ERR_INVALID_ARG),
    (dict(ks=float("inf")), pda.PDA_ERR_INVALID_ARG),
    (dict(S=70000), pda.PDA_ERR_UNSUPPORTED),
])
def test_decode_rejects_before_launch(lib, kw, status):
    assert call(lib, **kw) == status


def test_decode_zero_sequences_is_a_noop(lib):
    assert call(lib, S=0, out=None, q=None, k=None, v=None, tables=None, lens=None) == pda.PDA_OK


def test_bounded_wait_rejects_bad_limits(lib):
    assert lib.pda_test_bounded_wait(0, None) == pda.PDA_ERR_INVALID_ARG
    assert lib.pda_test_bounded_wait(2000001, None) == pda.PDA_ERR_INVALID_ARG


def test_query_status_null_pointer(lib):
    assert lib.pda_query_device_status(None, ctypes.POINTER(ctypes.c_int)()) == pda.PDA_ERR_INVALID_ARG


def test_workspace_info_null_pointers(lib):
    n = ctypes.c_int(0)
    b = ctypes.c_longlong(0)
    assert lib.pda_workspace_info(None, None, ctypes.byref(n)) == pda.PDA_ERR_INVALID_ARG
    assert lib.pda_workspace_info(None, ctypes.byref(b), None) == pda.PDA_ERR_INVALID_ARG


def test_reserve_rejects_bad_args(lib):
    assert lib.pda_reserve(4, 8, 2, 16, 24, None) == pda.PDA_ERR_INVALID_ARG
    assert lib.pda_reserve(-1, 8, 2, 16, 16, None) == pda.PDA_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(pda.PdaError, match="not built"):
        _binding.load(str(tmp_path / "missing.so"))


# ------------------------------------------- pda_decode_host: host-side checks

def host_call(lib, lens, table, NB=4, H=8, Hk=2, bs=16):
    import numpy as np
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    table = np.ascontiguousarray(table, dtype=np.int32)
    S, MB = table.shape
    q = np.zeros((S, H, 128), np.uint16)
    out = np.zeros_like(q)
    k = np.zeros((NB, Hk, 8, bs, 16), np.uint8)
    v = np.zeros((NB, Hk, 128, bs), np.uint8)
    return lib.pda_decode_host(out.ctypes.data, q.ctypes.data, k.ctypes.data, v.ctypes.data, table.ctypes.data,
                               lens.ctypes.data, S, H, Hk, 128, bs, MB, NB, 0.1, 0.05, 0.05, None)


@pytest.mark.parametrize("lens,table", [
    ([17, 5], [[0, 4, 0], [1, 0, 0]]),       # entry 4 of a 4-block pool, read by sequence 0
    ([17, 5], [[0, 1, 0], [-1, 0, 0]]),      # negative entry read by sequence 1
    ([49, 0], [[0, 1, 2], [0, 0, 0]]),       # 49 tokens need 4 entries of a 3-entry row
    ([-1, 0], [[0, 0, 0], [0, 0, 0]]),       # negative length
])
def test_decode_host_checks_tables_before_any_copy(lib, lens, table):
    # Every entry a sequence reads is checked on the host against the pool;
    # these calls return before any CUDA call (no device is needed).
    assert host_call(lib, lens, table) == pda.PDA_ERR_INVALID_ARG


def test_decode_host_shares_the_size_checks(lib):
    import numpy as np
    t = np.zeros((2, 3), np.int32)
    assert host_call(lib, [1, 1], t, H=18, Hk=2) == pda.PDA_ERR_UNSUPPORTED      # GQA 9
    assert host_call(lib, [1, 1], t, bs=24) == pda.PDA_ERR_UNSUPPORTED
    assert host_call(lib, [1, 1], t, NB=0) == pda.PDA_ERR_INVALID_ARG
    assert lib.pda_decode_host(None, None, None, None, None, None, 0, 8, 2, 128, 16, 3, 4, 0.1, 0.05, 0.05,
                               None) == pda.PDA_OK


def test_plain_c_caller(lib, tmp_path):
    # The boundary is C: a C11 program includes the header on its own, links
    # libpda.so and calls host-side entry points.
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = tmp_path / "abi_c_check"
    libdir = os.path.dirname(pda.LIB_PATH)
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "abi_c_check.c"), "-L", libdir, "-lpda", "-Wl,-rpath," + libdir,
                    "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
