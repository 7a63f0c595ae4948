"""pda_decode_noalloc: the decode path for callers that cannot allocate device memory.

Such callers (a server that handed all device memory to its own pool at
start-up, code that must keep every device allocation under its own
allocator's control) cannot let the library grow a workspace with
cudaMallocAsync. pda_decode_noalloc keeps the split partials in a fixed array
compiled into the library instead. These tests call it through the C ABI and
check that it gives what pda_decode gives, call after call, and that it
refuses batches whose partials would not fit.

This file is named so that pytest collects it last; it must also pass alone
in a fresh process (it builds and loads the library itself).
"""

import ctypes

import pytest
import torch

import paged_kv_decode_pda_gb300 as pda
import workloads
from tests import gpu_util as U

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    torch.cuda.set_device(0)
    from paged_kv_decode_pda_gb300 import build
    build.build()
    pda.load()
    pda.set_split_override(0)
    yield
    pda.set_split_override(0)


def _close(a: torch.Tensor, b: torch.Tensor, label: str):
    """Same tolerance the parity tests use (max 8e-3, mean 2e-4), here between the two entry points."""
    d = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all(), label
    assert d.max().item() <= U.MAX_ABS, "%s: max diff %g" % (label, d.max().item())
    assert d.mean().item() <= U.MEAN_ABS, "%s: mean diff %g" % (label, d.mean().item())


def _both(batch, splits):
    cfg = batch.cfg
    pda.set_split_override(splits)
    try:
        ref = U.run_cuda(batch)
        out = torch.empty_like(batch.q)
        pda.decode_noalloc(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens, cfg.scale,
                           cfg.k_scale, cfg.v_scale, out=out)
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
    return ref, out


@pytest.mark.parametrize("splits", [0, 3])
def test_noalloc_matches_decode_on_two_calls_in_a_row(splits):
    # Two different batches back to back: the second call must not see the
    # first call's partials left in the shared array.
    first = workloads.make_batch(workloads.CONFIGS[workloads.SMALL], device=DEV)
    second = workloads.make_custom(5, 40, 8, [1, 77, 1024, 513, 300], block_size=16, seed=77, device=DEV)
    for i, batch in enumerate((first, second)):
        ref, out = _both(batch, splits)
        _close(out, ref, "call %d (splits %d)" % (i + 1, splits))
    assert pda.query_device_status() == 0


def noalloc_splits(cfg) -> int:
    """The split count pda_decode_noalloc plans: the heuristic at the per-unit
    kernel's 3 CTAs per SM, capped at the table width."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = pda.choose_splits(cfg.num_seqs, cfg.num_kv_heads, cfg.max_num_blocks_per_seq, cfg.block_size, sms, 3)
    return min(n, cfg.max_num_blocks_per_seq)


def test_noalloc_default_plan_splits_through_the_array():
    # With its own plan (no override) the small benchmark batch splits, so
    # its partials go through the static array; the result matches the oracle.
    cfg = workloads.CONFIGS[workloads.SMALL]
    assert noalloc_splits(cfg) > 1
    batch = workloads.make_batch(cfg, device=DEV)
    out = torch.empty_like(batch.q)
    pda.decode_noalloc(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens, cfg.scale,
                       cfg.k_scale, cfg.v_scale, out=out)
    torch.cuda.synchronize()
    U.compare(out, U.run_oracle(batch), "noalloc, own plan", literal=True)


def test_noalloc_allocates_no_device_memory():
    # A split call on a stream the library has never seen: no workspace
    # appears for that stream and the device's free memory does not move.
    batch = workloads.make_custom(6, 32, 8, [1024, 700, 999, 64, 1024, 513], seed=91, device=DEV)
    cfg = batch.cfg
    out = torch.empty_like(batch.q)
    s, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    pda.set_split_override(3)
    try:
        # first call: the library's module (and its array) may load lazily here
        pda.decode_noalloc(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens, cfg.scale,
                           cfg.k_scale, cfg.v_scale, out=out, stream=s)
        s.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        s2.wait_stream(s)
        for _ in range(3):
            pda.decode_noalloc(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens,
                               cfg.scale, cfg.k_scale, cfg.v_scale, out=out, stream=s2)
        s2.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
    finally:
        pda.set_split_override(0)
    assert pda.workspace_info(s) == (0, 0) and pda.workspace_info(s2) == (0, 0)
    assert free1 == free0, "device free memory moved by %d bytes" % (free0 - free1)


def test_noalloc_rejects_batches_beyond_its_buffer():
    # 256 seqs x 64 heads x 8 splits x 520 B = 68 MB > 16 MiB: refused before any launch.
    lib = pda.load()
    buf = torch.empty(1 << 16, dtype=torch.uint8, device=DEV)
    tables = torch.zeros(256 * 1024, dtype=torch.int32, device=DEV)
    lens = torch.zeros(256, dtype=torch.int32, device=DEV)
    pda.set_split_override(8)
    try:
        st = lib.pda_decode_noalloc(buf.data_ptr(), buf.data_ptr(), buf.data_ptr(), buf.data_ptr(),
                                    tables.data_ptr(), lens.data_ptr(), 256, 64, 8, 128, 16, 1024, 0.1, 0.05, 0.05,
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    finally:
        pda.set_split_override(0)
    assert st == pda.PDA_ERR_NOALLOC_CAPACITY
    assert b"static buffer" in lib.pda_status_string(st)
