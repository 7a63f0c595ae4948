"""pda_set_block_check on GPU: block ids outside the pool are flagged and
read as block 0, never outside the pool.

The caches sit inside larger allocations with PAD spare blocks on both sides
and every bad id stays within that padding, so every read of these tests is
inside allocated memory whether or not the check works; the tests then see
whether it did.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_pda_gb300 as pda
import workloads
from tests import gpu_util as U

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PAD = 8
BAD_BLOCK = 64   # kStatusBadBlock


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    torch.cuda.set_device(0)
    from paged_kv_decode_pda_gb300 import build
    build.build()
    pda.load()
    pda.set_split_override(0)
    assert pda.query_device_status() == 0
    yield
    pda.set_block_check(0)
    pda.set_split_override(0)
    assert pda.query_device_status() == 0


def _padded(t):
    """t inside a [PAD + NB + PAD, ...] allocation; returns the inner view."""
    big = torch.zeros((t.shape[0] + 2 * PAD,) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
    big[PAD:PAD + t.shape[0]].copy_(t)
    return big, big[PAD:PAD + t.shape[0]]


def _case(S, seed, bs=16):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 400, S)
    batch = workloads.make_custom(S, 32, 8, lens.tolist(), block_size=bs, pool_factor=1.2, seed=seed, device=DEV)
    NB = batch.num_blocks
    tables = batch.block_tables.clone()
    bad = {}
    for s, b in ((1, NB + 3), (S // 2, -2), (S - 1, NB)):   # all within the padding
        i = int(rng.integers(0, (int(lens[s]) + bs - 1) // bs))
        tables[s, i] = b
        bad[s] = i
    return batch, tables, bad


@pytest.mark.parametrize("S,entry", [(6, "decode"), (300, "decode"), (6, "noalloc"), (300, "slot_scales")])
def test_bad_block_ids_are_flagged_and_read_as_block_zero(S, entry):
    batch, tables, bad = _case(S, seed=S + len(entry))
    cfg = batch.cfg
    k_big, k = _padded(batch.k_cache.view(torch.uint8))
    v_big, v = _padded(batch.v_cache.view(torch.uint8))
    pda.set_block_check(batch.num_blocks)
    try:
        if entry == "decode":
            out = pda.decode(batch.q, k, v, tables, batch.seq_lens, cfg.scale, cfg.k_scale, cfg.v_scale)
        elif entry == "noalloc":
            out = torch.empty_like(batch.q)
            pda.decode_noalloc(batch.q, k, v, tables, batch.seq_lens, cfg.scale, cfg.k_scale, cfg.v_scale, out=out)
        else:
            # the scale tables are indexed by block id too: padded alike
            ks_big, ks = _padded(torch.full((batch.num_blocks, cfg.num_kv_heads, cfg.block_size), cfg.k_scale,
                                            device=DEV))
            vs_big, vs = _padded(torch.full_like(ks, cfg.v_scale))
            out = pda.decode_slot_scales(batch.q, k, v, ks, vs, tables, batch.seq_lens, cfg.scale)
        code = pda.query_device_status()
    finally:
        pda.set_block_check(0)
    assert code & BAD_BLOCK, "status %d" % code
    # The kernel read block 0 in place of each bad id: that is the oracle's
    # answer for the table with those entries set to 0.
    raw = batch.raw()
    fixed = tables.cpu().numpy().copy()
    for s, i in bad.items():
        fixed[s, i] = 0
    raw["block_tables"] = fixed
    U.compare(out, oracle.decode(**raw, scale=cfg.scale, k_scale=cfg.k_scale, v_scale=cfg.v_scale),
              "block check, %s, %d seqs" % (entry, S))


def test_check_off_by_default_and_clean_tables_pass():
    batch = workloads.make_custom(40, 32, 8, [300] * 40, seed=5, device=DEV)
    cfg = batch.cfg
    plain = U.run_cuda(batch).clone()
    assert pda.query_device_status() == 0
    pda.set_block_check(batch.num_blocks)
    try:
        checked = U.run_cuda(batch)
        assert pda.query_device_status() == 0
    finally:
        pda.set_block_check(0)
    assert torch.equal(plain, checked)
