"""Long contexts on GPU: the serving lengths the pages run (a 40,960-token
model length, passkey prompts up to 32K) and beyond, against the oracle.

A few sequences of tens of thousands of tokens are far fewer work units than
resident CTA slots, so the planner splits each one into many page ranges and
the merge kernel combines them; some cases also force small and prime split
counts.
"""

import numpy as np
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
    assert pda.query_device_status() == 0


@pytest.mark.parametrize("lens,H,Hk,bs,splits", [
    ([40960, 32768], 32, 8, 16, 0),        # the pages' model length and passkey length
    ([40960, 1, 20000], 40, 8, 64, 0),      # ragged next to a tiny one, 64-token blocks
    ([131072], 64, 8, 16, 0),               # 128K tokens, one sequence
    ([32768, 32767], 16, 2, 32, 7),         # forced prime split count
    ([65536], 8, 8, 128, 1),                # no split: one CTA streams 512 pages per kv head
])
def test_long_context(lens, H, Hk, bs, splits):
    batch = workloads.make_custom(len(lens), H, Hk, lens, block_size=bs, pool_factor=1.1, seed=sum(lens) % 1000,
                                  device=DEV)
    cfg = batch.cfg
    planned = pda.plan_splits(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq,
                              cfg.block_size)
    pda.set_split_override(splits)
    try:
        out = U.run_cuda(batch)
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
    # the bars apply literally where every context is long (|o| small); a
    # one-token neighbour's rows carry the bf16 rounding of O(1) values
    stats = U.compare(out, U.run_oracle(batch), "long context %s splits %d (planned %d)" % (lens, splits, planned),
                      literal=min(lens) > 1000)
    print(lens, "planned splits", planned, stats)
    if splits == 0:
        assert planned > 1, "a few long sequences must be split"
