"""Every decode variant bench.py times, at the headline size and in bench.py's
own launch configuration (its variant closures), against the oracle on
sampled sequences.
"""

import numpy as np
import pytest
import torch

import bench
import oracle
import paged_kv_decode_pda_gb300 as pda
import workloads
from tests import gpu_util as U

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def headline():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    torch.cuda.set_device(0)
    from paged_kv_decode_pda_gb300 import build
    build.build()
    pda.load()
    pda.set_split_override(0)
    cfg = workloads.CONFIGS[workloads.HEADLINE]
    batch = workloads.make_batch(cfg, device=DEV)
    rng = np.random.default_rng(5)
    ids = sorted(set(rng.choice(cfg.num_seqs, size=12, replace=False).tolist()) | {0, cfg.num_seqs - 1})
    yield cfg, batch, ids
    assert pda.query_device_status() == 0


@pytest.mark.parametrize("variant", ["plain", "ex", "shuffled_v", "strided_nhd", "slot_scales"])
def test_bench_variant_full_size(headline, variant):
    cfg, batch, ids = headline
    stream = torch.cuda.Stream()
    nbytes = workloads.algorithmic_bytes(cfg, batch.seq_lens_host)
    call, out, _ = bench.make_variant_call(variant, cfg, batch, [(batch.k_cache, batch.v_cache)],
                                           torch.empty_like(batch.q), nbytes, stream)
    with torch.cuda.stream(stream):
        call(0)
    stream.synchronize()
    kw = dict(scale=cfg.scale, k_scale=cfg.k_scale, v_scale=cfg.v_scale, seq_ids=ids)
    if variant == "ex":
        # the closure's sinks and output scale
        sinks = torch.randn(cfg.num_heads, generator=torch.Generator().manual_seed(3)).float()
        exact = oracle.decode(**batch.raw(), sinks=sinks.numpy(), **kw)
        U.compare_e4m3(out[ids], exact, 0.0075, "bench variant ex")
    else:
        # shuffled V and token-major caches hold the same values as the native
        # batch; the per-slot tables hold the per-tensor scales
        U.compare(out[ids], oracle.decode(**batch.raw(), **kw), "bench variant " + variant, literal=True)
