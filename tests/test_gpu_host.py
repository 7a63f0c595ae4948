"""pda_decode_host on GPU: inputs and output in host memory.

The staged call runs the same kernels on byte-identical copies of the
inputs, so it must equal pda_decode bitwise; the host-side table checks
must stop a bad table before anything is copied or launched.
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
    assert pda.query_device_status() == 0


def _host(batch, pinned):
    t = dict(q=batch.q, k=batch.k_cache.view(torch.uint8), v=batch.v_cache.view(torch.uint8),
             tables=batch.block_tables, lens=batch.seq_lens)
    h = {k: v.detach().cpu().contiguous() for k, v in t.items()}
    return {k: (v.pin_memory() if pinned else v) for k, v in h.items()}


def _run_host(batch, h, pinned, stream=None):
    cfg = batch.cfg
    out = torch.empty(h["q"].shape, dtype=torch.bfloat16, pin_memory=pinned)
    pda.decode_host(h["q"], h["k"], h["v"], h["tables"], h["lens"], cfg.scale, cfg.k_scale, cfg.v_scale, out=out,
                    stream=stream)
    (stream or torch.cuda.current_stream()).synchronize()
    return out


@pytest.mark.parametrize("S,max_len,pinned,bs", [(8, 900, True, 16), (200, 700, True, 16), (60, 300, False, 16),
                                                  (40, 700, True, 64), (300, 500, True, 32)])
def test_host_call_equals_device_call(S, max_len, pinned, bs):
    lens = np.random.default_rng(S).integers(0, max_len + 1, S)
    lens[0] = 0
    batch = workloads.make_custom(S, 32, 8, lens.tolist(), block_size=bs, pool_factor=1.3, seed=S, device=DEV)
    dev_out = U.run_cuda(batch)
    torch.cuda.synchronize()
    h = _host(batch, pinned)
    s = torch.cuda.Stream()
    host_out = _run_host(batch, h, pinned, stream=s)
    assert torch.equal(host_out, dev_out.cpu())
    if S <= 60:
        U.compare(host_out, U.run_oracle(batch), "decode_host bs=%d" % bs)


def test_host_call_rejects_a_bad_table_and_runs_nothing():
    batch = workloads.make_custom(4, 16, 4, [40, 0, 17, 33], seed=3, device=DEV)
    h = _host(batch, True)
    out = torch.full(h["q"].shape, 7.0, dtype=torch.bfloat16).pin_memory()
    bad = h["tables"].clone()
    bad[2, 1] = batch.num_blocks          # entry read by sequence 2 (17 tokens = 2 pages)
    cfg = batch.cfg
    with pytest.raises(pda.PdaError) as e:
        pda.decode_host(h["q"], h["k"], h["v"], bad, h["lens"], cfg.scale, cfg.k_scale, cfg.v_scale, out=out)
    assert e.value.status == pda.PDA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(out == 7.0), "nothing may be written back after a refused call"
    # entries past a sequence's pages are never read, so they are not checked
    ok = h["tables"].clone()
    ok[1, :] = -5                          # sequence 1 has no tokens
    ok[2, 2:] = 1 << 30
    got = _run_host(batch, dict(h, tables=ok), True)
    U.compare(got, U.run_oracle(batch), "decode_host, unread table entries hold anything")
