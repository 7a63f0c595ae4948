"""pda_decode_ex on GPU: attention sinks and fused e4m3 output against the oracle."""

import numpy as np
import pytest
import torch

import oracle
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


def _batch(seed=41):
    return workloads.make_custom(6, 40, 8, [0, 1, 17, 300, 1024, 777], block_size=16, pool_factor=1.2, seed=seed,
                                 device=DEV)


def _sinks(H, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(H, generator=g) * 2).float()


@pytest.mark.parametrize("splits", [1, 3, 12])
def test_sinks_parity(splits):
    batch = _batch()
    cfg = batch.cfg
    sinks = _sinks(cfg.num_heads, 1)
    pda.set_split_override(splits)
    try:
        out = pda.decode_ex(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens, cfg.scale,
                            cfg.k_scale, cfg.v_scale, sinks=sinks.to(DEV))
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
    ref = oracle.decode(**batch.raw(), scale=cfg.scale, k_scale=cfg.k_scale, v_scale=cfg.v_scale,
                        sinks=sinks.numpy())
    U.compare(out, ref, "sinks, splits=%d" % splits)
    assert torch.all(out[0] == 0), "zero-length sequence must stay zero with a sink"


def test_ex_without_options_equals_decode():
    batch = _batch(43)
    cfg = batch.cfg
    a = pda.decode_ex(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens, cfg.scale,
                      cfg.k_scale, cfg.v_scale)
    b = U.run_cuda(batch)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("splits,with_sinks", [(1, False), (3, True), (12, False), (12, True)])
def test_fp8_output(splits, with_sinks):
    batch = _batch(47)
    cfg = batch.cfg
    sinks = _sinks(cfg.num_heads, 2) if with_sinks else None
    out_scale = 0.0075   # |o| up to ~3.4 -> codes up to 448
    pda.set_split_override(splits)
    try:
        out = pda.decode_ex(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens, cfg.scale,
                            cfg.k_scale, cfg.v_scale, sinks=sinks.to(DEV) if with_sinks else None,
                            output_scale=out_scale)
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
    exact = oracle.decode(**batch.raw(), scale=cfg.scale, k_scale=cfg.k_scale, v_scale=cfg.v_scale,
                          sinks=sinks.numpy() if with_sinks else None)
    U.compare_e4m3(out, exact, out_scale, "fp8 output, %d splits" % splits)
    got = out.view(torch.uint8).cpu().numpy()
    assert np.all(got[0] == 0)


def test_ex_rejects_bad_options():
    lib = pda.load()
    batch = _batch(49)
    cfg = batch.cfg
    args = [batch.q.data_ptr(), batch.q.data_ptr(), batch.k_cache.data_ptr(), batch.v_cache.data_ptr(),
            batch.block_tables.data_ptr(), batch.seq_lens.data_ptr(), cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads,
            128, 16, int(batch.block_tables.shape[1]), cfg.scale, cfg.k_scale, cfg.v_scale]
    assert lib.pda_decode_ex(*args, 0, None, 7, 1.0, None) == pda.PDA_ERR_INVALID_ARG
    assert lib.pda_decode_ex(*args, 0, None, pda.PDA_OUT_E4M3, 0.0, None) == pda.PDA_ERR_INVALID_ARG
    assert lib.pda_decode_ex(*args, 0, None, pda.PDA_OUT_E4M3, float("nan"), None) == pda.PDA_ERR_INVALID_ARG
    assert lib.pda_decode_ex(*args, 5, None, pda.PDA_OUT_BF16, 1.0, None) == pda.PDA_ERR_INVALID_ARG


# ------------------------------------------------------- shuffled V layout

def _shuffle_v(v):
    NB, Hk, D, bs = v.shape
    return v.reshape(NB, Hk, D, bs // 16, 16).permute(0, 1, 3, 2, 4).contiguous()


@pytest.mark.parametrize("bs,splits", [(16, 0), (32, 3), (64, 0), (64, 12), (128, 2)])
def test_shuffled_v_parity_and_equal_to_native(bs, splits):
    batch = workloads.make_custom(5, 32, 8, [1, 77, 1024, 513, 300], block_size=bs, pool_factor=1.3, seed=53 + bs,
                                  device=DEV)
    cfg = batch.cfg
    v_sh = _shuffle_v(batch.v_cache)
    pda.set_split_override(splits)
    try:
        a = pda.decode_ex(batch.q, batch.k_cache, v_sh, batch.block_tables, batch.seq_lens, cfg.scale, cfg.k_scale,
                          cfg.v_scale, v_shuffled=True)
        b = U.run_cuda(batch)
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
    assert torch.equal(a, b), "the two V layouts hold the same values"
    raw = batch.raw()
    raw["v_cache"] = v_sh.cpu().contiguous().view(torch.uint8).numpy()
    ref = oracle.decode(**raw, scale=cfg.scale, k_scale=cfg.k_scale, v_scale=cfg.v_scale, v_shuffled=True)
    U.compare(a, ref, "shuffled V bs=%d" % bs)


@pytest.mark.parametrize("bs", [16, 64])
def test_cache_write_shuffled_v_bit_exact(bs):
    g = torch.Generator().manual_seed(bs)
    T, Hk, NB = 100, 4, 8
    key = (torch.randn(T, Hk, 128, generator=g) * 2).to(torch.bfloat16)
    val = (torch.randn(T, Hk, 128, generator=g) * 2).to(torch.bfloat16)
    slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int64)
    kc = torch.randint(0, 256, (NB, Hk, 8, bs, 16), generator=g, dtype=torch.uint8)
    vc = torch.randint(0, 256, (NB, Hk, bs // 16, 128, 16), generator=g, dtype=torch.uint8)
    kr, vr = kc.numpy().copy(), vc.numpy().copy()
    oracle.reshape_and_cache(kr, vr, key.view(torch.int16).numpy().view(np.uint16),
                             val.view(torch.int16).numpy().view(np.uint16), slots.numpy(), k_scale=0.05,
                             v_scale=0.05, v_shuffled=True)
    kd, vd = kc.to(DEV), vc.to(DEV)
    pda.reshape_and_cache(key.to(DEV), val.to(DEV), kd, vd, slots.to(DEV), 0.05, 0.05, v_shuffled=True)
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().numpy(), kr) and np.array_equal(vd.cpu().numpy(), vr)
