"""pda_decode_strided on GPU: token-major caches (NHD family) against the oracle.

The three layouts the API page describes are built from one native batch by
pure data movement (torch permutes), so the oracle on the native batch gives
the exact result for each.
"""

import pytest
import torch

import paged_kv_decode_pda_gb300 as pda
import workloads
from tests import gpu_util as U

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
D = 128


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


def token_major(batch):
    """K, V as [NB, bs, Hk, D] uint8 (row of (block, token, head) = D bytes)."""
    k = batch.k_cache.view(torch.uint8)                      # [NB, Hk, D/16, bs, 16]
    NB, Hk, C, bs, _ = k.shape
    kt = k.permute(0, 3, 1, 2, 4).reshape(NB, bs, Hk, D).contiguous()
    vt = batch.v_cache.view(torch.uint8).permute(0, 3, 1, 2).contiguous()   # [NB, bs, Hk, D]
    return kt, vt


def layouts(batch):
    kt, vt = token_major(batch)
    NB, bs, Hk, _ = kt.shape
    # [NB, bs, Hk, D] for K and V separately
    nhd = (kt, vt, kt.data_ptr(), vt.data_ptr(), (bs * Hk * D, Hk * D, D), (bs * Hk * D, Hk * D, D))
    # [NB, 2, bs, Hk, D] (K and V halves of each block)
    two = torch.stack([kt, vt], dim=1).contiguous()
    doc = (two, None, two.data_ptr(), two.data_ptr() + bs * Hk * D, (2 * bs * Hk * D, Hk * D, D),
           (2 * bs * Hk * D, Hk * D, D))
    # [NB, Hk, bs, 2D]: K and V packed in the content dim
    packed = torch.cat([kt.permute(0, 2, 1, 3), vt.permute(0, 2, 1, 3)], dim=-1).contiguous()
    pk = (packed, None, packed.data_ptr(), packed.data_ptr() + D, (Hk * bs * 2 * D, 2 * D, bs * 2 * D),
          (Hk * bs * 2 * D, 2 * D, bs * 2 * D))
    return {"nhd": nhd, "block_split": doc, "packed": pk}


@pytest.mark.parametrize("layout", ["nhd", "block_split", "packed"])
@pytest.mark.parametrize("bs,splits", [(16, 0), (16, 3), (64, 0), (32, 12), (128, 1)])
def test_strided_parity(layout, bs, splits):
    batch = workloads.make_custom(5, 40, 8, [1, 77, 1024, 513, 300], block_size=bs, pool_factor=1.3,
                                  seed=61 + bs, device=DEV)
    cfg = batch.cfg
    keep, keep2, kp, vp, ks, vs = layouts(batch)[layout]
    pda.set_split_override(splits)
    try:
        out = pda.decode_strided(batch.q, kp, vp, batch.block_tables, batch.seq_lens, cfg.scale, cfg.k_scale,
                                 cfg.v_scale, num_kv_heads=cfg.num_kv_heads, block_size=bs,
                                 num_blocks=batch.num_blocks, k_strides=ks, v_strides=vs)
        ref_gpu = U.run_cuda(batch)
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
    U.compare(out, U.run_oracle(batch), "strided %s bs=%d" % (layout, bs))
    assert (out.float() - ref_gpu.float()).abs().max().item() <= 8e-3


@pytest.mark.parametrize("layout", ["nhd", "block_split", "packed"])
@pytest.mark.parametrize("bs,splits", [(16, 0), (16, 2), (32, 0), (64, 3), (80, 0), (128, 0)])
def test_strided_persistent_parity(layout, bs, splits):
    # 160 ragged sequences x 8 kv heads: more units than one wave, so the
    # persistent kernel runs them, its pages arriving through tensor maps.
    import numpy as np
    rng = np.random.default_rng(200 + bs)
    lens = rng.integers(1, 300, 160)
    lens[::13] = 0
    lens[5::17] = 1
    batch = workloads.make_custom(160, 32, 8, lens.tolist(), block_size=bs, pool_factor=1.2, seed=81 + bs,
                                  device=DEV)
    cfg = batch.cfg
    keep, keep2, kp, vp, ks, vs = layouts(batch)[layout]
    pda.set_split_override(splits)
    try:
        out = pda.decode_strided(batch.q, kp, vp, batch.block_tables, batch.seq_lens, cfg.scale, cfg.k_scale,
                                 cfg.v_scale, num_kv_heads=cfg.num_kv_heads, block_size=bs,
                                 num_blocks=batch.num_blocks, k_strides=ks, v_strides=vs)
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
    U.compare(out, U.run_oracle(batch), "strided persistent %s bs=%d splits=%d" % (layout, bs, splits))
    assert all(torch.all(out[s] == 0) for s in range(len(lens)) if lens[s] == 0)


def test_strided_headline_batch_full_size():
    cfg = workloads.CONFIGS[workloads.HEADLINE]
    batch = workloads.make_batch(cfg, device=DEV)
    keep, keep2, kp, vp, ks, vs = layouts(batch)["nhd"]
    out = pda.decode_strided(batch.q, kp, vp, batch.block_tables, batch.seq_lens, cfg.scale, cfg.k_scale,
                             cfg.v_scale, num_kv_heads=cfg.num_kv_heads, block_size=cfg.block_size,
                             num_blocks=batch.num_blocks, k_strides=ks, v_strides=vs)
    torch.cuda.synchronize()
    ids = [0, 17, 100, 255]
    U.compare(out[ids], U.run_oracle(batch, seq_ids=ids), "strided nhd headline", literal=True)


@pytest.mark.parametrize("layout", ["nhd", "block_split", "packed"])
@pytest.mark.parametrize("bs", [16, 64])
def test_strided_single_kv_head(layout, bs):
    # One kv head: the head dimension has extent 1 and shares the token
    # stride (NHD), so it must not be taken for an overlapping dimension.
    batch = workloads.make_custom(3, 7, 1, [404, 0, 199], block_size=bs, pool_factor=1.3, seed=71 + bs,
                                  device=DEV)
    cfg = batch.cfg
    keep, keep2, kp, vp, ks, vs = layouts(batch)[layout]
    out = pda.decode_strided(batch.q, kp, vp, batch.block_tables, batch.seq_lens, cfg.scale, cfg.k_scale,
                             cfg.v_scale, num_kv_heads=1, block_size=bs, num_blocks=batch.num_blocks,
                             k_strides=ks, v_strides=vs)
    torch.cuda.synchronize()
    U.compare(out, U.run_oracle(batch), "strided %s, one kv head, bs=%d" % (layout, bs))


def test_strided_rejects_bad_strides():
    batch = workloads.make_custom(2, 8, 2, [20, 5], seed=67, device=DEV)
    cfg = batch.cfg
    keep, keep2, kp, vp, ks, vs = layouts(batch)["nhd"]
    bad = [(ks[0], ks[1], 8), (ks[0], 64, ks[2]), (0, ks[1], ks[2])]
    for b in bad:
        with pytest.raises(pda.PdaError):
            pda.decode_strided(batch.q, kp, vp, batch.block_tables, batch.seq_lens, cfg.scale, cfg.k_scale,
                               cfg.v_scale, num_kv_heads=cfg.num_kv_heads, block_size=16,
                               num_blocks=batch.num_blocks, k_strides=b, v_strides=vs)
