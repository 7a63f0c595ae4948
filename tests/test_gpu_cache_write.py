"""GPU KV-cache write (pda_reshape_and_cache) against the oracle: cache bytes must match exactly."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_pda_gb300 as pda
from tests import gpu_util as U
import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _case(T, Hk, bs, NB, seed, scale_k=0.05, scale_v=0.07, pad_frac=0.2, special=False):
    g = torch.Generator().manual_seed(seed)
    key = torch.randn(T, Hk, 128, generator=g) * 2
    val = torch.randn(T, Hk, 128, generator=g) * 30
    if special:
        key[0, 0, :8] = torch.tensor([float("inf"), -float("inf"), float("nan"), 1e6, -1e6, 0.0, -0.0, 1e-30])
    key, val = key.to(torch.bfloat16), val.to(torch.bfloat16)
    slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int64)
    slots[torch.rand(T, generator=g) < pad_frac] = -1
    kc = torch.randint(0, 256, (NB, Hk, 8, bs, 16), generator=g, dtype=torch.uint8)
    vc = torch.randint(0, 256, (NB, Hk, 128, bs), generator=g, dtype=torch.uint8)
    return key, val, slots, kc, vc, scale_k, scale_v


@pytest.mark.parametrize("T,Hk,bs,NB,seed,special", [
    (1, 1, 16, 1, 0, False), (7, 8, 16, 4, 1, True), (256, 8, 16, 300, 2, False), (100, 4, 64, 5, 3, False),
    (33, 2, 32, 4, 4, True), (513, 8, 128, 9, 5, False),
    (5000, 8, 16, 400, 6, True),     # many 16-token groups with random slots
])
def test_cache_write_bit_exact(T, Hk, bs, NB, seed, special):
    key, val, slots, kc, vc, ks, vs = _case(T, Hk, bs, NB, seed, special=special)
    kc_ref, vc_ref = kc.numpy().copy(), vc.numpy().copy()
    oracle.reshape_and_cache(kc_ref, vc_ref, key.view(torch.int16).numpy().view(np.uint16),
                             val.view(torch.int16).numpy().view(np.uint16), slots.numpy(), k_scale=ks, v_scale=vs)
    kd, vd = kc.to(DEV), vc.to(DEV)
    pda.reshape_and_cache(key.to(DEV), val.to(DEV), kd, vd, slots.to(DEV), ks, vs)
    torch.cuda.synchronize()
    assert pda.query_device_status() == 0
    assert np.array_equal(kd.cpu().numpy(), kc_ref), "K cache bytes differ from the oracle"
    assert np.array_equal(vd.cpu().numpy(), vc_ref), "V cache bytes differ from the oracle"


@pytest.mark.parametrize("scale", [0.05, 0.0731, 1.0 / 3.0, 2.0 ** -7, 2.0e-39])
@pytest.mark.parametrize("slots_kind", ["runs", "scattered", "small"])
def test_cache_write_every_bf16_value_bit_exact(scale, slots_kind):
    # All 65,536 bf16 bit patterns (NaNs, infinities, subnormals, both zeros)
    # as K and as V, through every writer path: 4096 tokens in whole blocks
    # (16-byte V rows), 4096 tokens at scattered slots (a token at a time),
    # and 512 tokens at scattered slots (one warp per token: a small write).
    # Every code must equal the oracle's e4m3 code of the binary32 quotient.
    # 2e-39 is a (subnormal) scale whose reciprocal overflows.
    Hk, bs = 1, 16
    allv = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    g = torch.Generator().manual_seed(11)
    if slots_kind == "small":
        T, NB = 512, 64
        key = allv.reshape(T, Hk, 128)
        val = key.flip(0)
        slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int64)
    else:
        # 4096 tokens, each row holding 16 patterns 8 times over
        T, NB = 4096, 300
        key = allv.reshape(T, Hk, 16).repeat_interleave(8, dim=2)
        val = key.flip(0)
        if slots_kind == "runs":
            slots = torch.arange(T, dtype=torch.int64)
        else:
            slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int64)
    kc = torch.zeros(NB, Hk, 8, bs, 16, dtype=torch.uint8)
    vc = torch.zeros(NB, Hk, 128, bs, dtype=torch.uint8)
    kc_ref, vc_ref = kc.numpy().copy(), vc.numpy().copy()
    oracle.reshape_and_cache(kc_ref, vc_ref, key.contiguous().view(torch.int16).numpy().view(np.uint16),
                             val.contiguous().view(torch.int16).numpy().view(np.uint16), slots.numpy(),
                             k_scale=scale, v_scale=scale)
    kd, vd = kc.to(DEV), vc.to(DEV)
    pda.reshape_and_cache(key.contiguous().to(DEV), val.contiguous().to(DEV), kd, vd, slots.to(DEV), scale, scale)
    torch.cuda.synchronize()
    assert pda.query_device_status() == 0

    # e4m3fn has two NaN codes, 0x7F and 0xFF; a NaN input may map to either
    # (the oracle keeps the input's sign, the GPU writes 0x7F), so NaN codes
    # compare equal. Every other code must match exactly.
    def same_nan(a):
        return np.where((a & 0x7F) == 0x7F, 0x7F, a)
    kg, vg = kd.cpu().numpy(), vd.cpu().numpy()
    assert np.array_equal(same_nan(kg), same_nan(kc_ref)), "K codes differ from the oracle"
    assert np.array_equal(same_nan(vg), same_nan(vc_ref)), "V codes differ from the oracle"
    assert np.count_nonzero((kg & 0x7F) == 0x7F) == np.count_nonzero((kc_ref & 0x7F) == 0x7F)


def test_cache_write_out_of_pool_slot_is_skipped_and_flagged():
    key, val, slots, kc, vc, ks, vs = _case(4, 2, 16, 2, 7, pad_frac=0.0)
    slots[1] = 2 * 16 + 5       # past the pool
    kd, vd = kc.to(DEV), vc.to(DEV)
    pda.reshape_and_cache(key.to(DEV), val.to(DEV), kd, vd, slots.to(DEV), ks, vs)
    assert pda.query_device_status() != 0
    good = slots.clone()
    good[1] = -1
    kc_ref, vc_ref = kc.numpy().copy(), vc.numpy().copy()
    oracle.reshape_and_cache(kc_ref, vc_ref, key.view(torch.int16).numpy().view(np.uint16),
                             val.view(torch.int16).numpy().view(np.uint16), good.numpy(), k_scale=ks, v_scale=vs)
    assert np.array_equal(kd.cpu().numpy(), kc_ref) and np.array_equal(vd.cpu().numpy(), vc_ref)


def test_write_then_decode_matches_oracle():
    """Fill a cache token by token through the GPU writer, then decode it."""
    S, H, Hk, bs = 3, 16, 4, 16
    lens = [40, 17, 64]
    batch = workloads.make_custom(S, H, Hk, lens, block_size=bs, seed=8, device=DEV)
    g = torch.Generator().manual_seed(9)
    for s, L in enumerate(lens):
        key = torch.randn(L, Hk, 128, generator=g).to(torch.bfloat16).to(DEV)
        val = torch.randn(L, Hk, 128, generator=g).to(torch.bfloat16).to(DEV)
        row = batch.block_tables[s].long()
        t = torch.arange(L, device=DEV)
        slots = row[t // bs] * bs + t % bs
        pda.reshape_and_cache(key, val, batch.k_cache, batch.v_cache, slots, batch.cfg.k_scale, batch.cfg.v_scale)
    out = U.run_cuda(batch)
    U.compare(out, U.run_oracle(batch), "write-then-decode")


@pytest.mark.parametrize("bs,shuffled", [(16, False), (64, False), (64, True), (32, True)])
def test_cache_write_runs_bit_exact(bs, shuffled):
    """Prefill-like slots: whole aligned 16-slot runs (coalesced path) mixed
    with a misaligned run and a run broken by padding (per-token path)."""
    g = torch.Generator().manual_seed(100 + bs)
    Hk = 8
    n_whole = 4800 // bs                      # 4800 tokens in whole blocks
    NB = n_whole + 6
    blocks = torch.randperm(NB, generator=g)
    slots = []
    for b in blocks[:n_whole].tolist():       # whole blocks, in token order
        slots += list(range(b * bs, (b + 1) * bs))
    blocks = blocks[n_whole - 6:]             # keep the indices below as they were
    b = int(blocks[6])
    slots += list(range(b * bs + 3, b * bs + min(bs, 3 + 16)))   # misaligned run inside one block
    b = int(blocks[7])
    run = list(range(b * bs, b * bs + 16))
    run[5] = -1                                          # padding inside a run
    slots += run
    slots += [int(blocks[8]) * bs + 7]                   # ragged tail
    T = len(slots)
    used = [x for x in slots if x >= 0]
    assert len(set(used)) == len(used), "slots must be distinct"
    slots_t = torch.tensor(slots, dtype=torch.int64)
    key = (torch.randn(T, Hk, 128, generator=g) * 3).to(torch.bfloat16)
    val = (torch.randn(T, Hk, 128, generator=g) * 3).to(torch.bfloat16)
    kc = torch.randint(0, 256, (NB, Hk, 8, bs, 16), generator=g, dtype=torch.uint8)
    vshape = (NB, Hk, bs // 16, 128, 16) if shuffled else (NB, Hk, 128, bs)
    vc = torch.randint(0, 256, vshape, generator=g, dtype=torch.uint8)
    kr, vr = kc.numpy().copy(), vc.numpy().copy()
    oracle.reshape_and_cache(kr, vr, key.view(torch.int16).numpy().view(np.uint16),
                             val.view(torch.int16).numpy().view(np.uint16), slots_t.numpy(), k_scale=0.05,
                             v_scale=0.07, v_shuffled=shuffled)
    kd, vd = kc.to(DEV), vc.to(DEV)
    pda.reshape_and_cache(key.to(DEV), val.to(DEV), kd, vd, slots_t.to(DEV), 0.05, 0.07, v_shuffled=shuffled)
    torch.cuda.synchronize()
    assert pda.query_device_status() == 0
    assert np.array_equal(kd.cpu().numpy(), kr), "K bytes differ"
    assert np.array_equal(vd.cpu().numpy(), vr), "V bytes differ"
