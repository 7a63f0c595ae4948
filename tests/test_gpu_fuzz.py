"""Randomised GPU parity over the supported shape space, against the fp64 oracle.

Each case draws, from a fixed seed: the batch size, kv heads (1-32) and GQA
ratio (1-8), the block size (16-128), ragged lengths (zeros included), a
table wider than needed (a quarter of the cases draw it with replacement, so
blocks are shared and repeated), a split count (planned or forced) and an entry point
(plain, sinks, shuffled V, token-major, per-slot scales, e4m3 output with
sinks and either V layout, the no-allocation entry point); a third of the
cases scale the query rows by powers of two from 2^-40 to 2^4, and a third
draw V three times larger. Contexts stay short so that the oracle is quick;
the batch sizes reach both kernel shapes.

Upward scaling stops at 2^4: logits of magnitude X carry an fp32 rounding
of about X 2^-24, so once X reaches ~10^5 two tokens whose logits lie that
close are weighted a few tenths of a percent apart from the exact result.
Any fp32 softmax does that; tests/test_gpu_accuracy.py covers rows past
f16's range on fixed inputs.
"""

from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
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


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    Hk = int(rng.choice([1, 2, 3, 4, 8, 16, 32]))
    g = int(rng.integers(1, 9))
    bs = int(rng.choice([16, 32, 48, 64, 80, 96, 112, 128]))
    S = int(rng.choice([1, 3, 17, 60, 150, 300]))
    max_len = int(rng.choice([1, 20, 200, 600]))
    lens = rng.integers(0, max_len + 1, S)
    lens[rng.random(S) < 0.1] = 0
    pages = max(1, int((lens.max() + bs - 1) // bs))
    MB = pages + int(rng.integers(0, 2 * pages + 1))          # tables wider than needed
    splits = int(rng.choice([0, 0, 1, 2, 3, 7]))
    variant = str(rng.choice(["plain", "sinks", "shuffled_v", "token_major", "slot_scales", "e4m3_out",
                              "noalloc"]))
    shared = bool(rng.random() < 0.25)   # tables drawn with replacement: shared and repeated blocks
    # a third of the cases scale query rows by powers of two past f16's range
    # either way, and a third draw V three times larger (few-token outputs
    # then often land in [2, 4), where the bar is tight)
    q_exps = rng.choice([0, 4, -4, -8, -16, -40], size=(S, Hk * g)).tolist() if rng.random() < 1 / 3 else None
    v_gain = 3.0 if rng.random() < 1 / 3 else 1.0
    return dict(Hk=Hk, g=g, bs=bs, S=S, lens=lens.tolist(), MB=MB, splits=splits, variant=variant,
                shared=shared, seed=seed, q_exps=q_exps, v_gain=v_gain)


def _tail_case(seed):
    """A multi-wave batch of long ragged contexts: the persistent kernel with
    longest-first order, tail pieces of both shapes (shrinking or equal) and
    units on both sides of the 1024-token cut."""
    rng = np.random.default_rng(5000 + seed)
    Hk = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.integers(1, 9))
    bs = int(rng.choice([16, 16, 16, 32, 64, 128]))
    splits = int(rng.choice([0, 0, 2, 3])) if Hk >= 4 else int(rng.choice([2, 3, 4]))
    units_goal = int(rng.integers(500, 1600))
    S = max(1, units_goal // (Hk * max(splits, 1)))
    lo = int(rng.choice([1, 300, 900]))
    lens = rng.integers(lo, 3001, S)
    lens[rng.random(S) < 0.05] = 0
    pages = max(1, int((lens.max() + bs - 1) // bs))
    MB = pages + int(rng.integers(0, 3))
    variant = str(rng.choice(["plain", "sinks", "shuffled_v", "token_major", "slot_scales", "e4m3_out"]))
    # as in _case: a third with query rows past f16's range, a third with larger V
    q_exps = rng.choice([0, 4, -4, -8, -16, -40], size=(S, Hk * g)).tolist() if rng.random() < 1 / 3 else None
    v_gain = 3.0 if rng.random() < 1 / 3 else 1.0
    return dict(Hk=Hk, g=g, bs=bs, S=S, lens=lens.tolist(), MB=MB, splits=splits, variant=variant,
                shared=bool(rng.random() < 0.25), seed=seed, q_exps=q_exps, v_gain=v_gain)


@pytest.mark.parametrize("seed", range(int(os.environ.get("PDA_FUZZ_FIRST", "0")),
                                  int(os.environ.get("PDA_FUZZ_FIRST", "0")) + int(os.environ.get("PDA_FUZZ_CASES", "100"))))
def test_random_case(seed):
    _run_case(seed, _case(seed))


@pytest.mark.parametrize("seed", range(int(os.environ.get("PDA_FUZZ_TAIL_CASES", "24"))))
def test_random_multi_wave_case(seed):
    _run_case(10000 + seed, _tail_case(seed))


def _run_case(seed, c):
    H = c["Hk"] * c["g"]
    batch = workloads.make_custom(c["S"], H, c["Hk"], c["lens"], block_size=c["bs"], pool_factor=1.3,
                                  seed=2000 + seed, device=DEV, max_num_blocks_per_seq=c["MB"],
                                  v_scale=0.05 / c["v_gain"])
    batch.cfg = batch.cfg.with_(v_scale=0.05)
    if c["q_exps"] is not None:
        mult = torch.tensor(np.ldexp(1.0, np.array(c["q_exps"], dtype=np.int64)), dtype=torch.float32, device=DEV)
        batch.q = (batch.q.float() * mult[:, :, None]).to(torch.bfloat16)
    cfg = batch.cfg
    if c["shared"]:
        # prefix-cache style tables: sequences share physical blocks and a
        # sequence may name one block twice
        gen = torch.Generator(device=DEV).manual_seed(3000 + seed)
        batch.block_tables.copy_(torch.randint(0, batch.num_blocks, tuple(batch.block_tables.shape),
                                               generator=gen, device=DEV, dtype=torch.int32))
    raw = batch.raw()
    kw = dict(scale=cfg.scale, k_scale=cfg.k_scale, v_scale=cfg.v_scale)
    label = "case %d %s" % (seed, c)
    pda.set_split_override(c["splits"])
    try:
        v = c["variant"]
        if v == "plain":
            out = U.run_cuda(batch)
            ref = oracle.decode(**raw, **kw)
        elif v == "sinks":
            sinks = (torch.randn(H, generator=torch.Generator().manual_seed(seed)) * 2).float()
            out = pda.decode_ex(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens,
                                cfg.scale, cfg.k_scale, cfg.v_scale, sinks=sinks.to(DEV))
            ref = oracle.decode(**raw, **kw, sinks=sinks.numpy())
        elif v == "shuffled_v":
            NB, Hk, _, bs = batch.v_cache.shape
            v_sh = batch.v_cache.reshape(NB, Hk, D, bs // 16, 16).permute(0, 1, 3, 2, 4).contiguous()
            out = pda.decode_ex(batch.q, batch.k_cache, v_sh, batch.block_tables, batch.seq_lens, cfg.scale,
                                cfg.k_scale, cfg.v_scale, v_shuffled=True)
            raw_sh = dict(raw)
            raw_sh["v_cache"] = v_sh.cpu().contiguous().view(torch.uint8).numpy()
            ref = oracle.decode(**raw_sh, **kw, v_shuffled=True)
        elif v == "token_major":
            k = batch.k_cache.view(torch.uint8)
            NB, Hk, C, bs, _ = k.shape
            kt = k.permute(0, 3, 1, 2, 4).reshape(NB, bs, Hk, D).contiguous()
            vt = batch.v_cache.view(torch.uint8).permute(0, 3, 1, 2).contiguous()
            st = (bs * Hk * D, Hk * D, D)
            out = pda.decode_strided(batch.q, kt.data_ptr(), vt.data_ptr(), batch.block_tables, batch.seq_lens,
                                     cfg.scale, cfg.k_scale, cfg.v_scale, num_kv_heads=Hk, block_size=bs,
                                     num_blocks=NB, k_strides=st, v_strides=st)
            torch.cuda.synchronize()
            del kt, vt
            ref = oracle.decode(**raw, **kw)
        elif v == "e4m3_out":
            sinks = (torch.randn(H, generator=torch.Generator().manual_seed(seed)) * 2).float()
            use_sinks, shuffled = seed % 2 == 0, seed % 3 == 0
            vc = batch.v_cache
            if shuffled:
                NB, Hk, _, bs = vc.shape
                vc = vc.reshape(NB, Hk, D, bs // 16, 16).permute(0, 1, 3, 2, 4).contiguous()
            out_scale = 0.0075
            out = pda.decode_ex(batch.q, batch.k_cache, vc, batch.block_tables, batch.seq_lens, cfg.scale,
                                cfg.k_scale, cfg.v_scale, sinks=sinks.to(DEV) if use_sinks else None,
                                output_scale=out_scale, v_shuffled=shuffled)
            torch.cuda.synchronize()
            ref = oracle.decode(**raw, **kw, sinks=sinks.numpy() if use_sinks else None)
        elif v == "noalloc":
            out = torch.empty_like(batch.q)
            # Its split count: the override, or the heuristic's at 3 CTAs per
            # SM, at most the table width. Its partials take 520 bytes per
            # (sequence, head, split) of a 16 MiB array; more is refused
            # before any launch.
            sms = torch.cuda.get_device_properties(0).multi_processor_count
            n = min(c["splits"] or pda.choose_splits(c["S"], c["Hk"], c["MB"], c["bs"], sms, 3), c["MB"])
            refuse = n > 1 and c["S"] * H * n * 520 > 16 << 20
            try:
                pda.decode_noalloc(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens,
                                   cfg.scale, cfg.k_scale, cfg.v_scale, out=out)
            except pda.PdaError as e:
                assert refuse and e.status == pda.PDA_ERR_NOALLOC_CAPACITY, label
                return
            assert not refuse, label
            if c["splits"]:
                # the same split count through the allocating entry point: the
                # per-unit arithmetic is the same whichever kernel runs it
                again = U.run_cuda(batch)
                torch.cuda.synchronize()
                assert torch.equal(out, again), label
            ref = oracle.decode(**raw, **kw)
        else:
            NB, Hk, bs = batch.num_blocks, c["Hk"], c["bs"]
            gen = torch.Generator(device=DEV).manual_seed(seed)
            ks = (torch.rand(NB, Hk, bs, generator=gen, device=DEV) * 0.02 + 0.04).float()
            vs = (torch.rand(NB, Hk, bs, generator=gen, device=DEV) * 0.02 + 0.04).float()
            out = pda.decode_slot_scales(batch.q, batch.k_cache, batch.v_cache, ks, vs, batch.block_tables,
                                         batch.seq_lens, cfg.scale)
            ref = oracle.decode(**raw, scale=cfg.scale, k_scales=ks.cpu().numpy(), v_scales=vs.cpu().numpy())
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
    if c["variant"] == "e4m3_out":
        U.compare_e4m3(out, ref, 0.0075, label, min_equal=0.85)
        out = out.view(torch.uint8)
    else:
        U.compare(out, ref, label)
    lens = c["lens"]
    assert all(torch.all(out[s] == 0) for s in range(len(lens)) if lens[s] == 0), label
