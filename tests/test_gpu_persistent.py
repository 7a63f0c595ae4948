"""GPU parity of the persistent decode kernel against the fp64 oracle.

A batch whose grid does not fit one wave of 4 CTAs per SM runs on the
persistent kernel: one CTA per resident slot, work units taken from an
atomic queue, pages streamed across unit boundaries, each unit's query rows
and header carried in its first stage, the consumer warps' merge done in the
unit's last stage. The batches here have many short, ragged sequences
(zero lengths, partial pages, one-token contexts), so every CTA runs many
units back to back and the oracle still finishes in seconds.
"""

from __future__ import annotations

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


def _many(S, bs, seed, max_len=300, H=32, Hk=8):
    """S ragged sequences in [0, max_len): every 13th empty, some of one token."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, max_len, S)
    lens[::13] = 0
    lens[5::17] = 1
    return workloads.make_custom(S, H, Hk, lens.tolist(), block_size=bs, pool_factor=1.2, seed=seed, device=DEV)


def _kernel(batch):
    cfg = batch.cfg
    return pda.plan_kernel(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq,
                           cfg.block_size)


@pytest.mark.parametrize("bs,splits", [(16, 0), (16, 2), (16, 5), (32, 0), (32, 3), (48, 0), (64, 0), (64, 2),
                                       (80, 0), (96, 2), (112, 0), (128, 0), (128, 2)])
def test_persistent_parity(bs, splits):
    batch = _many(160, bs, seed=100 + bs + splits)
    pda.set_split_override(splits)
    try:
        assert _kernel(batch) == pda.PDA_KERNEL_PERSISTENT
        out = U.run_cuda(batch)
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
    stats = U.compare(out, U.run_oracle(batch), "persistent bs=%d splits=%d" % (bs, splits))
    lens = batch.seq_lens_host
    assert all(torch.all(out[s] == 0) for s in range(len(lens)) if lens[s] == 0), "empty sequences give zeros"
    print(bs, splits, stats)


@pytest.mark.parametrize("splits", [1, 3])
def test_persistent_bitwise_equals_per_unit_kernel(splits):
    # pda_decode_noalloc always runs the per-unit kernel; with the same split
    # count the per-unit arithmetic (stages, tiles, warp merge) is identical
    # (tail pieces off: a pieced unit folds its pieces instead).
    batch = _many(200, 16, seed=7, max_len=700)
    cfg = batch.cfg
    pda.set_split_override(splits)
    pda.set_tail_split(False)
    try:
        assert _kernel(batch) == pda.PDA_KERNEL_PERSISTENT
        a = U.run_cuda(batch)
        b = torch.empty_like(batch.q)
        pda.decode_noalloc(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens, cfg.scale,
                           cfg.k_scale, cfg.v_scale, out=b)
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
        pda.set_tail_split(True)
    assert torch.equal(a, b)


@pytest.mark.parametrize("S,Hk,MB,bs", [(16, 8, 64, 16), (64, 8, 64, 16), (256, 8, 256, 16), (128, 8, 128, 64),
                                       (77, 8, 8, 16), (2200, 8, 8, 16), (40, 4, 300, 32)])
def test_device_plan_matches_the_pure_planner(S, Hk, MB, bs):
    # On this device (its SM count, 3 persistent / 4 dense CTAs per SM) the
    # device-side plan equals the host-only planner's choice.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    kind, splits, launches = pda.choose_kernel(S, Hk, MB, bs, sms, 3, 4)
    H = 4 * Hk
    assert pda.plan_kernel(S, H, Hk, MB, bs) == kind
    assert pda.plan_splits(S, H, Hk, MB, bs) == splits
    assert pda.plan_launches(S, H, Hk, MB, bs) == launches


def test_launch_counts():
    # units beyond the resident slots are handed out longest first (one more
    # launch, up to 16384 units) and the units of the last partial round
    # are cut into pieces that the tail merge kernel folds (one more); a
    # split adds the merge launch
    batch = _many(160, 16, seed=3)
    cfg = batch.cfg
    args = (cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq, cfg.block_size)
    assert pda.plan_launches(*args) == 3
    pda.set_tail_split(False)
    try:
        assert pda.plan_launches(*args) == 2
    finally:
        pda.set_tail_split(True)
    pda.set_split_override(3)
    try:
        assert pda.plan_launches(*args) == 4
    finally:
        pda.set_split_override(0)
    assert pda.plan_launches(2200, 32, 8, 8, 16) == 1   # 17600 units: ticket order
    assert pda.plan_launches(0, 32, 8, 8, 16) == 0


def test_ticket_order_beyond_the_ordered_limit():
    # 2200 sequences x 8 kv heads = 17600 units: no order kernel, tickets in unit order
    batch = _many(2200, 16, seed=19, max_len=90)
    cfg = batch.cfg
    assert _kernel(batch) == pda.PDA_KERNEL_PERSISTENT
    assert pda.plan_launches(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq,
                             cfg.block_size) == 1
    out = U.run_cuda(batch)
    b = torch.empty_like(batch.q)
    pda.decode_noalloc(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens, cfg.scale,
                       cfg.k_scale, cfg.v_scale, out=b)
    torch.cuda.synchronize()
    assert torch.equal(out, b)
    U.compare(out, U.run_oracle(batch), "persistent, 17600 units")


def test_largest_batch_of_short_sequences():
    # 65,535 sequences (the largest batch) x 2 kv heads = 131,070 units of
    # 0-40 tokens: the persistent kernel in ticket order (past the ordered
    # limit), its queue counting 131,070 tickets. Sampled rows against the
    # oracle.
    S = 65535
    rng = np.random.default_rng(5)
    lens = rng.integers(0, 41, S)
    batch = workloads.make_custom(S, 8, 2, lens.tolist(), block_size=16, pool_factor=1.1, seed=6, device=DEV)
    cfg = batch.cfg
    assert _kernel(batch) == pda.PDA_KERNEL_PERSISTENT
    out = U.run_cuda(batch)
    torch.cuda.synchronize()
    ids = sorted(set(rng.choice(S, 400, replace=False).tolist()) | {0, S - 1, int(np.argmax(lens))})
    U.compare(out[ids], U.run_oracle(batch, seq_ids=ids), "65535 sequences")
    zero = [s for s in range(S) if lens[s] == 0]
    assert torch.all(out[zero] == 0)


@pytest.mark.parametrize("S", [40, 400])
def test_all_sequences_empty(S):
    # Every sequence has length 0: the dense per-unit kernel (40 sequences)
    # and the persistent kernel (400) must both write all-zero rows, with
    # and without splits.
    batch = workloads.make_custom(S, 32, 8, [0] * S, block_size=16, seed=S, device=DEV)
    for splits in (0, 3):
        pda.set_split_override(splits)
        try:
            out = torch.full_like(batch.q, 7.0)
            U.run_cuda(batch, out=out)
            torch.cuda.synchronize()
        finally:
            pda.set_split_override(0)
        assert torch.all(out == 0), "splits %d" % splits


def test_queue_resets_between_calls_and_graph_replays():
    # The work queue lives in the stream's workspace and each launch leaves
    # it at zero: calls of different sizes back to back, then graph replays.
    s = torch.cuda.Stream()
    batches = [_many(S, 16, seed=S) for S in (120, 300, 97)]
    s.wait_stream(torch.cuda.current_stream())   # the batches were made on the current stream
    for b in batches:
        assert _kernel(b) == pda.PDA_KERNEL_PERSISTENT
    first = []
    with torch.cuda.stream(s):
        for b in batches:
            first.append(U.run_cuda(b, stream=s).clone())
        again = [U.run_cuda(b, stream=s).clone() for b in reversed(batches)][::-1]
    s.synchronize()
    for x, y in zip(first, again):
        assert torch.equal(x, y)
    b = batches[1]
    cfg = b.cfg
    pda.reserve(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq, cfg.block_size,
                stream=s)
    out = torch.zeros_like(b.q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        U.run_cuda(b, out=out, stream=s)
    for _ in range(5):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, first[1])
    U.compare(first[1], U.run_oracle(b), "persistent, 300 sequences")


@pytest.mark.parametrize("splits", [2, 3])
def test_split_batch_in_a_graph_matches_eager(splits):
    # Order kernel, persistent kernel, the tail merge and the merge kernel
    # (programmatic dependents) captured together and replayed.
    b = _many(180, 16, seed=90 + splits, max_len=600)
    cfg = b.cfg
    pda.set_split_override(splits)
    try:
        assert pda.plan_launches(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq,
                                 cfg.block_size) == 4
        eager = U.run_cuda(b).clone()
        s = torch.cuda.Stream()
        pda.reserve(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq, cfg.block_size,
                    stream=s)
        out = torch.zeros_like(b.q)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            U.run_cuda(b, out=out, stream=s)
        for _ in range(3):
            out.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(out, eager)
    finally:
        pda.set_split_override(0)
    U.compare(eager, U.run_oracle(b), "persistent, %d splits" % splits)


def test_two_streams_run_their_queues_side_by_side():
    # Each stream has its own workspace, so its own work queue: two calls
    # that can overlap on the GPU must both give the single-stream result.
    a, b = _many(200, 16, seed=71), _many(260, 16, seed=72)
    ref_a, ref_b = U.run_cuda(a).clone(), U.run_cuda(b).clone()
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(s1):
            oa = U.run_cuda(a, stream=s1)
        with torch.cuda.stream(s2):
            ob = U.run_cuda(b, stream=s2)
        outs.append((oa, ob))
    torch.cuda.synchronize()
    for oa, ob in outs:
        assert torch.equal(oa, ref_a) and torch.equal(ob, ref_b)


def test_persistent_sinks_fp8_and_shuffled_v():
    batch = _many(150, 32, seed=61, H=40)
    cfg = batch.cfg
    assert _kernel(batch) == pda.PDA_KERNEL_PERSISTENT
    g = torch.Generator().manual_seed(9)
    sinks = (torch.randn(cfg.num_heads, generator=g) * 2).float()
    NB, Hk, D, bs = batch.v_cache.shape
    v_sh = batch.v_cache.reshape(NB, Hk, D, bs // 16, 16).permute(0, 1, 3, 2, 4).contiguous()
    a = pda.decode_ex(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens, cfg.scale,
                      cfg.k_scale, cfg.v_scale, sinks=sinks.to(DEV))
    b = pda.decode_ex(batch.q, batch.k_cache, v_sh, batch.block_tables, batch.seq_lens, cfg.scale, cfg.k_scale,
                      cfg.v_scale, sinks=sinks.to(DEV), v_shuffled=True)
    out_scale = 0.0075
    c = pda.decode_ex(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens, cfg.scale,
                      cfg.k_scale, cfg.v_scale, sinks=sinks.to(DEV), output_scale=out_scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b), "the two V layouts hold the same values"
    exact = oracle.decode(**batch.raw(), scale=cfg.scale, k_scale=cfg.k_scale, v_scale=cfg.v_scale,
                          sinks=sinks.numpy())
    U.compare(a, exact, "persistent with sinks")
    U.compare_e4m3(c, exact, out_scale, "persistent e4m3 output")


# ------------------------------------------------------------- tail pieces

def _uniform(S, H, Hk, ctx, bs=16, seed=0):
    return workloads.make_custom(S, H, Hk, [ctx] * S, block_size=bs, seed=seed, device=DEV)


@pytest.mark.parametrize("S,H,Hk,ctx,bs,splits,spread", [
    (80, 32, 8, 2048, 16, 0, 0),     # 640 units over 456 CTAs: the last 184 in shrinking pieces
    (80, 40, 8, 1024, 16, 0, 0),     # g = 5 (two PV passes): 64-page units in pieces of 26, 16 and 22 pages
    (40, 64, 8, 2048, 64, 2, 0),     # g = 8, 64-token blocks, 2 splits: pieces of splits, then the merge kernel
    (120, 32, 8, 1100, 16, 0, 0),    # a tail of 48 units: equal pieces of 18, 17, 17 and 17 pages
    (130, 32, 8, 2048, 16, 0, 0),    # a tail of 128 units: 8 equal pieces of 16 pages
    (120, 32, 8, 700, 16, 0, 0),     # 44-page units stay whole: the tail merge has nothing to fold
    (160, 32, 8, 900, 16, 0, 400),   # 900 to 1299 tokens: tail units on both sides of the 1024-token cut
    (700, 8, 1, 3000, 32, 0, 0),     # one kv head (g = 8), 32-token blocks: 244 tail units in shrinking pieces
    (128, 6, 2, 2766, 128, 2, 0),    # 128-token blocks, 2 splits of 11 pages in 5 equal pieces (2-3 pages)
    (33, 24, 8, 2735, 128, 2, 0),    # g = 3, 8 kv heads, the same cut on a 2-stage ring
])
def test_tail_pieces_parity(S, H, Hk, ctx, bs, splits, spread):
    """Units of the last, partial round are cut into pieces; the tail merge
    kernel folds them. Parity with the oracle, agreement with the same call
    without pieces, and the same bits call after call."""
    if spread:
        lens = [ctx + (i * 37) % spread for i in range(S)]
        batch = workloads.make_custom(S, H, Hk, lens, block_size=bs, seed=S + H + bs, device=DEV)
    else:
        batch = _uniform(S, H, Hk, ctx, bs=bs, seed=S + H + bs)
    cfg = batch.cfg
    pda.set_split_override(splits)
    try:
        kind = _kernel(batch)
        assert kind == pda.PDA_KERNEL_PERSISTENT
        a = U.run_cuda(batch).clone()
        b = U.run_cuda(batch).clone()
        pda.set_tail_split(False)
        c = U.run_cuda(batch).clone()
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
        pda.set_tail_split(True)
    assert torch.equal(a, b), "tail pieces must be deterministic"
    assert (a.float() - c.float()).abs().max().item() <= 4e-3
    U.compare(a, U.run_oracle(batch), "tail pieces S=%d H=%d bs=%d splits=%d (%s)" % (S, H, bs, splits, kind))
    assert pda.query_device_status() == 0


@pytest.mark.parametrize("S,splits,shuffled,kind", [
    (160, 0, False, pda.PDA_KERNEL_PERSISTENT),
    (160, 2, False, pda.PDA_KERNEL_PERSISTENT),
    (700, 0, True, pda.PDA_KERNEL_PERSISTENT),
    (60, 0, False, pda.PDA_KERNEL_PER_UNIT_DENSE),   # one wave, no split
    (2, 20, True, pda.PDA_KERNEL_PER_UNIT_DENSE),    # one wave, 20 splits: the merge kernel, no clusters
])
def test_page_gathers_bitwise_equal_to_page_copies(S, splits, shuffled, kind):
    """16-token pages reach the stages as four-page gathers or as one bulk
    copy per page: the same bytes, so the same bits, on the persistent
    kernel and on per-unit grids that do not merge in clusters. Ragged
    lengths give last stages of 1 to 3 pages (the gather repeats the first
    row into the unused slots), empty and one-token sequences."""
    batch = _many(S, 16, seed=300 + S + splits, max_len=700)
    cfg = batch.cfg
    pda.set_split_override(splits)
    try:
        assert _kernel(batch) == kind
    finally:
        pda.set_split_override(0)
    v = batch.v_cache
    if shuffled:  # [NB, Hk, bs/16, 128, 16]: the same values (bitwise the same outputs)
        NB, Hk, D, bs = v.shape
        v = v.reshape(NB, Hk, D, bs // 16, 16).permute(0, 1, 3, 2, 4).contiguous()

    def call():
        return pda.decode_ex(batch.q, batch.k_cache, v, batch.block_tables, batch.seq_lens, cfg.scale,
                             cfg.k_scale, cfg.v_scale, v_shuffled=shuffled)

    pda.set_split_override(splits)
    try:
        a = call().clone()
        pda.set_tma_gather(False)
        b = call().clone()
        torch.cuda.synchronize()
    finally:
        pda.set_tma_gather(True)
        pda.set_split_override(0)
    assert torch.equal(a, b)
    U.compare(a, U.run_oracle(batch), "page gathers S=%d splits=%d shuffled=%d" % (S, splits, shuffled))
    assert pda.query_device_status() == 0


def _slot_tables(batch, seed, junk=True):
    """Per-slot scales within +-20 % of the codes' scale; slots past each
    length hold NaN, which the kernels must never use."""
    cfg = batch.cfg
    NB, Hk, bs = batch.num_blocks, cfg.num_kv_heads, cfg.block_size
    g = torch.Generator(device=DEV).manual_seed(seed)
    ks = (torch.rand(NB, Hk, bs, generator=g, device=DEV) * 0.02 + 0.04).float()
    vs = (torch.rand(NB, Hk, bs, generator=g, device=DEV) * 0.02 + 0.04).float()
    if junk:
        for s, L in enumerate(batch.seq_lens_host):
            L = int(L)
            if L == 0:
                continue
            P = (L + bs - 1) // bs
            b = int(batch.block_tables[s, P - 1])
            n = L - (P - 1) * bs
            ks[b, :, n:] = float("nan")
            vs[b, :, n:] = float("nan")
    return ks, vs


@pytest.mark.parametrize("S,H,bs,splits,ctx", [
    (80, 32, 16, 0, 2048),    # 640 units: scale-row gathers, shrinking tail pieces
    (120, 40, 16, 0, 0),      # g = 5, ragged lengths: last stages of 1 to 3 pages
    (40, 32, 64, 2, 2048),    # 64-token blocks, 2 splits: a bulk copy per scale row, pieces of splits
    (100, 48, 32, 0, 0),      # g = 6, the widest group whose query rows leave room for the scale rows
])
def test_slot_scales_on_the_persistent_kernel(S, H, bs, splits, ctx):
    """Multi-wave per-slot-scale calls run on the persistent kernel, scale
    rows in the stages' side entries: oracle parity, the same bits call after
    call and with the gathers off, and the uncut call within rounding."""
    if ctx:
        batch = _uniform(S, H, 8, ctx, bs=bs, seed=S + H + bs)
    else:
        batch = _many(S, bs, seed=S + H + bs, max_len=2000, H=H)
    cfg = batch.cfg
    ks, vs = _slot_tables(batch, seed=S + bs)
    pda.set_split_override(splits)
    try:
        kind, nsplit, launches = pda.plan_slot_scales(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads,
                                                      cfg.max_num_blocks_per_seq, bs)
        assert kind == pda.PDA_KERNEL_PERSISTENT and nsplit == max(splits, 1)

        def call():
            return pda.decode_slot_scales(batch.q, batch.k_cache, batch.v_cache, ks, vs, batch.block_tables,
                                          batch.seq_lens, cfg.scale).clone()

        a, b = call(), call()
        pda.set_tma_gather(False)
        c = call()
        pda.set_tma_gather(True)
        pda.set_tail_split(False)
        d = call()
        torch.cuda.synchronize()
    finally:
        pda.set_tma_gather(True)
        pda.set_tail_split(True)
        pda.set_split_override(0)
    assert torch.equal(a, b), "deterministic"
    assert torch.equal(a, c), "gathers and bulk copies bring the same rows"
    assert (a.float() - d.float()).abs().max().item() <= 4e-3
    ref = oracle.decode(**batch.raw(), scale=cfg.scale, k_scales=ks.cpu().numpy(), v_scales=vs.cpu().numpy())
    U.compare(a, ref, "slot scales, persistent S=%d H=%d bs=%d splits=%d" % (S, H, bs, splits))
    assert pda.query_device_status() == 0


@pytest.mark.parametrize("S,H,Hk,bs,want", [
    (80, 64, 8, 16, pda.PDA_KERNEL_PER_UNIT),      # g = 8: no room beside the query rows
    (80, 40, 8, 128, pda.PDA_KERNEL_PER_UNIT),     # g = 5 at 128-token blocks (1 KiB of scale rows)
    (80, 32, 8, 128, pda.PDA_KERNEL_PERSISTENT),   # g = 4 at 128-token blocks
    (40, 32, 8, 16, pda.PDA_KERNEL_PER_UNIT),      # one wave: the per-unit kernel (cluster merges)
])
def test_slot_scale_kernel_choice(S, H, Hk, bs, want):
    kind, _, launches = pda.plan_slot_scales(S, H, Hk, 4096 // bs, bs)
    assert kind == want
    assert launches >= 1
    if want == pda.PDA_KERNEL_PER_UNIT:
        # still oracle parity on the per-unit kernel
        batch = _uniform(S, H, Hk, 300, bs=bs, seed=S + H)
        ks, vs = _slot_tables(batch, seed=H)
        out = pda.decode_slot_scales(batch.q, batch.k_cache, batch.v_cache, ks, vs, batch.block_tables,
                                     batch.seq_lens, batch.cfg.scale)
        torch.cuda.synchronize()
        ref = oracle.decode(**batch.raw(), scale=batch.cfg.scale, k_scales=ks.cpu().numpy(),
                            v_scales=vs.cpu().numpy())
        U.compare(out, ref, "slot scales, per-unit S=%d H=%d bs=%d" % (S, H, bs))


def test_tail_pieces_with_sinks_e4m3_output_and_strided_caches():
    # every persistent entry point takes the same pieces
    batch = _uniform(80, 32, 8, 2048, seed=11)
    assert _kernel(batch) == pda.PDA_KERNEL_PERSISTENT
    cfg = batch.cfg
    NB, Hk, bs = batch.num_blocks, cfg.num_kv_heads, cfg.block_size
    g = torch.Generator().manual_seed(3)
    sinks = (torch.randn(cfg.num_heads, generator=g) * 2).float()
    out_scale = 0.0075
    ex = pda.decode_ex(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens, cfg.scale,
                       cfg.k_scale, cfg.v_scale, sinks=sinks.to(DEV), output_scale=out_scale)
    kt = batch.k_cache.view(torch.uint8).permute(0, 3, 1, 2, 4).reshape(NB, bs, Hk, 128).contiguous()
    vt = batch.v_cache.view(torch.uint8).permute(0, 3, 1, 2).contiguous()
    st = (bs * Hk * 128, Hk * 128, 128)
    tm = pda.decode_strided(batch.q, kt.data_ptr(), vt.data_ptr(), batch.block_tables, batch.seq_lens, cfg.scale,
                            cfg.k_scale, cfg.v_scale, num_kv_heads=Hk, block_size=bs, num_blocks=NB,
                            k_strides=st, v_strides=st)
    torch.cuda.synchronize()
    raw = batch.raw()
    exact = oracle.decode(**raw, scale=cfg.scale, k_scale=cfg.k_scale, v_scale=cfg.v_scale, sinks=sinks.numpy())
    U.compare_e4m3(ex, exact, out_scale, "tail pieces, sinks + e4m3 out")
    U.compare(tm, U.run_oracle(batch), "tail pieces, token-major caches")
    assert pda.query_device_status() == 0
