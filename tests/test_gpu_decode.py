"""GPU parity of the CUDA decode path (through the C ABI) against the fp64 oracle."""

from __future__ import annotations

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


# ------------------------------------------------------------ full configs

@pytest.mark.parametrize("name", [workloads.SMALL, "40q8kv-64seq-ctx1024-bs16"])
def test_config_full_parity(name):
    batch = workloads.make_batch(workloads.CONFIGS[name], device=DEV)
    out = U.run_cuda(batch)
    torch.cuda.synchronize()
    stats = U.compare(out, U.run_oracle(batch), name, literal=True)
    print(name, stats)


@pytest.mark.parametrize("name", ["32q8kv-256seq-ctx4096-bs16", "40q8kv-256seq-ctx1to4000-bs16",
                                  "64q8kv-128seq-ctx8192-bs64"])
def test_config_full_size_every_sequence(name):
    """Full-size batch in the benchmark's launch configuration (planned split
    count and kernel), every element of every sequence against the oracle
    (the pages' error figures cover every element of 4 head layouts x 3 seeds
    over 1-4000-token contexts: vLLM pull request lishuoshuo-amd/vllm#3,
    "Kernel latency, accuracy runs and kernel error")."""
    cfg = workloads.CONFIGS[name]
    batch = workloads.make_batch(cfg, device=DEV)
    out = U.run_cuda(batch)
    torch.cuda.synchronize()
    ref = U.run_oracle(batch)
    stats = U.compare(out, ref, name, literal=True)
    print(name, "splits", pda.plan_splits(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads,
                                          cfg.max_num_blocks_per_seq, cfg.block_size), stats)


# -------------------------------------------------------------- edge cases

EDGE = [
    # (num_seqs, H, Hk, seq_lens, block_size)
    (1, 8, 8, [1], 16),
    (3, 8, 1, [15, 16, 17], 16),
    (4, 12, 4, [0, 1, 31, 33], 16),
    (2, 16, 2, [63, 64], 64),
    (3, 40, 8, [65, 1, 200], 64),
    (2, 6, 2, [257, 5], 32),
    (2, 14, 2, [100, 47], 48),
    (2, 7, 1, [129, 128], 128),
    (5, 64, 8, [3, 700, 16, 17, 1024], 16),
    (2, 4, 4, [0, 0], 16),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: "S%d_H%d_Hk%d_bs%d" % (c[0], c[1], c[2], c[4]))
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_edge_cases(case, splits):
    S, H, Hk, lens, bs = case
    batch = workloads.make_custom(S, H, Hk, lens, block_size=bs, pool_factor=1.5, seed=sum(lens) + H,
                                  device=DEV)
    pda.set_split_override(splits)
    try:
        out = U.run_cuda(batch)
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
    U.compare(out, U.run_oracle(batch), str(case))
    for s, L in enumerate(lens):
        if L == 0:
            assert torch.all(out[s] == 0)


def test_extra_table_columns_and_unused_pool_blocks():
    batch = workloads.make_custom(3, 8, 2, [40, 200, 17], block_size=16, pool_factor=2.0, seed=5, device=DEV,
                                  max_num_blocks_per_seq=40)
    out = U.run_cuda(batch)
    U.compare(out, U.run_oracle(batch), "wide table")


# ---------------------------------------------------------- split behaviour

def test_split_counts_agree():
    batch = workloads.make_custom(4, 32, 8, [1000, 513, 77, 1024], block_size=16, seed=9, device=DEV)
    ref = U.run_oracle(batch)
    outs = {}
    for n in (1, 2, 3, 7, 64):
        pda.set_split_override(n)
        try:
            outs[n] = U.run_cuda(batch).float()
            torch.cuda.synchronize()
        finally:
            pda.set_split_override(0)
        U.compare(outs[n], ref, "splits=%d" % n)
    for n in outs:
        assert (outs[n] - outs[1]).abs().max().item() <= 8e-3


def test_split_deterministic():
    batch = workloads.make_custom(8, 40, 8, [300] * 8, seed=4, device=DEV)
    for n in (1, 4):
        pda.set_split_override(n)
        try:
            a = U.run_cuda(batch)
            b = U.run_cuda(batch)
            torch.cuda.synchronize()
        finally:
            pda.set_split_override(0)
        assert torch.equal(a, b)


# --------------------------------------------------- gather / tail handling

def _permute_blocks(batch, seed):
    """Same logical cache, different physical placement."""
    NB = batch.num_blocks
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(NB, generator=g)           # new_id = perm[old_id]
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(NB)
    k2 = batch.k_cache[inv.to(batch.k_cache.device)].contiguous()
    v2 = batch.v_cache[inv.to(batch.v_cache.device)].contiguous()
    t2 = perm.to(torch.int32).to(batch.block_tables.device)[batch.block_tables.long()].contiguous()
    return workloads.Batch(batch.cfg, batch.q, k2, v2, t2, batch.seq_lens, batch.seq_lens_host)


@pytest.mark.parametrize("bs", [16, 64])
def test_gather_is_exact_under_block_permutation(bs):
    batch = workloads.make_custom(6, 32, 8, [1, 100, 513, 64, 1000, 17], block_size=bs, pool_factor=1.7, seed=11,
                                  device=DEV)
    for n in (1, 3):
        pda.set_split_override(n)
        try:
            a = U.run_cuda(batch)
            b = U.run_cuda(_permute_blocks(batch, 1))
            c = U.run_cuda(_permute_blocks(batch, 2))
            torch.cuda.synchronize()
        finally:
            pda.set_split_override(0)
        assert torch.equal(a, b) and torch.equal(a, c), "output depends on physical block ids"


@pytest.mark.parametrize("code", [0x7F, 0x7E, 0xFE])
def test_tail_slots_and_table_padding_are_ignored(code):
    lens = [19, 50, 16, 1, 33]
    batch = workloads.make_custom(5, 16, 4, lens, block_size=16, pool_factor=1.0, seed=12, device=DEV,
                                  max_num_blocks_per_seq=6)
    base = U.run_cuda(batch).clone()
    k2, v2, t2 = batch.k_cache.clone(), batch.v_cache.clone(), batch.block_tables.clone()
    kb, vb = k2.view(torch.uint8), v2.view(torch.uint8)
    for s, L in enumerate(lens):
        P = (L + 15) // 16
        n = L - (P - 1) * 16
        b = int(batch.block_tables[s, P - 1])
        kb[b, :, :, n:, :] = code
        vb[b, :, :, n:] = code
        t2[s, P:] = -1
    poisoned = workloads.Batch(batch.cfg, batch.q, k2, v2, t2, batch.seq_lens, batch.seq_lens_host)
    for n in (1, 2):
        pda.set_split_override(n)
        try:
            got = U.run_cuda(poisoned)
            ref = U.run_cuda(batch)
            torch.cuda.synchronize()
        finally:
            pda.set_split_override(0)
        assert torch.equal(got, ref)
    assert torch.equal(U.run_cuda(poisoned), base)


# -------------------------------------------------- streams, graphs, status

def test_side_stream_and_graph_capture():
    batch = workloads.make_custom(16, 32, 8, [1024] * 16, seed=13, device=DEV)
    cfg = batch.cfg
    eager = U.run_cuda(batch).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())   # the batch was made on the current stream
    pda.reserve(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq, cfg.block_size,
                stream=s)
    out = torch.empty_like(batch.q)
    with torch.cuda.stream(s):
        U.run_cuda(batch, out=out, stream=s)
    s.synchronize()
    assert torch.equal(out, eager)
    g = torch.cuda.CUDAGraph()
    out2 = torch.zeros_like(batch.q)
    with torch.cuda.graph(g, stream=s):
        U.run_cuda(batch, out=out2, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out2, eager)


def test_workspace_growth_during_capture_is_refused():
    pda.release()
    # 4 units x 32 splits: more splits than a cluster merges, so fp32 partials
    batch = workloads.make_custom(2, 8, 2, [8192, 8192], seed=14, device=DEV)
    cfg = batch.cfg
    assert pda.plan_splits(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq,
                           cfg.block_size) > 16
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    err = None
    try:
        with torch.cuda.graph(g, stream=s):
            try:
                U.run_cuda(batch, stream=s)
            except pda.PdaError as e:
                err = e
    except Exception:
        pass
    assert err is not None and err.status == pda.PDA_ERR_WORKSPACE


def test_cluster_merged_split_call_needs_no_workspace():
    # 2 to 16 splits in one wave merge inside their clusters: no partials, so
    # the call captures without pda_reserve and replays to the eager result.
    pda.release()
    batch = workloads.make_custom(2, 8, 2, [2048, 1500], seed=14, device=DEV)
    cfg = batch.cfg
    assert 2 <= pda.plan_splits(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq,
                                cfg.block_size) <= 16
    eager = U.run_cuda(batch).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    out = torch.zeros_like(batch.q)
    with torch.cuda.graph(g, stream=s):
        U.run_cuda(batch, out=out, stream=s)
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    assert pda.workspace_info(s) == (0, 0)
    assert torch.equal(out, eager)
    U.compare(eager, U.run_oracle(batch), "cluster merge, no workspace")


def test_graph_replay_after_workspace_growth():
    """A graph captured with a split call keeps its workspace address. A later,
    larger eager call on the same stream grows the workspace; the old buffer
    must stay allocated (retired, not freed) so the graph still replays to
    the eager result."""
    pda.release()
    small = workloads.make_custom(4, 32, 8, [900, 1000, 333, 1024], seed=17, device=DEV)
    big = workloads.make_custom(40, 64, 8, [4096] * 40, seed=18, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    cfg = small.cfg
    # 17 splits: more than a cluster merges, so the call keeps fp32 partials
    # in the workspace (and so does the big batch, persistent with 17 splits)
    pda.set_split_override(17)
    try:
        eager = U.run_cuda(small).clone()
        pda.reserve(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq, cfg.block_size,
                    stream=s)
        bytes0, retired0 = pda.workspace_info(s)
        assert bytes0 > 0 and retired0 == 0
        g = torch.cuda.CUDAGraph()
        out = torch.zeros_like(small.q)
        with torch.cuda.graph(g, stream=s):
            U.run_cuda(small, out=out, stream=s)
        with torch.cuda.stream(s):
            U.run_cuda(big, stream=s)      # grows the workspace of stream s
        s.synchronize()
        bytes1, retired1 = pda.workspace_info(s)
        assert bytes1 > bytes0 and retired1 == retired0 + 1
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
    finally:
        pda.set_split_override(0)
    assert torch.equal(out, eager)
    del g
    pda.release()
    assert pda.workspace_info(s) == (0, 0)


def test_bounded_wait_reports_and_context_survives():
    assert pda.query_device_status() == 0
    pda.bounded_wait_check(2000)
    code = pda.query_device_status()
    assert code != 0
    assert pda.query_device_status() == 0
    batch = workloads.make_custom(2, 8, 2, [40, 7], seed=15, device=DEV)
    U.compare(U.run_cuda(batch), U.run_oracle(batch), "after timeout")


def test_profile_events():
    batch = workloads.make_custom(4, 8, 2, [512] * 4, seed=16, device=DEV)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pda.set_profile_events(a, b)
    try:
        U.run_cuda(batch)
        b.synchronize()
        assert a.elapsed_time(b) > 0
    finally:
        pda.set_profile_events(None, None)


# ------------------------------------------------------- per-slot scales

@pytest.mark.parametrize("bs,splits", [(16, 0), (16, 3), (32, 0), (64, 0), (64, 2), (128, 0), (128, 2)])
def test_slot_scales_parity(bs, splits):
    import oracle
    lens = [1, 37, 300, 1024, 16]
    batch = workloads.make_custom(5, 32, 8, lens, block_size=bs, pool_factor=1.3, seed=21 + bs, device=DEV)
    NB, Hk = batch.num_blocks, 8
    # Per-slot scales within +-20 % of the scale the codes were made with (the
    # spread per-token quantisation of N(0,1) data gives), so values keep the
    # configs' range (tests/test_gpu_accuracy.py spreads them over 2^14).
    g = torch.Generator(device=DEV).manual_seed(5)
    ks = (torch.rand(NB, Hk, bs, generator=g, device=DEV) * 0.02 + 0.04).float()
    vs = (torch.rand(NB, Hk, bs, generator=g, device=DEV) * 0.02 + 0.04).float()
    # slots past each length hold junk scales, which must never be used
    for s, L in enumerate(lens):
        P = (L + bs - 1) // bs
        b = int(batch.block_tables[s, P - 1])
        n = L - (P - 1) * bs
        ks[b, :, n:] = float("nan")
        vs[b, :, n:] = float("nan")
    pda.set_split_override(splits)
    try:
        out = pda.decode_slot_scales(batch.q, batch.k_cache, batch.v_cache, ks, vs, batch.block_tables,
                                     batch.seq_lens, batch.cfg.scale)
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
    raw = batch.raw()
    ref = oracle.decode(**raw, scale=batch.cfg.scale, k_scales=ks.cpu().numpy(), v_scales=vs.cpu().numpy())
    U.compare(out, ref, "slot scales bs=%d" % bs)


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_slot_scale_row_gathers_bitwise_equal_to_pieces(bs):
    """Scale rows arrive as four-row gathers (16-token blocks) or one bulk
    copy per row (larger blocks), or, with the gathers off, as 16-byte
    cp.async pieces: the same bytes, so the same bits. Ragged lengths give
    last stages of fewer pages than a stage holds."""
    lens = [1, 15, 17, 63, 65, 200, 333, 1000, 0, 48]
    batch = workloads.make_custom(len(lens), 32, 8, lens, block_size=bs, pool_factor=1.3, seed=40 + bs, device=DEV)
    NB, Hk = batch.num_blocks, 8
    g = torch.Generator(device=DEV).manual_seed(6)
    ks = (torch.rand(NB, Hk, bs, generator=g, device=DEV) * 0.02 + 0.04).float()
    vs = (torch.rand(NB, Hk, bs, generator=g, device=DEV) * 0.02 + 0.04).float()

    def call():
        return pda.decode_slot_scales(batch.q, batch.k_cache, batch.v_cache, ks, vs, batch.block_tables,
                                      batch.seq_lens, batch.cfg.scale)

    a = call().clone()
    pda.set_tma_gather(False)
    try:
        b = call().clone()
        torch.cuda.synchronize()
    finally:
        pda.set_tma_gather(True)
    assert torch.equal(a, b)
    assert pda.query_device_status() == 0


def test_slot_scales_constant_table_matches_per_tensor():
    batch = workloads.make_custom(4, 40, 8, [100, 1000, 7, 513], seed=33, device=DEV)
    NB, Hk, bs = batch.num_blocks, 8, 16
    ks = torch.full((NB, Hk, bs), batch.cfg.k_scale, device=DEV)
    vs = torch.full((NB, Hk, bs), batch.cfg.v_scale, device=DEV)
    a = pda.decode_slot_scales(batch.q, batch.k_cache, batch.v_cache, ks, vs, batch.block_tables, batch.seq_lens,
                               batch.cfg.scale)
    b = U.run_cuda(batch)
    torch.cuda.synchronize()
    assert (a.float() - b.float()).abs().max().item() <= 4e-3
    U.compare(a, U.run_oracle(batch), "constant tables")


# ------------------------------------------------------------ merge kernels

@pytest.mark.parametrize("S,H,Hk,splits", [(8, 32, 8, 2), (8, 32, 8, 4), (8, 40, 8, 3), (6, 32, 8, 6), (8, 8, 8, 5),
                                            (8, 64, 8, 8), (8, 8, 1, 7), (4, 40, 8, 9), (4, 32, 8, 13),
                                            (4, 40, 8, 16), (4, 64, 8, 17), (2, 8, 1, 40)])
def test_merge_kernels_match_across_kernels(S, H, Hk, splits):
    """One-wave batches of 2 to 16 splits merge inside each unit's cluster
    of CTAs (one launch); more splits go through fp32 partials and the merge
    kernel, one warp per row up to 16 splits, four warps per row beyond.
    pda_decode_noalloc always uses the merge kernel. Both run the same tiles
    and the same fold: same split count, same bits, call after call and
    from a graph replayed twice; zero-length sequences, and splits left
    without pages by short sequences, give what the oracle gives."""
    lens = [1024, 0, 517, 16, 33, 1000, 0, 257][:S]
    batch = workloads.make_custom(S, H, Hk, lens, seed=H + splits, device=DEV, max_num_blocks_per_seq=64)
    cfg = batch.cfg
    pda.set_split_override(splits)
    try:
        assert pda.plan_kernel(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq,
                               cfg.block_size) == pda.PDA_KERNEL_PER_UNIT_DENSE
        assert pda.plan_launches(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq,
                                 cfg.block_size) == (1 if splits <= 16 else 2)
        ref = torch.empty_like(batch.q)
        pda.decode_noalloc(batch.q, batch.k_cache, batch.v_cache, batch.block_tables, batch.seq_lens, cfg.scale,
                           cfg.k_scale, cfg.v_scale, out=ref)
        outs = [U.run_cuda(batch).clone() for _ in range(3)]
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        pda.reserve(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq, cfg.block_size,
                    stream=s)
        g = torch.cuda.CUDAGraph()
        gout = torch.zeros_like(batch.q)
        with torch.cuda.graph(g, stream=s):
            U.run_cuda(batch, out=gout, stream=s)
        for _ in range(2):
            gout.zero_()
            with torch.cuda.stream(s):
                g.replay()
            s.synchronize()
            outs.append(gout.clone())
        torch.cuda.synchronize()
    finally:
        pda.set_split_override(0)
    for o in outs:
        assert torch.equal(o, ref)
    for i, L in enumerate(lens):
        if L == 0:
            assert torch.all(outs[0][i] == 0)
    U.compare(outs[0], U.run_oracle(batch), "merge H=%d splits=%d" % (H, splits))
    assert pda.query_device_status() == 0


@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("S", [6, 300])
def test_swizzled_v_pages_in_graphs(bs, S):
    """Native V pages of 32-, 64- and 128-token blocks load through a swizzled
    tensor map built on the host per call and passed by value to the kernel:
    a CUDA graph of the call (per-unit kernel for 6 sequences, persistent for
    300) replays to the eager result twice, and both match the oracle."""
    lens = np.random.default_rng(bs + S).integers(1, 3 * bs + 5, S).tolist()
    batch = workloads.make_custom(S, 32, 8, lens, block_size=bs, pool_factor=1.3, seed=bs * S, device=DEV)
    cfg = batch.cfg
    eager = U.run_cuda(batch).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    pda.reserve(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq, cfg.block_size, stream=s)
    g = torch.cuda.CUDAGraph()
    out = torch.zeros_like(batch.q)
    with torch.cuda.graph(g, stream=s):
        U.run_cuda(batch, out=out, stream=s)
    for _ in range(2):
        out.zero_()
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        assert torch.equal(out, eager)
    U.compare(eager, U.run_oracle(batch), "swizzled V bs=%d S=%d" % (bs, S))
