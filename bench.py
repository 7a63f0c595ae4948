"""Benchmark: fp8 paged decode attention on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]

``--gpus N`` runs N replicas, one process per GPU: under torchrun its
WORLD_SIZE must equal N; without a launcher, N > 1 starts torchrun itself.

A step is one ``pda_decode`` call (split plan, page gather, dequant, QK^T,
online softmax, PV, CTA merge, partial store / LSE merge) over one batch of
synthetic input already resident in HBM. Steps are captured in CUDA graphs
(the pages time "impl.forward in a CUDA graph, us per call") and replayed;
the timed region is bracketed by a barrier and device synchronisation and
timed with CUDA events on the replay stream. Under torchrun every rank is an
independent replica on its own GPU (decode attention has no exchange step):
the value is the bytes all ranks moved over the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle (the parity reference) on the
host cores instead, on bounded samples of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "µs/call and achieved HBM GB/s (% of GB300 peak) for fp8 paged decode attention"
UNIT = "GB/s"
# The pages' own figure for the same workload (32/8 heads, ctx 4096, 256
# sequences, fp8 cache, 16-token blocks): 362.53 us/call for the asm kernel
# on AMD MI355X, i.e. this many GB/s for the same byte count. Context only.
PAGES_GBS_SAME_WORKLOAD = 2_151_941_120 / 362.53e-6 / 1e9
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=workloads.HEADLINE, choices=sorted(workloads.CONFIGS))
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--variant", choices=["plain", "slot_scales", "ex", "shuffled_v", "strided_nhd"], default="plain",
                    help="decode entry point: pda_decode, pda_decode_slot_scales (per-slot tables), "
                         "pda_decode_ex with per-head sinks and e4m3 output, pda_decode_ex on the "
                         "shuffled V layout, or pda_decode_strided on [NB, bs, Hk, 128] K and V")
    ap.add_argument("--op", choices=["decode", "cache_write"], default="decode",
                    help="cache_write: time pda_reshape_and_cache on --tokens new tokens of the config's kv heads")
    ap.add_argument("--tokens", type=int, default=65536)
    ap.add_argument("--cw-slots", choices=["random", "blocks"], default="blocks",
                    help="cache_write slots: a random permutation of the pool, or whole blocks in token order "
                         "(a prefill)")
    ap.add_argument("--profile", type=int, default=0, metavar="N",
                    help="profiling mode: N plain pda_decode calls on the config, no timing, no JSON metric")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, ws: int, device) -> float:
    """Max of a per-rank scalar over all ranks (the slowest replica's time)."""
    if ws <= 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(bytes_per_step_local: int, steps: int, elapsed_ms_local: float, ws: int, device):
    """Whole-job GB/s: bytes all ranks moved (equal work per replica) over the slowest rank's time."""
    ms = reduce_max(elapsed_ms_local, ws, device)
    return ws * bytes_per_step_local * steps / (ms * 1e-3) / 1e9, ms


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Clock event reasons that void a timed region (sw_power_cap is kept and noted).
REJECT_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")

# Calls in the roofline graph, each bracketed by kernel events (independent
# of --steps). It runs right after the timed region, inside the same clock
# sampling window; the timed region itself carries no event nodes.
ROOFLINE_CALLS = 24

# Kernel function behind each decode instance name the library reports.
KERNEL_FUNCTION = {"per-unit (3 CTAs/SM)": "pda_split_decode_kernel", "per-unit dense (4 CTAs/SM)":
                   "pda_split_decode_kernel", "persistent": "pda_persistent_decode_kernel"}


def kernel_source_sha() -> str:
    """Hash of the device sources the decode kernel is compiled from (host code excluded).

    Comments and blank lines are left out, so editing a comment keeps the
    recorded ncu traffic valid; any change to the code itself changes the hash.
    """
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_pda_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith(".cuh"):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                text = f.read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            text = re.sub(r"//[^\n]*", "", text)
            text = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
            h.update(name.encode() + b"\0" + text.encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it is for this kernel source."""
    p = os.path.join(ROOT, "profiles", "decode_kernel_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("source_sha") != kernel_source_sha():
        return None
    ent = d.get("per_workload", {}).get(workload)
    if not ent:
        return None
    return float(ent["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clock / throttle sampling around the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="pda_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        load = [x for x, p in zip(sm, pw)] if sm else []
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "samples": len(rows), "reasons": sorted(reasons)}


# Arm Ltd. (implementer 0x41) part numbers of server cores, as /proc/cpuinfo
# reports them on Arm hosts that give no model name.
ARM_PARTS = {"0xd0c": "Neoverse-N1", "0xd40": "Neoverse-V1", "0xd49": "Neoverse-N2", "0xd4f": "Neoverse-V2",
             "0xd84": "Neoverse-V3", "0xd8e": "Neoverse-N3"}


def host_cpu_name() -> str:
    """The host CPU model as the OS reports it (x86 'model name'; on Arm the
    core's name from its part number when no name is given), with the online
    core count."""
    name = ""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model", "CPU part"):
            for line in info.splitlines():
                if line.startswith(key):
                    name = line.split(":", 1)[1].strip()
                    break
            if name:
                if key == "CPU part":
                    name = "Arm %s (part %s)" % (ARM_PARTS[name], name) if name in ARM_PARTS else "Arm part " + name
                break
    except OSError:
        pass
    return "%s (%d cores online)" % (name or platform.machine(), os.cpu_count() or 0)


def oracle_sample_rate(batch, budget_s: float, max_seqs: int | None = None, threads: int = 0):
    """Time the fp64 oracle on the first n sequences of the batch, n grown
    until about budget_s of wall time, on `threads` OpenMP threads (0: all);
    returns (GB/s, description, threads, n, seconds)."""
    import oracle

    cfg = batch.cfg
    raw = batch.raw()
    threads = threads or oracle.max_threads()
    n = 1
    S = cfg.num_seqs if max_seqs is None else min(cfg.num_seqs, max_seqs)
    while True:
        ids = list(range(n))
        t0 = time.perf_counter()
        oracle.decode(**raw, scale=cfg.scale, k_scale=cfg.k_scale, v_scale=cfg.v_scale, seq_ids=ids,
                      num_threads=threads)
        dt = time.perf_counter() - t0
        if dt >= budget_s or n >= S:
            break
        n = min(S, max(n + 1, int(n * min(8.0, budget_s / max(dt, 1e-3)))))
    lens = [batch.seq_lens_host[i] for i in ids]
    sub = workloads.algorithmic_bytes(cfg.with_(num_seqs=n), lens)
    desc = "%d of %d sequences (all %d heads, their full contexts), %.2f s, %d OpenMP threads" % (
        n, cfg.num_seqs, cfg.num_heads, dt, threads)
    return sub / dt / 1e9, desc, threads, n, dt


# ---------------------------------------------------------------- our arm

def run_ours(args, ws, rank, local):
    import paged_kv_decode_pda_gb300 as pda
    from paged_kv_decode_pda_gb300 import build

    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build.build()
    pda.load()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    cfg = workloads.CONFIGS[args.config]
    batch = workloads.make_batch(cfg, device=dev, seed=cfg.seed + rank)
    bytes_per_call = workloads.algorithmic_bytes(cfg, batch.seq_lens_host)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    kv_bytes = batch.k_cache.numel() + batch.v_cache.numel()
    replicas = max(1, math.ceil(3 * l2 / kv_bytes))
    caches = [(batch.k_cache, batch.v_cache)] + [(batch.k_cache.clone(), batch.v_cache.clone())
                                                 for _ in range(replicas - 1)]
    nsplit = pda.plan_splits(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq,
                             cfg.block_size)
    if args.variant != "slot_scales":   # token-major caches plan like page-major ones
        kernels_per_call = pda.plan_launches(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads,
                                             cfg.max_num_blocks_per_seq, cfg.block_size)
        kernel_id = pda.plan_kernel(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq,
                                    cfg.block_size)
    else:   # the per-slot-scale entry point plans for itself
        kernel_id, nsplit, kernels_per_call = pda.plan_slot_scales(
            cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq, cfg.block_size)
    kernel_kind = pda.KERNEL_NAMES[kernel_id]
    stream = torch.cuda.Stream(device=dev)
    out = torch.empty_like(batch.q)
    pda.reserve(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq, cfg.block_size,
                stream=stream)

    call, out, bytes_per_call = make_variant_call(args.variant, cfg, batch, caches, out, bytes_per_call, stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            call(i)
    stream.synchronize()
    assert pda.query_device_status(stream) == 0

    # Graphs: the timed region replays graphs of `chunk` plain calls (and one
    # for the remainder); the roofline graph holds ROOFLINE_CALLS calls, each
    # bracketed by kernel events (an event node costs the bracketed call its
    # overlap with its neighbours, so these calls stay out of the timed region).
    K = args.steps
    chunk = min(K, 100)
    ev_pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(ROOFLINE_CALLS)]

    def capture(n, with_events):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                if with_events:
                    pda.set_profile_events(*ev_pairs[i])
                call(i)
                pda.set_profile_events(None, None)
        return g

    # Can kernel events recorded inside a graph be timed on this stack? Probe once.
    mode = "graph"
    try:
        g_probe = capture(1, True)
        with torch.cuda.stream(stream):
            g_probe.replay()
        stream.synchronize()
        ev_pairs[0][0].elapsed_time(ev_pairs[0][1])
        del g_probe
    except Exception:
        mode = "eager"
        torch.cuda.synchronize()
    if mode == "graph":
        g_main = capture(chunk, False)
        rem = K % chunk
        g_rem = capture(rem, False) if rem else None
        g_roof = capture(ROOFLINE_CALLS, True)
        with torch.cuda.stream(stream):
            g_main.replay()
            g_roof.replay()
        stream.synchronize()

    def timed_region():
        sampler = ClockSampler(local)
        sampler.start()
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t_start.record(stream)
            if mode == "graph":
                for _ in range(K // chunk):
                    g_main.replay()
                if g_rem is not None:
                    g_rem.replay()
            else:
                # host enqueue (~10 us) stays far below the kernel time
                for i in range(K):
                    call(i)
            t_end.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        # roofline calls: the same calls, each with kernel events around the
        # decode kernel, right after the timed region
        with torch.cuda.stream(stream):
            if mode == "graph":
                g_roof.replay()
            else:
                for i in range(ROOFLINE_CALLS):
                    pda.set_profile_events(*ev_pairs[i])
                    call(i)
                    pda.set_profile_events(None, None)
        stream.synchronize()
        clocks = sampler.stop()
        return t_start, t_end, clocks

    t_start, t_end, clocks = timed_region()
    remeasured = False
    throttled = any(r in REJECT_REASONS for r in clocks.get("reasons", []))
    if reduce_max(1.0 if throttled else 0.0, ws, dev) > 0:   # every rank decides alike
        # a throttled run does not count: take the timed region once more
        t_start, t_end, clocks = timed_region()
        remeasured = True
    elapsed_ms = t_start.elapsed_time(t_end)
    kern_ms = sorted(a.elapsed_time(b) for a, b in ev_pairs)
    assert pda.query_device_status(stream) == 0

    value, elapsed_ms = aggregate_throughput(bytes_per_call, K, elapsed_ms, ws, dev)

    # ---- end to end through the public API from pinned host buffers
    e2e = None
    if args.e2e_steps > 0 and args.variant == "plain":
        host = {k: v.detach().cpu().pin_memory() for k, v in
                dict(q=batch.q, k=batch.k_cache, v=batch.v_cache, t=batch.block_tables, l=batch.seq_lens).items()}
        out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = out_host.numel() * out_host.element_size()

        def e2e_step():
            # one C-ABI call on host buffers: copies in, decode, copy out
            pda.decode_host(host["q"], host["k"], host["v"], host["t"], host["l"], cfg.scale, cfg.k_scale,
                            cfg.v_scale, out=out_host, stream=stream)

        with torch.cuda.stream(stream):
            e2e_step()
        stream.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.e2e_steps):
                e2e_step()
            e1.record(stream)
        stream.synchronize()
        e2e_value, e2e_ms = aggregate_throughput(bytes_per_call, args.e2e_steps, e0.elapsed_time(e1), ws, dev)
        e2e = {"value": e2e_value, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.e2e_steps,
               "path": "pinned host -> pda_decode_host (cudaMemcpyAsync of each input, pda_decode, "
                       "cudaMemcpyAsync of the output) -> pinned host"}
        del host

    # ---- a serving decode step: the KV cache stays resident; each step ships
    # q, one new K/V token per sequence, its slot, the tables and lengths,
    # writes the new tokens with pda_reshape_and_cache, decodes, and reads
    # the output back. Same metric (algorithmic decode bytes per step time).
    e2e_step_line = None
    if args.e2e_steps > 0 and args.variant == "plain":
        S, Hk = cfg.num_seqs, cfg.num_kv_heads
        g = torch.Generator().manual_seed(cfg.seed + 17)
        lens_h = torch.tensor(batch.seq_lens_host, dtype=torch.int64)
        last = torch.clamp(lens_h - 1, min=0)
        tables_h = batch.block_tables.cpu().to(torch.int64)
        slots_h = tables_h[torch.arange(S), last // cfg.block_size] * cfg.block_size + last % cfg.block_size
        slots_h[lens_h == 0] = -1
        parts = {"q": batch.q.detach().cpu(),
                 "k_new": (torch.randn(S, Hk, 128, generator=g) * 2).to(torch.bfloat16),
                 "v_new": (torch.randn(S, Hk, 128, generator=g) * 2).to(torch.bfloat16),
                 "slots": slots_h,
                 "t": batch.block_tables.cpu(),
                 "l": batch.seq_lens.cpu()}
        # One pinned host buffer and one device buffer hold all of a step's
        # inputs (256-byte aligned parts), so a step is a single copy in.
        offs, total = {}, 0
        for k, v in parts.items():
            offs[k] = total
            total += (v.numel() * v.element_size() + 255) // 256 * 256
        blob_h = torch.empty(total, dtype=torch.uint8).pin_memory()
        blob_d = torch.empty(total, dtype=torch.uint8, device=dev)

        def view(blob, k):
            v = parts[k]
            n = v.numel() * v.element_size()
            return blob[offs[k]:offs[k] + n].view(v.dtype).view(v.shape)

        for k, v in parts.items():
            view(blob_h, k).copy_(v)
        dev_bufs = {k: view(blob_d, k) for k in parts}
        out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        kc, vc = caches[0]
        h2d = total
        d2h = out_host.numel() * out_host.element_size()

        def serving_step():
            blob_d.copy_(blob_h, non_blocking=True)
            pda.reshape_and_cache(dev_bufs["k_new"], dev_bufs["v_new"], kc, vc, dev_bufs["slots"], cfg.k_scale,
                                  cfg.v_scale, stream=stream)
            pda.decode(dev_bufs["q"], kc, vc, dev_bufs["t"], dev_bufs["l"], cfg.scale, cfg.k_scale, cfg.v_scale,
                       out=out, stream=stream)
            out_host.copy_(out, non_blocking=True)

        with torch.cuda.stream(stream):
            for _ in range(3):
                serving_step()
        stream.synchronize()
        # A server replays its step as a CUDA graph (copies included).
        per_graph = 10
        step_mode = "graph"
        try:
            g_step = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_step, stream=stream):
                for _ in range(per_graph):
                    serving_step()
            with torch.cuda.stream(stream):
                g_step.replay()
            stream.synchronize()
        except Exception:
            step_mode = "eager"
            torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        n_steps = per_graph * max(2, args.e2e_steps)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n_steps // per_graph):
                if step_mode == "graph":
                    g_step.replay()
                else:
                    for _ in range(per_graph):
                        serving_step()
            e1.record(stream)
        stream.synchronize()
        assert pda.query_device_status(stream) == 0
        serial_ms = e0.elapsed_time(e1) / n_steps

        # Pipelined, as a server runs it: step i's inputs cross on a copy-in
        # stream while step i-1 decodes, and step i-1's output comes back on
        # a copy-out stream while step i decodes. Two device input buffers
        # and two outputs; events order every reuse.
        blob_d2 = [blob_d, torch.empty_like(blob_d)]
        dev_bufs2 = [dev_bufs, {k: view(blob_d2[1], k) for k in parts}]
        outs = [out, torch.empty_like(out)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_read = [torch.cuda.Event() for _ in range(2)]

        def pipelined(n):
            for i in range(n):
                b = i % 2
                if i >= 2:
                    s_in.wait_event(ev_done[b])      # step i-2 has finished reading buffer b
                with torch.cuda.stream(s_in):
                    blob_d2[b].copy_(blob_h, non_blocking=True)
                    ev_in[b].record(s_in)
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_read[b])    # step i-2's output has been read back
                db = dev_bufs2[b]
                pda.reshape_and_cache(db["k_new"], db["v_new"], kc, vc, db["slots"], cfg.k_scale, cfg.v_scale,
                                      stream=stream)
                pda.decode(db["q"], kc, vc, db["t"], db["l"], cfg.scale, cfg.k_scale, cfg.v_scale, out=outs[b],
                           stream=stream)
                ev_done[b].record(stream)
                s_out.wait_event(ev_done[b])
                with torch.cuda.stream(s_out):
                    out_host.copy_(outs[b], non_blocking=True)
                    ev_read[b].record(s_out)

        pipelined(4)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)
        pipelined(n_steps)
        stream.wait_stream(s_out)
        e1.record(stream)
        torch.cuda.synchronize()
        assert pda.query_device_status(stream) == 0
        v_step, ms_step = aggregate_throughput(bytes_per_call, n_steps, e0.elapsed_time(e1), ws, dev)
        e2e_step_line = {"value": v_step, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "ms_per_step": ms_step / n_steps, "steps": n_steps, "launch": "pipelined",
                         "serial_ms_per_step": serial_ms, "serial_launch": step_mode,
                         "path": "pinned host -> one cudaMemcpyAsync (q, new K/V tokens, slots, tables, lengths) -> "
                                 "pda_reshape_and_cache -> pda_decode -> cudaMemcpyAsync -> pinned host; "
                                 "KV cache resident in HBM; pipelined: copies of neighbouring steps overlap the "
                                 "decode on two copy streams"}
        del dev_bufs, dev_bufs2, blob_h, blob_d, blob_d2

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return

    peak, peak_kind = peaks()
    kern_median_ms = statistics.median(kern_ms)
    us_per_call = elapsed_ms * 1e3 / K
    # A call that is one kernel launch: the timed region's CUDA events give
    # that kernel's average launch duration directly (launch gaps included,
    # so never an underestimate), without the event nodes' cost to the
    # bracketed calls. Calls of several launches use the bracketed median.
    single_launch = kernels_per_call == 1
    kern_used_us = us_per_call if single_launch else kern_median_ms * 1e3
    achieved = bytes_per_call / (kern_used_us * 1e-6) / 1e9
    traffic = ncu_traffic(cfg.name) if args.variant == "plain" else None

    cpu = None
    if not args.no_cpu_baseline:
        rate, desc, cores, _, _ = oracle_sample_rate(batch, budget_s=10.0)
        rate1, desc1, _, _, _ = oracle_sample_rate(batch, budget_s=4.0, threads=1)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
               "one_core": {"value": rate1, "sample": desc1}, "host_cpu": host_cpu_name()}

    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": ws,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": elapsed_ms / K,
        "us_per_call": us_per_call,
        "frac_of_peak_hbm": value / ws / peak,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": value / ws / PAGES_GBS_SAME_WORKLOAD,
        "vs_baseline_note": "pages' asm kernel on AMD MI355X, 362.53 us/call for this workload (context only)",
        "dtype": "f16",
        "dtype_detail": "f16 MMA operands: e4m3 KV converted exactly, each bf16 q row shifted by a power of two "
                        "into f16's range (exact within 2^24 of the row's largest), probabilities as two f16 parts; "
                        "fp32 accumulation and softmax, bf16 out",
        "data": "synthetic (seeded N(0,1) q; K/V N(0,1) quantised to e4m3 with scale 0.05; shuffled block tables)",
        "config": {"workload": cfg.name, "variant": args.variant, "num_seqs": cfg.num_seqs, "num_heads": cfg.num_heads,
                   "num_kv_heads": cfg.num_kv_heads, "head_size": cfg.head_size, "block_size": cfg.block_size,
                   "ctx": cfg.ctx if cfg.ctx else list(cfg.ctx_range), "kv_splits": nsplit, "decode_kernel": kernel_kind,
                   "bytes_per_call": bytes_per_call,
                   "l2": "KV pool %.2f GB x %d replica(s) >= 3x L2 (%d MB); no flush needed" % (
                       kv_bytes / 1e9, replicas, l2 >> 20),
                   "timing": ("CUDA graphs of %d calls replayed" % chunk if mode == "graph" else
                              "eager launches (host enqueue << kernel time)") + "; CUDA events on the launch stream",
                   "parallelism": "replicas x%d" % ws},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_kind,
                     "kernel": KERNEL_FUNCTION[kernel_kind],
                     "timed_span": ("the timed region's CUDA events over its %d launches of the decode kernel "
                                    "(one launch per call)" % K) if single_launch else
                                   ("profile events around the decode kernel (with the unit-order kernel that "
                                    "precedes the persistent kernel and the tail merge kernel that follows it) "
                                    "of each of %d calls replayed as one graph "
                                    "right after the timed region, in the same clock window; achieved uses the "
                                    "median" % ROOFLINE_CALLS),
                     "kernel_us": kern_used_us,
                     "kernel_us_median": kern_median_ms * 1e3,
                     "kernel_us_min": kern_ms[0] * 1e3, "kernel_us_max": kern_ms[-1] * 1e3,
                     "kernel_us_mean": statistics.fmean(kern_ms) * 1e3,
                     "kernel_launches_timed": K if single_launch else len(kern_ms),
                     "bracketed_calls": len(kern_ms), "algorithmic_bytes_per_launch": bytes_per_call,
                     "call_frac": bytes_per_call / (us_per_call * 1e-6) / 1e9 / peak},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "e2e_serving_step": e2e_step_line,
        "clocks": dict(clocks, remeasured_after_throttle=remeasured),
        "gpu_launches": K * kernels_per_call,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------- reference arm

def run_reference(args, ws, rank, local):
    if rank != 0:
        return
    import oracle

    cfg = workloads.CONFIGS[args.config]
    batch = workloads.make_batch(cfg, device="cpu")
    raw = batch.raw()
    # Size each step so the whole run stays within about three minutes.
    budget_total = 120.0
    per_step = max(0.02, budget_total / max(1, args.steps + args.warmup))
    _, _, cores, n, dt = oracle_sample_rate(batch, budget_s=per_step)
    ids = list(range(n))
    lens = [batch.seq_lens_host[i] for i in ids]
    sample_bytes = workloads.algorithmic_bytes(cfg.with_(num_seqs=n), lens)

    def step():
        oracle.decode(**raw, scale=cfg.scale, k_scale=cfg.k_scale, v_scale=cfg.v_scale, seq_ids=ids,
                      num_threads=cores)

    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = sample_bytes * args.steps / total / 1e9
    desc = "%d of %d sequences (all %d heads, full contexts) per step, %d OpenMP threads" % (
        n, cfg.num_seqs, cfg.num_heads, cores)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (same generator and seed as the CUDA arm)",
        "config": {"workload": cfg.name, "sample": desc},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def make_variant_call(variant, cfg, batch, caches, out, bytes_per_call, stream):
    """The per-call closure for one decode variant, its output and its algorithmic bytes per call.

    ``caches`` is a list of (K, V) replicas in the native layout; call(i)
    reads replica i mod len(caches).
    """
    import paged_kv_decode_pda_gb300 as pda

    dev = batch.q.device
    replicas = len(caches)
    if variant == "slot_scales":
        # per-slot tables filled with the per-tensor scales (the pages' use)
        ks_t = torch.full((batch.num_blocks, cfg.num_kv_heads, cfg.block_size), cfg.k_scale, device=dev)
        vs_t = torch.full_like(ks_t, cfg.v_scale)
        pages_used = batch.pages_used()
        bytes_per_call += 2 * pages_used * cfg.block_size * 4 * cfg.num_kv_heads
    elif variant == "ex":
        sinks = torch.randn(cfg.num_heads, generator=torch.Generator().manual_seed(3)).float().to(dev)
        out = torch.empty(batch.q.shape, dtype=torch.float8_e4m3fn, device=dev)
        bytes_per_call -= out.numel()   # 1-byte instead of 2-byte output
        bytes_per_call += cfg.num_heads * 4
    elif variant == "shuffled_v":
        def shuffle(v):
            NB, Hk, D, bs = v.shape
            return v.reshape(NB, Hk, D, bs // 16, 16).permute(0, 1, 3, 2, 4).contiguous()
        caches = [(k, shuffle(v)) for k, v in caches]
    elif variant == "strided_nhd":
        def nhd(k, v):
            NB, Hk, C, bs, _ = k.shape
            kt = k.view(torch.uint8).permute(0, 3, 1, 2, 4).reshape(NB, bs, Hk, 128).contiguous()
            vt = v.view(torch.uint8).permute(0, 3, 1, 2).contiguous()
            return kt, vt
        caches = [nhd(k, v) for k, v in caches]
        hk, bsz = cfg.num_kv_heads, cfg.block_size
        nhd_strides = (bsz * hk * 128, hk * 128, 128)
    # The variant inputs above were made on torch's current stream; the calls
    # run on `stream`.
    torch.cuda.synchronize(dev)

    def call(i):
        kc, vc = caches[i % replicas]
        if variant == "strided_nhd":
            pda.decode_strided(batch.q, kc.data_ptr(), vc.data_ptr(), batch.block_tables, batch.seq_lens, cfg.scale,
                               cfg.k_scale, cfg.v_scale, num_kv_heads=hk, block_size=bsz,
                               num_blocks=batch.num_blocks, k_strides=nhd_strides, v_strides=nhd_strides, out=out,
                               stream=stream)
        elif variant == "shuffled_v":
            pda.decode_ex(batch.q, kc, vc, batch.block_tables, batch.seq_lens, cfg.scale, cfg.k_scale, cfg.v_scale,
                          v_shuffled=True, out=out, stream=stream)
        elif variant == "slot_scales":
            pda.decode_slot_scales(batch.q, kc, vc, ks_t, vs_t, batch.block_tables, batch.seq_lens, cfg.scale,
                                   out=out, stream=stream)
        elif variant == "ex":
            pda.decode_ex(batch.q, kc, vc, batch.block_tables, batch.seq_lens, cfg.scale, cfg.k_scale, cfg.v_scale,
                          sinks=sinks, output_scale=0.0075, out=out, stream=stream)
        else:
            pda.decode(batch.q, kc, vc, batch.block_tables, batch.seq_lens, cfg.scale, cfg.k_scale, cfg.v_scale,
                       out=out, stream=stream)

    return call, out, bytes_per_call


def run_profile(args):
    """N calls of one decode variant, untimed (what an ncu capture of this command sees)."""
    import paged_kv_decode_pda_gb300 as pda
    from paged_kv_decode_pda_gb300 import build

    torch.cuda.set_device(0)
    build.build()
    cfg = workloads.CONFIGS[args.config]
    batch = workloads.make_batch(cfg, device="cuda:0")
    stream = torch.cuda.current_stream()
    call, out, bytes_per_call = make_variant_call(args.variant, cfg, batch, [(batch.k_cache, batch.v_cache)],
                                                  torch.empty_like(batch.q),
                                                  workloads.algorithmic_bytes(cfg, batch.seq_lens_host), stream)
    for i in range(args.profile):
        call(i)
    torch.cuda.synchronize()
    code = pda.query_device_status()
    nsplit = pda.plan_splits(cfg.num_seqs, cfg.num_heads, cfg.num_kv_heads, cfg.max_num_blocks_per_seq,
                             cfg.block_size)
    print(json.dumps({"profile_calls": args.profile, "workload": cfg.name, "variant": args.variant,
                      "kv_splits": nsplit, "bytes_per_call": bytes_per_call,
                      "device_status": code}))
    if code:
        raise SystemExit(1)


def run_cache_write(args):
    """Time the KV-cache write (quantise + scatter) on one GPU; one JSON line."""
    import paged_kv_decode_pda_gb300 as pda
    from paged_kv_decode_pda_gb300 import build

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    cfg = workloads.CONFIGS[args.config]
    T, Hk, bs = args.tokens, cfg.num_kv_heads, cfg.block_size
    g = torch.Generator(device=dev).manual_seed(cfg.seed)
    NB = max(1, (T + bs - 1) // bs) * 2
    key = torch.randn(T, Hk, 128, generator=g, device=dev).to(torch.bfloat16)
    val = torch.randn(T, Hk, 128, generator=g, device=dev).to(torch.bfloat16)
    if args.cw_slots == "random":
        slots = torch.randperm(NB * bs, generator=g, device=dev)[:T].to(torch.int64)
    else:
        blocks = torch.randperm(NB, generator=g, device=dev)
        t = torch.arange(T, device=dev)
        slots = (blocks[t // bs] * bs + t % bs).to(torch.int64)
    kc = torch.zeros(NB, Hk, 8, bs, 16, dtype=torch.uint8, device=dev)
    vc = torch.zeros(NB, Hk, 128, bs, dtype=torch.uint8, device=dev)
    nbytes = T * Hk * 128 * (2 + 2 + 1 + 1) + T * 8
    stream = torch.cuda.Stream(device=dev)

    def call():
        pda.reshape_and_cache(key, val, kc, vc, slots, cfg.k_scale, cfg.v_scale, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            call()
    stream.synchronize()
    K = args.steps
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        for _ in range(min(K, 100)):
            call()
    reps = max(1, K // min(K, 100))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            gr.replay()
        e1.record(stream)
    stream.synchronize()
    n_calls = reps * min(K, 100)
    us = e0.elapsed_time(e1) * 1e3 / n_calls
    assert pda.query_device_status(stream) == 0
    peak, kind = peaks()
    print(json.dumps({"op": "cache_write", "metric": "us/call and GB/s of pda_reshape_and_cache", "value": nbytes / us / 1e3,
                      "unit": "GB/s", "us_per_call": us, "calls": n_calls, "tokens": T, "slots": args.cw_slots, "num_kv_heads": Hk,
                      "block_size": bs, "bytes_per_call": nbytes,
                      "roofline": {"bound": "hbm", "achieved": nbytes / us / 1e3, "peak": peak, "unit": "GB/s",
                                   "frac": nbytes / us / 1e3 / peak, "peak_source": kind}}), flush=True)


def spawn_replicas(n: int) -> int:
    """--gpus N > 1 without a launcher: run this command as N ranks under
    torchrun (one process per GPU, rendezvous on 127.0.0.1), rank 0 printing
    the JSON line; returns torchrun's exit status."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(n),
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.run(cmd).returncode


def main():
    args = parse()
    if args.gpus < 1:
        raise SystemExit("bench.py: --gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(spawn_replicas(args.gpus))
    ws, rank, local = dist_env()
    if ws != args.gpus:
        raise SystemExit("bench.py: --gpus %d but the launcher started %d rank(s) (WORLD_SIZE); "
                         "they must agree" % (args.gpus, ws))
    if args.profile:
        run_profile(args)
        return
    if args.op == "cache_write":
        if rank == 0:
            run_cache_write(args)
        return
    if args.impl == "reference":
        run_reference(args, ws, rank, local)
    else:
        run_ours(args, ws, rank, local)


if __name__ == "__main__":
    main()
