"""Benchmark of the delta-sync hot path on GB300: compress (trainer side) + verified in-place
apply (rollout side) of a synthetic BF16 checkpoint pair.

One step = bd_compress_batch over every tensor (XOR, classify, pack, checksum of new) followed
by bd_decompress_batch over every tensor (decode, scatter-XOR into the rollout copy, verify the
checksum).  The rollout copy alternates between old and new from step to step (XOR is an
involution), so every step is a full compress + a full verified apply, against checksum(new)
on odd steps and checksum(old) on even ones.

Prints one JSON line.  `value` is raw BF16 GB/s through the whole step (2 bytes per element
of one checkpoint divided by compress+apply time), summed over ranks for N > 1 (independent
replicas, weak scaling).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload dense7b] [--impl reference]

`--profile-case embed|layers|moe|dense|formats` runs a fixed small program for an ncu capture
instead (no timing, no JSON line), two rounds of: compress in each version, the full verified
apply and the incremental apply of each payload.  `embed`: the 32000x4096 embedding tensor of
dense7b in versions 1, 3 and 4 (the separate compress kernels), plus the standalone checksum, an
out-of-place apply and the apply without a workspace; `layers`: the 18 tensors of dense7b's first two layers in versions 1, 3
and 4 (the fused compress); `dense`: a 2^26-element tensor made by the 1 GiB workload's rule
(22% changed: the dense emit and apply) in versions 1 and 3, plus the checksum and an
out-of-place apply; `moe`: the 389 tensors of moe30b's layer 0 (cold experts with 0.64% of
their elements changed, 8 hot ones with 40%) in versions 1, 3 and 4; `formats`: the whole
--workload in versions 3 and 4.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "compress & apply GB/s of raw BF16 weights (% of HBM roofline); payload % raw"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0


def _peak_hbm() -> tuple[float, str]:
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _workload_specs(name: str) -> list[W.Spec]:
    if "@" in name:  # one tensor of a workload, e.g. sweep14336@rate0.02
        base, which = name.split("@", 1)
        return [s for s in W.specs(base) if s.name == which]
    return W.specs(name)


def _describe(name: str, specs: list[W.Spec]) -> str:
    n = sum(s.numel for s in specs)
    return f"{name}: {len(specs)} BF16 tensors, {n:,} elements ({2 * n / 1e9:.2f} GB per checkpoint)"


def _source_hash(files) -> str:
    """Hash of the named CUDA sources, to tell whether stored ncu counters still apply."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "lossless_bf16_weight_old_gb300", "csrc")
    for f in sorted(files):
        h.update(f.encode())
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic(workload: str, phase: str, n_total: int):
    """DRAM bytes (read + write) of one call of `phase` on this workload, from the committed
    ncu capture of the same kernels on a smaller case of the same kind, scaled by elements
    (profiles/dram_traffic.json); None when there is none for this workload or the kernels'
    sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f).get("phases", {}).get(phase, {})
    except (OSError, ValueError):
        return None
    if workload not in entry.get("scales_to", []):
        return None
    try:
        if entry.get("source_hash") != _source_hash(entry["sources"]):
            return None
    except (OSError, KeyError):
        return None
    return int(round(entry["bytes_per_element"] * n_total))


# ------------------------------------------------------------------------ multi-rank helpers

def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None) -> None:
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------------------ clocks

def _smi_id(dev, local: int) -> str:
    """nvidia-smi -i argument for this device: its UUID when torch exposes it."""
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    if uuid:
        u = str(uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------ oracle baseline

def _sample(specs: list[W.Spec], budget: int) -> list[W.Spec]:
    """Tensors of the workload in order, skipping any larger than the budget, until the
    budget of elements is reached (at least one tensor)."""
    out, tot = [], 0
    for s in specs:
        if tot + s.numel > budget:
            continue
        out.append(s)
        tot += s.numel
    return out or [min(specs, key=lambda s: s.numel)]


def oracle_baseline(specs: list[W.Spec], budget_elems: int, device) -> dict:
    """Times the CPU oracle (single thread) on a bounded sample of the workload's tensors."""
    import numpy as np
    import oracle
    oracle.build()
    sample = _sample(specs, budget_elems)
    t_enc = t_dec = 0.0
    elems = 0
    for s in sample:
        old, new = W.make_pair(s, device=device)
        o = old.reshape(-1).view(torch.int16).cpu().numpy().view(np.uint16)
        nw = new.reshape(-1).view(torch.int16).cpu().numpy().view(np.uint16)
        del old, new
        t0 = time.perf_counter()
        payload, ck = oracle.encode(o, nw)
        t1 = time.perf_counter()
        st, restored = oracle.decode(o, payload, ck)
        t2 = time.perf_counter()
        if st != oracle.OK or not np.array_equal(restored, nw):
            raise RuntimeError("oracle roundtrip failed")
        t_enc += t1 - t0
        t_dec += t2 - t1
        elems += o.size
    gbs = 2 * elems / (t_enc + t_dec) / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{len(sample)} tensors ({elems:,} elements) of the workload: "
                      f"encode {t_enc:.2f} s + decode {t_dec:.2f} s, single thread",
            "encode_gbs": round(2 * elems / t_enc / 1e9, 4),
            "decode_gbs": round(2 * elems / t_dec / 1e9, 4)}


# ---- the same oracle fanned out per tensor over the host's cores (spawned processes: a pool
# forked after CUDA is initialised can hang)

def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _shares(sample: list[W.Spec], workers: int) -> list[list[W.Spec]]:
    """Tensors split over workers, largest first onto the least loaded."""
    shares = [[] for _ in range(workers)]
    load = [0] * workers
    for s in sorted(sample, key=lambda s: -s.numel):
        i = load.index(min(load))
        shares[i].append(s)
        load[i] += s.numel
    return [sh for sh in shares if sh]


_FANOUT_PAIRS = []


def _fanout_init(share: list, barrier) -> None:
    """Worker start-up: build this worker's tensors on the CPU (outside any timing)."""
    import numpy as np
    torch.set_num_threads(1)
    import oracle  # noqa: F401  (loads the library once)
    for s in share:
        old, new = W.make_pair(s, device="cpu")
        _FANOUT_PAIRS.append((old.reshape(-1).view(torch.int16).numpy().view(np.uint16).copy(),
                              new.reshape(-1).view(torch.int16).numpy().view(np.uint16).copy()))
    if barrier is not None:
        barrier.wait()


def _fanout_run(_=None):
    """One pass of the oracle (encode + verified decode) over this worker's tensors."""
    import oracle
    t0 = time.perf_counter()
    elems = 0
    for o, nw in _FANOUT_PAIRS:
        payload, ck = oracle.encode(o, nw)
        st, _r = oracle.decode(o, payload, ck)
        if st != oracle.OK:
            raise RuntimeError("oracle roundtrip failed")
        elems += o.size
    return t0, time.perf_counter(), elems


def _fanout_worker(share: list, barrier, q) -> None:
    _fanout_init(share, barrier)
    q.put(_fanout_run())


def oracle_fanout(specs: list[W.Spec], budget_elems: int, workers: int | None = None) -> dict:
    """The CPU oracle on a bounded sample of the workload, one process per host core, each
    taking whole tensors: wall time from the first start to the last finish."""
    import multiprocessing as mp
    import oracle
    oracle.build()
    workers = workers or _host_cores()
    sample = _sample(specs, budget_elems)
    shares = _shares(sample, workers)
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(len(shares))
    q = ctx.Queue()
    procs = [ctx.Process(target=_fanout_worker, args=(sh, barrier, q)) for sh in shares]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=1800) for _ in procs]
    for pr in procs:
        pr.join(timeout=60)
    wall = max(r[1] for r in res) - min(r[0] for r in res)
    elems = sum(r[2] for r in res)
    return {"value": round(2 * elems / wall / 1e9, 4), "unit": "GB/s", "cores": len(shares),
            "kind": "oracle",
            "sample": f"{len(sample)} tensors ({elems:,} elements) of the workload over "
                      f"{len(shares)} processes, one per host core: {wall:.2f} s wall"}


def _fanout_loop(share: list, conn) -> None:
    """Persistent worker of the reference arm: builds its tensors, then runs one oracle pass
    per request until told to stop."""
    _fanout_init(share, None)
    conn.send("ready")
    while conn.recv() is not None:
        conn.send(_fanout_run())


def run_reference(args) -> None:
    """The reference arm: the CPU oracle as it stands, fanned out per tensor over the host's
    cores (one spawned process per core), same metric and unit as the GPU arm."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import multiprocessing as mp
    import oracle
    oracle.build()
    specs = _workload_specs(args.workload)
    # each step: one bounded sample of the workload's tensors, generated on the CPU by the
    # workers before timing starts
    sample = _sample(specs, args.ref_sample_elems)
    shares = _shares(sample, _host_cores())
    ctx = mp.get_context("spawn")
    pipes, procs = [], []
    for sh in shares:
        parent, child = ctx.Pipe()
        pr = ctx.Process(target=_fanout_loop, args=(sh, child))
        pr.start()
        pipes.append(parent)
        procs.append(pr)
    for c in pipes:
        if c.recv() != "ready":
            raise RuntimeError("reference worker failed to start")
    elems = sum(s.numel for s in sample)

    def step():
        for c in pipes:
            c.send("go")
        return [c.recv() for c in pipes]

    try:
        for _ in range(args.warmup):
            step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        dt = (time.perf_counter() - t0) / args.steps
    finally:
        for c in pipes:
            c.send(None)
        for pr in procs:
            pr.join(timeout=60)
    gbs = 2 * elems / dt / 1e9
    desc = (f"{len(sample)} tensors ({elems:,} elements) of {_describe(args.workload, specs)}, "
            f"over {len(shares)} processes")
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u16", "data": "synthetic",
            "config": {"workload": desc,
                       "where": f"host CPU, CPU oracle, one process per core ({len(shares)})"},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": len(shares),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------ GPU arm

def _host_mem_available() -> int:
    """Bytes of host memory this process may still use (the smaller of the free physical
    memory and the room left under a cgroup limit)."""
    try:
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError, AttributeError):
        avail = 1 << 62
    try:
        with open("/sys/fs/cgroup/memory.max") as f:
            lim = f.read().strip()
        with open("/sys/fs/cgroup/memory.current") as f:
            cur = int(f.read().strip())
        if lim != "max":
            avail = min(avail, int(lim) - cur)
    except (OSError, ValueError):
        pass
    return avail


L2_FLUSH_BYTES = 256 << 20     # twice the GB300's L2
E2E_GROUP_BYTES = 1 << 30      # old + new bytes per group of the e2e pipeline
STREAM_SLOT_BYTES = 64 << 20   # device slot of the streamed apply (two of them)
FLUSH_BELOW = 1 << 30          # flush L2 between timed runs when old + new are under 1 GiB


def run_ours(args) -> None:
    import lossless_bf16_weight_old_gb300 as bd

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    bd._lib.load()

    specs = _workload_specs(args.workload)
    ns = [s.numel for s in specs]
    n_total = sum(ns)
    k = len(specs)
    # flat buffers: old (trainer before), new (trainer after), rollout copy
    offs, o = [], 0
    for n in ns:
        offs.append(o)
        o += (n + 127) // 128 * 128
    O = torch.empty(o, dtype=torch.bfloat16, device=dev)
    N = torch.empty(o, dtype=torch.bfloat16, device=dev)
    for s, off, n in zip(specs, offs, ns):
        a, b = W.make_pair(s, device=dev)
        O[off:off + n].copy_(a.reshape(-1))
        N[off:off + n].copy_(b.reshape(-1))
        del a, b
    olds = [O[off:off + n] for off, n in zip(offs, ns)]
    news = [N[off:off + n] for off, n in zip(offs, ns)]
    Rb = O.clone()
    rolls = [Rb[off:off + n] for off, n in zip(offs, ns)]
    torch.cuda.synchronize()

    # small workloads: flush L2 (write twice its size) before every timed phase, outside the
    # phase's events; larger ones stream more than L2 by themselves
    flush = 4 * n_total < FLUSH_BELOW
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None

    # touched 32-byte sectors (16 elements) -- algorithmic write bytes of the in-place apply
    touched = 0
    for a, b in zip(olds, news):
        m = len(a) // 16 * 16
        diff = a.view(torch.int16) != b.view(torch.int16)
        touched += int(diff[:m].view(-1, 16).any(1).sum().item()) + int(diff[m:].any().item())
        del diff

    stream = torch.cuda.current_stream()
    # one workspace per direction, shared by every batch below (they run one after another)
    ws_c = torch.empty(max(bd.compress_workspace_size(ns), 256), dtype=torch.uint8, device=dev)
    ws_d = torch.empty(max(bd.decompress_workspace_size(ns), 256), dtype=torch.uint8,
                       device=dev)

    def sized_batch(src, dst, **kw):
        """A compress batch whose payload buffers have exactly the sizes the update needs
        (a first run with no room reports them)."""
        probe = bd.CompressBatch(src, dst, caps=[0] * k, workspace=ws_c, **kw)
        probe.run(stream)
        torch.cuda.synchronize()
        need = [int(v) for v in probe.sizes.tolist()]
        del probe
        b = bd.CompressBatch(src, dst, caps=need, workspace=ws_c, **kw)
        b.run(stream)
        torch.cuda.synchronize()
        if int(b.status.item()) != bd.OK:
            raise RuntimeError(f"compress status {int(b.status.item())}")
        return b, need

    comp, sizes = sized_batch(olds, news)
    payload_bytes = sum(sizes)
    ck_new = comp.checksums.clone()
    ck_old = torch.empty_like(ck_new)
    for i, a in enumerate(olds):
        ck_old[i:i + 1].copy_(bd.checksum(a))
    dec_to_new = bd.DecompressBatch(rolls, comp.payloads, sizes, ck_new, workspace=ws_d)
    dec_to_old = bd.DecompressBatch(rolls, comp.payloads, sizes, ck_old, workspace=ws_d)
    torch.cuda.synchronize()

    state = {"new": False}

    def step(evs=None, flush_l2=flush):
        if flush_l2:
            flush_buf.zero_()
        if evs is not None:
            evs[0].record(stream)
        comp.run(stream)
        if evs is not None:
            evs[1].record(stream)
        if flush_l2:
            flush_buf.zero_()
        if evs is not None:
            evs[2].record(stream)
        d = dec_to_old if state["new"] else dec_to_new
        d.run(stream)
        state["new"] = not state["new"]
        if evs is not None:
            evs[3].record(stream)
        return d

    clocks = ClockSampler(_smi_id(dev, local))
    clocks.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world, dev)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    last = None
    for i in range(args.steps):
        last = step(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world, dev)
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = start.elapsed_time(end)
    t_comp = [e[0].elapsed_time(e[1]) for e in evs]
    t_app = [e[2].elapsed_time(e[3]) for e in evs]

    # correctness of the timed work (outside the timed region)
    st_c, st_d = int(comp.status.item()), int(last.status.item())
    want = N if state["new"] else O
    if st_c != bd.OK or st_d != bd.OK or not torch.equal(Rb.view(torch.int16), want.view(torch.int16)):
        raise RuntimeError(f"timed steps did not verify: compress {st_c}, apply {st_d}")

    # small workloads: the same step with each call captured once in a CUDA graph and replayed
    # (one graph launch per phase instead of a dozen host-side launches), L2 flushed likewise
    graph_rep = None
    if flush:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graphs = {}
        for name, call in (("compress", comp), ("to_new", dec_to_new), ("to_old", dec_to_old)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                call.run(torch.cuda.current_stream())
            graphs[name] = g
        torch.cuda.synchronize()

        def g_step(evs=None):
            flush_buf.zero_()
            if evs is not None:
                evs[0].record(stream)
            graphs["compress"].replay()
            if evs is not None:
                evs[1].record(stream)
            flush_buf.zero_()
            if evs is not None:
                evs[2].record(stream)
            d = dec_to_old if state["new"] else dec_to_new
            graphs["to_old" if state["new"] else "to_new"].replay()
            state["new"] = not state["new"]
            if evs is not None:
                evs[3].record(stream)
            return d

        for _ in range(args.warmup):
            g_step()
        gevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
                for _ in range(args.steps)]
        for i in range(args.steps):
            last = g_step(gevs[i])
        torch.cuda.synchronize()
        want = N if state["new"] else O
        if (int(comp.status.item()) != bd.OK or int(last.status.item()) != bd.OK
                or not torch.equal(Rb.view(torch.int16), want.view(torch.int16))):
            raise RuntimeError("graph-replayed steps did not verify")
        gc = reduce_max(statistics.mean(e[0].elapsed_time(e[1]) for e in gevs), world, dev)
        ga = reduce_max(statistics.mean(e[2].elapsed_time(e[3]) for e in gevs), world, dev)
        graph_rep = {"compress_ms": round(gc, 4), "apply_ms": round(ga, 4),
                     "what": "the same step with the compress and each apply direction "
                             "captured once in a CUDA graph and replayed (same kernels, one "
                             "graph launch per phase), L2 flushed before each phase"}
        del graphs

    def timed(fn, steps):
        """Mean device time of fn over `steps` runs after the warm-up; with the L2 flushed
        before each run (outside its events) for small workloads."""
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        if flush:
            spans, out = [], None
            for _ in range(steps):
                flush_buf.zero_()
                t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                t0.record(stream)
                out = fn()
                t1.record(stream)
                spans.append((t0, t1))
            torch.cuda.synchronize()
            ms = sum(a.elapsed_time(b) for a, b in spans)
        else:
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(steps):
                out = fn()
            t1.record(stream)
            torch.cuda.synchronize()
            ms = t0.elapsed_time(t1)
        return reduce_max(ms, world, dev) / steps, out

    def alternate(table):
        def run():
            b = table[state["new"]]
            b.run(stream)
            state["new"] = not state["new"]
            return b
        return run

    def verified(name, last_batch):
        want = N if state["new"] else O
        if int(last_batch.status.item()) != bd.OK or not torch.equal(Rb.view(torch.int16),
                                                                     want.view(torch.int16)):
            raise RuntimeError(f"{name} did not verify")

    # the incremental apply (verified from the checksum of the resident weights; reads and
    # writes only the touched sectors), timed on its own after the step, alternating
    # directions like the step's apply
    inc = {True: bd.IncrementalBatch(rolls, comp.payloads, sizes, ck_new, ck_old, workspace=ws_d),
           False: bd.IncrementalBatch(rolls, comp.payloads, sizes, ck_old, ck_new, workspace=ws_d)}
    inc_ms, last_inc = timed(alternate(inc), args.steps)
    verified("incremental apply", last_inc)
    del inc

    # the full verified apply reading its payloads straight from mapped pinned host memory
    # (over the CPU-GPU link, no host-to-device copy), timed on its own
    h_offs, h_tot = [], 0
    for sz in sizes:
        h_offs.append(h_tot)
        h_tot += (sz + 255) // 256 * 256
    hbuf = bd.MappedHostBuffer(max(h_tot, 256))
    hview = hbuf.numpy()
    for p, o, sz in zip(comp.payloads, h_offs, sizes):
        hview[o:o + sz] = p[:sz].cpu().numpy()
    h_addrs = [hbuf.device_ptr + o for o in h_offs]
    hd = {True: bd.DecompressBatch(rolls, h_addrs, sizes, ck_old, workspace=ws_d),
          False: bd.DecompressBatch(rolls, h_addrs, sizes, ck_new, workspace=ws_d)}
    host_ms, last_h = timed(alternate(hd), args.steps)
    verified("apply from host payloads", last_h)
    del hd
    # the same host payloads streamed through two device slots (bd_decompress_batch_streamed):
    # the copy engines fill one slot while the other slot's tensors are applied
    slot = max(STREAM_SLOT_BYTES, max((z + 255) // 256 * 256 for z in sizes))
    sd = {True: bd.StreamedDecompressBatch(rolls, hbuf, h_offs, sizes, ck_old, slot_bytes=slot,
                                           workspace=ws_d),
          False: bd.StreamedDecompressBatch(rolls, hbuf, h_offs, sizes, ck_new, slot_bytes=slot,
                                            workspace=ws_d)}
    sd[False].staging = sd[True].staging   # one pair of slots (the calls run one after another)
    copy_stream = torch.cuda.Stream(device=dev)

    def streamed():
        b = sd[state["new"]]
        b.run(stream, copy_stream)
        state["new"] = not state["new"]
        return b

    str_ms, last_s = timed(streamed, args.steps)
    verified("streamed apply from host payloads", last_s)
    str_groups, acc = 0, slot
    for z in sizes:
        zz = (z + 255) // 256 * 256
        if acc + zz > slot:
            str_groups, acc = str_groups + 1, 0
        acc += zz
    del sd, hbuf

    # version 3 (compact position blocks) of the same update: compress bound to checksum(old),
    # the full verified apply, and the incremental apply -- backwards from a second payload of
    # the reverse update bound to checksum(new), so that both directions pass the base check
    def bound_format(**kw):
        fwd, s_f = sized_batch(olds, news, base_checksums=ck_old, **kw)
        bwd, s_b = sized_batch(news, olds, base_checksums=ck_new, **kw)
        c_ms, _ = timed(lambda: fwd.run(stream), args.steps)
        res = {"compress_ms": c_ms, "bytes": sum(s_f)}
        dec = {True: bd.DecompressBatch(rolls, bwd.payloads, s_b, ck_old, workspace=ws_d),
               False: bd.DecompressBatch(rolls, fwd.payloads, s_f, ck_new, workspace=ws_d)}
        incb = {True: bd.IncrementalBatch(rolls, bwd.payloads, s_b, ck_new, ck_old,
                                          workspace=ws_d),
                False: bd.IncrementalBatch(rolls, fwd.payloads, s_f, ck_old, ck_new,
                                           workspace=ws_d)}
        for name, table in (("apply", dec), ("incremental", incb)):
            ms, lastb = timed(alternate(table), args.steps)
            verified(f"{kw} {name}", lastb)
            res[name + "_ms"] = ms
        del fwd, bwd, dec, incb
        return res

    v3 = bound_format(compact=True)
    v4 = bound_format(rice=True)
    ow = bound_format(compact=True, overwrite=True)
    p3_bytes, p4_bytes = v3["bytes"], v4["bytes"]

    if flush:
        ms_step = statistics.mean(t_comp) + statistics.mean(t_app)
        ms_step = reduce_max(ms_step, world, dev)
    else:
        total_ms = reduce_max(total_ms, world, dev)
        ms_step = total_ms / args.steps
    raw = 2 * n_total
    value = world * raw / (ms_step * 1e-3) / 1e9
    peak, peak_kind = _peak_hbm()
    mc, ma = statistics.mean(t_comp), statistics.mean(t_app)
    comp_bytes = 4 * n_total + payload_bytes
    inc_bytes = payload_bytes + 2 * 32 * touched
    app_bytes = 2 * n_total + payload_bytes + 32 * touched
    comp_ach = comp_bytes / (mc * 1e-3) / 1e9
    app_ach = app_bytes / (ma * 1e-3) / 1e9
    dom = "compress" if mc >= ma else "apply"
    roof = {"bound": "hbm",
            "kernel": ("compress phase (bd_compress_batch: the fused compress kernel, then "
                       "emit_dense for the chunks too dense for a slot)" if dom == "compress" else
                       "apply phase (bd_decompress_batch: count scan + apply_chunks + apply_dense "
                       "+ apply_finish)"),
            "achieved": round(comp_ach if dom == "compress" else app_ach, 1),
            "peak": peak, "unit": "GB/s",
            "frac": round((comp_ach if dom == "compress" else app_ach) / peak, 4),
            "traffic": _traffic(args.workload, dom, n_total), "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback"}

    # e2e through the public API with host buffers: H2D old+new from pinned memory, compress,
    # verified apply, D2H of payloads + checksums + statuses
    e2e = None
    host_need = 4 * n_total + payload_bytes
    if host_need > _host_mem_available() // 2:
        e2e = {"value": None, "unit": "GB/s",
               "unavailable": f"pinned host copies of old and new ({host_need / 1e9:.0f} GB) "
                              f"exceed half of the host memory free to this process"}
    else:
        hO = torch.empty(O.shape, dtype=O.dtype, pin_memory=True)
        hN = torch.empty(N.shape, dtype=N.dtype, pin_memory=True)
        hO.copy_(O)
        hN.copy_(N)
        # groups of consecutive tensors (about E2E_GROUP_BYTES of old + new each): group g's
        # host-to-device copy runs on its own stream while group g-1 is compressed and applied,
        # and its payloads come back on a third stream once it is done
        groups, i0, acc = [], 0, 0
        for i, n in enumerate(ns):
            acc += 4 * n
            if acc >= E2E_GROUP_BYTES or i == k - 1:
                groups.append((i0, i + 1))
                i0, acc = i + 1, 0
        g_comp, g_dec, g_span, g_pay = [], [], [], []
        hoff = 0
        for (a0, a1) in groups:
            c = bd.CompressBatch(olds[a0:a1], news[a0:a1], caps=sizes[a0:a1], workspace=ws_c)
            g_comp.append(c)
            g_dec.append({False: bd.DecompressBatch(rolls[a0:a1], c.payloads, sizes[a0:a1],
                                                    ck_new[a0:a1], workspace=ws_d),
                          True: bd.DecompressBatch(rolls[a0:a1], c.payloads, sizes[a0:a1],
                                                   ck_old[a0:a1], workspace=ws_d)})
            g_span.append((offs[a0], offs[a1 - 1] + ns[a1 - 1]))
            pb = (c.payloads[-1].data_ptr() - c.payload_buf.data_ptr()) + sizes[a1 - 1]
            g_pay.append((hoff, pb))
            hoff += pb
        hP = torch.empty(max(hoff, 1), dtype=torch.uint8, pin_memory=True)
        hS = torch.empty(3 * k, dtype=torch.int64, pin_memory=True)
        # old and new come in on two streams (two copy engines), payloads go out on a third
        s_in = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
        s_out = torch.cuda.Stream(device=dev)
        ev_in = [[torch.cuda.Event() for _ in groups] for _ in s_in]
        ev_done = [torch.cuda.Event() for _ in groups]
        torch.cuda.synchronize()

        def e2e_step():
            for si in s_in:
                si.wait_stream(stream)   # the previous step's compute has read old and new
            for g, (a0, a1) in enumerate(groups):
                lo, hi = g_span[g]
                for si, ev, dst, src in zip(s_in, ev_in, (O, N), (hO, hN)):
                    with torch.cuda.stream(si):
                        dst[lo:hi].copy_(src[lo:hi], non_blocking=True)
                        ev[g].record(si)
                    stream.wait_event(ev[g])
                g_comp[g].run(stream)
                g_dec[g][state["new"]].run(stream)
                ev_done[g].record(stream)
                s_out.wait_event(ev_done[g])
                with torch.cuda.stream(s_out):
                    h0, pb = g_pay[g]
                    hP[h0:h0 + pb].copy_(g_comp[g].payload_buf[:pb], non_blocking=True)
                    hS[a0:a1].copy_(g_comp[g].sizes, non_blocking=True)
                    hS[k + a0:k + a1].copy_(g_comp[g].checksums, non_blocking=True)
                    hS[2 * k + a0:2 * k + a1].copy_(g_dec[g][state["new"]].statuses.to(torch.int64),
                                                    non_blocking=True)
            state["new"] = not state["new"]
            stream.wait_stream(s_out)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world, dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_steps = max(3, min(args.steps, 10))
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = reduce_max(e0.elapsed_time(e1), world, dev) / e2e_steps
        if any(int(v) != bd.OK for v in hS[2 * k:3 * k].tolist()):
            raise RuntimeError("e2e apply did not verify")
        want = N if state["new"] else O
        if not torch.equal(Rb.view(torch.int16), want.view(torch.int16)):
            raise RuntimeError("e2e apply did not restore")
        # the host link on its own in the same run: old and new copied in, both streams
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for si in s_in:
            si.wait_stream(stream)
        for si, dst, src in zip(s_in, (O, N), (hO, hN)):
            with torch.cuda.stream(si):
                dst.copy_(src, non_blocking=True)
        for si in s_in:
            stream.wait_stream(si)
        p1.record(stream)
        torch.cuda.synchronize()
        h2d_gbs = 4 * n_total / (p0.elapsed_time(p1) * 1e-3) / 1e9
        e2e = {"value": round(world * raw / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
               "ms_per_step": round(e_ms, 3), "steps": e2e_steps,
               "h2d_alone_gbs": round(h2d_gbs, 1),
               "h2d_bytes_per_step": 4 * n_total, "d2h_bytes_per_step": hoff + 8 * 3 * k,
               "overlap": f"{len(groups)} groups of tensors: old and new in on two streams, "
                          "compress + apply, payloads out on a third"}
        del hO, hN, hP, g_comp, g_dec

    cpu = None
    if rank == 0:
        cpu = oracle_baseline(specs, args.cpu_sample_elems, dev)
        cpu["fanout"] = oracle_fanout(specs, args.cpu_sample_elems)

    # tensor-table uploads (30 KiB each): the tensor table and the chunk, tile and (compress)
    # batch start arrays, each section 256-byte aligned
    blobs_c = -(-(128 * k + 3 * 8 * (k + 1) + 3 * 256) // 30720)
    blobs_d = -(-(128 * k + 2 * 8 * (k + 1) + 2 * 256) // 30720)
    # compress: uploads + the fused compress + emit_dense, or (a call with a tensor of more
    # batches than the fused compress takes -- the library's choice restated: about four
    # batches of up to 32 chunks per resident warp, at most 4096 batches per tensor) uploads +
    # encode_slots, two scans, emit and emit_dense; decompress: uploads + scan x2, both builds of
    # apply_chunks (one returns at once), apply_bitmap, apply_finish
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    chunks = [(n + 4095) // 4096 for n in ns]
    bch = max(1, min(32, sum(chunks) // (sms * 32 * 4)))
    fused = -(-max(chunks) // bch) <= 4096
    launches_per_step = (blobs_c + (2 if fused else 5)) + (blobs_d + 6)

    def frac(nbytes, ms):
        return round(nbytes / (ms * 1e-3) / 1e9 / peak, 4)

    def fmt_block(res, what, nbytes_payload=None):
        out = {"compress_ms": round(res["compress_ms"], 4), "apply_ms": round(res["apply_ms"], 4),
               "incremental_ms": round(res["incremental_ms"], 4), "what": what}
        if nbytes_payload is not None:
            out.update({
                "payload_pct": round(100 * nbytes_payload / raw, 4),
                "payload_vs_v1": round(nbytes_payload / payload_bytes, 4),
                "compress_roofline_frac": frac(4 * n_total + nbytes_payload, res["compress_ms"]),
                "apply_roofline_frac": frac(2 * n_total + nbytes_payload + 32 * touched,
                                            res["apply_ms"]),
                "incremental_roofline_frac": frac(nbytes_payload + 2 * 32 * touched,
                                                  res["incremental_ms"])})
        return out

    if rank == 0:
        rice = fmt_block(v4, "version-4 payloads (Rice-coded compact position blocks) of the "
                             "same update: bd_compress_versioned_batch format 4, "
                             "bd_decompress_batch in place, bd_decompress_incremental_batch in "
                             "place", p4_bytes)
        rice["payload_vs_v3"] = round(p4_bytes / p3_bytes, 4)
        line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "u16", "data": "synthetic",
                "config": {"workload": _describe(args.workload, specs),
                           "l2": (f"flushed before every timed phase ({L2_FLUSH_BYTES >> 20} MiB "
                                  "write outside the phase events); ms_per_step = compress + "
                                  "apply phase times") if flush else
                                 "inputs larger than L2 (no flush needed)",
                           "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
                "compress_gbs": round(raw / (mc * 1e-3) / 1e9, 2),
                "apply_gbs": round(raw / (ma * 1e-3) / 1e9, 2),
                "compress_ms": round(mc, 4), "apply_ms": round(ma, 4),
                "compress_roofline_frac": round(comp_ach / peak, 4),
                "apply_roofline_frac": round(app_ach / peak, 4),
                **({"graph_replay": dict(graph_rep, **{
                    "compress_gbs": round(raw / (graph_rep["compress_ms"] * 1e-3) / 1e9, 2),
                    "apply_gbs": round(raw / (graph_rep["apply_ms"] * 1e-3) / 1e9, 2),
                    "compress_roofline_frac": round(
                        comp_bytes / (graph_rep["compress_ms"] * 1e-3) / 1e9 / peak, 4),
                    "apply_roofline_frac": round(
                        app_bytes / (graph_rep["apply_ms"] * 1e-3) / 1e9 / peak, 4)})}
                   if graph_rep else {}),
                "apply_host_payload": {
                    "ms": round(host_ms, 4),
                    "gbs": round(raw / (host_ms * 1e-3) / 1e9, 2),
                    "what": "bd_decompress_batch in place with every payload in mapped pinned "
                            "host memory, read by the kernels over the CPU-GPU link"},
                "apply_streamed": {
                    "ms": round(str_ms, 4),
                    "gbs": round(raw / (str_ms * 1e-3) / 1e9, 2),
                    "slot_bytes": slot, "groups": str_groups,
                    "what": "bd_decompress_batch_streamed in place: the same pinned host "
                            "payloads copied into two device slots on a second stream while "
                            "the other slot's tensors are applied"},
                "apply_incremental": {
                    "ms": round(inc_ms, 4),
                    "gbs": round(raw / (inc_ms * 1e-3) / 1e9, 2),
                    "algorithmic_bytes": inc_bytes,
                    "roofline_frac": round(inc_bytes / (inc_ms * 1e-3) / 1e9 / peak, 4),
                    "what": "bd_decompress_incremental_batch in place: verified from the "
                            "checksums of the resident weights; algorithmic bytes = payload + "
                            "read and write of each touched 32-byte sector"},
                "compact": fmt_block(v3, "version-3 payloads (compact position blocks) of the "
                                         "same update: bd_compress_versioned_batch format 3, "
                                         "bd_decompress_batch in place, "
                                         "bd_decompress_incremental_batch in place", p3_bytes),
                "rice": rice,
                "overwrite": fmt_block(ow, "version-3 overwrite payloads (new field values "
                                           "instead of XOR masks; same size as the version-3 "
                                           "XOR payload) of the same update and of its reverse: "
                                           "bd_compress_versioned_batch format 3 | "
                                           "BD_FORMAT_OVERWRITE, bd_decompress_batch and "
                                           "bd_decompress_incremental_batch in place"),
                "compress_algorithmic_bytes": comp_bytes, "apply_algorithmic_bytes": app_bytes,
                "payload_pct": round(100 * payload_bytes / raw, 4),
                "touched_sector_pct": round(100 * touched / (raw / 32), 3),
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
                "gpu_launches": launches_per_step * args.steps}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_profile_case(args) -> None:
    """The fixed programs that the committed ncu summaries were captured from (one GPU).

    Each round of every case: compress in each version, the full verified apply of each
    payload in place (alternately to new and back to old), and the incremental apply of each
    payload from old; `embed` and `dense` also run the standalone checksum of old and one
    out-of-place full apply (the copy kernel).  Two rounds, so that a capture can skip the
    first."""
    import lossless_bf16_weight_old_gb300 as bd
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    case = args.profile_case
    if case == "embed":        # one 32000x4096 tensor: the separate compress kernels
        specs = [s for s in W.dense7b() if s.name == "embed"]
        versions = (1, 3, 4)
    elif case == "layers":     # dense7b's first two layers: the fused compress
        specs = [s for s in W.dense7b() if s.name.startswith(("layers.0.", "layers.1."))]
        versions = (1, 3, 4)
    elif case == "moe":        # moe30b's layer 0: sparse cold experts beside dense hot ones
        specs = [s for s in W.moe30b() if s.name.startswith("layers.0.")]
        versions = (1, 3, 4)
    elif case == "dense":      # a 2^26-element slice of the 1 GiB workload: the dense kernels
        specs = [W.Spec("w", (1 << 26,), kind="additive", tid=0)]
        versions = (1, 3)
    else:                      # "formats": a whole workload in versions 3 and 4
        specs = _workload_specs(args.workload)
        versions = (3, 4)
    olds, news = [], []
    for s in specs:
        a, b = W.make_pair(s, device=dev)
        olds.append(a.reshape(-1))
        news.append(b.reshape(-1))
    rolls = [o.clone() for o in olds]
    outs = [torch.empty_like(o) for o in olds] if case in ("embed", "dense") else None
    ck_old = torch.cat([bd.checksum(o).reshape(1) for o in olds])
    comp = {v: (bd.CompressBatch(olds, news) if v == 1 else
                bd.CompressBatch(olds, news, base_checksums=ck_old, compact=v == 3, rice=v == 4))
            for v in versions}
    sizes = {}
    for rnd in range(2):
        for v in versions:
            comp[v].run()
        torch.cuda.synchronize()
        for v in versions:
            sizes[v] = [int(x) for x in comp[v].sizes.tolist()]
        ck_new = comp[versions[0]].checksums
        state_new = False
        for r, o in zip(rolls, olds):
            r.copy_(o)
        done = []
        for v in versions:   # alternately to new and back to old
            dec = bd.DecompressBatch(rolls, comp[v].payloads, sizes[v],
                                     ck_old if state_new else ck_new)
            dec.run()
            done.append(dec)
            state_new = not state_new
        torch.cuda.synchronize()
        want = news if state_new else olds
        if any(int(x.status.item()) != bd.OK for x in done) or not all(
                torch.equal(r.view(torch.int16), w.view(torch.int16))
                for r, w in zip(rolls, want)):
            raise RuntimeError("profile case did not verify (full apply)")
        done = []
        for v in versions:
            for r, o in zip(rolls, olds):
                r.copy_(o)
            inc = bd.IncrementalBatch(rolls, comp[v].payloads, sizes[v], ck_old, ck_new)
            inc.run()
            done.append(inc)
        torch.cuda.synchronize()
        if any(int(x.status.item()) != bd.OK for x in done) or not all(
                torch.equal(r.view(torch.int16), w.view(torch.int16))
                for r, w in zip(rolls, news)):
            raise RuntimeError("profile case did not verify (incremental apply)")
        if outs is not None:
            cks = torch.cat([bd.checksum(o).reshape(1) for o in olds])
            oop = bd.DecompressBatch(olds, comp[1].payloads, sizes[1], ck_new, outs=outs)
            oop.run()
            torch.cuda.synchronize()
            if (bd.u64(cks) != bd.u64(ck_old) or int(oop.status.item()) != bd.OK or not all(
                    torch.equal(r.view(torch.int16), w.view(torch.int16))
                    for r, w in zip(outs, news))):
                raise RuntimeError("profile case did not verify (checksum, out of place)")
            # the entry point without a workspace (block-level decoder), out of place
            if case == "embed":
                lib = bd._lib.load()
                st = torch.full((1,), -1, dtype=torch.int32, device=dev)
                for o, p_, sz, ck, out in zip(olds, comp[1].payloads, sizes[1],
                                             torch.split(ck_new, 1), outs):
                    out.zero_()
                    rc = lib.bd_decompress_noalloc(o.data_ptr(), o.numel(), p_.data_ptr(), sz,
                                                   ck.data_ptr(), out.data_ptr(), st.data_ptr(),
                                                   torch.cuda.current_stream().cuda_stream)
                    if rc != bd.OK:
                        raise RuntimeError(f"bd_decompress_noalloc returned {rc}")
                torch.cuda.synchronize()
                if int(st.item()) != bd.OK or not all(
                        torch.equal(r.view(torch.int16), w.view(torch.int16))
                        for r, w in zip(outs, news)):
                    raise RuntimeError("profile case did not verify (no workspace)")
    print("profile case", case, "ok:",
          {v: sum(sizes[v]) for v in versions}, "payload bytes", flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="dense7b")
    p.add_argument("--cpu-sample-elems", type=int, default=1_000_000_000,
                   help="elements of the workload the CPU oracle baseline encodes+decodes")
    p.add_argument("--ref-sample-elems", type=int, default=400_000_000,
                   help="elements per step of the --impl reference arm")
    p.add_argument("--profile-case", choices=["embed", "layers", "moe", "dense", "formats"],
                   default=None,
                   help="run a fixed small program for an ncu capture instead of the bench")
    args = p.parse_args(argv)
    if args.profile_case:
        run_profile_case(args)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
