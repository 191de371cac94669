"""Benchmark of the simulated context-parallel attention layer on GB300.

One step = one pass of the whole hot path over one batch of synthetic input,
all U x A virtual ranks on this GPU: pack -> simulated all-to-all -> unpack
(AllGather placement) -> local-Q / global-KV attention -> reverse exchange.
Default workload: the Wan-like 480p AllGather-KV CP8 layer (local-Q
[1,4095,12,128] per rank against the gathered K/V [1,32760,12,128]).

`value` is the attention FLOPs of the step divided by the device time of the
whole step (inputs resident in HBM); `roofline` is the attention kernel alone
(CUDA events on its stream); `relayout` reports the pack/unpack GB/s;
`e2e` repeats the step through the same public API with every step's inputs
copied from pinned host memory and its output read back inside the timed
region (copies pipelined on their own streams against the compute).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Under torchrun (N > 1) every GPU runs its own replica of the layer (weak
scaling, no collective on the data path); the timed region is bracketed by a
barrier and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LQ/GKV attn TFLOP/s & % GB300 bf16 peak; QKV pack/unpack GB/s & % HBM"
# staging layouts of the exchange (values of ctx_layout in the C header)
LAYOUTS = {"tqkv": 0, "interleaved": 1}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha1(files=("attention.cu", "ptx.cuh")) -> str:
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "diffusion_transformer_context_gb300", "csrc")
    for fn in files:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


TRAFFIC_RECORDS = {
    # roofline object -> (committed ncu summary, kernel sources it was taken on)
    "attention": ("attn_traffic.json", ("attention.cu", "ptx.cuh")),
    "relayout": ("relayout_traffic.json", ("relayout.cu",)),
    "merge": ("merge_traffic.json", ("merge.cu", "ptx.cuh")),
}


def recorded_traffic(workload: str, kind: str = "attention"):
    """DRAM bytes per launch (attention) or per step (relayout: all its
    launches) from the committed ncu summary, or None if the kernel source
    changed since the counters were taken."""
    fname, files = TRAFFIC_RECORDS[kind]
    path = os.path.join(ROOT, "profiles", fname)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    entry = d.get(workload)
    if not entry or entry.get("source_sha1") != kernel_source_sha1(files):
        return None
    return entry.get("bytes_per_launch", entry.get("bytes_per_step"))


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3], parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        busy = [r for r in rows if r[2] > 0.25 * max(x[2] for x in rows)] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i, v in enumerate(r[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(busy)}


# ------------------------------------------------------------------ ranks

def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The slowest rank's time: every rank gets the maximum (all_reduce MAX)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def valid_keys(inp):
    """Per batch row, the gathered keys the masks leave valid: the image keys
    outside the image padding plus the text keys inside the text length."""
    wl = inp.wl
    img = [wl.S if inp.image_mask is None else int(inp.image_mask[b].sum()) for b in range(wl.B)]
    jnt = [wl.joint if inp.joint_mask is None else int(inp.joint_mask[b].sum()) for b in range(wl.B)]
    return [i + j for i, j in zip(img, jnt)]


def oracle_keys(inp, h_l):
    """The oracle's gathered K/V of head group 0 and its merged key mask."""
    import numpy as np
    import oracle
    import workloads

    wl, u16 = inp.wl, workloads.as_u16
    k, v = u16(inp.k[:, :, :h_l]), u16(inp.v[:, :, :h_l])
    if wl.joint:
        jk, jv = u16(inp.jk[:, :, :h_l]), u16(inp.jv[:, :, :h_l])
        k = np.concatenate([jk, k] if wl.joint_front else [k, jk], axis=1)
        v = np.concatenate([jv, v] if wl.joint_front else [v, jv], axis=1)
    mask = oracle.merge_joint_attn_mask(inp.image_mask, inp.joint_mask, wl.B, wl.S, wl.joint, wl.joint_front)
    return k, v, mask


def whole_job_tflops(flops_per_rank: float, world: int, ms: float) -> float:
    """Weak scaling: every rank does the same work; the job's throughput is
    all ranks' FLOPs over the slowest rank's time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


# ------------------------------------------------------------------ GPU arm

def run_gpu(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import workloads
    import diffusion_transformer_context_gb300 as ctx
    from diffusion_transformer_context_gb300.simulate import SimLayer

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = workloads.WORKLOADS[args.workload]
    inp = workloads.make_inputs(wl)
    sim = SimLayer(wl, device=dev, balanced=not args.unbalanced, layout=LAYOUTS[args.layout])
    sim.load(inp)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    if not args.eager:
        sim.capture()

    def run_phase(name):
        if args.eager:
            getattr(sim, name)(stream=stream)
        else:
            sim.replay(name)

    # one step, with events between its phases (exchange_in: pack + all-to-all
    # + unpack; attend: attention; exchange_out: reverse exchange)
    def timed_step(ev):
        for i, name in enumerate(sim.PHASES):
            ev[i].record(stream)
            run_phase(name)
        ev[len(sim.PHASES)].record(stream)

    def plain_step():
        for name in sim.PHASES:
            run_phase(name)

    for _ in range(args.warmup):
        plain_step()
    st = ctx.ctx_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {ctx.ctx_status_string(st)}")

    sampler = ClockSampler(local_rank) if (rank == 0 and not args.no_clocks) else None
    if sampler:
        sampler.start()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(sim.PHASES) + 1)] for _ in range(args.steps)]
    # Inputs smaller than L2 would stay cached from one step to the next:
    # then a buffer larger than L2 is written between steps (outside the
    # timed spans, which are the per-step event pairs).
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = sim.x.numel() * sim.x.element_size() < 2 * l2_bytes
    scrub = torch.empty(4 * l2_bytes, dtype=torch.uint8, device=dev) if flush else None
    barrier()
    for i in range(args.steps):
        if scrub is not None:
            scrub.fill_(i & 0xff)
        timed_step(evs[i])
    barrier()
    clocks = sampler.stop() if sampler else None
    st = ctx.ctx_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {ctx.ctx_status_string(st)}")
    total_ms = sum(ev[0].elapsed_time(ev[-1]) for ev in evs)
    parts = {name: [ev[i].elapsed_time(ev[i + 1]) for ev in evs] for i, name in enumerate(sim.PHASES)}
    total_ms = max_over_ranks(total_ms, world, dev)

    # ---------------------------------------------------------- e2e (host buffers)
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(sim, inp, args, world, dev, barrier)
    sim.l2_flushed = flush
    return sim, inp, total_ms, parts, clocks, e2e


def run_pack_line(args, dev, peaks, peak_kind):
    """The layout-only workload timed beside the default line: U = 4 ranks,
    each Q/K/V [1,1024,24,128], packed into staging buffers of the chosen
    layout ([4,3,1,1024,6,128] or [4,1,1024,6,384]) and, after the exchange,
    unpacked to [1,4096,6,128] per rank.

    `achieved` is the library's pack and unpack kernels in HBM terms. The
    work rotates over n buffer sets whose total is several times L2, so every
    read comes from HBM and every written line is written back inside the
    timed region (all but the last replay's). One CUDA graph holds the four
    ranks' packs (launches concurrent, as ranks run) of every set in turn,
    another the unpacks; each is replayed back to back, so graph launches
    are amortised over n sets as inside a layer's graph. The other staging
    layout is timed the same way and reported beside it. `copy_gbs` is a
    plain device copy of the same bytes per set timed the same way: the
    reference for transfers of this size. `step_gbs` is the whole simulated
    step (pack + all-to-all + unpack): there the staging buffers written by
    one kernel are read by the next from L2, so it is not an HBM figure."""
    import torch

    import workloads
    from diffusion_transformer_context_gb300.simulate import SimLayer

    wl = workloads.WORKLOADS["pack"]
    inp = workloads.make_inputs(wl)
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    main_layout = args.layout
    other_layout = "interleaved" if main_layout == "tqkv" else "tqkv"
    one = SimLayer(wl, device=dev, layout=LAYOUTS[main_layout])
    set_bytes = (one.x.numel() + one.send.numel() + one.recv.numel() + 3 * one.qg.numel()) * 2
    # a pack (or an unpack) touches half a set; between two uses of a buffer
    # the other sets' kernels move at least 4x L2 through the cache
    n_sets = 1 + -(-4 * l2_bytes // (set_bytes // 2))
    sims = {main_layout: [one] + [SimLayer(wl, device=dev, layout=LAYOUTS[main_layout]) for _ in range(n_sets - 1)],
            other_layout: [SimLayer(wl, device=dev, layout=LAYOUTS[other_layout]) for _ in range(n_sets)]}
    for sim in sims[main_layout] + sims[other_layout]:
        sim.load(inp)
        sim.step()  # library set-up outside any capture
    b_pack, b_unpack = one.pack_bytes(), one.unpack_bytes()
    b_step = b_pack + one.a2a_bytes() + b_unpack
    src = [torch.empty(b_pack // 4, dtype=torch.bfloat16, device=dev).fill_(1) for _ in range(n_sets)]
    dst = [torch.empty_like(x) for x in src]
    torch.cuda.synchronize(dev)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n_sets):
                fn(i)
        return g

    def copy_ranks(i):
        # the same bytes as four per-rank copies on the rank streams, as the packs run
        R = wl.ranks

        def one(g, s):
            n = src[i].numel() // R
            with torch.cuda.stream(s):
                dst[i][g * n:(g + 1) * n].copy_(src[i][g * n:(g + 1) * n])

        sims[main_layout][i]._per_rank(None, one)

    graphs = {"step": capture(lambda i: sims[main_layout][i].exchange_in()),
              "copy": capture(lambda i: dst[i].copy_(src[i])),
              "copy_ranks": capture(copy_ranks)}
    for lay, ss in sims.items():
        graphs["pack_" + lay] = capture(lambda i: ss[i].pack_ranks())
        graphs["unpack_" + lay] = capture(lambda i: ss[i].unpack_ranks())
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    reps = max(args.steps, 20)

    def timed_once(name):
        g = graphs[name]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / (reps * n_sets)  # per set

    # every graph warmed up first, then three rounds over all of them in turn
    # (median per graph), so that no figure depends on its place in the order
    for g in graphs.values():
        for _ in range(3):
            g.replay()
    samples = {n: [] for n in graphs}
    for _ in range(3):
        for n in graphs:
            samples[n].append(timed_once(n))

    def timed(name):
        return sorted(samples[name])[1]

    def rate(b, ms):
        return round(b / (ms * 1e-3) / 1e9, 1)

    def layout_figures(lay):
        ms_p, ms_u = timed("pack_" + lay), timed("unpack_" + lay)
        gbs = (b_pack + b_unpack) / ((ms_p + ms_u) * 1e-3) / 1e9
        staging = ([wl.U, 3, wl.B, wl.S_l, wl.h_l, wl.D] if lay == "tqkv"
                   else [wl.U, wl.B, wl.S_l, wl.h_l, 3 * wl.D])
        return {"staging": staging, "achieved": round(gbs, 1), "frac": round(gbs / peaks["hbm_gbs"], 4),
                "pack_gbs": rate(b_pack, ms_p), "unpack_gbs": rate(b_unpack, ms_u),
                "pack_ms": round(ms_p, 4), "unpack_ms": round(ms_u, 4),
                "traffic": recorded_traffic("pack_kernels" + ("" if lay == "tqkv" else "_" + lay), "relayout")}

    main = layout_figures(main_layout)
    other = layout_figures(other_layout)
    ms_step, ms_copy, ms_copy_ranks = timed("step"), timed("copy"), timed("copy_ranks")
    traffic = main.pop("traffic")
    return {"workload": "pack", "U": wl.U, "per_rank": [wl.B, wl.S_l, wl.H, wl.D], "staging_layout": main_layout,
            "staging": main["staging"], "bound": "hbm",
            "kernel": "relayout_kernel (4 packs; 4 unpacks)", "achieved": main["achieved"],
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": main["frac"],
            "peak_source": f"{peak_kind} hbm_gbs",
            **{k: main[k] for k in ("pack_gbs", "unpack_gbs", "pack_ms", "unpack_ms")},
            "algorithmic_bytes": {"pack": b_pack, "unpack": b_unpack},
            "copy_gbs": rate(b_pack, ms_copy),
            "copy_per_rank_gbs": rate(b_pack, ms_copy_ranks),
            "copy_note": "copy_gbs: one device copy of a set's bytes; copy_per_rank_gbs: the same bytes as one "
                         "copy per rank on the rank streams (the packs' launch pattern)",
            "timing": f"one CUDA graph over {n_sets} buffer sets of {set_bytes >> 20} MiB (L2 {l2_bytes >> 20} MiB), "
                      f"replayed {reps} times back to back: reads from HBM, write-back inside the timed region; "
                      f"median of 3 rounds over all graphs in turn",
            "gpu_launches_per_set": {"pack": wl.ranks, "unpack": wl.ranks},
            other_layout: other,
            "step_gbs": rate(b_step, ms_step), "step_ms": round(ms_step, 4),
            "step_note": "pack + simulated all-to-all + unpack; staging buffers re-read from L2",
            "traffic": traffic}


def run_e2e(sim, inp, args, world, dev, barrier):
    """The same steps with every step's inputs copied in from pinned host
    memory and its result copied back, all inside the timed region.

    Two copies of the layer (input, gathered and output buffers, graphs)
    take the steps in turn, the way a serving loop double-buffers: step i's
    input is copied in on its own stream while step i-1 computes (its buffer
    was last read by step i-2's exchange), and step i's result is read back
    on a third stream while the following steps compute (its buffer is next
    rewritten by step i+2, after that read-back)."""
    import torch

    from diffusion_transformer_context_gb300.simulate import SimLayer

    cs = torch.cuda.current_stream(dev)
    hs, ds = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    other = SimLayer(sim.wl, device=dev, balanced=not args.unbalanced, layout=sim.layout)
    other.load(inp)
    if not args.eager:
        other.capture()
    sims = [sim, other]
    host_x = torch.empty(sim.x.shape, dtype=sim.x.dtype).pin_memory()
    host_x.copy_(sim.x.cpu())

    def results_of(s):
        if not s.attention:
            return [s.qg, s.kg, s.vg], "exchange_in"  # the unpacked Q/K/V
        if s.wl.U > 1:
            return [s.y], "exchange_out"              # after the reverse exchange
        return [s.out], "attend"

    host_y = [torch.empty(r.shape, dtype=r.dtype).pin_memory() for r in results_of(sim)[0]]

    def phase(s, name):
        if args.eager:
            getattr(s, name)(stream=cs)
        else:
            s.replay(name)

    def ev():
        return torch.cuda.Event()

    x_free, out_free = [None, None], [None, None]  # per copy: its input read, its result read back

    def steps(n):
        for i in range(n):
            k = i & 1
            s = sims[k]
            results, rewrite = results_of(s)
            h2d_done, x_read, out_ready, d2h_done = ev(), ev(), ev(), ev()
            with torch.cuda.stream(hs):
                if x_free[k] is not None:
                    hs.wait_event(x_free[k])   # this copy's previous exchange has read its input
                s.x.copy_(host_x, non_blocking=True)
                h2d_done.record(hs)
            cs.wait_event(h2d_done)
            for name in s.PHASES:
                if name == rewrite and out_free[k] is not None:
                    cs.wait_event(out_free[k])  # this copy's previous read-back has left its result
                phase(s, name)
                if name == "exchange_in":
                    x_read.record(cs)
            out_ready.record(cs)
            with torch.cuda.stream(ds):
                ds.wait_event(out_ready)
                for h, r in zip(host_y, results):
                    h.copy_(r, non_blocking=True)
                d2h_done.record(ds)
            x_free[k], out_free[k] = x_read, d2h_done
        for k in range(2):
            if out_free[k] is not None:
                cs.wait_event(out_free[k])  # the last read-backs are inside the timed region

    steps(max(2, args.warmup))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(cs)
    hs.wait_event(e0)
    steps(args.steps)
    e1.record(cs)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    # after the timed region: the host copy of the last step's result equals the device result
    last = sims[(args.steps - 1) & 1]
    verified = all(torch.equal(h.to(dev), r) for h, r in zip(host_y, results_of(last)[0]))
    flops = sim.attn_flops(valid_keys(inp))
    return {"value": round(whole_job_tflops(flops * args.steps, world, e2e_ms), 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": host_x.numel() * host_x.element_size(),
            "d2h_bytes_per_step": sum(h.numel() * h.element_size() for h in host_y),
            "ms_per_step": round(e2e_ms / args.steps, 4),
            "pipeline": "H2D / compute / D2H on three streams; two copies of the layer take the steps in turn",
            "readback_verified": verified}


def cpu_baseline_sample(wl_name: str, seconds: float, seed: int = 1234):
    """Times the oracle as it stands on a bounded sample of the workload's
    attention rows (and the layout steps of one rank); returns a dict."""
    import numpy as np
    import oracle
    import workloads

    oracle.build()
    wl = workloads.WORKLOADS[wl_name]
    inp = workloads.make_inputs(wl)
    U, A = wl.U, wl.A
    u16 = workloads.as_u16
    # one rank's layout steps (pack + unpack), timed
    g = 0
    t = time.perf_counter()
    st = oracle.pack_qkv(u16(inp.shard(inp.q, g)), u16(inp.shard(inp.k, g)), u16(inp.shard(inp.v, g)), U)
    oracle.unpack_qkv(st, U)
    relayout_s = time.perf_counter() - t
    relayout_bytes = 2 * 2 * st.nbytes
    if not wl.attention:
        gbs = relayout_bytes / relayout_s / 1e9
        return {"value": round(gbs, 3), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                "sample": f"layout of one rank: {gbs:.2f} GB/s", "relayout_gbs": round(gbs, 3)}
    # attention: head group 0, gathered K/V, query rows of every rank
    h_l = wl.h_l
    q = u16(inp.q[:, :, :h_l])
    k, v, mask = oracle_keys(inp, h_l)
    Sk = k.shape[1]
    rng = np.random.default_rng(seed)

    def rows(n):
        return np.stack([rng.integers(0, wl.B, n), rng.integers(0, h_l, n), rng.integers(0, wl.S, n)], axis=1)

    def flops_of(bhi):
        if mask is None:
            return 4.0 * Sk * wl.D * len(bhi)
        return float(sum(4.0 * int(mask[b].sum()) * wl.D for b in bhi[:, 0]))

    t = time.perf_counter()
    probe = rows(max(16, 4 * oracle.num_threads()))
    oracle.attention_rows(q, k, v, probe, mask)
    per_row = max(1e-6, (time.perf_counter() - t) / len(probe))
    n = max(8, int(seconds / per_row))
    bhi = rows(n)
    t = time.perf_counter()
    oracle.attention_rows(q, k, v, bhi, mask)
    dt = time.perf_counter() - t
    return {"value": round(flops_of(bhi) / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{n} random query rows of {wl_name} (fp64 oracle, all keys each), {dt:.1f} s; "
                      f"layout of one rank: {relayout_bytes / relayout_s / 1e9:.2f} GB/s",
            "relayout_gbs": round(relayout_bytes / relayout_s / 1e9, 3)}


def shape_config(wl) -> dict:
    """The workload keys both arms report in `config`."""
    return {"workload": wl.name, "B": wl.B, "S": wl.S, "H": wl.H, "D": wl.D, "U": wl.U, "A": wl.A,
            "joint": wl.joint, "virtual_ranks": wl.U * wl.A}


def run_reference(args, rank):
    """--impl reference: the oracle, on the host cores, a bounded sample per step."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    import workloads

    oracle.build()
    wl = workloads.WORKLOADS[args.workload]
    inp = workloads.make_inputs(wl)
    u16 = workloads.as_u16
    if not wl.attention:
        run_reference_layout(args, wl, inp)
        return
    h_l = wl.h_l
    q = u16(inp.q[:, :, :h_l])
    k, v, mask = oracle_keys(inp, h_l)
    Sk = k.shape[1]
    rng = np.random.default_rng(1234)
    n_rows = args.ref_rows

    def one_step():
        bhi = np.stack([rng.integers(0, wl.B, n_rows), rng.integers(0, h_l, n_rows),
                        rng.integers(0, wl.S, n_rows)], axis=1)
        t = time.perf_counter()
        oracle.attention_rows(q, k, v, bhi, mask)
        dt = time.perf_counter() - t
        fl = float(sum(4.0 * (Sk if mask is None else int(mask[b].sum())) * wl.D for b in bhi[:, 0]))
        return fl, dt

    for _ in range(args.warmup):
        one_step()
    fl_tot = dt_tot = 0.0
    for _ in range(args.steps):
        fl, dt = one_step()
        fl_tot += fl
        dt_tot += dt
    value = fl_tot / dt_tot / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * dt_tot / args.steps, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**shape_config(wl), "sample_rows_per_step": n_rows},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": f"{n_rows} random query rows of {args.workload} per step, all keys"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_layout(args, wl, inp):
    """--impl reference on a layout-only workload: the oracle's pack and unpack
    of one rank per step, in GB/s of algorithmic read + write bytes."""
    import oracle
    import workloads

    u16 = workloads.as_u16
    shards = [[u16(inp.shard(t, g)) for t in (inp.q, inp.k, inp.v)] for g in range(wl.U * wl.A)]

    layout = LAYOUTS[args.layout]

    def one_step(g):
        t = time.perf_counter()
        st = oracle.pack_qkv_ex(*shards[g], wl.U, layout)
        oracle.unpack_qkv_ex(st, wl.U, layout)
        return 2 * 2 * st.nbytes, time.perf_counter() - t

    for i in range(args.warmup):
        one_step(i % len(shards))
    nb = dt = 0.0
    for i in range(args.steps):
        b, t = one_step(i % len(shards))
        nb += b
        dt += t
    value = nb / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * dt / args.steps, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u16 (bit copy)", "data": "synthetic",
            "config": {**shape_config(wl), "sample": "pack + unpack of one rank per step",
                       **({"staging_layout": args.layout} if args.layout != "tqkv" else {})},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": "pack + unpack of one rank per step"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_merge_bench(args):
    """--kernel lse_merge: the log-sum-exp merge of two key-segment attention
    outputs of the Wan-like 480p layer (8 ranks batched: [2, 1, 32760, 12, 128])."""
    import numpy as np
    import torch

    import workloads
    import diffusion_transformer_context_gb300 as ctx

    P, B, Sq, H, D = 2, 1, 32760, 12, 128
    gen = torch.Generator().manual_seed(workloads.SEED)
    o_host = workloads.randn((P, B, Sq, H, D), gen)
    l_host = torch.randn((P, B, H, Sq), generator=gen) * 3 + 10
    o, lse_p = o_host.cuda(), l_host.cuda()
    out = torch.empty((B, Sq, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    rows = B * Sq * H
    nbytes = P * rows * D * 2 + P * rows * 4 + rows * D * 2 + rows * 4
    for _ in range(args.warmup):
        ctx.ctx_lse_merge(o, lse_p, out, lse)
    torch.cuda.synchronize()
    sampler = None if args.no_clocks else ClockSampler(0)
    if sampler:
        sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        ctx.ctx_lse_merge(o, lse_p, out, lse)
    e1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    ms = e0.elapsed_time(e1) / args.steps
    gbs = nbytes / (ms * 1e-3) / 1e9
    # the same traffic mix without the merge arithmetic: an elementwise add of
    # the two segments' O (two reads and one write of the same O bytes), timed
    # the same way, as the reference for what this mix reaches on the device
    add_out = torch.empty_like(out)
    for _ in range(args.warmup):
        torch.add(o[0], o[1], out=add_out)
    e0.record()
    for _ in range(args.steps):
        torch.add(o[0], o[1], out=add_out)
    e1.record()
    torch.cuda.synchronize()
    add_bytes = 3 * rows * D * 2
    add_gbs = add_bytes / (e0.elapsed_time(e1) / args.steps * 1e-3) / 1e9
    # e2e: parts in from pinned host memory, merged output back
    oh, lh = o_host.pin_memory(), l_host.pin_memory()
    outh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e0.record()
    for _ in range(args.steps):
        o.copy_(oh, non_blocking=True)
        lse_p.copy_(lh, non_blocking=True)
        ctx.ctx_lse_merge(o, lse_p, out, lse)
        outh.copy_(out, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    peaks, kind = load_peaks()
    line = {"metric": "LSE merge of key-segment attention outputs, GB/s & % HBM", "value": round(gbs, 1),
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "lse_merge", "P": P, "B": B, "Sq": Sq, "H": H, "D": D,
                       "l2": "inputs_larger_than_l2"},
            "roofline": {"bound": "hbm", "kernel": "lse_merge_kernel", "achieved": round(gbs, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                         "peak_source": f"{kind} hbm_gbs", "algorithmic_bytes_per_launch": nbytes,
                         "traffic": recorded_traffic("wan480_two_segments", "merge"), "add_gbs": round(add_gbs, 1),
                         "add_note": "torch.add of the two segments' O (2 reads + 1 write of the same O bytes), "
                                     "timed the same way"},
            "gpu_launches": args.steps, "clocks": clocks,
            "e2e": {"value": round(nbytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": oh.numel() * 2 + lh.numel() * 4,
                    "d2h_bytes_per_step": outh.numel() * 2, "ms_per_step": round(e2e_ms, 4),
                    "pipeline": "copies and compute one after another"}}
    if not args.no_cpu_baseline:
        import oracle
        n = 4096  # rows of the sample
        ou = workloads.as_u16(o_host[:, :, :n // H])
        t = time.perf_counter()
        oracle.lse_merge(ou, l_host[:, :, :, :n // H].double().numpy())
        dt = time.perf_counter() - t
        sample_bytes = nbytes * (n // H) / Sq
        line["cpu_baseline"] = {"value": round(sample_bytes / dt / 1e9, 3), "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "sample": f"first {n // H} query rows of every head"}
    print(json.dumps(line), flush=True)


def run_attn_bench(args):
    """--kernel attn: one ctx_attn_lq_gkv call of --attn-shape B,Sq,Sk,H,D
    (seeded N(0,1) inputs in --dtype, no mask, scale 1/sqrt(D)), balanced
    schedule unless --unbalanced. L2 is flushed (a 256 MB write) before every
    timed launch and each launch is timed alone with CUDA events on the
    launching stream. Work: 4 * B * H * Sq * Sk * D FLOP per call."""
    import numpy as np
    import torch

    import workloads
    import diffusion_transformer_context_gb300 as ctx

    B, Sq, Sk, H, D = (int(x) for x in args.attn_shape.split(","))
    gen = torch.Generator().manual_seed(workloads.SEED)
    q_h = workloads.randn((B, Sq, H, D), gen, args.dtype)
    k_h = workloads.randn((B, Sk, H, D), gen, args.dtype)
    v_h = workloads.randn((B, Sk, H, D), gen, args.dtype)
    q, k, v = q_h.cuda(), k_h.cuda(), v_h.cuda()
    out = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    ws = None if args.unbalanced else ctx.attn_workspace(B, Sq, Sk, H, D)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flops = 4.0 * B * H * Sq * Sk * D

    def call():
        ctx.ctx_attn_lq_gkv(q, k, v, out, lse, workspace=ws)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    st = ctx.ctx_device_status()
    if st != 0:
        raise RuntimeError(f"device status: {ctx.ctx_status_string(st)}")
    sampler = None if args.no_clocks else ClockSampler(0)
    if sampler:
        sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e0, e1 in ev:
        flush.fill_(1)
        e0.record()
        call()
        e1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / args.steps
    tflops = flops / (ms * 1e-3) / 1e12
    # e2e: Q/K/V in from pinned host memory, O and LSE back, one step after another
    qp, kp, vp = (t.pin_memory() for t in (q_h, k_h, v_h))
    oh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    e0, e1 = ev[0]
    e0.record()
    for _ in range(args.steps):
        q.copy_(qp, non_blocking=True)
        k.copy_(kp, non_blocking=True)
        v.copy_(vp, non_blocking=True)
        call()
        oh.copy_(out, non_blocking=True)
        lh.copy_(lse, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    peaks, kind = load_peaks()
    line = {"metric": METRIC, "value": round(tflops, 3), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
            "config": {"workload": "attn", "B": B, "Sq": Sq, "Sk": Sk, "H": H, "D": D,
                       "l2": "flushed_between_steps",
                       "attn_schedule": "one CTA per unit" if ws is None else "persistent, key-split tail"},
            "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel", "achieved": round(tflops, 2),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(tflops / peaks["bf16_tflops"], 4),
                         "peak_source": f"{kind} bf16_tflops (burst)", "algorithmic_flops_per_launch": flops,
                         "launch_ms": round(ms, 4), "traffic": None},
            "gpu_launches": args.steps, "clocks": clocks,
            "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": 2 * (qp.numel() + kp.numel() + vp.numel()),
                    "d2h_bytes_per_step": 2 * oh.numel() + 4 * lh.numel(), "ms_per_step": round(e2e_ms, 4),
                    "pipeline": "copies and compute one after another"}}
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        u16 = workloads.as_u16
        rng = np.random.default_rng(workloads.SEED)
        n = 256
        bhi = np.stack([rng.integers(0, B, n), rng.integers(0, H, n), rng.integers(0, Sq, n)], axis=1)
        t = time.perf_counter()
        oracle.attention_rows(u16(q_h), u16(k_h), u16(v_h), bhi, dtype=args.dtype)
        dt = time.perf_counter() - t
        line["cpu_baseline"] = {"value": round(4.0 * Sk * D * n / dt / 1e12, 6), "unit": "TFLOP/s",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": f"{n} random query rows, all {Sk} keys each"}
    print(json.dumps(line), flush=True)


VARLEN_DOCS = (12288, 8192, 6144, 4096, 2048)  # tokens per packed document (sum 32768)


def run_varlen_bench(args):
    """--kernel varlen: packed variable-length documents under AllGather-KV.
    One packed sequence of 32768 tokens holds five documents (VARLEN_DOCS),
    12 heads, D = 128, over A = 8 ranks: every rank remaps the global query
    boundaries to its span of 4096 rows (ctx_varlen_remap, on the device) and
    attends the whole documents' keys (ctx_attn_varlen); the eight ranks'
    launches go out on parallel streams. Work: sum over documents of
    4 * len^2 * H * D FLOP per step."""
    import numpy as np
    import torch

    import workloads
    import diffusion_transformer_context_gb300 as ctx

    S, H, D, A = sum(VARLEN_DOCS), 12, 128, 8
    S_l = S // A
    gen = torch.Generator().manual_seed(workloads.SEED)
    q_h, k_h, v_h = (workloads.randn((S, H, D), gen) for _ in range(3))
    q, k, v = q_h.cuda(), k_h.cuda(), v_h.cuda()
    bounds = np.concatenate([[0], np.cumsum(VARLEN_DOCS)]).astype(np.int32)
    cu = torch.from_numpy(bounds).cuda()
    n_docs = len(VARLEN_DOCS)
    cu_loc = [torch.empty(n_docs + 1, dtype=torch.int32, device="cuda") for _ in range(A)]
    out = torch.empty((A, S_l, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((A, H, S_l), dtype=torch.float32, device="cuda")
    lanes = [torch.cuda.Stream() for _ in range(A)]
    flops = float(sum(4.0 * n * n * H * D for n in VARLEN_DOCS))
    # the eight simulated ranks share the GPU concurrently, so each call runs one CTA per
    # unit; one rank alone (as on its own GPU) is also timed with the balanced schedule
    ws0 = ctx.varlen_workspace(n_docs, S_l, H, D)

    def step():
        base = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(base)
        for r, s in enumerate(lanes):
            s.wait_event(fork)
            ctx.ctx_varlen_remap(cu, r * S_l, S_l, cu_loc[r], stream=s)
            ctx.ctx_attn_varlen(q[r * S_l:(r + 1) * S_l], k, v, cu_loc[r], cu, S_l, out[r], lse[r], stream=s)
            done = torch.cuda.Event()
            done.record(s)
            base.wait_event(done)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = ctx.ctx_device_status()
    if st != 0:
        raise RuntimeError(f"device status: {ctx.ctx_status_string(st)}")
    sampler = None if args.no_clocks else ClockSampler(0)
    if sampler:
        sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    ms = e0.elapsed_time(e1) / args.steps
    tflops = flops / (ms * 1e-3) / 1e12

    # one rank alone (a deployment runs one rank per GPU): rank 0, balanced and one CTA per unit
    def one_rank(ws):
        ctx.ctx_varlen_remap(cu, 0, S_l, cu_loc[0])
        for _ in range(3):
            ctx.ctx_attn_varlen(q[:S_l], k, v, cu_loc[0], cu, S_l, out[0], lse[0], workspace=ws)
        e0.record()
        for _ in range(args.steps):
            ctx.ctx_attn_varlen(q[:S_l], k, v, cu_loc[0], cu, S_l, out[0], lse[0], workspace=ws)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps

    lens0 = np.clip(np.minimum(bounds[1:], S_l) - bounds[:-1], 0, None)
    flops0 = float(sum(4.0 * int(lq) * int(n) * H * D for lq, n in zip(lens0, VARLEN_DOCS)))
    ms_bal, ms_unit = one_rank(ws0), one_rank(None)
    one_rank_line = {"rank": 0, "flops": flops0,
                     "balanced_tflops": round(flops0 / (ms_bal * 1e-3) / 1e12, 1),
                     "one_cta_per_unit_tflops": round(flops0 / (ms_unit * 1e-3) / 1e12, 1)}
    # e2e: the packed Q/K/V in from pinned host memory, every rank's output back.
    # Two buffer sets take the steps in turn (double-buffered as in the layer's
    # e2e): step i's input is copied in on its own stream while step i-1
    # computes, its output read back on a third stream while later steps compute.
    qh, kh, vh = (t.pin_memory() for t in (q_h, k_h, v_h))
    outh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    sets = [(q, k, v, out, lse, cu_loc)] + [
        (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(out),
         torch.empty_like(lse), [torch.empty_like(c) for c in cu_loc])]
    cs = torch.cuda.current_stream()
    hs, ds = torch.cuda.Stream(), torch.cuda.Stream()
    x_free, out_free = [None, None], [None, None]

    def e2e_steps(n):
        for i in range(n):
            b = i & 1
            sq, sk, sv, so, sl, sc = sets[b]
            h2d_done, x_read, d2h_done = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(hs):
                if x_free[b] is not None:
                    hs.wait_event(x_free[b])  # this set's previous step has read its inputs
                for dst, src in ((sq, qh), (sk, kh), (sv, vh)):
                    dst.copy_(src, non_blocking=True)
                h2d_done.record(hs)
            cs.wait_event(h2d_done)
            if out_free[b] is not None:
                cs.wait_event(out_free[b])  # this set's previous output has been read back
            fork = torch.cuda.Event()
            fork.record(cs)
            for r, st_ in enumerate(lanes):
                st_.wait_event(fork)
                ctx.ctx_varlen_remap(cu, r * S_l, S_l, sc[r], stream=st_)
                ctx.ctx_attn_varlen(sq[r * S_l:(r + 1) * S_l], sk, sv, sc[r], cu, S_l, so[r], sl[r], stream=st_)
                done = torch.cuda.Event()
                done.record(st_)
                cs.wait_event(done)
            x_read.record(cs)
            with torch.cuda.stream(ds):
                ds.wait_event(x_read)
                outh.copy_(so, non_blocking=True)
                d2h_done.record(ds)
            x_free[b], out_free[b] = x_read, d2h_done
        for b in range(2):
            if out_free[b] is not None:
                cs.wait_event(out_free[b])  # the last read-backs are inside the timed region

    e2e_steps(2)
    torch.cuda.synchronize()
    e0.record()
    e2e_steps(args.steps)
    e1.record()
    torch.cuda.synchronize()
    last = sets[(args.steps - 1) & 1][3]
    readback_ok = bool(torch.equal(outh.view(torch.int16), last.cpu().view(torch.int16)))
    e2e_ms = e0.elapsed_time(e1) / args.steps
    peaks, kind = load_peaks()
    line = {"metric": METRIC, "value": round(tflops, 3), "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "varlen", "documents": list(VARLEN_DOCS), "S": S, "H": H, "D": D, "A": A,
                       "l2": "inputs_larger_than_l2", "launch": "8 ranks on parallel streams",
                       "attn_schedule": "one CTA per unit (8 concurrent ranks)"},
            "one_rank": one_rank_line,
            "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel (varlen)", "achieved": round(tflops, 2),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(tflops / peaks["bf16_tflops"], 4),
                         "peak_source": f"{kind} bf16_tflops (burst)", "algorithmic_flops_per_step": flops,
                         "traffic": recorded_traffic("varlen_step")},
            "gpu_launches": 2 * A * args.steps, "clocks": clocks,
            "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": 3 * qh.numel() * 2, "d2h_bytes_per_step": outh.numel() * 2,
                    "ms_per_step": round(e2e_ms, 4), "readback_verified": readback_ok,
                    "pipeline": "H2D / compute / D2H on three streams; two buffer sets take the steps in turn"}}
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        d0 = VARLEN_DOCS[0]
        u16 = workloads.as_u16
        qd, kd, vd = (u16(t[:d0].unsqueeze(0)) for t in (q_h, k_h, v_h))
        rng = np.random.default_rng(workloads.SEED)
        n = 512
        bhi = np.stack([np.zeros(n, np.int64), rng.integers(0, H, n), rng.integers(0, d0, n)], axis=1)
        t = time.perf_counter()
        oracle.attention_rows(qd, kd, vd, bhi)
        dt = time.perf_counter() - t
        line["cpu_baseline"] = {"value": round(4.0 * d0 * D * n / dt / 1e12, 6), "unit": "TFLOP/s",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": f"{n} random query rows of the {d0}-token document, all its keys"}
    print(json.dumps(line), flush=True)


def run_per_rank(args, rank, world, local_rank):
    """--per-rank: one process per rank of the workload's U x A job (launched
    by torchrun with U*A processes, one GPU each): the library's kernels for
    every data step and NCCL all_to_all_single / all_gather between them
    (diffusion_transformer_context_gb300.ranks). Timed like the default line:
    W warm-up steps, K steps between barriers, the slowest rank's time;
    `value` = the attention FLOPs of all ranks / that time."""
    import torch
    import torch.distributed as dist

    import workloads
    from diffusion_transformer_context_gb300.ranks import Groups, RankLayer

    wl = workloads.WORKLOADS[args.workload]
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist.init_process_group("nccl", device_id=dev)
    try:
        G = Groups(wl.U, wl.A)
        inp = workloads.make_inputs(wl)
        layer = RankLayer(wl, G, dev, layout=LAYOUTS[args.layout])
        layer.load(*(inp.shard(t, rank).to(dev) for t in (inp.q, inp.k, inp.v)),
                   None if inp.jk is None else inp.jk.to(dev), None if inp.jv is None else inp.jv.to(dev),
                   inp.image_mask, inp.joint_mask)
        for _ in range(args.warmup):
            layer.step()
        dist.barrier()
        torch.cuda.synchronize(dev)
        sampler = ClockSampler(local_rank) if (rank == 0 and not args.no_clocks) else None
        if sampler:
            sampler.start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            layer.step()
        e1.record()
        dist.barrier()
        torch.cuda.synchronize(dev)
        clocks = sampler.stop() if sampler else None
        ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
        flops = layer.attn_flops(valid_keys(inp))
        total = torch.tensor([flops], dtype=torch.float64, device=dev)
        dist.all_reduce(total)
        U, S_l = wl.U, layer.S_l
        # this library's launches per rank and step (NCCL's own kernels not counted)
        launches = (4 if U > 1 else 2) + (1 if layer.mask is not None else 0)
        line = {"metric": METRIC, "value": round(float(total.item()) / (ms / args.steps * 1e-3) / 1e12, 3),
                "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True, "scaling": "strong",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {**shape_config(wl), "parallelism": f"ulysses{wl.U} x agkv{wl.A}, one rank per GPU (NCCL)",
                           "per_rank": [wl.B, S_l, wl.H, wl.D], "l2": "inputs_larger_than_l2"},
                "gpu_launches": launches * args.steps, "clocks": clocks, "e2e": None}
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="wan480")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-pack", action="store_true", help="skip the layout-only pack workload line")
    ap.add_argument("--layout", default="tqkv", choices=sorted(LAYOUTS),
                    help="staging layout of the exchange: [U,3,B,S_l,h_l,D] or [U,B,S_l,h_l,3D]")
    ap.add_argument("--per-rank", action="store_true",
                    help="one process per rank of the workload's U x A job (torchrun with U*A GPUs), NCCL between")
    ap.add_argument("--unbalanced", action="store_true", help="attention without a workspace (no unit split between CTAs)")
    ap.add_argument("--eager", action="store_true", help="launch every kernel from Python instead of CUDA graphs")
    ap.add_argument("--kernel", default=None, choices=["lse_merge", "varlen", "attn"], help="time one kernel alone")
    ap.add_argument("--attn-shape", default="1,4095,32760,12,128",
                    help="--kernel attn: B,Sq,Sk,H,D of the attention call")
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "fp16"], help="--kernel attn: input dtype")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=64)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours" and not os.environ.get("CTX_BENCH_ALLOW_SHORT_WARMUP"):
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.kernel == "lse_merge":
        if rank == 0:
            run_merge_bench(args)
        return
    if args.kernel == "varlen":
        if rank == 0:
            run_varlen_bench(args)
        return
    if args.kernel == "attn":
        if rank == 0:
            run_attn_bench(args)
        return
    if args.per_rank:
        run_per_rank(args, rank, world, local_rank)
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    sim, inp, total_ms, parts, clocks, e2e = run_gpu(args, rank, world, local_rank)
    peaks, peak_kind = load_peaks()
    K = args.steps
    attn_flops = sim.attn_flops(valid_keys(inp))
    ms_step = total_ms / K

    def avg(x):
        return sum(x) / len(x)

    relayout_bytes = sim.pack_bytes() + sim.a2a_bytes() + sim.unpack_bytes()
    relayout_ms = avg(parts["exchange_in"])
    relayout_gbs = relayout_bytes / (relayout_ms * 1e-3) / 1e9
    reverse_ms = avg(parts["exchange_out"])
    relayout_kernel = ("relayout_kernel (unpack of all ranks; at U = 1 a rank's staging buffer is its input)"
                       if sim.pack_view else "relayout_kernel (pack + all-to-all + unpack of all ranks)")
    relayout = {"bound": "hbm", "kernel": relayout_kernel,
                "achieved": round(relayout_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(relayout_gbs / peaks["hbm_gbs"], 4), "peak_source": f"{peak_kind} hbm_gbs",
                "ms": round(relayout_ms, 4), "algorithmic_bytes": relayout_bytes,
                "reverse_ms": round(reverse_ms, 4), "reverse_bytes": sim.reverse_bytes(),
                "traffic": recorded_traffic(args.workload + ("" if args.layout == "tqkv" else "_" + args.layout),
                                            "relayout"),
                "note": "inside the step: written rows drain from L2 during the next kernel, so an upper bound; "
                        "the `pack` object times the layout kernels with reads from HBM and timed write-backs"}
    config = {**shape_config(sim.wl),
              "l2": "flushed_between_steps" if sim.l2_flushed else "inputs_larger_than_l2",
              "parallelism": f"replicas{world}",
              "launch": "eager" if args.eager else "cuda graphs (one per phase)"}
    if args.layout != "tqkv":
        config["staging_layout"] = args.layout
    line = {"metric": METRIC, "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": config}
    if sim.attention:
        attn_ms = avg(parts["attend"])
        tflops = attn_flops / (attn_ms * 1e-3) / 1e12 if attn_ms > 0 else 0.0
        peak_tf = peaks["bf16_tflops"]
        config["attn_call"] = f"B'={sim.wl.U * sim.wl.B} Sq={sim.wl.S} Sk={sim.Sk} H={sim.h_l} D={sim.wl.D}"
        config["attn_schedule"] = "one CTA per unit" if sim.ws is None else "persistent, key-split tail"
        line.update({"value": round(whole_job_tflops(attn_flops, world, ms_step), 3), "unit": "TFLOP/s",
                     "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel", "achieved": round(tflops, 2),
                                  "peak": peak_tf, "unit": "TFLOP/s", "frac": round(tflops / peak_tf, 4),
                                  "peak_source": f"{peak_kind} bf16_tflops (burst)",
                                  "algorithmic_flops_per_launch": attn_flops, "launch_ms": round(attn_ms, 4),
                                  "traffic": recorded_traffic(args.workload)},
                     "relayout": relayout})
    else:
        # layout-only workload: the metric is the pack / unpack bandwidth in HBM terms (buffer
        # sets rotated so that reads come from HBM and write-backs land inside the timed region);
        # the step's own figure re-reads the staging buffers from L2 and is kept beside it
        pk = run_pack_line(args, torch.device("cuda", local_rank), peaks, peak_kind)
        relayout["note"] = "whole simulated step, L2 flushed between steps; staging buffers re-read from L2"
        line.update({"value": round(world * pk["achieved"], 1), "unit": "GB/s", "roofline": pk,
                     "step": relayout})
        if e2e is not None:
            e2e["value"] = round(world * relayout_bytes / (e2e["ms_per_step"] * 1e-3) / 1e9, 1)
            e2e["unit"] = "GB/s"
    line.update({"gpu_launches": sim.launches_per_step() * K, "clocks": clocks, "e2e": e2e})
    if sim.attention and not args.no_pack:
        # the pack/unpack target's own workload, after the timed region of the headline step
        line["pack"] = run_pack_line(args, torch.device("cuda", local_rank), peaks, peak_kind)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline_sample(args.workload, args.cpu_seconds)
        if not sim.attention:
            cb = {"value": cb["relayout_gbs"], "unit": "GB/s", "cores": cb["cores"], "kind": "oracle",
                  "sample": cb["sample"].split("; ")[-1]}
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
