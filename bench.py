"""Benchmark of the Vegas hot path: one verify + select + gamma-step sparse-draft iteration.

Default workload: one Llama-3-8B-shaped layer (B=1, H_q=32, H_kv=8, d=128,
n=32768, gamma=7, k=2048, Collect-2-Query), synthetic heavy-hitter data.

Timing discipline
  * the KV cache is replicated into enough copies that all of them together are
    larger than 4x L2; step i verifies + selects on copy i mod C and runs the gamma
    draft steps on copy (i + C/2) mod C, so every kernel reads HBM cold and the
    draft never profits from the verify pass that precedes it.  The draft uses
    that copy's own selection (made earlier on identical data), which is the
    method's order anyway: a draft phase follows the previous verification.
  * W untimed warm-up steps, then K steps between CUDA events on the launching
    stream, bracketed by a barrier and device synchronisation; rank 0 prints the
    max over ranks.  Per-phase events inside the timed region give the verify
    call's duration for the roofline figure.
  * nvidia-smi samples clocks and throttle reasons during the timed region.

`--impl reference` times the fp64 CPU oracle on the same workload (the only
reference implementation there is); `--gpus N` under torchrun runs N independent
replicas (the path has no data-path exchange: sequences are independent).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs per verify+select+sparse-draft iteration"
UNIT = "us/iteration"


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline sample")
    ap.add_argument("--e2e-steps", type=int, default=None)
    return ap.parse_args()


# ------------------------------------------------------------------ distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for nm, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ helpers
def workload_desc(w) -> str:
    n = f"n={w.n}" if w.n is not None else f"n~U[{w.ragged[0]},{w.ragged[1]}]"
    rows = "Collect-2-Query" if w.select_rows == "c2" else "all rows"
    return (f"{w.name}: B={w.B} H_q={w.Hq} H_kv={w.Hkv} d={w.d} {n} gamma={w.gamma} k={w.k} "
            f"select on {rows}" + (f" (+{w.extra_rows} overlap)" if w.extra_rows else "")
            + (f", {w.layers} layers" if w.layers > 1 else ""))


def algorithmic_bytes(w, lengths) -> dict:
    """KV bytes one iteration must read: the prefix once for verify, k + s + 1 slots per draft step."""
    per_tok = w.Hkv * w.d * 2 * 2
    verify = int(sum(lengths)) * per_tok
    draft = 0
    for n in lengths:
        cnt = min(w.k, int(n))
        for s in range(w.gamma):
            draft += (cnt + s + 1) * per_tok
    return {"verify": verify, "draft": draft, "per_token": per_tok}


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


VERIFY_SOURCES = ("verify_attn.cu", "attn_frag.cuh", "vg_common.cuh", "vg_internal.h")


def strip_c_comments(src: str) -> str:
    """C/C++ source without its comments and blank lines (string and character
    literals kept as they are), so that editing a comment leaves the code's hash."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(ln.rstrip() for ln in "".join(out).split("\n") if ln.strip())


def verify_source_sha() -> str:
    """sha256 over the code (comments left out) the verify kernel is compiled from."""
    h = hashlib.sha256()
    for f in VERIFY_SOURCES:
        src = open(os.path.join(ROOT, "self_speculative_sparse_gb300", "csrc", f), encoding="utf-8").read()
        h.update(strip_c_comments(src).encode())
    return h.hexdigest()


def profiled_traffic(workload: str):
    """Per-launch DRAM bytes of the verify kernel from the committed ncu summary, if it
    was taken on the current sources (the summary records their sha256)."""
    prof = os.path.join(ROOT, "profiles", f"verify_attn_{workload}.md")
    if not os.path.exists(prof):
        return None
    sha = verify_source_sha()
    vals = {}
    for line in open(prof):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256") != sha:
        return None
    try:
        return int(float(vals["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None



def pack_views(state, names, copy_values: bool):
    """One device byte buffer holding the state's tensors `names` (each slot 256-byte
    aligned); the state's attributes become views into it (values copied if asked)."""
    import torch

    offs, off = [], 0
    for nm in names:
        t = getattr(state, nm)
        offs.append(off)
        off = (off + t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(off, dtype=torch.uint8, device=getattr(state, names[0]).device)
    for nm, o in zip(names, offs):
        t = getattr(state, nm)
        v = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        if copy_values:
            v.copy_(t)
        setattr(state, nm, v)
    return buf

# ------------------------------------------------------------------ CPU oracle timing
def oracle_iteration_time(w, pool, budget_s: float, max_reps: int = 1000):
    """Time the fp64 oracle on whole iterations of sequence 0 of the workload."""
    import numpy as np
    import oracle
    from oracle import widen_bf16
    o, n = int(pool["seq_offset"][0]), int(pool["prefix_len"][0])
    K, V = widen_bf16(pool["K"][o:o + n]), widen_bf16(pool["V"][o:o + n])
    q = widen_bf16(pool["q_verify"][0])
    kn, vn = widen_bf16(pool["k_new"][0]), widen_bf16(pool["v_new"][0])
    qd, kd, vd = (widen_bf16(pool[x][:, 0]) for x in ("q_draft", "k_draft", "v_draft"))
    rows0 = w.rows(w.select_rows)
    rows1 = w.rows(w.extra_rows) if w.extra_rows else None
    times = []
    t_end = time.perf_counter() + budget_s
    while len(times) < max_reps:
        t0 = time.perf_counter()
        oracle.iteration(q, K, V, kn, vn, qd, kd, vd, w.k, rows0, rows1)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() > t_end:
            break
    return times


def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    import synth
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    if w.layers > 1 or w.B > 1:
        w_sample = synth.scaled(w, B=1, layers=1, n=int(w.lengths()[0]), ragged=None)
    else:
        w_sample = w
    pool = w_sample.layer_pool(0)
    for _ in range(args.warmup):
        oracle_iteration_time(w_sample, pool, 0.0, max_reps=1)
    times = []
    for _ in range(args.steps):
        times += oracle_iteration_time(w_sample, pool, 0.0, max_reps=1)
    # one oracle iteration covers one sequence of one layer; scale to the workload
    scale = w.B * w.layers if (w.layers > 1 or w.B > 1) else 1
    per_iter_us = statistics.mean(times) * 1e6 * scale
    sample = (f"{args.steps} oracle iterations of sequence 0 (n={int(pool['prefix_len'][0])}), "
              f"scaled x{scale} to the workload" if scale > 1 else
              f"{args.steps} full oracle iterations of the workload")
    line = {
        "impl": "reference", "metric": METRIC, "value": per_iter_us, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_iter_us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_desc(w)},
        "cpu_baseline": {"value": per_iter_us, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": per_iter_us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, local, world):
    import numpy as np
    import torch
    import synth
    from self_speculative_sparse_gb300 import build as vbuild
    from self_speculative_sparse_gb300 import binding as vb
    from self_speculative_sparse_gb300.runtime import LayerState

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    vbuild.build()
    w = synth.WORKLOADS[args.workload]
    multi = w.layers > 1
    pool = w.layer_pool(0)
    lengths = pool["prefix_len"]
    nbytes = {k: v * w.layers for k, v in algorithmic_bytes(w, lengths).items()}
    layer_bytes = int(pool["K"].nbytes + pool["V"].nbytes)
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    if multi:
        # every layer resident (each far larger than L2): the model's own order streams them
        ncopy = w.layers
        states = [LayerState(w, pool, device=f"cuda:{local}")]
        for layer in range(1, w.layers):
            states.append(LayerState(w, w.layer_pool(layer), device=f"cuda:{local}"))
    else:
        # rotating copies of the one layer, so every kernel reads its cache cold
        ncopy = max(3, -(-4 * l2 // layer_bytes) + 1)
        states = [LayerState(w, pool, device=f"cuda:{local}") for _ in range(ncopy)]
    stream = torch.cuda.current_stream()
    tl = [torch.full((w.B,), s + 1, dtype=torch.int32, device=f"cuda:{local}") for s in range(w.gamma)]

    def draft_phase(st):  # on the current stream (the capture stream inside a graph capture)
        for s in range(w.gamma):
            st.draft_step(s, tl[s])

    # every copy gets one full iteration first, so each has its own selection
    for st in states:
        st.iteration(stream=stream, select_extra=False)
    torch.cuda.synchronize()
    for st in states:
        if st.check_status() != 0:
            raise RuntimeError(f"device status {st.check_status()}")

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            fn()
        return g

    half = ncopy // 2

    def step(i):
        if multi:  # the model's order: verify every layer, select, then each draft step over the layers
            for st in states:
                st.verify()
                st.select()
            for s in range(w.gamma):
                for st in states:
                    st.draft_step(s, tl[s])
            return
        # one layer: verify + select on copy i, the draft phase on copy i + ncopy/2
        a, b = states[i % ncopy], states[(i + half) % ncopy]
        a.verify()
        a.select()
        draft_phase(b)

    def phase_calls(i, which):  # the same calls as step(i), one phase only
        if multi:
            for st in states:
                if which == "v":
                    st.verify()
                elif which == "s":
                    st.select()
            if which == "d":
                for s in range(w.gamma):
                    for st in states:
                        st.draft_step(s, tl[s])
            return
        if which == "v":
            states[i % ncopy].verify()
        elif which == "s":
            states[i % ncopy].select()
        else:
            draft_phase(states[(i + half) % ncopy])

    # One graph per timed run (a serving loop replays captured decode steps, so the
    # host's launch cost stays off the GPU timeline); warm-up steps in a graph of their own.
    g_warm = capture(lambda: [step(i) for i in range(args.warmup)])
    g_run = capture(lambda: [step(args.warmup + i) for i in range(args.steps)])
    # per-phase breakdown: the same calls, one phase at a time, K back to back
    g_v = capture(lambda: [phase_calls(args.warmup + i, "v") for i in range(args.steps)])
    g_s = capture(lambda: [phase_calls(args.warmup + i, "s") for i in range(args.steps)])
    g_d = capture(lambda: [phase_calls(args.warmup + i, "d") for i in range(args.steps)])
    torch.cuda.synchronize()
    for g in (g_run, g_v, g_s, g_d):  # each graph's first launch (it uploads the graph), untimed
        g.replay()
    torch.cuda.synchronize()

    # ---- headline: K steps between two events, right after the W warm-up steps (the
    # sampler's start-up pause would otherwise leave the GPU idle just before them)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    g_warm.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g_run.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_total = e0.elapsed_time(e1)
    # ---- per-phase events
    ph = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    ph[0].record(stream)
    g_v.replay()
    ph[1].record(stream)
    g_s.replay()
    ph[2].record(stream)
    g_d.replay()
    ph[3].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps
    t_verify = ph[0].elapsed_time(ph[1]) * 1e3 / args.steps
    t_select = ph[1].elapsed_time(ph[2]) * 1e3 / args.steps
    t_draft = ph[2].elapsed_time(ph[3]) * 1e3 / args.steps
    # ---- K steps launched eagerly (no graph): one vg_iteration call per step (the
    # model's per-layer calls for the multi-layer workload); the mean from two events
    # around them, the spread from a second pass with an event between steps
    def eager_step(i):
        if multi:
            step(i)
        else:
            states[i % ncopy].iteration(stream=stream, select_extra=False)

    torch.cuda.synchronize()
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ee[0].record(stream)
    for i in range(args.steps):
        eager_step(args.warmup + i)
    ee[1].record(stream)
    torch.cuda.synchronize()
    eager_mean = ee[0].elapsed_time(ee[1]) * 1e3 / args.steps
    es = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    es[0].record(stream)
    for i in range(args.steps):
        eager_step(args.warmup + i)
        es[i + 1].record(stream)
    torch.cuda.synchronize()
    eager_steps = sorted(es[i].elapsed_time(es[i + 1]) * 1e3 for i in range(args.steps))

    def pct(v, q):
        return v[min(len(v) - 1, int(round(q * (len(v) - 1))))]
    # ---- secondary: the draft phase with its gathered entries warm in L2 (K draft
    # phases on one cache copy), where the headline reads every step cold
    draft_warm = None
    if not multi:
        g_dw = capture(lambda: [draft_phase(states[0]) for _ in range(args.steps)])
        g_dw.replay()
        torch.cuda.synchronize()
        ew = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ew[0].record(stream)
        g_dw.replay()
        ew[1].record(stream)
        torch.cuda.synchronize()
        draft_warm = ew[0].elapsed_time(ew[1]) * 1e3 / args.steps / max(1, w.gamma)
    # ---- cost of the fused logit aggregation: the verify call with no scores, with the
    # Collect-2-Query rows and with all rows (same rotation, K back-to-back calls)
    R = w.gamma + 1
    variants = {"no_scores": 0, "collect2": (1 | (1 << w.gamma)), "all_rows": (1 << R) - 1}

    def verify_masked(st, m0):
        vb.vg_verify_attn(st.dims, st.cache, st.q_verify, st.k_new, st.v_new, st.prefix_len, m0, 0,
                          st.scores0 if m0 else None, None, st.score_stride, st.out_verify, st.ws,
                          dev_status=st.status)

    score_cost = {}
    if not multi:
        gv = {nm: capture(lambda m0=m0: [verify_masked(states[(args.warmup + i) % ncopy], m0)
                                         for i in range(args.steps)]) for nm, m0 in variants.items()}
        for nm, g in gv.items():
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            ev[0].record(stream)
            g.replay()
            ev[1].record(stream)
            torch.cuda.synchronize()
            score_cost[nm] = ev[0].elapsed_time(ev[1]) * 1e3 / args.steps
        base = score_cost["no_scores"]
        for nm in ("collect2", "all_rows"):
            score_cost[nm + "_overhead_pct"] = 100.0 * (score_cost[nm] - base) / base
    bad = [(i, st.check_status()) for i, st in enumerate(states) if st.check_status() != 0]
    if bad:
        raise RuntimeError(f"device status (copy, code): {bad}")

    # ---- end to end through the public C ABI (vg_iteration) with host buffers.  A
    # step's inputs sit in one pinned host buffer and one device buffer (the tensors
    # the call reads are views into it), so one copy brings them in; the outputs the
    # same way, one copy out.
    e2e_steps = args.e2e_steps or args.steps
    in_names = ("q_verify", "k_new", "v_new", "q_draft", "k_draft", "v_draft")
    out_names = ("out_verify", "idx", "count", "out_draft")
    e2e_states = states if multi else states[:ncopy]
    staged = []
    for a in e2e_states:
        dev_in = pack_views(a, in_names, copy_values=True)
        dev_out = pack_views(a, out_names, copy_values=False)
        host_in = torch.empty_like(dev_in, device="cpu").pin_memory()
        host_in.copy_(dev_in)
        host_out = torch.empty_like(dev_out, device="cpu").pin_memory()
        staged.append((a, dev_in, host_in, dev_out, host_out))
    bi = sum(getattr(states[0], nm).numel() * getattr(states[0], nm).element_size() for nm in in_names)
    bo = sum(getattr(states[0], nm).numel() * getattr(states[0], nm).element_size() for nm in out_names)
    bi, bo = bi * (w.layers if multi else 1), bo * (w.layers if multi else 1)

    # Copies run on streams of their own, as a serving loop overlaps them: a step's inputs
    # go in while the step before it computes, its results come out while the next one
    # computes.  Events keep each staging buffer safe: its inputs are overwritten only
    # after the call that read them has finished, its results only after they were read.
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    nslot = len(staged)
    ev_in = [torch.cuda.Event() for _ in range(nslot)]
    ev_done = [torch.cuda.Event() for _ in range(nslot)]
    ev_read = [torch.cuda.Event() for _ in range(nslot)]
    used = [False] * nslot

    # each buffer set's iteration captured once (vg_iteration_plan_create), launched per step
    plans = [a.plan(select_extra=False) for a, *_ in staged]

    def e2e_step(i):
        for sl in (range(nslot) if multi else [i % ncopy]):
            a, dev_in, host_in, dev_out, host_out = staged[sl]
            if used[sl]:
                s_in.wait_event(ev_done[sl])
            with torch.cuda.stream(s_in):
                dev_in.copy_(host_in, non_blocking=True)
            ev_in[sl].record(s_in)
            stream.wait_event(ev_in[sl])
            if used[sl]:
                stream.wait_event(ev_read[sl])
            plans[sl].launch(stream)
            ev_done[sl].record(stream)
            s_out.wait_event(ev_done[sl])
            with torch.cuda.stream(s_out):
                host_out.copy_(dev_out, non_blocking=True)
            ev_read[sl].record(s_out)
            used[sl] = True

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    barrier(world)
    for pl in plans:
        pl.close()
    bad = [(i, st.check_status()) for i, st in enumerate(e2e_states) if st.check_status() != 0]
    if bad:
        raise RuntimeError(f"device status after the end-to-end steps (copy, code): {bad}")

    us_iter = ms_step * 1e3 / world  # whole-job: iterations of all ranks per unit time
    peaks = measured_peaks()
    verify_gbs = nbytes["verify"] / (t_verify * 1e-6) / 1e9
    kv_gbs = (nbytes["verify"] + nbytes["draft"]) / (ms_step * 1e-3) / 1e9
    launches_per_step = (2 + 1 + 2 * w.gamma) * (w.layers if multi else 1)
    line = {
        "metric": METRIC, "value": us_iter, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(w),
                   "l2": (f"{w.layers} resident layers of {layer_bytes / 1e6:.0f} MB each (L2 {l2 / 1e6:.0f} MB): "
                          f"verify over every layer, then each draft step over every layer" if multi else
                          f"{ncopy} rotating cache copies of {layer_bytes / 1e6:.0f} MB (> 4x L2 of "
                          f"{l2 / 1e6:.0f} MB); draft on a different copy than the verify before it"),
                   "timing": ("K steps replayed as one CUDA graph, CUDA events around it; the graph is launched "
                              "once untimed first (its upload), the W warm-up steps run just before it"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "kv_bytes_per_iteration": nbytes["verify"] + nbytes["draft"],
        "kv_gbs": kv_gbs, "kv_pct_of_hbm": 100.0 * kv_gbs / peaks["hbm_gbs"],
        "eager_launches_us": {"mean": eager_mean, "p10": pct(eager_steps, 0.1), "p50": pct(eager_steps, 0.5),
                              "p90": pct(eager_steps, 0.9),
                              "note": "per rank, no CUDA graph: vg_iteration per step (its kernels launched one "
                                      "by one; the multi-layer workload: its per-layer calls in the model's "
                                      "order); percentiles over steps timed with an event between steps"},
        "draft_step_l2_warm_us": draft_warm,
        "phases_us": {"verify_call": t_verify, "select": t_select, "draft_gamma_steps": t_draft,
                      "per_draft_step": t_draft / max(1, w.gamma)},
        "phases_note": "sums over the layers of one step" if multi else "one layer",
        "verify_call_by_score_rows_us": score_cost,
        "roofline": {"kernel": "vg_verify_attn (verify_kernel + combine)", "bound": "hbm",
                     "achieved": verify_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": verify_gbs / peaks["hbm_gbs"], "peak_source": peaks["source"],
                     "traffic": profiled_traffic(w.name),
                     "algorithmic_bytes": nbytes["verify"]},
        "e2e": {"value": e2e_s / e2e_steps * 1e6 / world, "unit": UNIT, "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo,
                "api": "vg_iteration_plan_launch (each buffer set's iteration captured once at set-up)",
                "copies": "pinned host buffers; one copy in and one out per step, on streams of their own "
                          "that overlap the neighbouring steps' compute; host clock around all steps"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        times = oracle_iteration_time(w, pool, args.cpu_seconds)
        # sequence 0 of layer 0 is timed; the whole workload's time is scaled by prefix
        # tokens (the verification dominates the oracle's work) and by layers
        n0 = int(lengths[0])
        scale = w.layers * float(sum(int(n) for n in lengths)) / n0
        line["cpu_baseline"] = {"value": statistics.mean(times) * 1e6 * scale, "unit": UNIT, "cores": cpu_threads(),
                                "kind": "oracle",
                                "sample": f"{len(times)} fp64 oracle iterations of sequence 0 (n={n0}; verify, "
                                          f"both score masks, top-k, {w.gamma} draft steps)"
                                          + (f", scaled x{scale:.2f} to the workload's prefix tokens and layers"
                                             if scale != 1.0 else ", which is the whole workload")}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, local, world = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, local, world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
