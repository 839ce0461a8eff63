"""Benchmark of the Vegas hot path: one verify + select + gamma-step sparse-draft iteration.

Default workload: the full iteration loop, 32 layers of Llama-3-8B-shaped heads
(H_q=32, H_kv=8, d=128) over B=8 sequences with ragged prefix lengths
n ~ U[4096, 65536], gamma=6, k=2048, Collect-2-Query selection; synthetic
heavy-hitter data.  The same line carries per-phase figures of the one-layer
workloads (llama8b n=32768; long70b n=131072; batched B=16 n=16384).

Timing discipline
  * Multi-layer workload: every layer stays resident (each is far larger than L2)
    and a step runs the model's order: verify and select on every layer, then each
    draft step over every layer.  One-layer workloads: the KV cache is replicated
    into enough copies that all of them together exceed 4x L2; step i verifies +
    selects on copy i mod C and runs the gamma draft steps on copy (i + C/2) mod C,
    so every kernel reads HBM cold and the draft never profits from the verify pass
    before it (the draft uses that copy's own earlier selection, the method's order).
  * W untimed warm-up steps, then K steps between CUDA events on the launching
    stream, bracketed by a barrier and device synchronisation; rank 0 prints the
    max over ranks.  Per-phase graphs (K verify calls, K selections, K draft phases
    on the same rotation) give the three roofline fractions: the verify call, the
    fused verify+select pass, and the draft phase.
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
DEFAULT_WORKLOAD = "loop32"
SECONDARY = "llama8b,long70b,batched"


def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--secondary", default=None,
                    help="comma-separated one-layer workloads measured per phase beside the headline "
                         f"(default: {SECONDARY} when the headline is {DEFAULT_WORKLOAD}; 'none' to skip)")
    ap.add_argument("--secondary-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline sample")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None,
                    help="only the first N layers of a multi-layer workload (small profiling captures)")
    return ap.parse_args(argv)


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
    """KV bytes one layer's iteration must read: the prefix once for verify, k + s + 1
    slots per draft step (the selection, then the draft tokens so far)."""
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


VERIFY_SOURCES = ("verify_attn.cu", "vg_common.cuh", "vg_internal.h")
DRAFT_SOURCES = ("sparse_draft.cu", "attn_frag.cuh", "vg_common.cuh", "vg_internal.h")


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


def source_sha(files=VERIFY_SOURCES) -> str:
    """sha256 over the code (comments left out) a kernel is compiled from."""
    h = hashlib.sha256()
    for f in files:
        src = open(os.path.join(ROOT, "self_speculative_sparse_gb300", "csrc", f), encoding="utf-8").read()
        h.update(strip_c_comments(src).encode())
    return h.hexdigest()


def verify_source_sha() -> str:
    return source_sha(VERIFY_SOURCES)


def profiled_traffic(kernel: str, workload: str, files) -> int | None:
    """Per-launch DRAM bytes of a kernel from its committed ncu summary
    (profiles/<kernel>_<workload>.md), if it was taken on the current sources (the
    summary records their sha256)."""
    prof = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(prof):
        return None
    vals = {}
    for line in open(prof):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256") != source_sha(files):
        return None
    try:
        return int(float(vals["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


def roofline_parts(w, S, fr, peaks, verify_launches) -> dict:
    """The three roofline fractions (verify call, fused verify + select, draft phase),
    each with the per-launch DRAM traffic of its dominant kernel where a committed ncu
    summary of the current sources has it (else null)."""
    parts = {k: {"bound": "hbm", "achieved": v["achieved_gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                 "frac": v["frac"]} for k, v in fr.items()}
    vt = profiled_traffic("verify_attn", w.name, VERIFY_SOURCES)
    for k in ("verify_call", "verify_select"):
        parts[k].update({"kernel": "verify_kernel", "traffic": vt,
                         "algorithmic_bytes_per_launch": S.nbytes["verify"] / verify_launches})
    parts["draft_phase"].update({"kernel": "draft_kernel",
                                 "traffic": profiled_traffic("draft_attn", w.name, DRAFT_SOURCES),
                                 "algorithmic_bytes_per_launch": S.nbytes["draft"] / (w.gamma * verify_launches)})
    return parts


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


def overlap_fraction(a, b, k) -> float:
    """|A ∩ B| / k of two selections (a reported statistic of the bench)."""
    import numpy as np
    if k <= 0:
        return 1.0
    return len(np.intersect1d(a, b)) / float(k)


# ------------------------------------------------------------------ CPU oracle timing
def oracle_iteration_time(w, pool, budget_s: float, max_reps: int = 1000):
    """Time the fp64 oracle on whole iterations of sequence 0 of the workload."""
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


def oracle_scale(w, lengths, n0: int) -> float:
    """Factor from one oracle iteration of sequence 0 to the whole workload: prefix tokens
    (the verification dominates the oracle's work) and layers."""
    return w.layers * float(sum(int(n) for n in lengths)) / n0


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    import synth
    if rank != 0:
        return
    w = synth.WORKLOADS[args.workload]
    lengths = w.lengths()
    if w.layers > 1 or w.B > 1:
        w_sample = synth.scaled(w, B=1, layers=1, n=int(lengths[0]), ragged=None)
    else:
        w_sample = w
    pool = w_sample.layer_pool(0)
    for _ in range(args.warmup):
        oracle_iteration_time(w_sample, pool, 0.0, max_reps=1)
    times = []
    for _ in range(args.steps):
        times += oracle_iteration_time(w_sample, pool, 0.0, max_reps=1)
    n0 = int(pool["prefix_len"][0])
    scale = oracle_scale(w, lengths, n0)
    per_iter_us = statistics.mean(times) * 1e6 * scale
    sample = (f"{args.steps} oracle iterations of sequence 0 (n={n0}), scaled x{scale:.2f} to the workload's "
              f"prefix tokens and layers" if scale != 1.0 else
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
class Setup:
    """A workload resident on the GPU, with the step and per-phase call sequences."""

    def __init__(self, w, local: int):
        import torch
        from self_speculative_sparse_gb300.runtime import LayerState
        self.w = w
        self.multi = w.layers > 1
        dev = f"cuda:{local}"
        self.pool = w.layer_pool(0)
        self.lengths = self.pool["prefix_len"]
        self.layer_bytes = int(self.pool["K"].nbytes + self.pool["V"].nbytes)
        self.l2 = torch.cuda.get_device_properties(local).L2_cache_size
        if self.multi:
            # every layer resident (each far larger than L2): the model's own order streams them
            self.ncopy = w.layers
            self.states = [LayerState(w, self.pool, device=dev)]
            for layer in range(1, w.layers):
                self.states.append(LayerState(w, w.layer_pool(layer), device=dev))
        else:
            # rotating copies of the one layer, so every kernel reads its cache cold
            self.ncopy = max(3, -(-4 * self.l2 // self.layer_bytes) + 1)
            self.states = [LayerState(w, self.pool, device=dev) for _ in range(self.ncopy)]
        self.stream = torch.cuda.current_stream()
        self.side = torch.cuda.Stream(device=dev)  # (the multi-layer step's selections)
        self.tl = [torch.full((w.B,), s + 1, dtype=torch.int32, device=dev) for s in range(w.gamma)]
        self.half = self.ncopy // 2
        # per layer: the prefix once for verify, the selection + draft tokens per draft step
        self.nbytes = {k: v * w.layers for k, v in algorithmic_bytes(w, self.lengths).items()}
        # every copy gets one full iteration first, so each has its own selection
        for st in self.states:
            st.iteration(stream=self.stream, select_extra=False)
        torch.cuda.synchronize()
        self.check("set-up")

    def check(self, when: str) -> None:
        bad = [(i, st.check_status()) for i, st in enumerate(self.states) if st.check_status() != 0]
        if bad:
            raise RuntimeError(f"device status at {when} (copy, code): {bad}")

    def draft_phase(self, st) -> None:
        for s in range(self.w.gamma):
            st.draft_step(s, self.tl[s])

    def step(self, i: int) -> None:
        if self.multi:
            # The model's order: verify every layer, then each draft step over the layers.
            # A layer's selection is needed only by the draft phase, so it runs on a second
            # stream beside the next layers' verification (the next layer's verify depends
            # on this layer's output, not on its selection); the draft phase joins it.
            # (The fork and the join go through the stream current at the call - the
            # capturing one inside a graph capture - so the side stream joins the capture.)
            import torch
            cur = torch.cuda.current_stream()
            for st in self.states:
                st.verify()
                ev = torch.cuda.Event()
                ev.record(cur)
                self.side.wait_event(ev)
                st.select(stream=self.side)
            done = torch.cuda.Event()
            done.record(self.side)
            cur.wait_event(done)
            for s in range(self.w.gamma):
                for st in self.states:
                    st.draft_step(s, self.tl[s])
            return
        # one layer: verify + select on copy i, the draft phase on copy i + ncopy/2
        a, b = self.states[i % self.ncopy], self.states[(i + self.half) % self.ncopy]
        a.verify()
        a.select()
        self.draft_phase(b)

    def phase_calls(self, i: int, which: str) -> None:
        """The calls of step(i) for one phase only: 'v' verify, 's' select, 'd' draft."""
        if self.multi:
            for st in self.states:
                if which == "v":
                    st.verify()
                elif which == "s":
                    st.select()
            if which == "d":
                for s in range(self.w.gamma):
                    for st in self.states:
                        st.draft_step(s, self.tl[s])
            return
        if which == "v":
            self.states[i % self.ncopy].verify()
        elif which == "s":
            self.states[i % self.ncopy].select()
        else:
            self.draft_phase(self.states[(i + self.half) % self.ncopy])

    def verify_masked(self, i: int, m0: int) -> None:
        """The verify call of step(i) with one score mask (or none)."""
        from self_speculative_sparse_gb300 import binding as vb
        sts = self.states if self.multi else [self.states[i % self.ncopy]]
        for st in sts:
            vb.vg_verify_attn(st.dims, st.cache, st.q_verify, st.k_new, st.v_new, st.prefix_len, m0, 0,
                              st.scores0 if m0 else None, None, st.score_stride, st.out_verify, st.ws,
                              dev_status=st.status)


def capture(fn):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        fn()
    return g


def time_graph_us(g, stream, reps: int) -> float:
    """Mean µs per rep of a graph holding `reps` reps: launched once untimed (its upload),
    then once between two events on the launching stream."""
    import torch
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / reps


def phase_times(S: Setup, first: int, steps: int) -> dict:
    """Per-phase µs of one step (sums over the layers of a multi-layer workload)."""
    t = {}
    for which, nm in (("v", "verify_call"), ("s", "select"), ("d", "draft_gamma_steps")):
        g = capture(lambda which=which: [S.phase_calls(first + i, which) for i in range(steps)])
        t[nm] = time_graph_us(g, S.stream, steps)
        del g
    t["per_draft_step"] = t["draft_gamma_steps"] / max(1, S.w.gamma)
    return t


def score_cost(S: Setup, first: int, steps: int) -> dict:
    """The verify call without scores, with the Collect-2-Query rows and with all rows."""
    w = S.w
    R = w.gamma + 1
    variants = {"no_scores": 0, "collect2": (1 | (1 << w.gamma)), "all_rows": (1 << R) - 1}
    out = {}
    for nm, m0 in variants.items():
        g = capture(lambda m0=m0: [S.verify_masked(first + i, m0) for i in range(steps)])
        out[nm] = time_graph_us(g, S.stream, steps)
        del g
    base = out["no_scores"]
    for nm in ("collect2", "all_rows"):
        out[nm + "_overhead_pct"] = 100.0 * (out[nm] - base) / base
    return out


def fractions(S: Setup, ph: dict, peak: float) -> dict:
    """Three HBM fractions, each recomputable from phases_us and the algorithmic bytes:
    the verify call alone, the fused verify+select pass, and the draft phase."""
    vb_, db_ = S.nbytes["verify"], S.nbytes["draft"]
    def f(nbytes, us):
        gbs = nbytes / (us * 1e-6) / 1e9
        return {"achieved_gbs": gbs, "frac": gbs / peak, "bytes": nbytes, "us": us}
    return {"verify_call": f(vb_, ph["verify_call"]),
            "verify_select": f(vb_, ph["verify_call"] + ph["select"]),
            "draft_phase": f(db_, ph["draft_gamma_steps"])}


def selection_stats(S: Setup, score_us: dict, ph: dict, iter_us: float) -> dict:
    """Selection overhead (score emission + top-k) as a share of the iteration, and the
    overlap of the Collect-2-Query selection with the all-rows selection where both run."""
    import torch
    w = S.w
    mask_key = "collect2" if w.select_rows == "c2" else "all_rows"
    emit = score_us[mask_key] - score_us["no_scores"]
    out = {"score_emission_us": emit, "select_us": ph["select"],
           "selection_overhead_pct": 100.0 * (emit + ph["select"]) / iter_us,
           "note": "(verify with the selection mask - verify without scores + top-k) / iteration"}
    # the query-agnostic comparison policy (a sliding window of the last k positions)
    # against the verification-guided selection of the same layer
    from self_speculative_sparse_gb300 import binding as vb
    st = S.states[0]
    idx_w = torch.empty_like(st.idx)
    cnt_w = torch.empty_like(st.count)
    vb.vg_window_select(st.prefix_len, w.B, st.max_len, st.k, idx_w, cnt_w, dev_status=st.status)
    torch.cuda.synchronize()
    iv, cv, iw = st.idx.cpu().numpy(), st.count.cpu().numpy(), idx_w.cpu().numpy()
    ovw = [overlap_fraction(iv[b, :int(cv[b])], iw[b, :int(cv[b])], int(cv[b])) for b in range(w.B)]
    out["overlap_window_vs_" + w.select_rows] = {"mean": float(sum(ovw) / len(ovw)), "min": float(min(ovw)),
                                                 "sequences": len(ovw)}
    if w.extra_rows:
        ov = []
        for st in S.states[:1]:
            st.iteration(stream=S.stream, select_extra=True)
            torch.cuda.synchronize()
            idx, idx1 = st.idx.cpu().numpy(), st.idx1.cpu().numpy()
            cnt = st.count.cpu().numpy()
            for b in range(w.B):
                c = int(cnt[b])
                ov.append(overlap_fraction(idx[b, :c], idx1[b, :c], c))
        out["overlap_" + w.select_rows + "_vs_" + w.extra_rows] = {
            "mean": float(sum(ov) / len(ov)), "min": float(min(ov)), "sequences": len(ov)}
    return out


def secondary_line(name: str, local: int, steps: int, peak: float) -> dict:
    import synth
    import torch
    w = synth.WORKLOADS[name]
    S = Setup(w, local)
    ph = phase_times(S, 0, steps)
    sc = score_cost(S, 0, steps)
    g_run = capture(lambda: [S.step(i) for i in range(steps)])
    it_us = time_graph_us(g_run, S.stream, steps)
    del g_run
    S.check("secondary " + name)
    out = {"workload": workload_desc(w), "us_per_iteration": it_us, "phases_us": ph,
           "fractions_of_hbm": fractions(S, ph, peak), "verify_call_by_score_rows_us": sc,
           "selection": selection_stats(S, sc, ph, it_us)}
    del S
    torch.cuda.empty_cache()
    return out


ACCEPT_VOCAB = 151936  # a Qwen3-family vocabulary (the pages' models)


def accept_timing(w, local: int, steps: int, peak: float) -> dict:
    """The acceptance step after verification (greedy and speculative sampling) on
    synthetic logits of the workload's batch and gamma, vocabulary ACCEPT_VOCAB."""
    import torch
    import synth
    from self_speculative_sparse_gb300 import binding as vb
    B, gamma, V = w.B, w.gamma, ACCEPT_VOCAB
    inp = synth.accept_inputs(B, gamma, V, seed=7)
    dev = f"cuda:{local}"
    # copies of the inputs, rotated per step, that together exceed twice the L2
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    per = sum(v.nbytes for v in inp.values())
    ncopy = max(2, -(-2 * l2 // per))
    ts = [{k: torch.from_numpy(v).to(dev) for k, v in inp.items()} for _ in range(ncopy)]
    na = torch.empty(B, dtype=torch.int32, device=dev)
    nt = torch.empty(B, dtype=torch.int32, device=dev)
    ws = torch.empty(vb.vg_accept_workspace_size(B, gamma, V), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    out = {"workload": f"B={B} gamma={gamma} V={V}, fp32 logits; inputs rotated over {ncopy} copies (> 2x L2)"}
    for mode, nm in ((vb.VG_ACCEPT_GREEDY, "greedy"), (vb.VG_ACCEPT_SAMPLE, "sample")):
        def call(i):
            t = ts[i % ncopy]
            vb.vg_accept(B, gamma, V, t["p_logits"], t["q_logits"], t["x"], t["u"], t["u_res"], mode, na, nt, None,
                         ws, dev_status=status)
        call(0)
        torch.cuda.synchronize()
        g = capture(lambda: [call(i) for i in range(steps)])
        us = time_graph_us(g, stream, steps)
        del g
        rows = B * (gamma + 1) + (B * gamma if mode == vb.VG_ACCEPT_SAMPLE else 0)
        nbytes = rows * V * 4 + (B * 2 * V * 4 if mode == vb.VG_ACCEPT_SAMPLE else 0)
        gbs = nbytes / (us * 1e-6) / 1e9
        out[nm] = {"us": us, "bytes": nbytes, "achieved_gbs": gbs, "frac": gbs / peak,
                   "mean_accepted": float(na.float().mean().item())}
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} in the acceptance step")
    return out


def run_ours(args, rank, local, world):
    import torch
    import synth
    from self_speculative_sparse_gb300 import build as vbuild

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    vbuild.build()
    w = synth.WORKLOADS[args.workload]
    if args.layers:
        w = synth.scaled(w, layers=min(w.layers, args.layers))
    S = Setup(w, local)
    stream, multi, ncopy = S.stream, S.multi, S.ncopy

    # One graph per timed run (a serving loop replays captured decode steps, so the
    # host's launch cost stays off the GPU timeline); warm-up steps in a graph of their own.
    g_warm = capture(lambda: [S.step(i) for i in range(args.warmup)])
    g_run = capture(lambda: [S.step(args.warmup + i) for i in range(args.steps)])
    torch.cuda.synchronize()
    g_run.replay()  # the graph's first launch (it uploads the graph), untimed
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
    clk = clocks.stop()
    del g_warm, g_run
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps
    ph = phase_times(S, args.warmup, args.steps)

    # ---- K steps launched eagerly (no graph): one vg_iteration call per step (the
    # model's per-layer calls for the multi-layer workload); the mean from two events
    # around them, the spread from a second pass with an event between steps
    def eager_step(i):
        if multi:
            S.step(i)
        else:
            S.states[i % ncopy].iteration(stream=stream, select_extra=False)

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
        g_dw = capture(lambda: [S.draft_phase(S.states[0]) for _ in range(args.steps)])
        draft_warm = time_graph_us(g_dw, stream, args.steps) / max(1, w.gamma)
        del g_dw
    sc = score_cost(S, args.warmup, args.steps)
    S.check("timed runs")

    # ---- end to end through the public C ABI with host buffers.  A step's inputs sit
    # in one pinned host buffer and one device buffer (the tensors the call reads are
    # views into it), so one copy brings them in; the outputs the same way, one copy out.
    e2e_steps = args.e2e_steps or args.steps
    in_names = ("q_verify", "k_new", "v_new", "q_draft", "k_draft", "v_draft")
    out_names = ("out_verify", "idx", "count", "out_draft")
    staged = []
    for a in S.states:
        dev_in = pack_views(a, in_names, copy_values=True)
        dev_out = pack_views(a, out_names, copy_values=False)
        host_in = torch.empty_like(dev_in, device="cpu").pin_memory()
        host_in.copy_(dev_in)
        host_out = torch.empty_like(dev_out, device="cpu").pin_memory()
        staged.append((a, dev_in, host_in, dev_out, host_out))
    st0 = S.states[0]
    bi = sum(getattr(st0, nm).numel() * getattr(st0, nm).element_size() for nm in in_names)
    bo = sum(getattr(st0, nm).numel() * getattr(st0, nm).element_size() for nm in out_names)
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

    # each buffer set's iteration captured once (vg_iteration_plan_create), launched per
    # step; the multi-layer workload runs its step's per-layer calls in the model's order
    # (as the timed graph does), its layers' inputs in before and results out after
    plans = [] if multi else [a.plan(select_extra=False) for a, *_ in staged]
    ev_all = torch.cuda.Event()
    # (the multi-layer step's public calls captured once, as a serving loop captures its
    # decode step, and replayed per step; the capture reads the staged buffers' views)
    g_e2e = capture(lambda: S.step(0)) if multi else None

    def e2e_step_multi(i):
        for sl in range(nslot):
            a, dev_in, host_in, dev_out, host_out = staged[sl]
            if used[sl]:
                s_in.wait_event(ev_done[sl])
            with torch.cuda.stream(s_in):
                dev_in.copy_(host_in, non_blocking=True)
            ev_in[sl].record(s_in)
            stream.wait_event(ev_in[sl])
            if used[sl]:
                stream.wait_event(ev_read[sl])
        g_e2e.replay()
        ev_all.record(stream)
        for sl in range(nslot):
            a, dev_in, host_in, dev_out, host_out = staged[sl]
            ev_done[sl] = ev_all
            s_out.wait_event(ev_all)
            with torch.cuda.stream(s_out):
                host_out.copy_(dev_out, non_blocking=True)
            ev_read[sl].record(s_out)
            used[sl] = True

    def e2e_step(i):
        if multi:
            e2e_step_multi(i)
            return
        for sl in [i % ncopy]:
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
    del g_e2e
    S.check("end-to-end steps")

    us_iter = ms_step * 1e3 / world  # whole-job: iterations of all ranks per unit time
    peaks = measured_peaks()
    fr = fractions(S, ph, peaks["hbm_gbs"])
    kv_gbs = (S.nbytes["verify"] + S.nbytes["draft"]) / (ms_step * 1e-3) / 1e9
    launches_per_step = S.states[0].launches_per_iteration(tail_from_device=True) * (w.layers if multi else 1)
    verify_launches = w.layers if multi else 1
    line = {
        "metric": METRIC, "value": us_iter, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(w),
                   "l2": (f"{w.layers} resident layers of {S.layer_bytes / 1e6:.0f} MB each (L2 "
                          f"{S.l2 / 1e6:.0f} MB): verify over every layer (each layer's selection on a second "
                          f"stream beside the next layers' verification), then each draft step over every layer"
                          if multi else
                          f"{ncopy} rotating cache copies of {S.layer_bytes / 1e6:.0f} MB (> 4x L2 of "
                          f"{S.l2 / 1e6:.0f} MB); draft on a different copy than the verify before it"),
                   "timing": ("K steps replayed as one CUDA graph, CUDA events around it; the graph is launched "
                              "once untimed first (its upload), the W warm-up steps run just before it"),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "kv_bytes_per_iteration": S.nbytes["verify"] + S.nbytes["draft"],
        "kv_gbs": kv_gbs, "kv_pct_of_hbm": 100.0 * kv_gbs / peaks["hbm_gbs"],
        "eager_launches_us": {"mean": eager_mean, "p10": pct(eager_steps, 0.1), "p50": pct(eager_steps, 0.5),
                              "p90": pct(eager_steps, 0.9),
                              "note": "per rank, no CUDA graph: vg_iteration per step (its kernels launched one "
                                      "by one; the multi-layer workload: its per-layer calls in the model's "
                                      "order); percentiles over steps timed with an event between steps"},
        "draft_step_l2_warm_us": draft_warm,
        "phases_us": ph,
        "phases_note": "sums over the layers of one step" if multi else "one layer",
        "fractions_of_hbm": fr,
        "verify_call_by_score_rows_us": sc,
        "selection": selection_stats(S, sc, ph, ms_step * 1e3),
        "roofline": {"kernel": "vg_verify_attn (verify_kernel + combine), the largest share of the step",
                     "bound": "hbm", "achieved": fr["verify_call"]["achieved_gbs"], "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": fr["verify_call"]["frac"], "peak_source": peaks["source"],
                     "traffic": profiled_traffic("verify_attn", w.name, VERIFY_SOURCES),
                     "algorithmic_bytes_per_launch": S.nbytes["verify"] / verify_launches,
                     "launch_us": ph["verify_call"] / verify_launches,
                     "parts": roofline_parts(w, S, fr, peaks, verify_launches)},
        "e2e": {"value": e2e_s / e2e_steps * 1e6 / world, "unit": UNIT, "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo,
                "api": ("vg_verify_attn / vg_topk_select / vg_sparse_draft_attn per layer in the model's order, "
                        "captured once as a CUDA graph of the step and launched per step" if multi else
                        "vg_iteration_plan_launch (each buffer set's iteration captured once at set-up)"),
                "copies": "pinned host buffers; one copy in and one out per step, on streams of their own "
                          "that overlap the neighbouring steps' compute; host clock around all steps"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
    }
    pool, lengths = S.pool, S.lengths
    del staged, plans, S
    torch.cuda.empty_cache()

    if rank == 0:
        line["accept_step_us"] = accept_timing(w, local, args.steps, peaks["hbm_gbs"])
    names = args.secondary if args.secondary is not None else (SECONDARY if args.workload == DEFAULT_WORKLOAD
                                                               else "none")
    if rank == 0 and names != "none":
        line["workloads"] = {}
        for nm in [x for x in names.split(",") if x and x != args.workload]:
            line["workloads"][nm] = secondary_line(nm, local, args.secondary_steps, peaks["hbm_gbs"])
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        times = oracle_iteration_time(w, pool, args.cpu_seconds)
        n0 = int(lengths[0])
        scale = oracle_scale(w, lengths, n0)
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
