"""Benchmark of one hybrid speculative-decoding round on GB300.

A step is one whole round on the device: n-gram lookup over every history,
pricing and batch-wide allocation (one fused kernel, spec_draft_and_price), and
chain verification over the full-vocabulary target rows of the allocated slots
(spec_verify_chain).  The workload is the
batch-128 mixed editing / chat configuration (context 4096, budget 256,
V = 151936 bf16 logits, T = 0); its logits are synthetic, laid out exactly as
the allocation asks (the target forward itself is not part of the path).

Timing: one CUDA graph holds a pass of 30 rounds rotating over the input
sets (the launches in order on one stream) and one more holds the rounds of K
past the last whole pass (all K when K < 30); each graph runs once untimed,
then W warm-up steps, then K steps of graph replays (passes, then the tail)
between a barrier and a device synchronisation,
with CUDA events on the launching stream around them (replays keep the device
queue ahead of the host, so the events time the kernels, not host launch
gaps); three input sets rotate so that every step reads logits that are not
in L2 (3 x 117 MB > 129 MB).
`value` = verified draft tokens per second (sum of verify_len per step);
rows/s, per-kernel times, the verify kernel's HBM roofline fraction, an
end-to-end figure through host buffers, the oracle's CPU time and the SM
clocks seen during the timed region ride along on the same JSON line.

--impl reference times the oracle (plain single-threaded C) on the host
cores on bounded samples of the same workload and prints the same metric.
Under torchrun each rank runs its own batch (weak scaling, no collective on
the data path); rank 0 prints.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft tokens/sec and verify rows/sec at V=151936, BS 4/128; % HBM roofline"
UNIT = "tokens/s"
WORKLOAD = "mixed_bs128"
NBUF = 3


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


KERNEL_SOURCES = ["speculative_decoding_draft_spec_gb300/csrc/verify.cu",
                  "speculative_decoding_draft_spec_gb300/csrc/common.cuh"]


def source_hash(paths):
    """sha256 of the sources with comments and blank space removed: a change to the
    code changes it, a change to a comment does not."""
    import hashlib
    import re

    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


def measured_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu summary
    (profiles/traffic.json), or None when the kernel's sources changed since (or
    no capture of that launch exists)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel, {}).get(workload)
    if not rec or rec.get("source_sha256") != source_hash(KERNEL_SOURCES):
        return None
    return rec["dram_bytes_per_launch"]


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_over_ranks(ms, tokens, rows, world, device="cpu"):
    """Whole-job figures of a weak-scaling run: the slowest rank's time and the
    tokens and rows of every rank (one all-reduce each; the path itself
    exchanges nothing)."""
    if world == 1:
        return ms, tokens, rows
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor([tokens, rows], dtype=torch.int64, device=device)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n[0].item()), int(n[1].item())


def build_workload(rank):
    import workloads as W

    return W.mixed_bs128(seed=1002 + rank)


def config_json(cfg, extra=None):
    d = {"workload": f"{WORKLOAD}: B={cfg['B']}, V={cfg['V']}, context 4096, budget {cfg['budget']}, "
                     f"lambda {cfg['lam']}, T=0, bf16 logits",
         "batch": cfg["B"], "vocab": cfg["V"], "context": 4096, "budget": cfg["budget"], "temperature": 0.0,
         "l2": f"{NBUF} rotating input sets (logits {NBUF} x > L2/3); no flush"}
    if extra:
        d.update(extra)
    return d


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) around a timed region: the sampler waits
    for its first sample before the region starts and for one taken after it
    ends, and keeps the last sample before the region, every sample inside it
    and the first after it (a region shorter than the interval is bracketed by
    its neighbours)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def _read(self):
        for ln in self.proc.stdout:
            if ln.strip():
                self._stamped.append((time.monotonic(), ln))

    def _wait(self, pred, limit=5.0):
        t = time.monotonic()
        while not pred() and time.monotonic() - t < limit:
            time.sleep(0.005)

    def __enter__(self):
        self._stamped = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()
        self._wait(lambda: len(self._stamped) > 0)
        self.t0 = time.monotonic()
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        t1 = time.monotonic()
        self._wait(lambda: any(t > t1 for t, _ in list(self._stamped)))
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self._thread.join(timeout=5)
        st = list(self._stamped)
        before = [x for x in st if x[0] < self.t0][-1:]
        inside = [x for x in st if self.t0 <= x[0] <= t1]
        after = [x for x in st if x[0] > t1][:1]
        self.lines = [ln for _, ln in before + inside + after]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- oracle baseline
def oracle_round(cfg, lay, logits, reqs):
    """The oracle's round over the requests `reqs` (lookup, batch pricing, their verification)."""
    import oracle as O

    sub = np.asarray(reqs)
    ng = O.ngram_propose(cfg["hist"][sub], cfg["hist_len"][sub], cfg["n_min"], cfg["n_max"], cfg["L"],
                         cfg["copy_cap"])
    if len(sub) == cfg["B"]:
        O.price_and_allocate(cfg["d"], cfg["c"], cfg["d_len"], ng.g, ng.g_len, ng.match_n, ng.agree,
                             ng.copy_len, cfg["coef"], cfg["lam"], cfg["budget"], cfg["max_verify_len"],
                             cfg["policy"], cfg["draft_greedy"])
    rows = [np.arange(lay.row_off[r], lay.row_off[r + 1]) for r in sub]
    ro = np.concatenate([[0], np.cumsum([len(x) for x in rows])]).astype(np.int32)
    O.verify_chain(logits[np.concatenate(rows)], ro, lay.chain[sub], lay.verify_len[sub])
    return int(lay.verify_len[sub].sum())


def oracle_layout(cfg):
    import oracle as O

    ng = O.ngram_propose(cfg["hist"], cfg["hist_len"], cfg["n_min"], cfg["n_max"], cfg["L"], cfg["copy_cap"])
    return O.price_and_allocate(cfg["d"], cfg["c"], cfg["d_len"], ng.g, ng.g_len, ng.match_n, ng.agree,
                                ng.copy_len, cfg["coef"], cfg["lam"], cfg["budget"], cfg["max_verify_len"],
                                cfg["policy"], cfg["draft_greedy"])


def host_cpu():
    """The host the oracle runs on: its architecture, CPU model (lscpu) and the
    number of cores the process may use."""
    import platform

    info = {"arch": platform.machine(), "cores_available": len(os.sched_getaffinity(0))
            if hasattr(os, "sched_getaffinity") else os.cpu_count(), "cpu_count": os.cpu_count()}
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            k, _, v = ln.partition(":")
            if k.strip() in ("Model name", "Vendor ID", "Socket(s)", "Core(s) per socket"):
                info[k.strip().lower().replace(" ", "_").replace("(s)", "s")] = v.strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return info


def cpu_baseline(cfg, lay, logits, seconds=10.0):
    tokens, t0, n = 0, time.perf_counter(), 0
    while time.perf_counter() - t0 < seconds:
        tokens += oracle_round(cfg, lay, logits, range(cfg["B"]))
        n += 1
    dt = time.perf_counter() - t0
    return {"value": tokens / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} full oracle rounds of the {WORKLOAD} batch ({dt:.1f} s, single-threaded C)",
            "host": host_cpu()}


def run_reference(args):
    import workloads as W

    rank, world, _ = dist_env()
    if rank != 0:
        return
    cfg = build_workload(0)
    lay = oracle_layout(cfg)
    logits = W.compact_logits(cfg, lay.row_off, lay.verify_len)
    # size each step so that the whole run stays within ~2 minutes
    t0 = time.perf_counter()
    oracle_round(cfg, lay, logits, range(cfg["B"]))
    t_full = time.perf_counter() - t0
    per_step = 100.0 / max(1, args.steps + args.warmup)
    s = int(max(1, min(cfg["B"], cfg["B"] * per_step / t_full)))
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        oracle_round(cfg, lay, logits, rng.choice(cfg["B"], s, replace=False))
    tok, t0 = 0, time.perf_counter()
    for _ in range(args.steps):
        tok += oracle_round(cfg, lay, logits, np.sort(rng.choice(cfg["B"], s, replace=False)))
    dt = time.perf_counter() - t0
    v = tok / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_json(cfg, {"sample_requests_per_step": s}),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{s} of {cfg['B']} requests per step (lookup + verify), batch pricing",
                             "host": host_cpu()},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm
def make_rounds(S, torch, W, cfg, nbuf):
    """nbuf ChainRounds holding the workload, their logits laid out as the
    device allocation asks (the allocation is run once to learn the layout)."""
    from speculative_decoding_draft_spec_gb300.round import ChainRound

    B, K, L, V = cfg["B"], cfg["K"], cfg["L"], cfg["V"]
    max_rows = B * (L + 1)
    rounds = []
    for _ in range(nbuf):
        rnd = ChainRound(B, cfg["hist"].shape[1], K, L, V, torch.bfloat16, max_rows, cfg["coef"], cfg["n_min"],
                         cfg["n_max"], cfg["copy_cap"])
        rnd.load(cfg["hist"], cfg["hist_len"], cfg["d"], cfg["c"], cfg["d_len"])
        rounds.append(rnd)
    rounds[0].draft_and_price(cfg["lam"], cfg["budget"], cfg["max_verify_len"], cfg["policy"], True)
    torch.cuda.synchronize()
    row_off = rounds[0].row_off.cpu().numpy()
    vlen = rounds[0].verify_len.cpu().numpy()
    n_rows, n_tok = int(row_off[-1]), int(vlen.sum())
    logits = W.compact_logits(cfg, row_off, vlen)
    lt = torch.from_numpy(logits.view(np.int16)).view(torch.bfloat16).to("cuda")
    for rnd in rounds:
        rnd.logits[:n_rows].copy_(lt)
    torch.cuda.synchronize()
    return rounds, n_rows, n_tok, logits


PASS_STEPS = 30  # steps per replay of a pass graph


def step_plan(n, nset, per):
    """How n steps run: (replays of the pass graph, sets of the single-step
    graphs after them).  A pass holds `per` steps (a multiple of nset) on sets
    0, 1, .., so step i runs on set i % nset either way."""
    assert per % nset == 0
    return n // per, [i % nset for i in range(n % per)]


def capture(torch, fn):
    """fn(stream) captured into a CUDA graph, after one run on a side stream."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn(torch.cuda.current_stream())
    return g


def timed_parts(torch, sets, names, steps, warmup, barrier=lambda: None, sampler=None, launches=30):
    """`sets` holds, per input set, one function per component of a step (in
    step order), each taking the stream to launch on.

    The timed region: one CUDA graph holds a pass of about PASS_STEPS steps
    (a whole number of rotations over the sets, step i on set i % len(sets),
    each step's launches in order on one stream, so consecutive steps run back
    to back as they would inside a captured decode step, without a graph
    launch between them), and one more graph holds the steps of `steps` past
    the last whole pass (for steps < PASS_STEPS, all of them).  Each graph
    runs once untimed, then W untimed steps, then `steps` timed steps between
    a barrier and a device synchronisation: whole passes, then the tail graph;
    CUDA events on the launching stream around the region.

    Per-component times: for each component, one graph of `launches`
    back-to-back launches of it, cycling over the sets, replayed after the
    timed region and timed with events around each replay; its mean per
    launch (the kernels' own time, with the device's gap between consecutive
    kernels but without host launch gaps).

    Returns the region's elapsed ms and the mean us per launch of each
    component."""
    import contextlib

    stream = torch.cuda.current_stream()
    nset = len(sets)
    steps_g = [capture(torch, lambda st, fns=fns: [f(st) for f in fns]) for fns in sets]
    per = nset * max(1, PASS_STEPS // nset)
    pass_g = capture(torch, lambda st: [f(st) for i in range(per) for f in sets[i % nset]])
    _, tail = step_plan(steps, nset, per)
    tail_g = capture(torch, lambda st: [f(st) for i in tail for f in sets[i]]) if tail else None

    def run(n, tail_graph=None):
        passes, singles = step_plan(n, nset, per)
        for _ in range(passes):
            pass_g.replay()
        if tail_graph is not None:
            tail_graph.replay()
        else:
            for i in singles:
                steps_g[i].replay()

    # warm-up: every graph the timed region replays runs once first (so no
    # graph upload falls inside it), then the W warm-up steps
    pass_g.replay()
    if tail_g is not None:
        tail_g.replay()
    run(warmup)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with (sampler if sampler is not None else contextlib.nullcontext()):
        t_start.record(stream)
        run(steps, tail_g)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier()
    comp = {}
    reps = 10
    for j, name in enumerate(names):
        g = capture(torch, lambda st, j=j: [sets[i % nset][j](st) for i in range(launches)])
        for _ in range(2):
            g.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        comp[name] = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3 / launches
    return t_start.elapsed_time(t_end), comp


def round_parts(S, torch, cfg, rnd):
    """The two launches of one round on `rnd`'s inputs, as functions of the
    stream: spec_draft_and_price and spec_verify_chain (T = 0)."""
    def draft(stream):
        S.spec_draft_and_price(rnd.hist, rnd.hist_len, rnd.n_min, rnd.n_max, rnd.copy_cap, rnd.g, rnd.g_len,
                               rnd.match_n, rnd.agree, rnd.copy_len, rnd.d, rnd.c, rnd.d_len, rnd.est, cfg["lam"],
                               cfg["budget"], cfg["max_verify_len"], cfg["policy"], True, rnd.chain, rnd.S,
                               rnd.chain_len, rnd.source, rnd.verify_len, rnd.row_off, rnd.point_mass, rnd.ws,
                               stream)

    def verify(stream):
        S.spec_verify_chain(rnd.logits, rnd.row_off, rnd.max_rows, rnd.chain, rnd.verify_len, rnd.out_tokens,
                            rnd.n_accepted, rnd.n_emitted, rnd.ws, point_mass=rnd.point_mass, temperature=0.0,
                            stream=stream)

    return [draft, verify]


def timed_rounds(S, torch, cfg, rounds, steps, warmup, barrier=lambda: None, sampler=None):
    """The chain round (draft + price, verify) timed over graph replays of
    whole passes over the input sets (timed_parts); returns the elapsed ms and
    the mean per-kernel us."""
    sets = [round_parts(S, torch, cfg, rnd) for rnd in rounds]
    return timed_parts(torch, sets, ["draft_price", "verify"], steps, warmup, barrier, sampler)


EDIT_RATES = (0.0, 0.15, 0.30, 0.45, 0.60, 0.70)
BS4_SETS = 10  # rotating input sets: 10 x (19.5 MB of target rows (+ 8.5 MB of draft rows)) > L2


def measure_bs4(S, torch, W, steps, warmup, hbm, rate, probabilistic=False):
    """The batch-4 code-editing configuration with all four requests at one edit
    rate: draft + price, then chain verification of the allocated rows.

    T = 0: greedy drafts (proposed policy).  T = 1 with probabilistic drafting
    (extension policy): the drafter's 7 tokens are sampled on the device from
    its bf16 rows (spec_sample_drafts) before draft + price, and the sampled
    verification (spec_verify_chain_drafted) takes the draft rows' statistics
    from that call instead of reading them again; the sampling step counter is held
    fixed so that every round has the same layout (the work does not depend on
    the drawn values), and verification's Philox step is the input set's
    index.  Same timing as the batch-128 round, over ten rotating input sets.
    Also reports the accepted drafts per round (summed over the batch, mean
    over the sets) and the share of requests whose chain is the n-gram one."""
    from speculative_decoding_draft_spec_gb300.round import ChainRound

    T = 1.0 if probabilistic else 0.0
    cfg = W.edit_bs4(temperature=T, probabilistic=probabilistic, edit_rates=[rate] * 4)
    B, K, L, V = cfg["B"], cfg["K"], cfg["L"], cfg["V"]
    greedy = not probabilistic
    dl = None
    if probabilistic:
        dl = torch.from_numpy(cfg["draft_logits"].view(np.int16)).view(torch.bfloat16).to("cuda")
    rounds = []
    for _ in range(BS4_SETS):
        rnd = ChainRound(B, cfg["hist"].shape[1], K, L, V, torch.bfloat16, B * (L + 1), cfg["coef"], cfg["n_min"],
                         cfg["n_max"], cfg["copy_cap"], with_draft=probabilistic)
        rnd.load(cfg["hist"], cfg["hist_len"], cfg["d"], cfg["c"], cfg["d_len"])
        if probabilistic:
            rnd.draft_logits.copy_(dl)
        rounds.append(rnd)

    def sample(rnd, st):
        S.spec_sample_drafts(rnd.draft_logits, 1.0, rnd.d, rnd.ws, seed=0, step=0, stream=st)

    first = rounds[0]
    if probabilistic:
        sample(first, None)
    first.draft_and_price(cfg["lam"], cfg["budget"], cfg["max_verify_len"], cfg["policy"], greedy)
    torch.cuda.synchronize()
    row_off = first.row_off.cpu().numpy()
    vlen = first.verify_len.cpu().numpy()
    source = first.source.cpu().numpy()
    n_rows, n_tok = int(row_off[-1]), int(vlen.sum())
    lt = torch.from_numpy(W.compact_logits(cfg, row_off, vlen).view(np.int16)).view(torch.bfloat16).to("cuda")
    for rnd in rounds:
        rnd.logits[:n_rows].copy_(lt)
    sets = []
    for k, rnd in enumerate(rounds):
        parts = [lambda st, rnd=rnd: sample(rnd, st)] if probabilistic else []
        parts += [lambda st, rnd=rnd: rnd.draft_and_price(cfg["lam"], cfg["budget"], cfg["max_verify_len"],
                                                          cfg["policy"], greedy, st),
                  lambda st, rnd=rnd, k=k: rnd.verify(temperature=T, seed=0, step=k, stream=st,
                                                      drafted=probabilistic)]
        sets.append(parts)
    names = (["sample_drafts"] if probabilistic else []) + ["draft_price", "verify"]
    ms, comp = timed_parts(torch, sets, names, steps, warmup)
    torch.cuda.synchronize()
    accepted = statistics.mean(int(r.n_accepted.sum().item()) for r in rounds)
    q_rows = 0
    if probabilistic:  # draft rows whose statistics verification reuses: sampled positions within verify_len
        pm = first.point_mass.cpu().numpy()
        q_rows = int(sum(int((pm[r, :min(int(vlen[r]), K)] == 0).sum()) for r in range(B)))
    ver_bytes = n_rows * V * 2  # verification streams the target rows only
    out = {"edit_rate": rate, "value": n_tok * steps / (ms * 1e-3), "unit": UNIT,
           "rows_per_s": n_rows * steps / (ms * 1e-3), "us_per_round": 1e3 * ms / steps, "steps": steps,
           "verified_tokens_per_step": n_tok, "verify_rows_per_step": n_rows, "draft_rows_reused": q_rows,
           "accepted_per_step": accepted, "ngram_chain_share": float(np.isin(source, (1, 2)).mean()),
           "components_us": {k: round(v, 3) for k, v in comp.items()},
           "verify_roofline_frac": round(ver_bytes / (comp["verify"] * 1e-6) / 1e9 / hbm, 4),
           "status_clean": all(int(r.ws.status()) == 0 for r in rounds)}
    wl = f"edit_bs4 {'probabilistic ' if probabilistic else ''}rate {rate:.2f}"
    out["verify_traffic"] = measured_traffic(
        "verify_rows_kernel<bf16, sampled>" if probabilistic else "verify_rows_kernel<bf16, greedy>", wl)
    out["verify_algorithmic_bytes"] = ver_bytes
    if probabilistic:
        out["extension_tail_share"] = float(((source == 3) & (first.chain_len.cpu().numpy() > K)).mean())
        out["sample_drafts_roofline_frac"] = round(B * K * V * 2 / (comp["sample_drafts"] * 1e-6) / 1e9 / hbm, 4)
        out["sample_drafts_traffic"] = measured_traffic("verify_rows_kernel<bf16, drafting>", wl)
        out["resample_traffic"] = measured_traffic("resample_kernel<bf16>", wl)
    del rounds
    return out


def measure_bs4_sweep(S, torch, W, steps, warmup, hbm, probabilistic=False):
    """measure_bs4 at each edit rate of the configuration's sweep."""
    per = [measure_bs4(S, torch, W, steps, warmup, hbm, r, probabilistic) for r in EDIT_RATES]
    T = 1 if probabilistic else 0
    what = ("drafts sampled on the device, extension policy" if probabilistic else "greedy drafts, proposed policy")
    return {"workload": f"edit_bs4: B=4, V=151936 bf16, history 2048, budget 64, lambda 0.04, T={T}, {what}; "
                        "edit rate swept over {0,15,30,45,60,70}% (all four requests at one rate)",
            "by_edit_rate": per, "l2": f"{BS4_SETS} rotating input sets per rate (> L2)"}


def measure_long_sampled(S, torch, W, steps, warmup, hbm):
    """The batch-64 long-context workload: draft + price over 32768-token
    histories (clusters of CTAs per request), then sampled chain verification
    at T = 0.7 over fp32 logits materialised as 16 rows per request; two input
    sets (2 x 622 MB > L2)."""
    from speculative_decoding_draft_spec_gb300.round import ChainRound

    cfg = W.long_bs64()
    B, K, L, V, rows = cfg["B"], cfg["K"], cfg["L"], cfg["V"], cfg["rows_per_request"]
    ro = torch.as_tensor(cfg["row_off_materialised"]).to("cuda")
    logits = torch.from_numpy(W.materialised_logits(cfg)).to("cuda")
    rounds = []
    for k in range(2):
        rnd = ChainRound(B, cfg["hist"].shape[1], K, L, V, torch.float32, B * rows, cfg["coef"], cfg["n_min"],
                         cfg["n_max"], cfg["copy_cap"])
        rnd.load(cfg["hist"], cfg["hist_len"], cfg["d"], cfg["c"], cfg["d_len"])
        rnd.logits.copy_(logits)
        rounds.append(rnd)
    del logits
    stream = torch.cuda.current_stream()

    sets = [[lambda st, rnd=rnd: rnd.draft_and_price(cfg["lam"], cfg["budget"], cfg["max_verify_len"], cfg["policy"],
                                                     True, st),
             lambda st, rnd=rnd, k=k: rnd.verify(temperature=cfg["temperature"], seed=0, step=k, row_off=ro,
                                                 stream=st)]
            for k, rnd in enumerate(rounds)]
    ms, comp = timed_parts(torch, sets, ["draft_price", "verify"], steps, warmup)
    vlen = rounds[0].verify_len.cpu().numpy()
    n_tok = int(vlen.sum())
    n_rows = int((vlen + 1).sum())
    achieved = n_rows * V * 4 / (comp["verify"] * 1e-6) / 1e9
    return {"workload": "long_bs64: B=64, history 32768, n <= 4, budget 512, lambda 0.3, T=0.7, fp32 logits "
                        "materialised as 16 rows per request",
            "value": n_tok * steps / (ms * 1e-3), "unit": UNIT, "rows_per_s": n_rows * steps / (ms * 1e-3),
            "ms_per_step": ms / steps, "steps": steps, "verified_tokens_per_step": n_tok,
            "verify_rows_per_step": n_rows, "components_us": {k: round(v, 3) for k, v in comp.items()},
            "verify_roofline_frac": round(achieved / hbm, 4),
            "verify_algorithmic_bytes": n_rows * V * 4,
            "verify_traffic": measured_traffic("verify_rows_kernel<fp32, sampled>", "long_bs64"),
            "status_clean": all(int(r.ws.status()) == 0 for r in rounds),
            "l2": "2 rotating input sets (2 x 622 MB > L2)"}


def measure_tree(S, torch, W, steps, warmup, hbm, width=16):
    """The tree round, batch 32 trees of `width` rows (bf16 V = 151936): the
    candidate tree built on the device from the drafter's block and the n-gram
    chain (spec_build_tree), then greedy tree verification (spec_verify_tree)
    of logits that plant a true path of mean accept length 3 (capped by the
    tree); enough rotating logit sets to hold over 300 MB (two at width 16,
    eight at width 4), so no step reads rows still in L2."""
    cfg = W.tree_bs32(width=width)
    B, V, n = cfg["B"], cfg["V"], cfg["width"]
    dev = lambda a, dt=None: torch.as_tensor(np.ascontiguousarray(a)).to("cuda") if dt is None else \
        torch.as_tensor(np.ascontiguousarray(a)).to("cuda", dt)
    blk = [dev(cfg[k]) for k in ("anchor", "cand_tok", "cand_score", "ng_tok", "ng_len", "ng_score", "ng_adj")]
    i32 = dict(dtype=torch.int32, device="cuda")
    tok2, par2, cid2 = (torch.empty((B, n), **i32) for _ in range(3))
    nrow = torch.empty(B, **i32)
    ws_b = S.Workspace(B, 1, 1, 1)
    S.spec_build_tree(*blk, n, tok2, par2, cid2, nrow, ws_b)
    torch.cuda.synchronize()
    node_off_h, tok_h, par_h = W.flatten_trees(tok2.cpu().numpy(), par2.cpu().numpy(), nrow.cpu().numpy())
    rows = int(node_off_h[-1])
    logits, _ = W.tree_logits(node_off_h, tok_h, par_h, V)
    lt = torch.from_numpy(logits.view(np.int16)).view(torch.bfloat16).to("cuda")
    nset = max(2, -(-300_000_000 // (rows * V * 2)))
    sets = [lt] + [lt.clone() for _ in range(nset - 1)]
    node_off = dev(node_off_h)
    # the verify reads the builder's rows in place: [B x n] with every tree full
    assert np.all(nrow.cpu().numpy() == n)
    path, out = torch.empty((B, n), **i32), torch.empty((B, n), **i32)
    acc = torch.empty(B, **i32)
    ws = S.Workspace(B, rows, 1, V)
    stream = torch.cuda.current_stream()

    build = lambda st: S.spec_build_tree(*blk, n, tok2, par2, cid2, nrow, ws_b, st)
    sets = [[build, lambda st, lg=lg: S.spec_verify_tree(lg, node_off, rows, tok2, par2, n, path, acc, out, ws, st)]
            for lg in sets]
    ms, comp = timed_parts(torch, sets, ["build", "verify"], steps, warmup)
    accepted = int(acc.sum().item())
    return {"width": n,
            "workload": f"tree_bs32: B=32, block of 8 picks with top-4 candidates plus a 15-token n-gram chain, "
                        f"trees of {n} rows, bf16 V=151936, planted mean accept length 3 (capped by the tree)",
            "tree_rows_per_s": rows * steps / (ms * 1e-3), "accepted_tokens_per_s": accepted * steps / (ms * 1e-3),
            "ms_per_step": ms / steps, "steps": steps, "rows_per_step": rows, "accepted_per_step": accepted,
            "components_us": {k: round(v, 3) for k, v in comp.items()},
            "verify_roofline_frac": round(rows * V * 2 / (comp["verify"] * 1e-6) / 1e9 / hbm, 4),
            "status_clean": int(ws.status()) == 0 and int(ws_b.status()) == 0,
            "l2": f"{nset} rotating logit sets ({nset} x {rows * V * 2 / 1e6:.1f} MB > L2)"}


def measure_tree_widths(S, torch, W, steps, warmup, hbm):
    """measure_tree at each tree width of the configuration (4, 8, 12, 16 rows)."""
    per = [measure_tree(S, torch, W, steps, warmup, hbm, w) for w in (4, 8, 12, 16)]
    top = dict(per[-1])
    top["by_width"] = per
    return top


def measure_tree_fill(S, torch, W, steps, warmup, hbm):
    """The filled tree round, batch 32 (bf16 V = 151936): n-gram chains from the
    anchor and from each of the 8 picks made on the device from the requests'
    4096-token texts (spec_ngram_fill), the candidate tree built from the block
    and the 9 chains per request (spec_build_tree), then greedy tree
    verification of 16 rows per request (spec_verify_tree); two logit sets
    (2 x 156 MB > L2)."""
    cfg = W.tree_fill_bs32(width=16)
    B, V, n, P = cfg["B"], cfg["V"], cfg["width"], cfg["P"]
    dev = lambda a: torch.as_tensor(np.ascontiguousarray(a)).to("cuda")
    hist, hist_len, cand_tok = dev(cfg["hist"]), dev(cfg["hist_len"]), dev(cfg["cand_tok"])
    blk = [dev(cfg[k]) for k in ("anchor", "cand_tok", "cand_score")]
    sc = [dev(cfg[k]) for k in ("ng_score", "ng_adj")]
    i32 = dict(dtype=torch.int32, device="cuda")
    ng_tok, ng_ev = (torch.empty((B, P + 1, cfg["Lg"]), **i32) for _ in range(2))
    ng_len = torch.empty((B, P + 1), **i32)
    tok2, par2, cid2 = (torch.empty((B, n), **i32) for _ in range(3))
    nrow = torch.empty(B, **i32)
    ws_b = S.Workspace(B, 1, 1, 1)

    def fill(st):
        S.spec_ngram_fill(hist, hist_len, cand_tok, cfg["n_min"], cfg["copy_cap"], cfg["max_depth"], ng_tok, ng_len,
                          ng_ev, ws_b, st)

    def build(st):
        S.spec_build_tree(*blk, ng_tok, ng_len, *sc, n, tok2, par2, cid2, nrow, ws_b, st)

    fill(None)
    build(None)
    torch.cuda.synchronize()
    node_off_h, tok_h, par_h = W.flatten_trees(tok2.cpu().numpy(), par2.cpu().numpy(), nrow.cpu().numpy())
    rows = int(node_off_h[-1])
    logits, _ = W.tree_logits(node_off_h, tok_h, par_h, V)
    lt = torch.from_numpy(logits.view(np.int16)).view(torch.bfloat16).to("cuda")
    lsets = [lt, lt.clone()]
    node_off = dev(node_off_h)
    assert np.all(nrow.cpu().numpy() == n)
    path, out = torch.empty((B, n), **i32), torch.empty((B, n), **i32)
    acc = torch.empty(B, **i32)
    ws = S.Workspace(B, rows, 1, V)
    sets = [[fill, build, lambda st, lg=lg: S.spec_verify_tree(lg, node_off, rows, tok2, par2, n, path, acc, out,
                                                                ws, st)]
            for lg in lsets]
    ms, comp = timed_parts(torch, sets, ["fill", "build", "verify"], steps, warmup)
    accepted = int(acc.sum().item())
    chain_tokens = int(ng_len.sum().item())
    return {"workload": "tree_fill_bs32: B=32, 4096-token texts, n-gram chains from the anchor and 8 picks "
                        "(passage copy >= 4 tokens, else the most frequent follower of 3; depth 32), block of 8 "
                        "picks with top-4 candidates, trees of 16 rows, bf16 V=151936",
            "tree_rows_per_s": rows * steps / (ms * 1e-3), "accepted_tokens_per_s": accepted * steps / (ms * 1e-3),
            "ms_per_step": ms / steps, "steps": steps, "rows_per_step": rows, "accepted_per_step": accepted,
            "chain_tokens_per_step": chain_tokens,
            "components_us": {k: round(v, 3) for k, v in comp.items()},
            "verify_roofline_frac": round(rows * V * 2 / (comp["verify"] * 1e-6) / 1e9 / hbm, 4),
            "status_clean": int(ws.status()) == 0 and int(ws_b.status()) == 0,
            "l2": "2 rotating logit sets (2 x 156 MB > L2)"}


def run_gpu(args):
    import torch

    import speculative_decoding_draft_spec_gb300 as S
    import workloads as W

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    S.build()
    cfg = build_workload(rank)
    B, L, V = cfg["B"], cfg["L"], cfg["V"]
    rounds, n_rows, n_tok, logits = make_rounds(S, torch, W, cfg, NBUF)
    kw = dict(lam=cfg["lam"], budget=cfg["budget"], max_verify_len=cfg["max_verify_len"])

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    clk = ClockSampler(local)
    ms, comp = timed_rounds(S, torch, cfg, rounds, args.steps, args.warmup, barrier, clk)
    ms, job_tok, job_rows = reduce_over_ranks(ms, n_tok, n_rows, world, "cuda")
    ok = all(int(r.ws.status()) == 0 for r in rounds)
    if args.legs == "timed":
        if rank == 0:
            print(json.dumps({"legs": "timed", "ms_per_step": ms / args.steps, "components_us": comp,
                              "status_clean": ok}), flush=True)
        return
    stream = torch.cuda.current_stream()

    # end to end through the public API with host buffers: H2D of the step's inputs
    # (histories, drafter chain, confidences, logits) from pinned memory, the round,
    # D2H of the emitted tokens and counts
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    h_hist, h_len, h_d, h_c = pin(cfg["hist"]), pin(cfg["hist_len"]), pin(cfg["d"]), pin(cfg["c"])
    h_logits = torch.from_numpy(logits.view(np.int16)).pin_memory()
    h_out = torch.empty((B, L + 1), dtype=torch.int32).pin_memory()
    h_na = torch.empty(B, dtype=torch.int32).pin_memory()
    e_steps = max(3, min(args.steps, 50))
    rnd = rounds[0]
    h2d = sum(x.numel() * x.element_size() for x in (h_hist, h_len, h_d, h_c, h_logits))
    d2h = h_out.numel() * 4 + h_na.numel() * 4
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for it in range(e_steps + 2):
        if it == 2:
            e0.record(stream)
        rnd.hist.copy_(h_hist, non_blocking=True)
        rnd.hist_len.copy_(h_len, non_blocking=True)
        rnd.d.copy_(h_d, non_blocking=True)
        rnd.c.copy_(h_c, non_blocking=True)
        rnd.logits[:n_rows].view(torch.int16).copy_(h_logits, non_blocking=True)
        rnd.run(**kw)
        h_out.copy_(rnd.out_tokens, non_blocking=True)
        h_na.copy_(rnd.n_accepted, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_over_ranks(e0.elapsed_time(e1) / e_steps, 0, 0, world, "cuda")[0]

    # budget sizing for a later step (spec_size_budget), from this batch's survivals;
    # the pipeline runs it on a side stream, here it is timed alone
    bsz = S.Workspace(1, 1, 1, 1)
    b_out = torch.zeros(1, dtype=torch.int32, device="cuda")
    l_out = torch.zeros(1, dtype=torch.float32, device="cuda")
    _, sz = timed_parts(torch, [[lambda st: S.spec_size_budget(rounds[0].S, rounds[0].chain_len, cfg["max_verify_len"],
                                                              256.0, 1.0, b_out, l_out, bsz, st)]],
                        ["size_budget"], 3, args.warmup)
    sizing = {"us": round(sz["size_budget"], 3),
              "slots": int(np.minimum(rounds[0].chain_len.cpu().numpy(), cfg["max_verify_len"]).sum()),
              "C0": 256.0, "p": 1.0, "b_star": int(b_out.item()), "lambda": float(l_out.item())}

    hbm, peak_kind = peaks()
    bs4 = measure_bs4_sweep(S, torch, W, min(args.steps, 3000), args.warmup, hbm)
    bs4_prob = measure_bs4_sweep(S, torch, W, min(args.steps, 2000), args.warmup, hbm, probabilistic=True)
    long_sampled = measure_long_sampled(S, torch, W, min(args.steps, 1000), args.warmup, hbm)
    tree = measure_tree_widths(S, torch, W, min(args.steps, 2000), args.warmup, hbm)
    tree_fill = measure_tree_fill(S, torch, W, min(args.steps, 2000), args.warmup, hbm)
    if rank != 0:
        return
    verify_us = comp["verify"]
    alg_bytes = n_rows * V * 2
    achieved = alg_bytes / (verify_us * 1e-6) / 1e9
    cpu = cpu_baseline(cfg, oracle_layout(cfg), logits, seconds=args.cpu_seconds) if args.cpu_seconds > 0 else None
    line = {
        "metric": METRIC, "value": job_tok * args.steps / (ms * 1e-3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_json(cfg),
        "rows_per_s": job_rows * args.steps / (ms * 1e-3),
        "verified_tokens_per_step": n_tok, "verify_rows_per_step": n_rows,
        "components_us": {k: round(v, 3) for k, v in comp.items()},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4),
                     "traffic": measured_traffic("verify_rows_kernel<bf16, greedy>", WORKLOAD),
                     "peak_kind": peak_kind,
                     "kernel": "verify_rows_kernel<bf16, greedy>", "algorithmic_bytes": alg_bytes},
        "cpu_baseline": cpu,
        "e2e": {"value": job_tok / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
        "bs4": bs4,
        "bs4_probabilistic": bs4_prob,
        "long_bs64_sampled": long_sampled,
        "tree_bs32": tree,
        "tree_fill_bs32": tree_fill,
        "budget_sizing": sizing,
        "status_clean": ok,
    }
    print(json.dumps(line), flush=True)


def run_once():
    """One launch each of the tree n-gram fill and the tree builder (the
    filled-tree workload: 32 requests, 4096-token texts, chains from the anchor
    and 8 picks, trees of 16 rows) and of draft sampling (batch-4 code editing,
    4 x 7 bf16 draft rows, T = 1), then the chain verifications of
    once_verify_launches, for a profiler."""
    import torch

    import speculative_decoding_draft_spec_gb300 as S
    import workloads as W

    S.build()
    i32 = dict(dtype=torch.int32, device="cuda")
    dev = lambda a: torch.as_tensor(np.ascontiguousarray(a)).cuda()
    c = W.tree_fill_bs32(width=16)
    B, P, Lg = c["B"], c["cand_tok"].shape[1], c["Lg"]
    ws = S.Workspace(B, 1, 1, 1)
    tok, ev = (torch.empty((B, P + 1, Lg), **i32) for _ in range(2))
    ln = torch.empty((B, P + 1), **i32)
    S.spec_ngram_fill(dev(c["hist"]), dev(c["hist_len"]), dev(c["cand_tok"]), c["n_min"], c["copy_cap"],
                      c["max_depth"], tok, ln, ev, ws)
    blk = [dev(c[k]) for k in ("anchor", "cand_tok", "cand_score")] + [tok, ln] + \
          [dev(c[k]) for k in ("ng_score", "ng_adj")]
    tt, tp, tc = (torch.empty((B, 16), **i32) for _ in range(3))
    nr = torch.empty(B, **i32)
    S.spec_build_tree(*blk, 16, tt, tp, tc, nr, ws)
    e = W.edit_bs4(temperature=1.0, probabilistic=True)
    dl = torch.from_numpy(e["draft_logits"].view(np.int16)).view(torch.bfloat16).cuda()
    ws2 = S.Workspace(e["B"], e["B"] * (e["L"] + 1), e["K"], e["V"])
    y = torch.empty((e["B"], e["K"]), **i32)
    S.spec_sample_drafts(dl, 1.0, y, ws2, seed=0, step=0)
    torch.cuda.synchronize()
    ok = int(ws.status()) == 0 and int(ws2.status()) == 0
    rows = once_verify_launches(S, torch, W)
    print(json.dumps({"legs": "once", "tree_rows": int(nr.sum()), "verify_rows": rows, "status_clean": ok}),
          flush=True)


def once_verify_launches(S, torch, W):
    """One chain verification each, after its round's draft + price: batch-4 code
    editing at the 30 % edit rate at T = 0 (bf16 rows), the same at T = 1 with
    drafts sampled on the device (bf16 target rows, the draft rows' statistics
    from the drafting call; the sampled kernel and the max(0, p - q) draw, which
    reads the draft row), and the batch-64 long-context workload
    at T = 0.7 (fp32, 16 rows per request), for a profiler.  Returns the verify
    rows of each."""
    from speculative_decoding_draft_spec_gb300.round import ChainRound

    out = {}
    c = W.edit_bs4(edit_rates=[0.3] * 4)
    rnd = ChainRound(c["B"], c["hist"].shape[1], c["K"], c["L"], c["V"], torch.bfloat16, c["B"] * (c["L"] + 1),
                     c["coef"], c["n_min"], c["n_max"], c["copy_cap"])
    rnd.load(c["hist"], c["hist_len"], c["d"], c["c"], c["d_len"])
    rnd.draft_and_price(c["lam"], c["budget"], c["max_verify_len"], c["policy"], True)
    ro, vl = rnd.row_off.cpu().numpy(), rnd.verify_len.cpu().numpy()
    n = int(ro[-1])
    rnd.logits[:n].copy_(torch.from_numpy(W.compact_logits(c, ro, vl).view(np.int16)).view(torch.bfloat16))
    rnd.verify(temperature=0.0)
    torch.cuda.synchronize()
    out["edit_bs4 rate 0.30"] = n
    c = W.edit_bs4(temperature=1.0, probabilistic=True, edit_rates=[0.3] * 4)
    rnd = ChainRound(c["B"], c["hist"].shape[1], c["K"], c["L"], c["V"], torch.bfloat16, c["B"] * (c["L"] + 1),
                     c["coef"], c["n_min"], c["n_max"], c["copy_cap"], with_draft=True)
    rnd.load(c["hist"], c["hist_len"], c["d"], c["c"], c["d_len"])
    rnd.draft_logits.copy_(torch.from_numpy(c["draft_logits"].view(np.int16)).view(torch.bfloat16))
    S.spec_sample_drafts(rnd.draft_logits, 1.0, rnd.d, rnd.ws, seed=0, step=0)
    rnd.draft_and_price(c["lam"], c["budget"], c["max_verify_len"], c["policy"], False)
    ro, vl = rnd.row_off.cpu().numpy(), rnd.verify_len.cpu().numpy()
    n = int(ro[-1])
    rnd.logits[:n].copy_(torch.from_numpy(W.compact_logits(c, ro, vl).view(np.int16)).view(torch.bfloat16))
    rnd.verify(temperature=1.0, seed=0, step=0, drafted=True)
    torch.cuda.synchronize()
    out["edit_bs4 probabilistic rate 0.30"] = n
    c = W.long_bs64()
    rows = c["rows_per_request"]
    rnd = ChainRound(c["B"], c["hist"].shape[1], c["K"], c["L"], c["V"], torch.float32, c["B"] * rows, c["coef"],
                     c["n_min"], c["n_max"], c["copy_cap"])
    rnd.load(c["hist"], c["hist_len"], c["d"], c["c"], c["d_len"])
    rnd.logits.copy_(torch.from_numpy(W.materialised_logits(c)))
    rnd.draft_and_price(c["lam"], c["budget"], c["max_verify_len"], c["policy"], True)
    rnd.verify(temperature=c["temperature"], seed=0, step=0,
               row_off=torch.as_tensor(c["row_off_materialised"]).cuda())
    torch.cuda.synchronize()
    out["long_bs64"] = int((rnd.verify_len.cpu().numpy() + 1).sum())
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--legs", default="all", choices=["all", "timed", "once"],
                    help="timed: only the warm-up and timed loop; once: one launch each of the tree "
                         "fill, tree builder and draft sampling kernels and of the batch-4 greedy, batch-4 "
                         "sampled and long-context sampled verifications (both for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.legs == "once":
        run_once()
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
