"""Benchmark of the ISD verify-and-propose step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload c64]

One step = isd_verify_propose (every stage of the hot path: the verify
decisions, the correction or bonus draws and the next stride's proposals, one
call of two kernels) over one batch of synthetic logits resident in HBM: C=64
sequences, stride L=8, V=151936, bf16, T=1 by default.  Prints ONE JSON line
(rank 0).  At N=1 the line also carries, measured after the headline in the
same run: the Gumbel-max sampler on the same batch, the other workloads
(greedy, highconc, ragged) and the step under top-k 50 / top-p 0.95
(`configs`), and the oracle's check of a sample of the headline's outputs
(`parity`).

Metric: verified stride-positions per second (sum of L_i per step / step
time); the line also carries logit GB/s against the measured HBM peak.
N > 1 (torchrun, one process per GPU): every rank runs its own replica of the
batch (the step has no cross-GPU exchange), value = all ranks' positions /
max-over-ranks time.

--impl reference times the fp64 CPU oracle (the only other implementation of
this step) on a bounded sample of the same workload, on the host cores.
"""
import argparse
import hashlib
import json

import numpy as np
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC_BASE = "verified stride-positions/sec and logit GB/s (% of B300 HBM peak)"
SUB_STEPS = 200  # timed steps of each sub-record


def metric_for(batch):
    """The metric's name with the workload's batch and vocabulary sizes."""
    return f"{METRIC_BASE}, C={batch.num_seqs} V={batch.vocab}"


UNIT = "positions/s"
REFERENCE_BUDGET_S = 120.0  # seconds for a whole --impl reference run
FALLBACK_HBM_GBS = 6400.0
L2_FLUSH_BYTES = 256 << 20
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c64", choices=["c64", "greedy", "highconc", "ragged"])
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="the workload's recipe at another batch size C (a sweep point; no sub-records)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--separate", action="store_true",
                    help="time isd_verify then isd_propose (two launches) instead of isd_verify_propose")
    ap.add_argument("--row", choices=["step", "kv", "filtered"], default="step",
                    help="kv: time the KV-slot commit of the stationary batch (isd_kv_commit); "
                         "filtered: time the step under top-k 50 / top-p 0.95 (isd_verify_filtered + "
                         "isd_propose_filtered)")
    return ap.parse_args()


def workload_config(batch, extra):
    Ls = batch.strides()
    cfg = {"workload": f"{batch.name}: {batch.meta['description']}", "num_seqs": batch.num_seqs,
           "sum_stride": int(sum(Ls)), "vocab": batch.vocab,
           "logits": str(batch.dtype).replace("torch.", ""), "seed": batch.seed, "offset": batch.offset,
           "data_seed": batch.meta["data_seed"]}
    cfg.update(extra)
    return cfg


def algorithmic_bytes(batch, accept_len, valid):
    """Logit bytes the step must read: for every sequence its p_k and q_k rows
    (k <= L_i; greedy sequences read no q), the final anchor row where every
    proposal was accepted, and the qnew rows of sequences whose proposals are
    drawn.  The re-read of a rejected row pair is not counted."""
    esz = 2 if str(batch.dtype).endswith("bfloat16") else 4
    row = esz * batch.vocab
    Ls = batch.strides()
    temps = batch.temperature.cpu().tolist()
    verify = propose = 0
    for i, L in enumerate(Ls):
        a = int(accept_len[i])
        per = L if temps[i] == 0.0 else 2 * L
        verify += row * (per + (1 if a == L else 0))
        if int(valid[i]):
            propose += row * L
    return verify, propose


def accepted_share(batch, accept_len):
    """Accepted proposals over verified ones in this batch: the share of
    positions on the common acceptance path (the pages report about 78 % on
    their serving runs; here it is a property of the synthetic logits)."""
    Ls = batch.strides()
    total = sum(Ls)
    return sum(max(0, int(a)) for a in accept_len) / total if total else 0.0


def reread_bytes(batch, accept_len):
    """Bytes of the rejected row pairs the correction reads a second time
    (p_j and q_j of every T > 0 sequence that rejects), reported beside the
    algorithmic bytes, not in them: they should come from L2."""
    esz = 2 if str(batch.dtype).endswith("bfloat16") else 4
    temps = batch.temperature.cpu().tolist()
    rejecting = sum(1 for i, L in enumerate(batch.strides()) if temps[i] > 0 and 0 <= int(accept_len[i]) < L)
    return 2 * rejecting * batch.vocab * esz


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank runs: what the compiler sees."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":  # string or character literal, copied whole
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
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


# The sources that build and launch the verify kernel: its translation unit,
# the host file that sizes its grid, workspace and cache policy, and the
# local headers they include.  Profiled DRAM counters stay valid while these
# are unchanged.
PROFILED_SOURCES = ("isd_verify.cu", "isd_api.cu")


def profiled_source_files():
    """PROFILED_SOURCES and the local headers they include, recursively."""
    csrc = os.path.join(ROOT, "speculative_verify_accept_02_b300", "csrc")
    seen = []

    def visit(path):
        path = os.path.normpath(path)
        if path in seen:
            return
        seen.append(path)
        with open(path, encoding="utf-8") as f:
            text = f.read()
        for inc in re.findall(r'^[ \t]*#[ \t]*include[ \t]+"([^"]+)"', text, re.M):
            visit(os.path.join(os.path.dirname(path), inc))

    for name in PROFILED_SOURCES:
        visit(os.path.join(csrc, name))
    return sorted(seen)


def kernel_source_hash():
    """Hash of the code (comments and blank lines ignored) of the files that
    build and launch the verify kernel."""
    h = hashlib.sha256()
    for path in profiled_source_files():
        with open(path, encoding="utf-8") as f:
            h.update(os.path.relpath(path, ROOT).encode() + _strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per isd_verify call from the committed ncu summary, if it was
    taken on the current kernel sources; else None."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    entry = t.get(workload)
    if not entry or entry.get("source_hash") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_verify")


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons while running."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index):
        import torch
        self.proc = None
        self.lines = []
        try:
            ident = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = ident if ident.startswith("GPU-") else f"GPU-{ident}"
        except Exception:
            ident = str(device_index)
        self.cmd = ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
                    "-lms", "200", "-i", ident]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(self.REASONS, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# The fp64 oracle as it stands (CPU baseline, reference arm)
# ---------------------------------------------------------------------------

def _host_inputs(batch):
    from speculative_verify_accept_02_b300 import workloads
    return dict(p=workloads.host_logits(batch.p), q=workloads.host_logits(batch.q),
                qnew=workloads.host_logits(batch.qnew), tokens=batch.tokens.cpu().numpy(),
                offs=batch.seq_offsets.cpu().numpy(), temp=batch.temperature.cpu().numpy())


def _oracle_step(h, batch, seqs, nthreads=0):
    import oracle
    v = oracle.verify(h["p"], h["q"], batch.vocab, h["tokens"], h["offs"], h["temp"], batch.seed,
                      batch.offset, seqs=seqs, nthreads=nthreads)
    oracle.propose(h["qnew"], batch.vocab, h["offs"], h["temp"], batch.seed, batch.offset,
                   accept_len=v["accept_len"], seqs=seqs, nthreads=nthreads)


def _oracle_filtered_step(h, batch, seqs, nthreads=0):
    """The oracle's filtered step (top-k 50, top-p 0.95) on the whole sub-batch
    (its filtered functions take every sequence)."""
    import oracle
    tp = float(np.float32(FILTER_TOP_P))
    v = oracle.verify_filtered(h["p"], h["q"], batch.vocab, h["tokens"], h["offs"], h["temp"], batch.seed,
                               batch.offset, FILTER_TOP_K, tp)
    oracle.propose_filtered(h["qnew"], batch.vocab, h["offs"], h["temp"], batch.seed, batch.offset,
                            FILTER_TOP_K, tp, accept_len=v["accept_len"])


def time_oracle(batch, seconds, nthreads=0, seqs=None):
    """oracle verify+propose on the batch (or the sequences `seqs`), repeated
    for about `seconds`, on `nthreads` threads (0: all the host's)."""
    import oracle
    h = _host_inputs(batch)
    seqs = list(range(batch.num_seqs)) if seqs is None else list(seqs)
    Ls = batch.strides()
    positions = sum(Ls[i] for i in seqs)
    before = oracle.threads()
    reps = 0
    t0 = time.perf_counter()
    while True:
        _oracle_step(h, batch, seqs, nthreads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    used = oracle.threads(nthreads)
    if nthreads:  # the thread count sticks: put the earlier one back (an empty call sets it)
        oracle.verify(np.zeros((1, 1), np.float32), np.zeros((1, 1), np.float32), 1, np.zeros(0, np.int32),
                      np.zeros(1, np.int32), np.zeros(0, np.float32), 0, 0, nthreads=before)
    return positions * reps / el, used, reps, el, positions


def _sample_batch(batch, seqs, kp):
    """A sub-batch of the workload: sequences `seqs`, each cut to its first kp
    positions (a shorter stride; its anchor rows p_1..p_{kp+1} are the
    sequence's own)."""
    import torch
    from speculative_verify_accept_02_b300 import workloads
    o = batch.seq_offsets.tolist()
    prow, qrow, Ls = [], [], []
    for i in seqs:
        L = min(kp, o[i + 1] - o[i])
        prow += [o[i] + i + k for k in range(L + 1)]
        qrow += [o[i] + k for k in range(L)]
        Ls.append(L)
    offs = torch.tensor([0] + list(np.cumsum(Ls)), dtype=torch.int32)
    sub = workloads.Batch(batch.name, batch.vocab, batch.ld, batch.dtype, offs, batch.temperature[seqs].clone(),
                          batch.tokens[qrow].clone(), batch.p[prow].clone(), batch.q[qrow].clone(),
                          batch.qnew[qrow].clone(), batch.seed, batch.offset, dict(batch.meta))
    return sub, sum(Ls)


def run_reference_kv(args):
    """The oracle's KV commit on the --row kv workload (C=64 sequences,
    stride 8, accept lengths uniform on 0..7), timed per commit on the host."""
    import oracle
    from speculative_verify_accept_02_b300 import workloads
    C, M = KV_NUM_SEQS, KV_MASKS
    W, K = max(3, args.warmup), args.steps
    n = W + K
    ld = n * (M + 1) + 2 * M + 2
    state = workloads.make_kv_state(C, ld, C * ld, 0, seed=7)
    accept = np.random.default_rng(7).integers(0, M + 1, (n, C)).astype(np.int32)
    for j in range(W):
        oracle.kv_commit(state, accept[j], M)
    t0 = time.perf_counter()
    refused = sum(1 for j in range(W, n) if oracle.kv_commit(state, accept[j], M) != 0)
    us = 1e6 * (time.perf_counter() - t0) / K
    desc = f"every commit of the stationary batch ({C} sequences, {M} masks), one thread"
    line = {"impl": "reference", "metric": f"KV-slot commits/sec (isd_kv_commit), C={C} stride {M + 1}",
            "value": 1e6 / us, "unit": "commits/s", "n_gpus": args.gpus, "steps": K, "warmup": W,
            "ms_per_step": us / 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int32", "data": "synthetic",
            "config": {"workload": f"stationary batch of {C} sequences, {M} masks, accept lengths uniform on 0..{M}",
                       "refused_commits": refused, "sample": desc},
            "cpu_baseline": {"value": 1e6 / us, "unit": "commits/s", "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": 1e6 / us, "unit": "commits/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return  # the oracle runs once, on rank 0
    if args.row == "kv":
        run_reference_kv(args)
        return
    import oracle
    from speculative_verify_accept_02_b300 import workloads
    filtered = args.row == "filtered"
    stepper = _oracle_filtered_step if filtered else _oracle_step
    batch = workloads.make(args.workload, device="cpu", num_seqs=args.num_seqs)
    # The sample per step is sized so that the whole run (warm-up and timed
    # steps) takes about REFERENCE_BUDGET_S: up to 8 whole sequences, or one
    # sequence cut to fewer positions when a whole one is already too slow.
    one, _ = _sample_batch(batch, [0], 1 << 30)
    h1 = _host_inputs(one)
    t0 = time.perf_counter()
    stepper(h1, one, [0])
    t_seq = time.perf_counter() - t0
    t_step = REFERENCE_BUDGET_S / max(1, args.steps + args.warmup)
    L0 = batch.strides()[0]
    if t_seq <= t_step:
        ns = int(min(8, max(1, t_step // t_seq)))
        seqs = list(range(0, batch.num_seqs, max(1, batch.num_seqs // ns)))[:ns]
        kp = 1 << 30
    else:
        seqs = [0]
        kp = max(1, int(L0 * t_step / t_seq))
    sub, positions = _sample_batch(batch, seqs, kp)
    h = _host_inputs(sub)
    idx = list(range(len(seqs)))
    for _ in range(args.warmup):
        stepper(h, sub, idx)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        stepper(h, sub, idx)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = positions / (ms / 1e3)
    desc = (f"{len(seqs)} of {batch.num_seqs} sequences" + (f", cut to {kp} positions" if kp < L0 else "")
            + f" ({positions} positions) per step, "
            + (f"verify+propose under top-k {FILTER_TOP_K} / top-p {FILTER_TOP_P}" if filtered else "verify+propose"))
    metric = (f"verified stride-positions/sec under top-k {FILTER_TOP_K} / top-p {FILTER_TOP_P}, "
              f"C={batch.num_seqs} V={batch.vocab}") if filtered else metric_for(batch)
    line = {"impl": "reference", "metric": metric, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(batch, {"sample": desc}),
            # the filtered oracle runs row by row on one thread
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1 if filtered else oracle.threads(),
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# The CUDA path
# ---------------------------------------------------------------------------

def slowest_rank(ms, device, distributed):
    """The job's time: the largest of the ranks' times (one all-reduce)."""
    import torch
    if not distributed:
        return float(ms)
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(positions_per_rank, world, steps, ms):
    """Whole-job positions per second: every replica verifies its own batch."""
    return positions_per_rank * world * steps / (ms / 1e3)


def time_calls(call, flush, stream, K):
    """K calls, each bracketed by its own events on `stream`, the L2 flushed
    before each outside them: the calls' durations in ms."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def sub_record(batch, ms, kernel_bytes, peak, accept_len=None):
    """One workload's figures: step time, positions per second, the step's
    algorithmic logit bytes over its average duration against the peak."""
    avg_s = sum(ms) / len(ms) / 1e3
    rec = {"workload": f"{batch.name}: {batch.meta['description']}", "step_us": 1e3 * statistics.median(ms),
           "step_us_best": 1e3 * min(ms), "positions_per_s": batch.total / avg_s,
           "roofline": {"achieved_gbs": kernel_bytes / avg_s / 1e9, "frac": kernel_bytes / avg_s / 1e9 / peak,
                        "algorithmic_bytes": kernel_bytes},
           "steps": len(ms)}
    if accept_len is not None:
        rec["accepted_share"] = accepted_share(batch, accept_len)
    return rec


def fused_sub_records(dev, stream, flush, peak, K, head_batch):
    """The Gumbel-max sampler on the headline batch, then the other workloads
    through the same fused call (inverse-CDF draws), each timed as the
    headline (K steps, L2 flushed between them)."""
    import torch
    from speculative_verify_accept_02_b300 import isd_verify_propose, isd_verify_propose_workspace_bytes, workloads
    from speculative_verify_accept_02_b300.api import workspace
    out = {}
    for key, name, sampler in (("gumbel", None, "gumbel"), ("greedy", "greedy", "icdf"),
                               ("highconc", "highconc", "icdf"), ("ragged", "ragged", "icdf")):
        b = head_batch if name is None else workloads.make(name, device=dev)
        ws = workspace(isd_verify_propose_workspace_bytes(b.num_seqs, b.total, b.vocab, b.dtype), dev)
        res = {}

        def call():
            res["out"] = isd_verify_propose(b.p, b.q, b.tokens, b.qnew, b.seq_offsets, b.temperature, b.seed,
                                            b.offset, vocab=b.vocab, total=b.total, ws=ws, stream=stream,
                                            sampler=sampler)
        for _ in range(3):
            call()
        torch.cuda.synchronize(dev)
        v, pr = res["out"]
        acc = v.accept_len.cpu().tolist()
        vb, pb = algorithmic_bytes(b, acc, pr.valid.cpu().tolist())
        rec = sub_record(b, time_calls(call, flush, stream, K), vb + pb, peak, acc)
        rec["step"] = f"isd_verify_propose ({'Gumbel-max' if sampler == 'gumbel' else 'inverse-CDF'} draws)"
        out[key] = rec
        del b, ws, res
        torch.cuda.empty_cache()
    return out


def filtered_sub_record(dev, stream, flush, peak, K, batch):
    """The step under top-k 50 / top-p 0.95 on the headline batch:
    isd_verify_filtered then isd_propose_filtered; the roofline is the verify
    call's (every p and q row streamed once)."""
    import torch
    from speculative_verify_accept_02_b300 import (isd_propose_filtered, isd_propose_filtered_workspace_bytes,
                                                   isd_verify_filtered, isd_verify_filtered_workspace_bytes)
    from speculative_verify_accept_02_b300.api import workspace
    C, total, V = batch.num_seqs, batch.total, batch.vocab
    k, tp = FILTER_TOP_K, FILTER_TOP_P
    vws = workspace(isd_verify_filtered_workspace_bytes(C, total, k), dev)
    pws = workspace(isd_propose_filtered_workspace_bytes(C, total, k), dev)
    res = {}

    def verify():
        res["v"] = isd_verify_filtered(batch.p, batch.q, batch.tokens, batch.seq_offsets, batch.temperature,
                                       batch.seed, batch.offset, top_k=k, top_p=tp, vocab=V, total=total, ws=vws,
                                       stream=stream)

    def step():
        verify()
        isd_propose_filtered(batch.qnew, batch.seq_offsets, batch.temperature, batch.seed, batch.offset,
                             res["v"].accept_len, top_k=k, top_p=tp, vocab=V, total=total, ws=pws, stream=stream)
    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    acc = res["v"].accept_len.cpu().tolist()
    vbytes = filtered_verify_bytes(batch)
    rec = sub_record(batch, time_calls(step, flush, stream, K), vbytes, peak, acc)
    vms = time_calls(verify, flush, stream, K)
    avg_s = sum(vms) / len(vms) / 1e3
    rec["roofline"] = {"achieved_gbs": vbytes / avg_s / 1e9, "frac": vbytes / avg_s / 1e9 / peak,
                       "algorithmic_bytes": vbytes, "kernel": "isd_verify_filtered (top-k lists, then decisions)",
                       "avg_launch_us": avg_s * 1e6}
    rec["step"] = f"isd_verify_filtered + isd_propose_filtered, top-k {k}, top-p {tp}"
    return rec


def oracle_parity(batch, vout, pout):
    """The oracle's check of a sample of the headline's outputs (the first
    sequence, the last four and eight at random), by the comparison the GPU
    tests make: the counts of compared sequences and exempted decisions."""
    import oracle
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from parity import Report, compare_propose, compare_verify
    h = _host_inputs(batch)
    C = batch.num_seqs
    rng = np.random.default_rng(11)
    seqs = sorted(set([0] + list(range(max(0, C - 4), C)) + list(rng.choice(C, size=min(C, 8), replace=False))))
    gv = dict(accept_len=vout.accept_len.cpu().numpy(), out_tokens=vout.out_tokens.cpu().numpy(),
              ratio=vout.ratio.cpu().numpy(), alpha=vout.alpha.cpu().numpy())
    gp = dict(proposals=pout.proposals.cpu().numpy(), valid=pout.valid.cpu().numpy())
    ov = oracle.verify(h["p"], h["q"], batch.vocab, h["tokens"], h["offs"], h["temp"], batch.seed, batch.offset,
                       seqs=seqs)
    rep = compare_verify(ov, gv, h["offs"], seqs=seqs, report=Report())
    agree = [i for i in seqs if ov["accept_len"][i] == gv["accept_len"][i]]
    op = oracle.propose(h["qnew"], batch.vocab, h["offs"], h["temp"], batch.seed, batch.offset,
                        accept_len=gv["accept_len"], seqs=agree)
    compare_propose(op, gp, h["offs"], seqs=agree, report=rep)
    out = {k: v for k, v in rep.summary().items() if k != "cut_skips"}
    out["failures"] = len(rep.failures)
    out["sample"] = [int(i) for i in seqs]
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    from speculative_verify_accept_02_b300 import (_lib, build, isd_propose, isd_propose_workspace_bytes,
                                                   isd_verify, isd_verify_propose,
                                                   isd_verify_propose_workspace_bytes, isd_verify_workspace_bytes,
                                                   workloads)
    from speculative_verify_accept_02_b300.api import ProposeOut, VerifyOut, workspace

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    distributed = world > 1
    dev = torch.device("cuda", local if distributed else 0)
    torch.cuda.set_device(dev)
    if distributed:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        build.build()
    if distributed:
        dist.barrier()
    _lib.load()

    batch = workloads.make(args.workload, device=dev, num_seqs=args.num_seqs)
    C, total, V = batch.num_seqs, batch.total, batch.vocab
    i32, f32 = torch.int32, torch.float32
    vout = VerifyOut(torch.empty(C, dtype=i32, device=dev), torch.empty(total + C, dtype=i32, device=dev),
                     torch.empty(total, dtype=f32, device=dev), torch.empty(C, dtype=f32, device=dev))
    pout = ProposeOut(torch.empty(total, dtype=i32, device=dev), torch.empty(C, dtype=torch.uint8, device=dev))
    vws = workspace(isd_verify_workspace_bytes(C, total, V, batch.dtype), dev)
    pws = workspace(isd_propose_workspace_bytes(C, total, V, batch.dtype), dev)
    fws = workspace(isd_verify_propose_workspace_bytes(C, total, V, batch.dtype), dev)
    fused = not args.separate
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def verify(b):
        isd_verify(b["p"], b["q"], b["tokens"], b["seq_offsets"], b["temperature"], batch.seed, batch.offset,
                   vocab=V, total=total, out=vout, ws=vws, stream=stream)

    def propose(b):
        isd_propose(b["qnew"], b["seq_offsets"], b["temperature"], batch.seed, batch.offset,
                    accept_len=vout.accept_len, vocab=V, total=total, out=pout, ws=pws, stream=stream)

    def step(b):
        """One step: the fused call (one launch), or the two calls."""
        if fused:
            isd_verify_propose(b["p"], b["q"], b["tokens"], b["qnew"], b["seq_offsets"], b["temperature"],
                               batch.seed, batch.offset, vocab=V, total=total, out=vout, pout=pout, ws=fws,
                               stream=stream)
        else:
            verify(b)
            propose(b)

    names = ("p", "q", "qnew", "tokens", "seq_offsets", "temperature")
    resident = {n: getattr(batch, n) for n in names}
    for _ in range(max(3, args.warmup)):
        step(resident)
    torch.cuda.synchronize(dev)
    acc_host = vout.accept_len.cpu().tolist()
    vbytes, pbytes = algorithmic_bytes(batch, acc_host, pout.valid.cpu().tolist())
    rbytes = reread_bytes(batch, acc_host)

    # Timed region: K steps, each bracketed by its own events; the L2 flush
    # between steps lies outside them.
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(dev.index)
    if distributed:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with sampler:
        t_wall = time.perf_counter()
        for k in range(K):
            flush.zero_()
            ev[k][0].record(stream)
            if fused:
                step(resident)
                ev[k][1].record(stream)
            else:
                verify(resident)
                ev[k][1].record(stream)
                propose(resident)
            ev[k][2].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    if distributed:
        dist.barrier()
    per_step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    step_ms = sum(per_step_ms)
    verify_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    total_ms = slowest_rank(step_ms, dev, distributed)
    ms_per_step = total_ms / K
    value = job_throughput(total, world, K, total_ms)
    logit_gbs = (vbytes + pbytes) * world * K / (total_ms / 1e3) / 1e9
    peak, peak_kind = load_peaks()
    verify_avg_s = verify_ms / K / 1e3
    # The roofline kernel is the verify kernel; fused, it also streams the
    # qnew rows it draws proposals from.
    kernel_bytes = vbytes + (pbytes if fused else 0)
    achieved = kernel_bytes / verify_avg_s / 1e9

    # End to end through the public API: every step copies its inputs from
    # pinned host memory, runs, and reads every result back.
    host_in = {n: resident[n].cpu().pin_memory() for n in names}
    dev_in = {n: torch.empty_like(resident[n]) for n in names}
    results = (vout.accept_len, vout.out_tokens, vout.ratio, vout.alpha, pout.proposals, pout.valid)
    host_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in results]
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = sum(x.numel() * x.element_size() for x in host_out)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.e2e_steps)]
    for k in range(args.e2e_steps):
        e2e_ev[k][0].record(stream)
        for n in names:
            dev_in[n].copy_(host_in[n], non_blocking=True)
        step(dev_in)
        for hbuf, dbuf in zip(host_out, results):
            hbuf.copy_(dbuf, non_blocking=True)
        e2e_ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e_ev) / args.e2e_steps
    e2e_value = job_throughput(total, world, 1, slowest_rank(e2e_ms, dev, distributed))

    if rank != 0:
        dist.destroy_process_group()
        return
    configs = None
    if not distributed and fused and args.workload == "c64" and args.num_seqs is None:
        # The other figures of the record, after the headline: the Gumbel-max
        # sampler, the other workloads, the filtered step.
        sub_k = min(K, SUB_STEPS)
        configs = fused_sub_records(dev, stream, flush, peak, sub_k, batch)
        configs["filtered"] = filtered_sub_record(dev, stream, flush, peak, sub_k, batch)
    cpu = None
    parity = None
    if not distributed:  # the CPU baseline is taken at N=1 only
        rate, threads, reps, el, pos = time_oracle(batch, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"full batch ({pos} positions) verify+propose, {reps} repetition(s) in {el:.1f} s"}
        # the same oracle on one core, on the batch's first sequences (a bounded sample)
        one = list(range(min(batch.num_seqs, max(1, threads))))
        rate1, _, reps1, el1, pos1 = time_oracle(batch, args.cpu_seconds, nthreads=1, seqs=one)
        cpu["single_core"] = {"value": rate1, "unit": UNIT, "cores": 1,
                              "sample": f"{len(one)} sequences ({pos1} positions) verify+propose, "
                                        f"{reps1} repetition(s) in {el1:.1f} s"}
        # the same oracle checks a sample of the headline's outputs (the timed
        # steps' inputs, seed and offset)
        parity = oracle_parity(batch, vout, pout)
    line = {
        "metric": metric_for(batch), "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": workload_config(batch, {
            "l2": f"flushed by a {L2_FLUSH_BYTES >> 20} MiB write between timed steps",
            "parallelism": f"replicas x{world}", "step": "isd_verify_propose (one call: stream kernel, draw kernel)" if fused else "isd_verify + isd_propose",
            "accepted_share": accepted_share(batch, acc_host)}),
        "logit_gbs": logit_gbs, "hbm_frac": logit_gbs / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": profiled_traffic(args.workload),
                     "kernel": ("isd_verify_propose: stream_kernel, then draw_kernel launched behind it"
                                if fused else "isd_verify: stream_kernel, then draw_kernel launched behind it"),
                     "algorithmic_bytes": kernel_bytes, "reread_bytes": rbytes,
                     "peak_source": f"{peak_kind} hbm_gbs", "avg_launch_us": verify_avg_s * 1e6},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "step_us": {"median": 1e3 * statistics.median(per_step_ms), "best": 1e3 * min(per_step_ms)},
        "gpu_launches": (2 if fused else 3) * K,  # stream + draw kernels (+ propose_kernel) per step
        "configs": configs,
        "parity": parity,
        "clocks": sampler.summary(),
        "wall_s_timed": t_wall,
    }
    print(json.dumps(line), flush=True)
    if distributed:
        dist.destroy_process_group()


KV_NUM_SEQS, KV_MASKS = 64, 7


def run_kv(args):
    """Commits per second of isd_kv_commit on a stationary batch of C=64
    sequences at stride 8 (M=7 masks), one launch per commit.  Each commit
    takes a fresh accept length per sequence, uniform on 0..7 (read only
    where proposals are pending); the state evolves as in a decode run.
    The floor is the same kernel on an empty batch (launch and one pass of
    its checks): the commit cannot be faster."""
    import torch
    from speculative_verify_accept_02_b300 import _lib, build, isd_kv_commit, workloads
    if int(os.environ.get("RANK", "0")) != 0:
        return
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    _lib.load()
    C, M = KV_NUM_SEQS, KV_MASKS
    K, W, E = args.steps, max(3, args.warmup), args.e2e_steps
    n = K + W + E
    ld = n * (M + 1) + 2 * M + 2
    state = workloads.make_kv_state(C, ld, C * ld, 0, seed=7).to_torch(dev)
    rng = np.random.default_rng(7)
    accept = torch.from_numpy(rng.integers(0, M + 1, (n, C)).astype(np.int32)).to(dev)
    status = torch.empty(n, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for j in range(W):
        isd_kv_commit(state, accept[j], M, status=status[j:j + 1], stream=stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(dev.index)
    torch.cuda.synchronize(dev)
    with sampler:
        for k in range(K):
            flush.zero_()
            ev[k][0].record(stream)
            isd_kv_commit(state, accept[W + k], M, status=status[W + k:W + k + 1], stream=stream)
            ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
    us = 1e3 * sum(a.elapsed_time(b) for a, b in ev) / K
    # e2e: the step's accept lengths come from the host, the status goes back
    host_acc = accept[W + K:].cpu().pin_memory()
    host_status = torch.empty(1, dtype=torch.int32, pin_memory=True)
    dev_acc = torch.empty(C, dtype=torch.int32, device=dev)
    e2e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(E)]
    for k in range(E):
        e2e[k][0].record(stream)
        dev_acc.copy_(host_acc[k], non_blocking=True)
        isd_kv_commit(state, dev_acc, M, status=status[W + K + k:W + K + k + 1], stream=stream)
        host_status.copy_(status[W + K + k:W + K + k + 1], non_blocking=True)
        e2e[k][1].record(stream)
    torch.cuda.synchronize(dev)
    e2e_us = 1e3 * sum(a.elapsed_time(b) for a, b in e2e) / max(1, E)
    refused = int((status != 0).sum().item())
    # floor: the same kernel on an empty batch
    empty = workloads.make_kv_state(0, 1, 1, [], seed=0).to_torch(dev)
    none = torch.empty(0, dtype=torch.int32, device=dev)
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for k in range(K):
        flush.zero_()
        fev[k][0].record(stream)
        isd_kv_commit(empty, none, M, status=status[:1], stream=stream)
        fev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    floor_us = 1e3 * sum(a.elapsed_time(b) for a, b in fev) / K
    line = {
        "metric": f"KV-slot commits/sec (isd_kv_commit), C={C} stride {M + 1}", "value": 1e6 / us,
        "unit": "commits/s", "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": us / 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": f"stationary batch of {C} sequences, {M} masks, accept lengths uniform on 0..{M}",
                   "l2": f"flushed by a {L2_FLUSH_BYTES >> 20} MiB write between timed commits",
                   "refused_commits": refused},
        "floor": {"kind": "the same kernel on an empty batch", "us": floor_us, "frac": floor_us / us},
        "e2e": {"value": 1e6 / e2e_us, "unit": "commits/s", "h2d_bytes_per_step": C * 4, "d2h_bytes_per_step": 4},
        "gpu_launches": K,
        "clocks": sampler.summary(),
    }
    print(json.dumps(line), flush=True)


FILTER_TOP_K, FILTER_TOP_P = 50, 0.95


def filtered_verify_bytes(batch):
    """Logit bytes isd_verify_filtered must read: every p row (sum L + C)
    and every q row (sum L), once each."""
    esz = 2 if str(batch.dtype).endswith("bfloat16") else 4
    return (2 * batch.total + batch.num_seqs) * batch.vocab * esz


def run_filtered(args):
    """Positions per second of the step under the evaluation setting's
    filters (top-k 50, top-p 0.95) on the bench workload: isd_verify_filtered
    then isd_propose_filtered with its accept lengths, L2 flushed between
    steps.  The roofline is the verify call's: every p and q row is streamed
    once by its top-k kernel."""
    import torch
    from speculative_verify_accept_02_b300 import (_lib, build, isd_propose_filtered,
                                                   isd_propose_filtered_workspace_bytes, isd_verify_filtered,
                                                   isd_verify_filtered_workspace_bytes, workloads)
    from speculative_verify_accept_02_b300.api import ProposeOut, VerifyOut, workspace
    if int(os.environ.get("RANK", "0")) != 0:
        return
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    _lib.load()
    batch = workloads.make(args.workload, device=dev, num_seqs=args.num_seqs)
    C, total, V = batch.num_seqs, batch.total, batch.vocab
    k, tp = FILTER_TOP_K, FILTER_TOP_P
    i32, f32 = torch.int32, torch.float32
    vout = VerifyOut(torch.empty(C, dtype=i32, device=dev), torch.empty(total + C, dtype=i32, device=dev),
                     torch.empty(total, dtype=f32, device=dev), torch.empty(C, dtype=f32, device=dev))
    pout = ProposeOut(torch.empty(total, dtype=i32, device=dev), torch.empty(C, dtype=torch.uint8, device=dev))
    vws = workspace(isd_verify_filtered_workspace_bytes(C, total, k), dev)
    pws = workspace(isd_propose_filtered_workspace_bytes(C, total, k), dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def verify(b):
        isd_verify_filtered(b["p"], b["q"], b["tokens"], b["seq_offsets"], b["temperature"], batch.seed,
                            batch.offset, top_k=k, top_p=tp, vocab=V, total=total, out=vout, ws=vws, stream=stream)

    def propose(b):
        isd_propose_filtered(b["qnew"], b["seq_offsets"], b["temperature"], batch.seed, batch.offset,
                             vout.accept_len, top_k=k, top_p=tp, vocab=V, total=total, out=pout, ws=pws,
                             stream=stream)

    names = ("p", "q", "qnew", "tokens", "seq_offsets", "temperature")
    resident = {n: getattr(batch, n) for n in names}
    W, K = max(3, args.warmup), args.steps
    for _ in range(W):
        verify(resident)
        propose(resident)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(dev.index)
    torch.cuda.synchronize(dev)
    with sampler:
        for j in range(K):
            flush.zero_()
            ev[j][0].record(stream)
            verify(resident)
            ev[j][1].record(stream)
            propose(resident)
            ev[j][2].record(stream)
        torch.cuda.synchronize(dev)
    step_ms = sum(e[0].elapsed_time(e[2]) for e in ev) / K
    verify_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    verify_bytes = filtered_verify_bytes(batch)
    peak, peak_kind = load_peaks()
    achieved = verify_bytes / (verify_ms / 1e3) / 1e9
    # e2e: inputs from pinned host memory, every result read back
    host_in = {n: resident[n].cpu().pin_memory() for n in names}
    dev_in = {n: torch.empty_like(resident[n]) for n in names}
    results = (vout.accept_len, vout.out_tokens, vout.ratio, vout.alpha, pout.proposals, pout.valid)
    host_out = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in results]
    E = max(1, args.e2e_steps)
    e2e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(E)]
    for j in range(E):
        e2e[j][0].record(stream)
        for n in names:
            dev_in[n].copy_(host_in[n], non_blocking=True)
        verify(dev_in)
        propose(dev_in)
        for hbuf, dbuf in zip(host_out, results):
            hbuf.copy_(dbuf, non_blocking=True)
        e2e[j][1].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e) / E
    line = {
        "metric": f"verified stride-positions/sec under top-k {k} / top-p {tp}, C={C} V={V}",
        "value": total / (step_ms / 1e3),
        "unit": UNIT, "n_gpus": 1, "steps": K, "warmup": W, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(batch, {"top_k": k, "top_p": tp, "kept_ids_arithmetic": "f64",
                                          "l2": f"flushed by a {L2_FLUSH_BYTES >> 20} MiB write between timed steps",
                                          "step": "isd_verify_filtered + isd_propose_filtered (four launches)"}),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "kernel": "isd_verify_filtered (top-k selection + decisions)",
                     "algorithmic_bytes": verify_bytes, "peak_source": f"{peak_kind} hbm_gbs",
                     "avg_launch_us": verify_ms * 1e3},
        "e2e": {"value": total / (e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in host_in.values()),
                "d2h_bytes_per_step": sum(x.numel() * x.element_size() for x in host_out)},
        "gpu_launches": 4 * K,
        "clocks": sampler.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.row == "kv":
        run_kv(args)
    elif args.row == "filtered":
        run_filtered(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
