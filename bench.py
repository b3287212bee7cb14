#!/usr/bin/env python3
"""Benchmark of batched speculative-decoding verification on GB300.

One step is one verification round: one call of the library over a whole
batch of B sequences (the headline workload is sampling at B=256, V=128256,
K=5).  The timed loop rotates through several input sets whose required bytes
together exceed the L2 cache, so every step streams from HBM.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on the
host cores instead (the reference arm); under torchrun every rank runs its own
batch (weak scaling) and the time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
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

METRIC = "verify rounds/s and achieved HBM GB/s (% roofline) at B=256,V=128256,K=5"
UNIT = "rounds/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0      # the ~8 TB/s nominal HBM3e figure, a second denominator
PRE_STEPS = 3                 # untimed steps issued just before the timed ones
DEFAULT_MODE = {1: "sample", 2: "greedy", 3: "sample", 4: "round", 5: "sample"}
KERNEL_SOURCES = [
    "speculative_decoding_verification_08_gb300/csrc/sv_device.cuh",
    "speculative_decoding_verification_08_gb300/csrc/sv_tma.cuh",
    "speculative_decoding_verification_08_gb300/csrc/sv_item.cuh",
    "speculative_decoding_verification_08_gb300/csrc/sv_logits.cuh",
    "speculative_decoding_verification_08_gb300/csrc/sv_alpha.cuh",
    "speculative_decoding_verification_08_gb300/csrc/specverify.cu",
]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--mode", choices=["sample", "greedy", "round", "alpha", "logits"],
                    default=None,
                    help="alpha: the acceptance-rate diagnostic; logits: sampling from logits "
                         "(log of the workload's probabilities, temperature 1)")
    ap.add_argument("--sets", type=int, default=0,
                    help="input sets rotated through (0: at least 4, and enough that their "
                         "required bytes exceed 4x L2)")
    ap.add_argument("--graph", action="store_true", help="replay the steps from a CUDA graph")
    ap.add_argument("--ctas-per-sm", type=int, default=0, help="persistent grid residency (0 = max)")
    ap.add_argument("--e2e-steps", type=int, default=60)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-copy", action="store_true",
                    help="end-to-end leg copies all inputs to the device each step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--seed", type=int, default=0,
                    help="offset of the input sets' seeds (0: the documented inputs)")
    ap.add_argument("--trace", action="store_true",
                    help="build the trace variant of the library, record --trace-launches "
                         "consecutive launches of the item kernel after the warm-up and print "
                         "their timeline (no timing line)")
    ap.add_argument("--trace-launches", type=int, default=4)
    ap.add_argument("--trace-out", default="",
                    help="also save the raw trace records (.npy) to this path")
    a = ap.parse_args(argv)
    if a.mode is None:
        a.mode = DEFAULT_MODE[a.config]
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    return a


# ---------------------------------------------------------------------------
# distributed helpers (host logic; covered by a gloo test)

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(cfg: int, set_index: int, rank: int, offset: int = 0) -> int:
    """Seed of input set `set_index` on `rank`: every rank verifies its own
    batch; `offset` (--seed) moves every set to other inputs."""
    from speculative_decoding_verification_08_gb300.inputs import SEED_BASE
    return SEED_BASE + cfg + 1000 * set_index + 100000 * rank + 10_000_000 * offset


class nvtx_range:
    """An NVTX range (for ncu --nvtx filtering); nothing if torch lacks NVTX."""

    def __init__(self, name: str):
        self.name = name

    def __enter__(self):
        try:
            import torch
            torch.cuda.nvtx.range_push(self.name)
            self.pushed = True
        except Exception:
            self.pushed = False
        return self

    def __exit__(self, *exc):
        if self.pushed:
            import torch
            torch.cuda.nvtx.range_pop()
        return False


def reduce_max(x: float, device=None) -> float:
    """Maximum of x over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate_rounds_per_s(steps: int, world: int, max_elapsed_s: float) -> float:
    """Whole-job rounds/s: every rank ran `steps` rounds of its own batch."""
    return steps * world / max_elapsed_s


# ---------------------------------------------------------------------------
# required (algorithmic) bytes: the rows and gathers the rule must touch

def required_bytes(mode_arr, n_arr, K: int, V: int) -> int:
    """Greedy sequence: rows 0..n of p (4V each) + tokens + outputs.  Sampling
    sequence: a 64-byte gather pair per tested position, the row pair p_n, q_n
    (8V) on rejection or the row p_K (4V) when all K are accepted, tokens,
    uniforms and outputs."""
    total = 0
    for m, n in zip(mode_arr, n_arr):
        n = int(n)
        if int(m) == 0:
            total += (n + 1) * 4 * V + 4 * K + 8
        else:
            tested = min(n + 1, K)
            rows = 8 * V if n < K else 4 * V
            total += 64 * tested + rows + 4 * K + 4 * K + 8 + 8
    return total


def logits_bytes(n_arr, K: int, V: int) -> int:
    """Sampling from logits reads the row pair (zp_i, zq_i) of every tested
    position once for its normalisers, then the rejected pair again (8V) or the
    bonus row zp_K twice (8V), plus tokens, uniforms and outputs."""
    total = 0
    for n in n_arr:
        tested = min(int(n) + 1, K)
        total += (tested + 1) * 8 * V + 8 * K + 16
    return total


def alpha_bytes(B: int, K: int, V: int) -> int:
    """The acceptance-rate diagnostic must read rows p_0..p_{K-1} and
    q_0..q_{K-1} of every sequence in full once (its second sweep over a row
    pair, for the minima after the totals, is served by L2) and writes B*K + B
    doubles."""
    return 8 * V * B * K + 8 * (B * K + B)


def dense_bytes(mode_arr, K: int, V: int) -> int:
    """Bytes of every row a rule could read (no early exit)."""
    total = 0
    for m in mode_arr:
        total += (K + 1) * 4 * V + (K * 4 * V if int(m) == 1 else 0)
    return total


def h2d_copy_gbs(host, dev, nbytes: int = 256 << 20, reps: int = 10) -> float:
    """Host-to-device bandwidth of a plain copy from page-locked memory (the
    copy engine over the host link), for the end-to-end leg's ceiling."""
    import torch
    x = host.reshape(-1)[: nbytes // host.element_size()]
    y = torch.empty(x.shape, dtype=x.dtype, device=dev)
    for _ in range(2):
        y.copy_(x, non_blocking=True)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        y.copy_(x, non_blocking=True)
    e1.record()
    torch.cuda.synchronize(dev)
    return reps * x.numel() * x.element_size() / (e0.elapsed_time(e1) * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# clocks during the timed region

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                self.samples.append(dict(t=ts + frac, sm=float(parts[2]), sm_max=float(parts[3]),
                                         reasons=[r for r, v in zip(REASONS, parts[6:10])
                                                  if v.lower().startswith("active")]))
            except (ValueError, IndexError):
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        inside = [s for s in self.samples if t0 <= s["t"] <= t1]
        note = "samples inside the timed region"
        if not inside:
            inside = [s for s in self.samples if t0 - 0.25 <= s["t"] <= t1 + 0.25]
            note = "timed region shorter than the sampling period; samples within 0.25 s of it"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.samples[-1]["sm_max"], "reasons": [],
                    "samples": 0, "note": "no sample near the timed region"}
        reasons = sorted({r for s in inside for r in s["reasons"]})
        return {"sm_mhz": statistics.median(s["sm"] for s in inside),
                "sm_max_mhz": max(s["sm_max"] for s in inside), "reasons": reasons,
                "samples": len(inside), "note": note}


# ---------------------------------------------------------------------------
# roofline denominators and ncu traffic

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, mode: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel sources changed since it was taken or nothing matches."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    entry = d.get("entries", {}).get(f"{workload}|{mode}")
    return None if entry is None else entry.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)

def host_inputs(cfg: int, seed: int):
    import torch
    from speculative_decoding_verification_08_gb300.inputs import make_inputs
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    bt = make_inputs(cfg, dev, seed=seed)
    host = bt.numpy()
    del bt
    if dev == "cuda":
        torch.cuda.empty_cache()
    return host


def time_oracle(host, mode: str, K: int, seconds: float, nthreads: int, max_rounds=None,
                seqs=None):
    """Runs the oracle over (a subset of) the batch until `seconds` pass; returns
    (rounds/s scaled to the full batch, sequences per round, rounds run)."""
    import numpy as np
    import oracle
    p, q, t, ua, ur, md = host
    B = p.shape[0]
    if seqs is not None and seqs < B:
        sl = slice(0, seqs)
        p, t, ua, ur, md = p[sl], t[sl], ua[sl], ur[sl], md[sl]
        q = None if q is None else q[sl]
    nb = p.shape[0]
    if mode == "logits":
        p, q = np.log(p), np.log(q)
    rounds = 0
    t0 = time.perf_counter()
    while True:
        if mode == "greedy":
            oracle.verify_greedy(p, t, nthreads=nthreads)
        elif mode == "sample":
            oracle.verify_sample(p, q, t, ua, ur, nthreads=nthreads)
        elif mode == "alpha":
            oracle.alpha(p, q)   # single-threaded
        elif mode == "logits":
            oracle.verify_sample_logits(p, q, t, ua, ur, 1.0)   # single-threaded
        else:
            oracle.verify_round(md, p, q, t, ua, ur, nthreads=nthreads)
        rounds += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_rounds is not None and rounds >= max_rounds):
            break
    return rounds * nb / B / el, nb, rounds, el


def oracle_parity(sets, outs, keep, mode: str, K: int, V: int):
    """Part of the CPU-baseline leg: runs the oracle on every rotated input set
    and compares the CUDA path's outputs of that set with it.  Returns
    (parity summary, required bytes per set computed from the oracle's
    n_accepted).  A decision mismatch (n_accepted, a greedy token, a drawn
    token outside the boundary band, or an alpha beyond 1e-6) is counted, not
    raised, so that the line still prints; main() then exits non-zero."""
    import numpy as np
    import oracle
    from oracle.compare import classify, compare_logits
    out = {"sets": len(sets), "sequences": 0, "draws": 0, "decision_mismatches": 0,
           "boundary_mismatches": 0, "boundary_cases": []}
    req = []
    for i, bt in enumerate(sets):
        p, q, t, ua, ur, md = bt.numpy()
        B = p.shape[0]
        n_gpu = outs[i][0].cpu().numpy()
        x_gpu = outs[i][1].cpu().numpy()
        out["sequences"] += B
        if mode == "alpha":
            a0, e0 = oracle.alpha(p, q)
            a1 = keep[i][0].cpu().numpy()
            out["decision_mismatches"] += int((np.abs(a1 - a0) > 1e-6).sum())
            out["max_alpha_error"] = max(out.get("max_alpha_error", 0.0),
                                         float(np.abs(a1 - a0).max()))
            req.append(alpha_bytes(B, K, V))
            continue
        if mode == "logits":
            zp, zq = np.log(p), np.log(q)
            n0, x0, _ = oracle.verify_sample_logits(zp, zq, t, ua, ur, 1.0)
            out["draws"] += B
            try:
                expl = compare_logits(zp, zq, 1.0, t, ua, ur, n0, x0, n_gpu, x_gpu)
                out["logits_near_threshold_accepts"] = out.get(
                    "logits_near_threshold_accepts", 0) + sum(k == "accept" for _, k in expl)
                out["boundary_mismatches"] += sum(k == "draw" for _, k in expl)
            except AssertionError:
                out["decision_mismatches"] += 1
            req.append(logits_bytes(n0, K, V))
            continue
        nth = os.cpu_count() or 1
        if mode == "greedy":
            n0, x0, _ = oracle.verify_greedy(p, t, nthreads=nth)
            rule = np.zeros(B, dtype=np.uint8)
        elif mode == "sample":
            n0, x0, _ = oracle.verify_sample(p, q, t, ua, ur, nthreads=nth)
            rule = np.ones(B, dtype=np.uint8)
        else:
            n0, x0, _ = oracle.verify_round(md, p, q, t, ua, ur, nthreads=nth)
            rule = md
        c = classify(p, q, ur, rule, K, n0, x0, n_gpu, x_gpu)
        out["draws"] += int((rule == 1).sum())
        out["decision_mismatches"] += len(c["n"]) + len(c["greedy"]) + len(c["unexplained"])
        out["boundary_mismatches"] += len(c["boundary"])
        out["boundary_cases"] += [(i,) + tuple(x) for x in c["boundary"]][:20]
        req.append(required_bytes(rule, n0, K, V))
    out["boundary_band"] = "|u*R - C_k| <= 1e-9 R (drawn tokens only)"
    return out, req


def workload_config(args, B, K, V, extra=None):
    from speculative_decoding_verification_08_gb300.inputs import CONFIGS
    cfg = {"workload": CONFIGS[args.config]["name"], "B": B, "V": V, "K": K, "mode": args.mode,
           "input_sets": args.sets if args.sets > 0 else 4}
    if extra:
        cfg.update(extra)
    return cfg


def run_reference(args):
    """Reference arm: the CPU oracle on the host cores, same workload and metric."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from speculative_decoding_verification_08_gb300.inputs import CONFIGS
    c = CONFIGS[args.config]
    B, K, V = c["B"], c["K"], c["V"]
    host = host_inputs(args.config, rank_seed(args.config, 0, 0, args.seed))
    ncpu = os.cpu_count() or 1
    # calibrate: sequences per step so that warmup + steps stay within ~2 minutes
    _, _, _, el = time_oracle(host, args.mode, K, 0.0, ncpu, max_rounds=1)
    per_seq = el / B
    budget = 120.0 / max(1, args.steps + args.warmup)
    seqs = int(max(ncpu, min(B, budget / max(per_seq, 1e-9))))
    time_oracle(host, args.mode, K, 0.0, ncpu, max_rounds=args.warmup, seqs=seqs)
    rps, nb, rounds, el = time_oracle(host, args.mode, K, float("inf"), ncpu,
                                      max_rounds=args.steps, seqs=seqs)
    sample = (f"{nb} of the {B} sequences of input set 0 per step, {rounds} steps, "
              f"{el:.3g} s on {ncpu} threads; value scaled to full {B}-sequence rounds")
    line = {
        "impl": "reference", "metric": METRIC, "value": rps, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / rps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": workload_config(args, B, K, V),
        "cpu_baseline": {"value": rps, "unit": UNIT, "cores": ncpu, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": rps, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the CUDA path

def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch
    import torch.distributed as dist

    import speculative_decoding_verification_08_gb300 as sv
    from speculative_decoding_verification_08_gb300.inputs import CONFIGS, make_inputs

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    sv.build()
    lib = sv.load()
    if args.trace:
        # the same calls through a trace build of the library (SV_TRACE=1)
        import tempfile
        from speculative_decoding_verification_08_gb300 import _build
        out = os.path.join(tempfile.mkdtemp(prefix="specverify_trace"), "libspecverify_trace.so")
        lib = sv._declare(ctypes.CDLL(_build.build_trace(out)))
    if args.ctas_per_sm:
        sv.set_ctas_per_sm(args.ctas_per_sm)

    c = CONFIGS[args.config]
    B, K, V = c["B"], c["K"], c["V"]
    ws = sv.Workspace(B, K, V, dev)
    stream = torch.cuda.Stream(dev)          # every timed launch goes to this stream
    sh = ctypes.c_void_p(stream.cuda_stream)
    P = lambda x: ctypes.c_void_p(0 if x is None else x.data_ptr())
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    sets, outs, calls, keep = [], [], [], []

    def add_sets(count):
        """Appends input sets and their precomputed C-ABI argument lists (the
        timed loop is one C call per step)."""
        for s_idx in range(len(sets), len(sets) + count):
            bt = make_inputs(args.config, dev, seed=rank_seed(args.config, s_idx, rank, args.seed))
            n = torch.empty(B, dtype=torch.int32, device=dev)
            nx = torch.empty(B, dtype=torch.int32, device=dev)
            sets.append(bt)
            outs.append((n, nx))
            if args.mode == "logits":
                zp, zq = torch.log(bt.p), torch.log(bt.q)
                keep.append((zp, zq))
                calls.append((lib.sv_verify_sample_logits,
                              (P(zp), V, P(zq), V, P(bt.t), P(bt.u_acc), P(bt.u_res), B, K, V,
                               ctypes.c_float(1.0), P(n), P(nx), ws.ptr, ws.nbytes, sh)))
            elif args.mode == "alpha":
                a_out = torch.empty(B, K, dtype=torch.float64, device=dev)
                e_out = torch.empty(B, dtype=torch.float64, device=dev)
                keep.append((a_out, e_out))
                calls.append((lib.sv_alpha,
                              (P(bt.p), V, P(bt.q), V, B, K, V, P(a_out), P(e_out), ws.ptr,
                               ws.nbytes, sh)))
            elif args.mode == "greedy":
                calls.append((lib.sv_verify_greedy,
                              (P(bt.p), V, P(bt.t), B, K, V, P(n), P(nx), ws.ptr, ws.nbytes, sh)))
            elif args.mode == "sample":
                calls.append((lib.sv_verify_sample,
                              (P(bt.p), V, P(bt.q), V, P(bt.t), P(bt.u_acc), P(bt.u_res), B, K,
                               V, P(n), P(nx), ws.ptr, ws.nbytes, sh)))
            else:
                calls.append((lib.sv_verify_round,
                              (P(bt.mode), P(bt.p), V, P(bt.q), V, P(bt.t), P(bt.u_acc),
                               P(bt.u_res), B, K, V, P(n), P(nx), None, None, 0, ws.ptr,
                               ws.nbytes, sh)))
        # the sets were made on torch's current stream and the calls run on
        # `stream`: finish them (and release nothing still in use) first
        torch.cuda.synchronize(dev)

    def step(k):
        fn, a = calls[k % len(calls)]
        rc = fn(*a)
        if rc != 0:
            raise RuntimeError(f"verify call failed: {sv.status_string(rc)}")

    def warm_up():
        with nvtx_range("warmup"):
            for k in range(max(args.warmup, len(calls))):   # every set's outputs at least once
                step(k)
            torch.cuda.synchronize(dev)

    def required_per_launch():
        """Algorithmic bytes per launch, from each set's n_accepted; with the
        per-set figures, the histogram of n and the dense bytes."""
        req, dense, nhist = [], [], np.zeros(K + 1, dtype=np.int64)
        for bt, (n, _) in zip(sets if args.mode != "alpha" else [], outs):
            md = bt.mode.cpu().numpy() if args.mode == "round" else np.full(
                B, 0 if args.mode == "greedy" else 1)   # logits: sampling
            nn = n.cpu().numpy()
            nhist += np.bincount(nn, minlength=K + 1)[:K + 1]
            req.append(logits_bytes(nn, K, V) if args.mode == "logits"
                       else required_bytes(md, nn, K, V))
            dense.append(dense_bytes(md, K, V))
        if args.mode == "alpha":
            req = dense = [alpha_bytes(B, K, V)]
        return float(np.mean(req)), req, dense, nhist

    add_sets(args.sets if args.sets > 0 else 4)
    warm_up()
    req_per_launch, req, dense, nhist = required_per_launch()
    if args.sets == 0 and len(sets) * req_per_launch < 4 * l2:
        # more sets, so that consecutive launches never find their rows in L2
        # (bounded by a memory budget; the line says so if that is not enough)
        per_set = max(1.0, float(np.mean(dense)) * (3 if args.mode == "logits" else 1))
        want = int(np.ceil(4.4 * l2 / max(req_per_launch, 1.0)))   # sets differ a little
        want = min(want, 4096, max(len(sets), int(40e9 // per_set)))
        add_sets(want - len(sets))
        warm_up()
        req_per_launch, req, dense, nhist = required_per_launch()
    torch.cuda.empty_cache()
    if args.trace:
        # consecutive launches (the next input sets of the rotation) with the
        # buffer cleared before the first
        sv.trace_reset(stream, lib)
        for k in range(max(1, args.trace_launches)):
            step(k)
        records = sv.trace_read(stream, lib)
        if args.trace_out:
            np.save(args.trace_out, records)
        if rank == 0:
            print(json.dumps({"trace": sv.trace_timeline(records),
                              "config": workload_config(args, B, K, V), "mode": args.mode}))
        return 0
    status = ws.status(stream)
    kernels_per_step = sv.last_kernel_count()
    grid_ctas = int(sv.last_grid_size())     # of the timed launches (the e2e leg may differ)
    l2_resident = len(sets) * req_per_launch < 4 * l2

    graph = None
    if args.graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(len(calls)):
                step(k)
        graph = g

    clocks = ClockSampler(dev.index or 0) if rank == 0 else None
    time.sleep(0.3 if clocks else 0.0)
    barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # three untimed steps right before the start event (the input sets that
    # precede set 0 in the rotation), so that the timed steps start on a busy
    # GPU: neither the idle time above nor the host's first enqueue falls
    # inside the timed region
    with nvtx_range("warmup"):
        if graph is None:
            for k in range(-PRE_STEPS, 0):
                step(k % len(calls))
        else:
            with torch.cuda.stream(stream):
                graph.replay()
    t_wall0 = time.time()
    with nvtx_range("timed"):
        e0.record(stream)
        if graph is None:
            for k in range(args.steps):
                step(k)
            launches = args.steps
        else:
            reps = max(1, args.steps // len(calls))
            with torch.cuda.stream(stream):
                for _ in range(reps):
                    graph.replay()
            launches = reps * len(calls)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier()
    el_ms = e0.elapsed_time(e1)
    max_ms = reduce_max(el_ms, dev)
    if clocks:
        clocks.stop()
    steps_done = launches
    rounds_per_s = aggregate_rounds_per_s(steps_done, world, max_ms / 1000.0)
    ms_per_step = max_ms / steps_done
    kernel_us = el_ms * 1000.0 / steps_done
    peak, peak_kind = hbm_peak()
    workload = c["name"]
    traffic = ncu_traffic(workload, args.mode)

    # end to end through the public API: pinned host inputs -> device -> result
    e2e = None
    if not args.no_e2e and rank == 0 and args.mode in ("sample", "greedy"):
        hv = sv.HostVerifier(B, K, V, dev, sampling=args.mode == "sample",
                             mapped=not args.e2e_copy)
        bt = sets[0]
        hp = bt.p.cpu().pin_memory()
        hq = bt.q.cpu().pin_memory() if args.mode == "sample" else None
        ht, hua, hur = (bt.t.cpu().pin_memory(), bt.u_acc.cpu().pin_memory(),
                        bt.u_res.cpu().pin_memory())
        run = (lambda: hv.sample(hp, hq, ht, hua, hur)) if args.mode == "sample" else (
            lambda: hv.greedy(hp, ht))
        for _ in range(3):
            run()
        n_e2e = max(1, min(args.e2e_steps, args.steps))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            run()
        t1 = time.perf_counter()
        assert np.array_equal(hv.n_host.numpy(), outs[0][0].cpu().numpy())
        link = h2d_copy_gbs(hp, dev)
        rate = hv.h2d_bytes() * n_e2e / (t1 - t0) / 1e9
        e2e = {"value": n_e2e / (t1 - t0), "unit": UNIT,
               "h2d_bytes_per_step": hv.h2d_bytes(),
               "d2h_bytes_per_step": hv.d2h_bytes(), "steps": n_e2e,
               "link": {"achieved_gbs": rate, "copy_engine_h2d_gbs": link,
                        "frac": rate / link,
                        "note": "input bytes that crossed the host link per second, against a "
                                "plain pinned-to-device copy of 256 MB measured alongside"},
               "transfer": ("inputs in pinned host memory read in place by the kernels over "
                            "the host link (only the rows the rule needs)" if hv.mapped else
                            "all inputs copied host to device every step")}
        del hv, hp, hq

    cpu = None
    parity = None
    req_source = ("n_accepted of the CUDA path (the oracle did not run: no CPU-baseline leg "
                  "on this rank)") if args.mode != "alpha" else "fixed by the sizes"
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        host = sets[0].numpy()
        ncpu = os.cpu_count() or 1
        threaded = args.mode not in ("alpha", "logits")   # those oracles are single-threaded
        secs = args.cpu_seconds / 2 if threaded else args.cpu_seconds
        rps, nb, rounds, el = time_oracle(host, args.mode, K, secs, ncpu)
        used = ncpu if threaded else 1
        cpu = {"value": rps, "unit": UNIT, "cores": used, "kind": "oracle",
               "sample": f"{rounds} full rounds ({nb} sequences each) of input set 0, "
                         f"{el:.1f} s on {used} thread{'s' if used > 1 else ''}"}
        if threaded:   # the same oracle on one thread, for the per-core figure
            rps1, _, rounds1, el1 = time_oracle(host, args.mode, K, secs, 1)
            cpu["value_1thread"] = rps1
            cpu["sample"] += f"; {rounds1} rounds in {el1:.1f} s on 1 thread"
        # the same oracle on every rotated input set: parity of the timed
        # launches' outputs, and the required bytes from the oracle's n
        parity, req_oracle = oracle_parity(sets, outs, keep, args.mode, K, V)
        req_per_launch = float(np.mean(req_oracle))
        req_source = "n_accepted of the oracle on the same inputs"
    achieved = req_per_launch / (kernel_us * 1e-6) / 1e9

    if rank == 0:
        clk = clocks.summary(t_wall0, t_wall1) if clocks else None
        line = {
            "metric": METRIC, "value": rounds_per_s, "unit": UNIT, "n_gpus": world,
            "steps": steps_done, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; see inputs.py)",
            "config": workload_config(args, B, K, V, {
                "input_sets": len(sets),
                "l2": (f"rotating {len(sets)} input sets; {len(sets) * req_per_launch / 1e6:.0f} MB"
                       f" required bytes per rotation = {len(sets) * req_per_launch / l2:.1f}x "
                       f"L2 ({l2 / 1e6:.0f} MB)"),
                "launch": "cuda graph" if graph is not None else "one C-ABI call per step",
                "grid_ctas": grid_ctas}),
            "seq_rounds_per_s": rounds_per_s * B,
            "achieved_gbs": achieved * world,
            "required_bytes_per_round": req_per_launch,
            "dense_bytes_per_round": float(np.mean(dense)),
            "n_accepted_hist": nhist.tolist(),
            "required_bytes_from": req_source,
            "parity": parity,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind,
                         "peak_nominal_gbs": NOMINAL_HBM_GBS,
                         "frac_nominal": achieved / NOMINAL_HBM_GBS,
                         "traffic": traffic, "kernel_us": kernel_us,
                         **({"note": "L2-resident rotation: not an HBM figure"}
                            if l2_resident else {})},
            "gpu_launches": launches * kernels_per_step,
            "status_bits": status,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "impl": "gb300",
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    if parity is not None and parity["decision_mismatches"]:
        print(f"bench: {parity['decision_mismatches']} outputs differ from the oracle beyond "
              "the boundary band", file=sys.stderr)
        return 1
    return 0


if __name__ == "__main__":
    sys.exit(main())
