"""Benchmark of the GB300 verify-and-sample step.

One step = one full verify round (LM-head contraction over the whole
vocabulary, softmax normalisers, left-to-right accept tests, residual or
bonus draw) for the Llama-3.1-8B-shaped LM head (V=128256, d=4096, B=1,
K=4, T=1) on synthetic inputs, through the C ABI.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--drafts model|ngram]

``--drafts ngram`` times the prompt-lookup variant instead: each step runs
the GPU n-gram drafter over a synthetic 4096-token context and verifies its
drafts as point masses (no draft logits are streamed).  ``--top-k`` and
``--top-p`` time truncated sampling (the same settings for target and
draft), which adds the per-row cut kernel to each step.  ``--tree`` times
greedy tree verification of a Medusa-like tree (3 levels of 3 branches, 39
nodes) at the same shape.  ``--fp8`` times the step with an FP8 E4M3 LM head
(weights and hidden states quantised per row, fp32 scales).

``--sweep`` runs the batch sweep of the 8B shape instead (B in
{1,2,4,8,16,32,64} x K in {3,4,5}, T=1, alpha ~0.7; ``--sweep-points
16x4,64x5`` picks points) and prints one JSON line per point with the
round rate, the contraction's time and its fractions of the HBM and the
tensor-core rooflines, to show where the step leaves the memory-bound
regime.

Prints one JSON line (rank 0).  Metric: verify rounds/s; ``roofline`` is
the LM-head contraction kernel's algorithmic bytes over its CUDA-event
duration against the measured HBM copy bandwidth; ``e2e`` is the same
metric through spec_verify_run_host with host buffers; ``cpu_baseline``
times the CPU oracle on a bounded sample.  ``--impl reference`` times the
CPU oracle alone (the reference arm).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "spec-verify rounds/s and % of HBM roofline at V=128256, d=4096, K=4, B=1"
UNIT = "rounds/s"
L2_BYTES = 129 * 1024 * 1024
NOMINAL_HBM_GBS = 8000.0
KERNEL_SRCS = [os.path.join(ROOT, "speculative_decoding_verification_22_gb300", "csrc", f)
               for f in ("sv_lmhead_tc.cu", "sv_internal.cuh", "sv_kernels.h")]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "lmhead_tc_llama8b.md")
TRAFFIC_FILE_FP8 = os.path.join(ROOT, "profiles", "lmhead_tc_llama8b_fp8.md")
TRAFFIC_FILE_B8K7 = os.path.join(ROOT, "profiles", "lmhead_tc_llama8b_b8k7.md")


# ---------------------------------------------------------------------------
# host-side helpers (no GPU needed; covered by the CPU tests)
# ---------------------------------------------------------------------------

def algorithmic_bytes(V, d, B, K, greedy=False, elt=2, point_mass=False, ctx_tokens=0):
    """Bytes one verify round must move: W_lm + q_logits + hidden + draft
    tokens + uniforms + outputs (q and uniforms are not read when greedy; q
    is absent for point-mass drafts, whose drafter reads ctx_tokens int32
    context tokens per sequence)."""
    w = elt * V * d
    q = 0 if (greedy or point_mass) else 4 * B * K * V
    w += 4 * B * ctx_tokens
    h = elt * B * (K + 1) * d
    small = 4 * B * K + (0 if greedy else 4 * B * (K + 1)) + 4 * B * (K + 1) + 4 * B
    return w + q + h + small


def contraction_bytes(V, d, B, K, greedy=False, elt=2, point_mass=False):
    """Algorithmic bytes of the contraction kernel alone: W_lm, hidden and
    (sampling with draft logits) the draft logits it streams for the softmax
    partials; with 1-byte (FP8) elements also the fp32 row scales."""
    q = 0 if (greedy or point_mass) else 4 * B * K * V
    scales = 4 * V + 4 * B * (K + 1) if elt == 1 else 0
    return elt * V * d + elt * B * (K + 1) * d + q + scales


CTX_TOKENS = 4096


def make_contexts(B, V, seed, device, length=CTX_TOKENS, doc=3072):
    """Synthetic prompt-lookup contexts: a random `doc`-token document, then
    spans of 8-32 tokens copied from random places in it, up to `length`
    tokens, so the last tokens recur earlier (as when an answer quotes its
    input).  Returns tokens [B, length] int32 and lengths [B]."""
    import torch
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    ctx = torch.empty((B, length), dtype=torch.int32)
    for b in range(B):
        ctx[b, :doc] = torch.randint(0, V, (doc,), generator=g, dtype=torch.int32)
        pos = doc
        while pos < length:
            n = int(torch.randint(8, 33, (1,), generator=g))
            s0 = int(torch.randint(0, doc - n, (1,), generator=g))
            n = min(n, length - pos)
            ctx[b, pos:pos + n] = ctx[b, s0:s0 + n]
            pos += n
    lens = torch.full((B,), length, dtype=torch.int32)
    return ctx.to(device), lens.to(device)


def n_input_sets(set_bytes, minimum=4, cap=256):
    """Rotating input sets whose total is at least twice the L2 size."""
    return int(min(cap, max(minimum, math.ceil(2 * L2_BYTES / max(set_bytes, 1)))))


def aggregate(elapsed_s: float, rounds: int, group=None):
    """Max elapsed time and total rounds over all ranks (weak scaling: each
    rank runs its own rounds on its own W replica)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_s, rounds
    dev = torch.device("cuda", torch.cuda.current_device()) \
        if dist.get_backend(group) == "nccl" else torch.device("cpu")
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    n = torch.tensor([rounds], dtype=torch.int64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(n, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), int(n.item())


REASON_COLS = {
    "clocks_event_reasons.hw_slowdown": "hw_slowdown",
    "clocks_event_reasons.hw_thermal_slowdown": "hw_thermal_slowdown",
    "clocks_event_reasons.sw_thermal_slowdown": "sw_thermal_slowdown",
    "clocks_event_reasons.sw_power_cap": "sw_power_cap",
}


def parse_clocks(text: str):
    """Summarise an nvidia-smi --format=csv clock log: median SM clock under
    load (samples above 30% of max power draw or any, if none), max clock,
    and every throttle reason seen Active."""
    rows = list(csv.reader(io.StringIO(text)))
    if not rows:
        return None
    head = [h.strip().split(" [")[0] for h in rows[0]]
    idx = {h: i for i, h in enumerate(head)}
    sm, smax, power, reasons = [], [], [], set()
    for r in rows[1:]:
        if len(r) != len(head):
            continue
        try:
            col = "clocks.sm" if "clocks.sm" in idx else "clocks.current.sm"
            sm.append(float(r[idx[col]].split()[0]))
            smax.append(float(r[idx["clocks.max.sm"]].split()[0]))
            power.append(float(r[idx["power.draw"]].split()[0]))
        except (KeyError, ValueError, IndexError):
            continue
        for col, name in REASON_COLS.items():
            if col in idx and r[idx[col]].strip() == "Active":
                reasons.add(name)
    if not sm:
        return None
    pmax = max(power) if power else 0.0
    loaded = [s for s, p in zip(sm, power) if p >= 0.3 * pmax] or sm
    return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
            "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_hash():
    """First 16 hex digits of the SHA-256 of the contraction kernel's sources."""
    h = hashlib.sha256()
    for f in KERNEL_SRCS:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(path=TRAFFIC_FILE):
    """DRAM bytes per launch of the contraction kernel from the committed
    ncu summary of this workload, or None if the kernel source changed since
    the capture (or there is none)."""
    if path is None:
        return None
    try:
        text = open(path).read()
        src = kernel_source_hash()
    except OSError:
        return None
    traffic, sha = None, None
    for line in text.splitlines():
        if line.startswith("dram_bytes_per_full_launch:"):
            traffic = int(float(line.split(":", 1)[1].split()[0]))
        if line.startswith("kernel_source_sha256_16:"):
            sha = line.split(":", 1)[1].strip()
    return traffic if (sha == src and traffic) else None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


class ClockSampler:
    def __init__(self, out_path=None):
        self.proc = None
        self.out = out_path

    def start(self, uuid=None):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             + ",".join(REASON_COLS))
        cmd = ["nvidia-smi", f"--query-gpu={q}", "--format=csv", "-lms", "200"]
        if uuid:
            cmd += ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        if self.out:
            with open(self.out, "w") as f:
                f.write(out)
        return parse_clocks(out)


# ---------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_rate(wl, W_np, inputs, budget_s, w_scale=None):
    """Times the CPU oracle (one thread) on this workload.  Full rounds while
    they fit the budget; otherwise a vocabulary slice of the contraction,
    which is >99.9% of an oracle round at this shape, scaled to a round."""
    import oracle
    import spec_inputs as si
    h = si.to_oracle(inputs["hidden"]).reshape(wl.B * (wl.K + 1), wl.d)
    t0 = time.perf_counter()
    rows = 1024
    oracle.logits(h, W_np, 0, rows)
    per_row = (time.perf_counter() - t0) / rows
    round_est = per_row * wl.V
    if round_est <= budget_s / 2:
        q = inputs.get("q_logits")
        qa = None if q is None else si.to_oracle(q)
        if w_scale is not None:   # FP8 LM head
            fn = oracle.verify_fp8
            args = (si.to_oracle(inputs["hidden8"]), si.to_oracle(inputs["h_scale"]), W_np,
                    si.to_oracle(w_scale), si.to_oracle(inputs["draft"]), qa,
                    si.to_oracle(inputs["uniforms"]), wl.T)
        else:
            fn = oracle.verify
            args = (si.to_oracle(inputs["hidden"]), W_np, si.to_oracle(inputs["draft"]), qa,
                    si.to_oracle(inputs["uniforms"]), wl.T)
        n, t0 = 0, time.perf_counter()
        while True:
            fn(*args)
            n += 1
            el = time.perf_counter() - t0
            if el >= budget_s / 2 or n >= 1000:
                break
        return n / el, f"{n} full oracle rounds", n
    rows = max(1024, int(wl.V * (budget_s / 2) / round_est))
    rows = min(rows, wl.V)
    t0 = time.perf_counter()
    oracle.logits(h, W_np, 0, rows)
    el = time.perf_counter() - t0
    frac = rows / wl.V
    return frac / el, (f"contraction over {rows} of {wl.V} vocabulary rows "
                       f"({frac:.3f} of a round), scaled to one round"), frac


def host_cpu():
    """CPU model and logical core count of the host running the oracle."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        import platform
        model = platform.processor() or platform.machine()
    return {"cpu_model": model, "nproc": os.cpu_count()}


def parity_sample(wl, W_np, sets, out_tok, out_n, ran, T, w_scale=None, max_sets=32):
    """The oracle on up to max_sets of the rounds this run timed, in parallel
    on the host's cores (one round per thread).  Returns the rounds' parity
    against the GPU's outputs with the flagged rounds (a uniform within 1e-6
    of an accept threshold, or of an edge of the final draw's CDF) and the
    oracle's all-core rate."""
    import concurrent.futures
    import numpy as np
    import oracle
    import spec_inputs as si
    idx = list(ran)[:max(1, min(max_sets, 2 * (os.cpu_count() or 1)))]
    host = []
    for i in idx:
        s = sets[i]
        h = {k: si.to_oracle(s[k]) for k in ("draft", "q_logits", "uniforms")}
        if w_scale is not None:
            h["hidden8"], h["h_scale"] = si.to_oracle(s["hidden8"]), si.to_oracle(s["h_scale"])
        else:
            h["hidden"] = si.to_oracle(s["hidden"])
        host.append(h)
    ws = None if w_scale is None else si.to_oracle(w_scale)

    def one(h):
        if ws is not None:
            return oracle.verify_fp8(h["hidden8"], h["h_scale"], W_np, ws, h["draft"],
                                     h["q_logits"], h["uniforms"], T)
        return oracle.verify(h["hidden"], W_np, h["draft"], h["q_logits"], h["uniforms"], T)

    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        refs = list(ex.map(one, host))
    el = time.perf_counter() - t0
    band = 1e-6 if T > 0 else 1e-7
    rounds = mism = unflagged = fa = fd = 0
    for i, ref in zip(idx, refs):
        gt, gn = out_tok[i].cpu().numpy(), out_n[i].cpu().numpy()
        bad = np.any(gt != ref["tokens"], axis=1) | (gn != ref["n_accepted"])
        flag = ref["dist"] <= band
        rounds += len(gn)
        mism += int(bad.sum())
        unflagged += int((bad & ~flag).sum())
        fa += int((ref["dist_accept"] <= band).sum())
        fd += int((ref["dist_draw"] <= band).sum())
    parity = {"rounds": rounds, "mismatched_rounds": mism, "unflagged_mismatches": unflagged,
              "flagged_accept": fa, "flagged_draw": fd, "flag_band": band,
              "note": "sample of this run's timed rounds; the large-sample rates come from "
                      "the parity tests"}
    all_cores = {"value": len(idx) / el, "unit": UNIT, "threads": threads,
                 "sample": f"{len(idx)} full oracle rounds, one per thread"}
    return parity, all_cores


def reference_arm(args, wl, dev):
    import torch
    import spec_inputs as si
    W = si.make_weights(wl, seed=1, device=dev)
    inputs = si.make_round(wl, W, seed=2)
    W_np = si.to_oracle(W)
    budget_per_step = max(0.05, 150.0 / max(1, args.steps + args.warmup))
    import oracle
    h = si.to_oracle(inputs["hidden"]).reshape(wl.B * (wl.K + 1), wl.d)
    t0 = time.perf_counter()
    oracle.logits(h, W_np, 0, 1024)
    per_row = (time.perf_counter() - t0) / 1024
    rows = int(min(wl.V, max(256, budget_per_step / per_row)))
    full = rows == wl.V
    args_full = (si.to_oracle(inputs["hidden"]), W_np, si.to_oracle(inputs["draft"]),
                 si.to_oracle(inputs["q_logits"]), si.to_oracle(inputs["uniforms"]), wl.T)

    def step(i):
        if full:
            oracle.verify(*args_full)
        else:
            v0 = (i * rows) % (wl.V - rows + 1)
            oracle.logits(h, W_np, v0, v0 + rows)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    el = time.perf_counter() - t0
    frac = rows / wl.V
    value = args.steps * frac / el
    sample = ("full oracle rounds" if full else
              f"each step: the oracle's contraction over {rows} of {wl.V} vocabulary rows "
              f"({frac:.4f} of a round, >99.9% of a round's oracle time), scaled to rounds")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl),
            "cpu_baseline": dict({"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                                  "sample": sample}, **host_cpu()),
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def medusa_tree(levels=3, branches=3):
    """Parents of a full tree, level by level (each node's parent precedes it)."""
    par, level = [], [-1]
    for _ in range(levels):
        nxt = []
        for p in level:
            for _ in range(branches):
                par.append(p)
                nxt.append(len(par) - 1)
        level = nxt
    return par


def workload_config(wl, extra=None, drafts="model", top_k=0, top_p=1.0, tree=False,
                    fp8=False):
    what = (f"draft acceptance ~{wl.alpha}" if drafts == "model" else
            f"prompt-lookup drafts (n-gram 5..2) over a {CTX_TOKENS}-token synthetic context, "
            "verified as point masses")
    if tree:
        what = (f"greedy tree verification of a 3x3x3 tree ({wl.K} nodes; first child of "
                "each node follows the target's choice)")
    if top_k or top_p < 1.0:
        what += f", truncated sampling top-k {top_k} top-p {top_p} on both sides"
    if fp8:
        what += ", FP8 E4M3 LM head and hidden states (fp32 row scales)"
    cfg = {"workload": f"Llama-3.1-8B-shaped LM-head verify round, V={wl.V}, d={wl.d}, "
                       f"B={wl.B}, K={wl.K}, T={wl.T}, {what}",
           "V": wl.V, "d": wl.d, "B": wl.B, "K": wl.K, "T": wl.T,
           "weights": "bf16 N(0, 0.02^2)", "alpha_target": wl.alpha}
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

SWEEP_B = (1, 2, 4, 8, 16, 32, 64)
SWEEP_K = (3, 4, 5)


def sweep_points(spec=None):
    """(B, K) points of the batch sweep: all of SWEEP_B x SWEEP_K, or the
    'BxK,BxK' list given."""
    if not spec:
        return [(b, k) for b in SWEEP_B for k in SWEEP_K]
    out = []
    for item in spec.split(","):
        b, k = item.lower().split("x")
        out.append((int(b), int(k)))
    return out


def regime(hbm_frac, tensor_frac):
    """Which roofline a point is closer to: the bound whose fraction is
    larger is the one the kernel is pressing against."""
    return "tensor" if tensor_frac > hbm_frac else "hbm"


def batch_sweep(args, dev):
    """One JSON line per (B, K) point of the 8B-shape batch sweep."""
    import torch
    import spec_inputs as si
    import speculative_decoding_verification_22_gb300 as sv
    peaks, peak_src = measured_peaks()
    base = si.workload("sweep")
    W = si.make_weights(base, seed=1, device=dev)
    steps = max(20, min(args.steps, 400))
    for B, K in sweep_points(args.sweep_points):
        wl = si.workload("sweep", B=B, K=K)
        set_bytes = 2 * B * (K + 1) * wl.d + 4 * B * K * wl.V + 8 * B * (K + 1)
        nsets = min(8, n_input_sets(set_bytes))
        sets = [si.make_round(wl, W, seed=30_000 + 100 * B + 10 * K + i) for i in range(nsets)]
        eng = sv.SpecVerify(wl.V, wl.d, B, K, "bf16", device=dev)
        stream = torch.cuda.Stream(device=dev)
        sv.spec_verify_set_stream(eng.h, stream)
        ot = [torch.empty((B, K + 1), dtype=torch.int32, device=dev) for _ in range(nsets)]
        on = [torch.empty((B,), dtype=torch.int32, device=dev) for _ in range(nsets)]

        def run(i):
            s = sets[i % nsets]
            sv.spec_verify_run(eng.h, s["hidden"], W, s["draft"], s["q_logits"], s["uniforms"],
                               wl.T, ot[i % nsets], on[i % nsets])

        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for i in range(max(args.warmup, nsets)):
                run(i)
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for i in range(steps):
                run(i)
            e1.record(stream)
        torch.cuda.synchronize()
        el = e0.elapsed_time(e1) / 1e3
        sv.spec_verify_timing(eng.h, True)
        with torch.cuda.stream(stream):
            for i in range(steps):
                run(i)
        ms_k1, n_k1 = sv.spec_verify_timing_read(eng.h)
        sv.spec_verify_timing(eng.h, False)
        code = eng.status()
        tokens = float((torch.stack(on).cpu().numpy() + 1).sum(axis=1).mean())
        eng.close()
        if code != sv.SV_OK:
            raise RuntimeError(f"B={B} K={K}: {sv.spec_verify_strerror(code)}")
        k1_s = ms_k1 / 1e3 / n_k1
        k1_bytes = contraction_bytes(wl.V, wl.d, B, K)
        flops = 2.0 * B * (K + 1) * wl.d * wl.V
        hbm = k1_bytes / k1_s / 1e9 / peaks["hbm_gbs"]
        tc = flops / k1_s / 1e12 / peaks["bf16_tflops"]
        rate = steps / el
        print(json.dumps({
            "mode": "sweep", "unit": UNIT, "B": B, "K": K, "rows": B * (K + 1),
            "value": rate, "ms_per_step": 1e3 * el / steps,
            "emitted_tokens_per_s": rate * tokens, "emitted_tokens_per_round": tokens,
            "contraction_us": k1_s * 1e6, "contraction_bytes": k1_bytes,
            "contraction_gflop": flops / 1e9, "flop_per_byte": flops / k1_bytes,
            "hbm_frac": hbm, "tensor_frac": tc, "pressing_on": regime(hbm, tc),
            "peaks": f"{peak_src}: hbm {peaks['hbm_gbs']} GB/s, bf16 {peaks['bf16_tflops']} TF/s",
            "steps": steps, "data": "synthetic"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="llama8b")
    ap.add_argument("--drafts", default="model", choices=["model", "ngram"])
    ap.add_argument("--top-k", type=int, default=0)
    ap.add_argument("--top-p", type=float, default=1.0)
    ap.add_argument("--tree", action="store_true")
    ap.add_argument("--fp8", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--clock-log", default=None)
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--sweep-points", default=None)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    import torch
    import torch.distributed as dist
    import spec_inputs as si

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = si.workload(args.workload)
    if args.tree:
        tree_par = medusa_tree()
        wl = si.workload(args.workload, K=len(tree_par), T=0.0)

    if args.sweep and args.impl != "reference":
        if rank == 0:
            batch_sweep(args, dev)
        if world > 1:
            dist.destroy_process_group()
        return

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args, wl, dev)), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    import speculative_decoding_verification_22_gb300 as sv

    T = wl.T
    ngram = args.drafts == "ngram"
    fp8 = args.fp8
    if fp8:
        W8, w_scale = si.make_fp8_weights(wl, seed=1 + 1000 * rank, device=dev)
        W = W8
    else:
        W = si.make_weights(wl, seed=1 + 1000 * rank, device=dev)
    set_bytes = (2 * wl.B * (wl.K + 1) * wl.d + 4 * wl.B * wl.K
                 + (4 * wl.B * CTX_TOKENS if ngram else 4 * wl.B * wl.K * wl.V)
                 + 4 * wl.B * (wl.K + 1))
    nsets = n_input_sets(set_bytes)
    if fp8:
        sets = [si.make_fp8_round(wl, W8, w_scale, seed=10_000 + 1000 * rank + i)
                for i in range(nsets)]
        for s in sets:
            s["hidden"] = s["hidden8"]
    else:
        sets = [si.make_round(wl, W, seed=10_000 + 1000 * rank + i) for i in range(nsets)]
    if args.tree:
        par_t = torch.tensor(tree_par, dtype=torch.int32, device=dev).repeat(wl.B, 1)
        for s in sets:
            # node tokens: the first child of each node follows the target's
            # choice (plain torch matmul, input shaping only), others random
            L = (s["hidden"].float() @ W.float().T)
            arg = L.argmax(dim=-1)
            tok = s["draft"].clone()
            for j, pj in enumerate(tree_par):
                if j % 3 == 0:
                    tok[:, j] = arg[:, pj + 1].to(torch.int32)
            s["draft"], s["parents"] = tok.contiguous(), par_t.contiguous()
            s["nodes"] = torch.empty((wl.B, wl.K), dtype=torch.int32, device=dev)
    if ngram:
        for i, s in enumerate(sets):
            s["q_logits"] = None
            s["ctx"], s["lens"] = make_contexts(wl.B, wl.V, 20_000 + 1000 * rank + i, dev)
            s["draft"] = torch.empty((wl.B, wl.K), dtype=torch.int32, device=dev)
            s["dlen"] = torch.empty((wl.B,), dtype=torch.int32, device=dev)
    # every input set read once on the device before the warm-up, as inputs
    # that an earlier step of a pipeline has just written would be: the
    # first read of a tensor long after it was written measured about 1 us
    # per round slower over a 20-round timed region (the first run of a
    # process), and a single pass over the sets removes that
    touch = torch.zeros((), dtype=torch.float32, device=dev)
    for s in sets:
        for v in s.values():
            if torch.is_tensor(v) and v.is_cuda and v.numel():
                touch += v.float().sum()
    torch.cuda.synchronize()
    eng = sv.SpecVerify(wl.V, wl.d, wl.B, wl.K, "fp8" if fp8 else "bf16", device=dev)
    stream = torch.cuda.Stream(device=dev)
    sv.spec_verify_set_stream(eng.h, stream)
    # one (16-byte aligned) output pair per input set
    out_tok = [torch.empty((wl.B, wl.K + 1), dtype=torch.int32, device=dev)
               for _ in range(nsets)]
    out_n = [torch.empty((wl.B,), dtype=torch.int32, device=dev) for _ in range(nsets)]
    torch.cuda.synchronize()

    def run_set(i):
        s = sets[i]
        if ngram:
            sv.spec_ngram_draft(s["ctx"], s["lens"], wl.K, 2, 5, s["draft"], s["dlen"],
                                stream=torch.cuda.current_stream())
        if fp8:
            sv.spec_verify_run_fp8(eng.h, s["hidden8"], s["h_scale"], W8, w_scale, s["draft"],
                                   s["q_logits"], s["uniforms"], T, out_tok[i], out_n[i])
        elif args.tree:
            sv.spec_verify_tree_greedy(eng.h, s["hidden"], W, s["draft"], s["parents"],
                                       out_tok[i], s["nodes"], out_n[i])
        elif truncated:
            sv.spec_verify_run_truncated(eng.h, s["hidden"], W, s["draft"], s["q_logits"],
                                         s["uniforms"], T, args.top_k, args.top_p, args.top_k,
                                         args.top_p, out_tok[i], out_n[i])
        else:
            sv.spec_verify_run(eng.h, s["hidden"], W, s["draft"], s["q_logits"],
                               s["uniforms"], T, out_tok[i], out_n[i])

    truncated = T > 0 and (0 < args.top_k < wl.V or args.top_p < 1.0)
    launches_per_run = (sv.spec_verify_launches_per_run(eng.h, T) + (1 if ngram else 0)
                        + (1 if truncated else 0))
    # the clocks are sampled from before the warm-up to after the kernel
    # timing pass, so that a short timed region still has samples around it
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(args.clock_log)
    sampler.start(uuid)
    time.sleep(0.3)

    # warm-up: exactly args.warmup untimed rounds, cycling through the sets
    used = set()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            run_set(i % nsets)
            used.add(i % nsets)
    # (the status word is checked after the timed region: it holds the
    # first error of any round since the last read)

    # timed: exactly args.steps rounds (the sets after the warm-up's, so a
    # round does not find its inputs in L2).  Long runs are cut into five
    # contiguous windows whose rates give the median and spread; an event
    # between two rounds costs the overlap of one round's tail with the
    # next round's start (a few us), so short runs are timed as one window.
    steps = args.steps
    nwin = min(5, steps) if steps >= 500 else 1
    bounds = [steps * w // nwin for w in range(nwin + 1)]
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(nwin + 1)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for w in range(nwin):
            for i in range(bounds[w], bounds[w + 1]):
                j = (args.warmup + i) % nsets
                run_set(j)
                used.add(j)
            evs[w + 1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed = evs[0].elapsed_time(evs[-1]) / 1e3
    win_rates = [(bounds[w + 1] - bounds[w]) / (evs[w].elapsed_time(evs[w + 1]) / 1e3)
                 for w in range(nwin)]
    code = eng.status()
    if code != sv.SV_OK:
        raise RuntimeError(f"device status after timing: {sv.spec_verify_strerror(code)}")
    max_el, total_rounds = aggregate(elapsed, steps)
    value = total_rounds / max_el
    windows = {"windows": nwin, "rounds_per_window": [bounds[w + 1] - bounds[w]
                                                      for w in range(nwin)],
               "median_rounds_per_s": statistics.median(win_rates),
               "min_rounds_per_s": min(win_rates), "max_rounds_per_s": max(win_rates),
               "note": "rank-local windows of the one timed region (one window below 500 "
                       "rounds)"}

    # emitted tokens per round over the input sets
    ran = sorted(used)
    n_host = torch.stack([out_n[i] for i in ran]).cpu().numpy()   # [sets run, B]
    tokens_per_round = float((n_host + 1).sum(axis=1).mean())

    # contraction kernel timing (CUDA events on the launching stream)
    kt_steps = min(steps, 2000)
    sv.spec_verify_timing(eng.h, True)
    with torch.cuda.stream(stream):
        for i in range(kt_steps):
            run_set(i % nsets)
    ms_k1, n_k1 = sv.spec_verify_timing_read(eng.h)
    sv.spec_verify_timing(eng.h, False)
    clocks = sampler.stop()
    k1_s = ms_k1 / 1e3 / n_k1
    peaks, peak_src = measured_peaks()
    k1_bytes = contraction_bytes(wl.V, wl.d, wl.B, wl.K, greedy=T == 0, point_mass=ngram,
                                 elt=1 if fp8 else 2)
    achieved = k1_bytes / k1_s / 1e9
    # the whole round's algorithmic bytes (FP8: 1-byte elements plus the
    # fp32 row scales)
    step_bytes = algorithmic_bytes(wl.V, wl.d, wl.B, wl.K, greedy=T == 0, point_mass=ngram,
                                   elt=1 if fp8 else 2, ctx_tokens=CTX_TOKENS if ngram else 0)
    if fp8:
        step_bytes += 4 * wl.V + 4 * wl.B * (wl.K + 1)
    # ncu captures exist for the default workload and its FP8 variant only
    plain = not (ngram or truncated or args.tree)
    traffic_file = None
    if plain and args.workload == "llama8b":
        traffic_file = TRAFFIC_FILE_FP8 if fp8 else TRAFFIC_FILE
    elif plain and args.workload == "llama8b_b8k7" and not fp8:
        traffic_file = TRAFFIC_FILE_B8K7
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "traffic": recorded_traffic(traffic_file),
                "peak_source": f"{peak_src} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                "kernel": "lmhead_tc_kernel (LM-head contraction + softmax partials)",
                "kernel_us": k1_s * 1e6, "algorithmic_bytes_per_launch": k1_bytes,
                "frac_of_nominal_8TBs": achieved / NOMINAL_HBM_GBS,
                "step_frac_of_measured": step_bytes * value / world / 1e9 / peaks["hbm_gbs"]}

    # end to end through the host-buffer entry point (prompt lookup: the
    # context, hidden states and uniforms copied in from pinned memory, the
    # drafter and the verify call, the outputs copied back, every step)
    e2e_steps = min(steps, 1000)
    keys = ("hidden", "ctx", "lens", "uniforms") if ngram else (
        "hidden", "draft", "q_logits", "uniforms")
    pin = [{k: sets[i][k].cpu().pin_memory() for k in keys} for i in range(min(nsets, 8))]
    ht = torch.empty((wl.B, wl.K + 1), dtype=torch.int32).pin_memory()
    hn = torch.empty((wl.B,), dtype=torch.int32).pin_memory()
    if args.tree:
        keys = ("hidden", "draft", "parents")
        pin = [{k: sets[i][k].cpu().pin_memory() for k in keys} for i in range(min(nsets, 8))]
    if fp8:
        keys = ("hidden8", "h_scale", "draft", "q_logits", "uniforms")
        pin = [{k: sets[i][k].cpu().pin_memory() for k in keys} for i in range(min(nsets, 8))]
    if ngram or truncated or args.tree or fp8:
        dbuf = {k: torch.empty_like(sets[0][k]) for k in keys}
        if ngram:
            dbuf.update(draft=torch.empty_like(sets[0]["draft"]),
                        dlen=torch.empty_like(sets[0]["dlen"]))
        # outputs of their own: the timed rounds' outputs stay for the
        # parity sample
        dtok, dn = torch.empty_like(out_tok[0]), torch.empty_like(out_n[0])

    def e2e_step(p):
        if fp8:
            with torch.cuda.stream(stream):
                for k in keys:
                    dbuf[k].copy_(p[k], non_blocking=True)
                sv.spec_verify_run_fp8(eng.h, dbuf["hidden8"], dbuf["h_scale"], W8, w_scale,
                                       dbuf["draft"], dbuf["q_logits"], dbuf["uniforms"], T,
                                       dtok, dn)
                ht.copy_(dtok, non_blocking=True)
                hn.copy_(dn, non_blocking=True)
            stream.synchronize()
            return
        if args.tree:
            with torch.cuda.stream(stream):
                for k in keys:
                    dbuf[k].copy_(p[k], non_blocking=True)
                sv.spec_verify_tree_greedy(eng.h, dbuf["hidden"], W, dbuf["draft"],
                                           dbuf["parents"], dtok, sets[0]["nodes"], dn)
                ht.copy_(dtok, non_blocking=True)
                hn.copy_(dn, non_blocking=True)
            stream.synchronize()
            return
        if not ngram and not truncated:
            sv.spec_verify_run_host(eng.h, p["hidden"], W, p["draft"], p["q_logits"],
                                    p["uniforms"], T, ht, hn)
            return
        if not ngram:
            # truncated sampling: the host buffers copied in, the step, the
            # outputs copied back (through the public entry points)
            with torch.cuda.stream(stream):
                for k in keys:
                    dbuf[k].copy_(p[k], non_blocking=True)
                sv.spec_verify_run_truncated(eng.h, dbuf["hidden"], W, dbuf["draft"],
                                             dbuf["q_logits"], dbuf["uniforms"], T, args.top_k,
                                             args.top_p, args.top_k, args.top_p, dtok, dn)
                ht.copy_(dtok, non_blocking=True)
                hn.copy_(dn, non_blocking=True)
            stream.synchronize()
            return
        with torch.cuda.stream(stream):
            for k in keys:
                dbuf[k].copy_(p[k], non_blocking=True)
            sv.spec_ngram_draft(dbuf["ctx"], dbuf["lens"], wl.K, 2, 5, dbuf["draft"],
                                dbuf["dlen"], stream=stream)
            sv.spec_verify_run(eng.h, dbuf["hidden"], W, dbuf["draft"], None,
                               dbuf["uniforms"], T, dtok, dn)
            ht.copy_(dtok, non_blocking=True)
            hn.copy_(dn, non_blocking=True)
        stream.synchronize()

    for i in range(3):
        e2e_step(pin[i % len(pin)])
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(pin[i % len(pin)])
    e2e_el = time.perf_counter() - t0
    _, e2e_total = aggregate(e2e_el, e2e_steps)
    e2e_max, _ = aggregate(e2e_el, e2e_steps)
    h2d = sum(pin[0][k].numel() * pin[0][k].element_size() for k in pin[0])
    d2h = ht.numel() * 4 + hn.numel() * 4
    e2e_serial = {"value": e2e_total / e2e_max, "unit": UNIT, "h2d_bytes_per_step": h2d,
                  "d2h_bytes_per_step": d2h,
                  "how": "spec_verify_run_host: copies in, the step, copies out, synchronise"}
    e2e = dict(e2e_serial)
    if not (ngram or truncated or args.tree or fp8):
        # the same rounds through the double-buffered host entry points: a
        # round's input copies overlap the previous round's kernels
        hts = [torch.empty((wl.B, wl.K + 1), dtype=torch.int32).pin_memory() for _ in range(2)]
        hns = [torch.empty((wl.B,), dtype=torch.int32).pin_memory() for _ in range(2)]

        def pipelined(n):
            busy = []
            for i in range(n):
                slot, p = i % 2, pin[i % len(pin)]
                if slot in busy:
                    busy.remove(slot)
                    if sv.spec_verify_wait_host(eng.h, slot) != sv.SV_OK:
                        raise RuntimeError("device status in a host round")
                sv.spec_verify_submit_host(eng.h, slot, p["hidden"], W, p["draft"],
                                           p["q_logits"], p["uniforms"], T, hts[slot],
                                           hns[slot])
                busy.append(slot)
            for slot in busy:
                if sv.spec_verify_wait_host(eng.h, slot) != sv.SV_OK:
                    raise RuntimeError("device status in a host round")

        pipelined(4)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        pipelined(e2e_steps)
        p_el = time.perf_counter() - t0
        _, p_total = aggregate(p_el, e2e_steps)
        p_max, _ = aggregate(p_el, e2e_steps)
        e2e = {"value": p_total / p_max, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "how": "spec_verify_submit_host / spec_verify_wait_host, two slots: each "
                      "round's copies in overlap the previous round's kernels; outputs "
                      "copied back and waited for every round"}

    cpu = None
    parity = None
    if rank == 0:
        W_np = si.to_oracle(W)
        rate, sample, _ = oracle_rate(wl, W_np, sets[0], args.cpu_budget,
                                      w_scale=w_scale if fp8 else None)
        cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample}
        cpu.update(host_cpu())
        if not (ngram or truncated or args.tree):
            # the oracle on a sample of this run's own rounds, one round per
            # host thread: the rounds' parity and flags, and an all-core rate
            parity, all_cores = parity_sample(wl, W_np, sets, out_tok, out_n, ran, T,
                                              w_scale if fp8 else None)
            cpu["all_cores"] = all_cores

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * max_el / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3 (fp32 accumulate)" if fp8 else "bf16",
            "data": "synthetic",
            "config": workload_config(wl, {
                "l2": f"inputs larger than L2: W_lm {2 * wl.V * wl.d} B per round plus "
                      f"{nsets} rotating input sets ({nsets * set_bytes} B)",
                "launch": "direct launches on one stream (programmatic dependent launch)",
                "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
                drafts=args.drafts, top_k=args.top_k, top_p=args.top_p, tree=args.tree,
                fp8=fp8),
            "emitted_tokens_per_round": tokens_per_round,
            "emitted_tokens_per_s": value * tokens_per_round,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "timed_windows": windows,
            "parity_sample": parity,
            "e2e": e2e,
            "e2e_serial": e2e_serial,
            "gpu_launches": launches_per_run * steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    eng.close()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
