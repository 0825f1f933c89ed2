"""Benchmark of the batched verify-and-accept step (one JSON line on rank 0).

A step is one spec_verify call -- the streaming launch that reads every
logit row once, then the draw launch that folds the statistics, runs the
acceptance scan and draws the replacement or bonus token -- over one batch
of the B=64, K=4, V=128256 bf16 workload (Zipf-like logits, T = 1), inputs
resident in HBM.
Input copies rotate so that every step reads data L2 has evicted (each
copy's logits, 147.75 MB, exceed the 129 MB L2); a workload too small for
that is timed one call at a time with an L2 flush before each.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME | --workload all]

Under torchrun every rank verifies its own batch (its own seed) with no
collective on the data path: weak scaling, value = all ranks' positions / the
slowest rank's time.  ``--impl reference`` times the float64 CPU oracle on
the host cores instead (rank 0 only).  ``--workload all`` prints one line for
each of the five synthetic workloads.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "spec_verify verified positions/s and HBM GB/s (% of roofline), B=64 K=4 V=128256"
WORKLOAD = "llama3_stochastic"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--copies", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="warm-up and timed steps only (for ncu captures); prints ms/step")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def rank_seed(seed: int, rank: int) -> int:
    """Every rank verifies its own batch: weak scaling, no shared data."""
    return seed + rank


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time (gloo all-reduce on a CPU tensor)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def row_lengths(w):
    """Drafted tokens each batch row verifies (K, or the ragged K_b)."""
    kb = getattr(w, "k_per_row", None)
    return np.full(w.B, w.K, np.int64) if kb is None else np.asarray(kb, np.int64)


def algorithmic_bytes(w, accepted):
    """Bytes the path must move for one batch: the target rows 0..K_b of
    every row, the draft rows 0..K_b-1 of rows with T > 0, and the re-read of
    the sampled position's rows (2 rows on a rejection, 1 for a bonus; none
    for greedy rows).  K_b = K unless the workload is ragged."""
    elt = w.elt
    V = w.V
    kb = row_lengths(w)
    stoch = w.temperature != 0
    pass1 = int(((kb + 1) * V * elt).sum()) + int((kb * stoch).sum()) * V * elt
    rej = int(((accepted < kb) & (accepted >= 0) & stoch).sum())
    bonus = int(((accepted == kb) & stoch).sum())
    pass2 = (2 * rej + bonus) * V * elt
    return pass1, pass2


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the GPU runs steps."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = open(os.path.join("/tmp", f"sv_clocks_{os.getpid()}.csv"), "w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.seek(0)
        rows = [l.strip().split(", ") for l in self.out if l.strip()]
        self.out.close()
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


_ORACLE_ROWS = None
_ORACLE_CACHE = {}


def _oracle_init(rows):
    global _ORACLE_ROWS
    _ORACLE_ROWS = rows


def _workload_init(name, seed, keep):
    """Worker start: rebuild the rows the timing loop cycles over (the
    generator draws every row from streams of its own)."""
    global _ORACLE_ROWS
    _ORACLE_ROWS = (name, seed)
    from speculative_decoding_verification_25_gb300 import synth
    for r in range(keep):
        _ORACLE_CACHE[r] = synth.make(name, seed=seed, rows=[r])


def _oracle_row(r):
    from oracle import oracle
    w = _ORACLE_CACHE.get(r)
    if w is None:
        from speculative_decoding_verification_25_gb300 import synth
        name, seed = _ORACLE_ROWS
        w = synth.make(name, seed=seed, rows=[r])
    if w.k_per_row is not None:
        return oracle.spec_verify_ragged(w.target, w.draft, w.draft_tokens, w.uniforms,
                                         w.temperature, w.k_per_row, dtype=w.dtype)
    return oracle.spec_verify(w.target, w.draft, w.draft_tokens, w.uniforms, w.temperature,
                              dtype=w.dtype)


def _oracle_timed(idx):
    return _oracle_row(idx % len(_ORACLE_CACHE)).accepted_len


def cpu_baseline(w, seed, gpu, budget_s=12.0, keep=16):
    """The float64 oracle, as it stands, on the host cores (one spawn worker
    per core).  It first verifies every row of the batch once, and those
    results give the parity counts of the GPU outputs ``gpu`` (accepted,
    out_tokens, logp, logq); then it cycles over the first ``keep`` rows for
    about ``budget_s`` -- the timed sample.  Returns (cpu_baseline, parity)."""
    import multiprocessing as mp
    from oracle import oracle
    from oracle.parity import check_structure, compare
    cores = os.cpu_count() or 1
    keep = min(keep, w.B)
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores, initializer=_workload_init, initargs=(w.name, seed, keep)) as pool:
        parts = pool.map(_oracle_row, range(w.B), chunksize=1)
        t0 = time.perf_counter()
        done = 0
        for _ in pool.imap_unordered(_oracle_timed, range(int(budget_s * cores * 100)), chunksize=1):
            done += 1
            if time.perf_counter() - t0 > budget_s:
                break
        dt = time.perf_counter() - t0
        pool.terminate()
    cat = lambda f: np.concatenate([getattr(p, f) for p in parts])
    ref = oracle.BatchResult(cat("accepted_len"), cat("out_tokens"), cat("logp"), cat("logq"),
                             cat("ratio_margin"), cat("cdf_margin"), sum((p.mode for p in parts), []))
    acc, out, lp, lq = gpu
    rep = compare(ref, acc, out, lp, lq, w.temperature)
    parity = {"rows": rep.rows, "greedy_rows": rep.greedy_rows,
              "stochastic_rows": rep.stochastic_rows, "ambiguous_rows": rep.ambiguous_rows,
              "mismatched_rows": rep.mismatched_rows,
              "mismatched_frac": rep.mismatched_rows / max(1, rep.rows),
              "max_logprob_err": rep.max_logprob_err, "rule_failures": len(rep.failures),
              "structure_failures": len(check_structure(acc, out, w.draft_tokens, w.V)),
              "oracle": "float64 numpy, every row of the timed batch"}
    pos_per_row = float((row_lengths(w)[:keep] + 1).mean())
    cpu = {"value": done * pos_per_row / dt, "unit": "positions/s", "cores": cores,
           "kind": "oracle",
           "sample": f"{done} row verifications cycling over rows 0..{keep - 1} of the "
                     f"{w.name} batch (K={w.K}, V={w.V}), float64 numpy, {cores} spawn "
                     f"workers, {dt:.1f} s wall"}
    return cpu, parity


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from speculative_decoding_verification_25_gb300 import synth
    from oracle import oracle
    w = synth.make(args.workload, seed=args.seed, rows=range(8))
    rows_per_step = 2

    kb = row_lengths(w)

    def step(i):
        r = [(2 * i + k) % w.B for k in range(rows_per_step)]
        if w.parents is not None:
            oracle.verify_tree_greedy(w.target[r], w.draft_tokens[r], w.parents[r], dtype=w.dtype)
        elif w.k_per_row is not None:
            oracle.spec_verify_ragged(w.target[r], w.draft[r], w.draft_tokens[r], w.uniforms[r],
                                      w.temperature[r], w.k_per_row[r], dtype=w.dtype)
        else:
            oracle.spec_verify(w.target[r], w.draft[r], w.draft_tokens[r], w.uniforms[r],
                               w.temperature[r], dtype=w.dtype)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    positions = sum(int(kb[(2 * i + k) % w.B]) + 1 for i in range(args.steps)
                    for k in range(rows_per_step))
    val = positions / dt
    cfg = synth.WORKLOADS[args.workload]
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "positions/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload} B={cfg['B']} K={cfg['K']} V={cfg['V']} "
                               f"{cfg['dtype']}", "B": cfg["B"], "K": cfg["K"], "V": cfg["V"],
                   "logits": cfg["dtype"], "step_sample_rows": rows_per_step},
        "cpu_baseline": {"value": val, "unit": "positions/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows_per_step} rows of the batch per step, one process"},
        "e2e": {"value": val, "unit": "positions/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


FIVE = ("tiny_stochastic", "greedy_batch", "llama3_stochastic", "long_draft_mixed_t",
        "large_vocab_stress")


def _json_default(o):
    """numpy scalars in the JSON line"""
    if isinstance(o, np.integer):
        return int(o)
    if isinstance(o, np.floating):
        return float(o)
    raise TypeError(f"not JSON serializable: {type(o).__name__}")


def run_ours(args):
    import torch
    import torch.distributed as dist

    from speculative_decoding_verification_25_gb300 import build as b

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("gloo")
    b.build()
    torch.cuda.set_device(local)
    names = FIVE if args.workload == "all" else (args.workload,)
    for name in names:
        line = bench_workload(args, name, rank, world, local)
        if rank == 0 and line is not None:
            print(json.dumps(line, default=_json_default), flush=True)
    if world > 1:
        dist.destroy_process_group()


def bench_workload(args, name, rank, world, local):
    """Time one workload; returns the JSON line (rank 0) or None."""
    import torch
    import torch.distributed as dist

    from speculative_decoding_verification_25_gb300 import _native as N
    from speculative_decoding_verification_25_gb300 import api, synth

    dev = torch.device("cuda", local)
    seed = rank_seed(args.seed, rank)
    w = synth.make(name, seed=seed, workers=synth.default_workers())
    dt_torch = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    dtype_code = N.SV_BF16 if w.dtype == "bf16" else N.SV_F32
    B, K, V = w.B, w.K, w.V

    def host_logits(a):
        t = torch.from_numpy(a.view(np.int16) if w.dtype == "bf16" else a)
        return t.view(dt_torch) if w.dtype == "bf16" else t

    ragged = w.k_per_row is not None
    host = dict(target=host_logits(w.target).pin_memory(), draft=host_logits(w.draft).pin_memory(),
                draft_tokens=torch.from_numpy(w.draft_tokens).pin_memory(),
                uniforms=torch.from_numpy(w.uniforms).pin_memory(),
                temperature=torch.from_numpy(w.temperature).pin_memory())
    if ragged:
        host["k_per_row"] = torch.from_numpy(np.ascontiguousarray(w.k_per_row, np.int32)).pin_memory()

    # Cold inputs: the bytes touched between two uses of one copy must be at
    # least twice the L2.  Rotate enough copies when that takes few; else
    # time one call at a time with a flush of 2 x L2 before each.
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    p1_all, _ = algorithmic_bytes(w, np.zeros(B, np.int64))
    need = 1 + -(-2 * l2 // max(1, p1_all))
    rotate = need <= 64
    n_copies = max(args.copies, need) if rotate else 1
    copies = [{k: v.to(dev) for k, v in host.items()} for _ in range(n_copies)]
    flush = None if rotate else torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    ws_bytes = N.spec_verify_workspace_bytes(B, K, V, dtype_code)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    outt = torch.empty(B, K + 1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def call(c, lp=None, lq=None):
        if ragged:
            st = N.spec_verify_ragged_raw(c["target"].data_ptr(), c["draft"].data_ptr(), dtype_code,
                                          c["draft_tokens"].data_ptr(), c["uniforms"].data_ptr(),
                                          c["temperature"].data_ptr(), c["k_per_row"].data_ptr(),
                                          B, K, V, acc.data_ptr(), outt.data_ptr(), lp, lq,
                                          ws.data_ptr(), ws_bytes, sh)
        else:
            st = N.spec_verify_raw(c["target"].data_ptr(), c["draft"].data_ptr(), dtype_code,
                                   c["draft_tokens"].data_ptr(), c["uniforms"].data_ptr(),
                                   c["temperature"].data_ptr(), B, K, V, acc.data_ptr(),
                                   outt.data_ptr(), lp, lq, ws.data_ptr(), ws_bytes, sh)
        if st != N.SV_OK:
            raise N.SpecVerifyError(st)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()

    # ---- warm-up, then the timed region (device events on the launching stream)
    for i in range(args.warmup):
        if flush is not None:
            flush.fill_(i & 0xff)
        call(copies[i % len(copies)])
    sampler = ClockSampler(local)
    sampler.start()
    clock_t0 = time.perf_counter()
    barrier()
    if rotate:
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(args.steps):
            call(copies[i % len(copies)])
        ev1.record(stream)
        barrier()
        t_ms = ev0.elapsed_time(ev1)
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(i & 0xff)          # evict the inputs from L2 (outside the events)
            evs[i][0].record(stream)
            call(copies[0])
            evs[i][1].record(stream)
        barrier()
        t_ms = sum(a.elapsed_time(e) for a, e in evs)
    t_ms = max_over_ranks(t_ms, world)
    gpu_launches = 2 * args.steps
    accepted = acc.cpu().numpy()
    if args.profile:
        sampler.stop()
        if rank == 0:
            print(json.dumps({"profile": True, "workload": name, "ms_per_step": t_ms / args.steps}),
                  flush=True)
        return None

    # keep the GPU on the same steps for >= 1.5 s so the clock samples see load
    i = 0
    while time.perf_counter() - clock_t0 < 1.5:
        if flush is not None:
            flush.fill_(i & 0xff)
        call(copies[i % len(copies)])
        i += 1
        if i % 200 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()

    # ---- end to end through the public call with host buffers
    d2h_acc = torch.empty(B, dtype=torch.int32).pin_memory()
    d2h_tok = torch.empty(B, K + 1, dtype=torch.int32).pin_memory()
    dst = copies[0]
    e2e_steps = max(10, min(args.steps, 100))

    def e2e_step():
        for k in host:
            dst[k].copy_(host[k], non_blocking=True)
        r = api.spec_verify(dst["target"], dst["draft"], dst["draft_tokens"], dst["uniforms"],
                            dst["temperature"], k_per_row=dst.get("k_per_row"), workspace=ws)
        d2h_acc.copy_(r.accepted_len, non_blocking=True)
        d2h_tok.copy_(r.out_tokens, non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e2e_steps
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = d2h_acc.numel() * 4 + d2h_tok.numel() * 4

    # ---- the streaming launch alone (spec_verify_row_stats), back to back on
    # the same cold inputs: the pass's own throughput, outside the step
    n_rs = max(args.steps, 50)
    kpr = lambda c: c["k_per_row"].data_ptr() if ragged else 0
    r0 = torch.cuda.Event(enable_timing=True)
    r1 = torch.cuda.Event(enable_timing=True)
    barrier()
    if rotate:
        r0.record(stream)
        for i in range(n_rs):
            c = copies[i % len(copies)]
            if N.spec_verify_row_stats_raw(c["target"].data_ptr(), c["draft"].data_ptr(), dtype_code,
                                           c["temperature"].data_ptr(), kpr(c), B, K, V,
                                           ws.data_ptr(), ws_bytes, sh) != N.SV_OK:
                raise RuntimeError("spec_verify_row_stats failed")
        r1.record(stream)
        barrier()
        rs_ms = r0.elapsed_time(r1) / n_rs
    else:
        rs_ms = 0.0
        for i in range(n_rs):
            flush.fill_(i & 0xff)
            r0.record(stream)
            c = copies[0]
            if N.spec_verify_row_stats_raw(c["target"].data_ptr(), c["draft"].data_ptr(), dtype_code,
                                           c["temperature"].data_ptr(), kpr(c), B, K, V,
                                           ws.data_ptr(), ws_bytes, sh) != N.SV_OK:
                raise RuntimeError("spec_verify_row_stats failed")
            r1.record(stream)
            barrier()
            rs_ms += r0.elapsed_time(r1)
        rs_ms /= n_rs
    rs_ms = max_over_ranks(rs_ms, world)

    # ---- the plug step: on its own, and fused into the verify launch
    max_len = 4096
    seqs = torch.zeros(B, max_len, dtype=torch.int32, device=dev)
    lens = torch.zeros(B, dtype=torch.int32, device=dev)
    n_plug = 50
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    barrier()
    p0.record(stream)
    for _ in range(n_plug):
        if N.spec_verify_plug_raw(acc.data_ptr(), outt.data_ptr(), B, K, seqs.data_ptr(),
                                  lens.data_ptr(), max_len, None, None, sh) != N.SV_OK:
            raise RuntimeError("plug failed")
    p1.record(stream)
    barrier()
    plug_us = p0.elapsed_time(p1) / n_plug * 1e3
    fused_us = None
    if rotate:
        n_fused = max(args.steps, 50)
        lens.zero_()
        barrier()
        p0.record(stream)
        for i in range(n_fused):
            c = copies[i % len(copies)]
            if N.spec_verify_and_plug_raw(
                    c["target"].data_ptr(), c["draft"].data_ptr(), dtype_code,
                    c["draft_tokens"].data_ptr(), c["uniforms"].data_ptr(),
                    c["temperature"].data_ptr(), c["k_per_row"].data_ptr() if ragged else None,
                    B, K, V, acc.data_ptr(), outt.data_ptr(), None, None, seqs.data_ptr(),
                    lens.data_ptr(), max_len, None, ws.data_ptr(), ws_bytes, sh) != N.SV_OK:
                raise RuntimeError("spec_verify_and_plug failed")
            if (i + 1) % 64 == 0:
                lens.zero_()
        p1.record(stream)
        barrier()
        fused_us = p0.elapsed_time(p1) / n_fused * 1e3

    # ---- the outputs the parity block checks (one call with log-probabilities)
    lp = torch.empty(B, K, dtype=torch.float32, device=dev)
    lq = torch.empty(B, K, dtype=torch.float32, device=dev)
    call(copies[0], lp.data_ptr(), lq.data_ptr())
    torch.cuda.synchronize(dev)
    gpu_out = (acc.cpu().numpy(), outt.cpu().numpy(), lp.cpu().numpy(), lq.cpu().numpy())
    dev_flags = api.device_errors(ws)

    if rank != 0:
        del copies, host
        return None

    ms_per_step = t_ms / args.steps
    # verified positions: K_b + 1 per row (the target positions the step checks)
    positions = int((row_lengths(w) + 1).sum()) * world
    value = positions / (ms_per_step * 1e-3)
    p1_bytes, p2_bytes = algorithmic_bytes(w, accepted)
    hbm, peak_src = peaks()
    step_gbs = (p1_bytes + p2_bytes) / (ms_per_step * 1e-3) / 1e9
    # the streaming kernel a ragged batch of up to 2048 rows runs is the compact one
    k1 = "sv_row_stats_compact_kernel" if ragged and B <= 2048 else "sv_row_stats_kernel"
    t1, t2 = stored_traffic(name, k1), stored_traffic(name, "sv_draw_kernel")
    roofline = {"bound": "hbm", "achieved": step_gbs, "peak": hbm, "unit": "GB/s",
                "frac": step_gbs / hbm, "traffic": t1 + t2 if t1 and t2 else None,
                "kernel": f"the whole step: {k1} + sv_draw_kernel, back to back",
                "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peak_src == "measured" else "fallback",
                "bytes_per_launch": p1_bytes + p2_bytes,
                "bytes": "every logit row read once + the sampled position's rows re-read "
                         "(2 rows at a rejection, 1 for a bonus; accepted_len of this batch)",
                "ms_per_launch": ms_per_step}
    cpu, parity = (None, None)
    if not args.no_cpu_baseline:
        cpu, parity = cpu_baseline(w, seed, gpu_out)
    if rotate:
        l2_label = (f"{len(copies)} rotating input copies, {p1_all / 1e6:.2f} MB read per step: "
                    f"{(len(copies) - 1) * p1_all / 1e6:.0f} MB touched between two uses of a copy "
                    f"(>= 2 x the {l2 / 1e6:.0f} MB L2)")
    else:
        l2_label = (f"{p1_all / 1e6:.3f} MB read per step: each call timed alone (events around "
                    f"it) after writing a {2 * l2 / 1e6:.0f} MB buffer (2 x L2)")
    line = {
        "metric": METRIC, "value": value, "unit": "positions/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"{name} B={B} K={K} V={V} {w.dtype} logits",
                   "B": B, "K": K, "V": V, "logits": w.dtype,
                   "T": describe_temperatures(w.temperature),
                   "k_per_row": ("ragged: K_b uniform in 0..%d, mean %.2f" % (K, float(w.k_per_row.mean()))
                                 if ragged else f"every row {K}"),
                   "l2": l2_label,
                   "parallelism": f"{world} independent replicas, own batch per GPU"},
        "roofline": roofline,
        "parity": parity,
        "cpu_baseline": cpu,
        "e2e": {"value": positions / (e2e_ms * 1e-3), "unit": "positions/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": gpu_launches,
        "clocks": clocks,
        "extra": {"rows_per_s": B * world / (ms_per_step * 1e-3),
                  "streaming_pass_alone": {
                      "us_per_launch": rs_ms * 1e3,
                      "gb_per_s": p1_all / (rs_ms * 1e-3) / 1e9,
                      "frac": p1_all / (rs_ms * 1e-3) / 1e9 / hbm,
                      "how": ("spec_verify_row_stats launched back to back on the rotating copies, "
                              "events around the loop" if rotate else
                              "spec_verify_row_stats timed one launch at a time after a 2 x L2 flush")},
                  "gb_per_s": step_gbs,
                  "frac_of_nominal_8tbs": step_gbs / 8000.0,
                  "pass1_bytes": p1_bytes, "resample_bytes": p2_bytes,
                  "plug_us_per_call": plug_us,
                  "verify_and_plug_us_per_step": fused_us,
                  "emitted_tokens_per_step": int((accepted + 1).sum()),
                  "mean_accepted_len": float(accepted.mean()),
                  "device_flags": dev_flags},
    }
    del copies, host
    return line


def describe_temperatures(T):
    T = np.asarray(T)
    greedy = int((T == 0).sum())
    if greedy == len(T):
        return "0 (greedy) all rows"
    vals = np.unique(T[T != 0])
    body = f"{vals[0]:g} all tempered rows" if len(vals) == 1 else \
        f"{vals.min():.2f}..{vals.max():.2f} over tempered rows"
    return body + (f", {greedy} greedy rows" if greedy else "")


def stored_traffic(workload, kernel="sv_row_stats_kernel"):
    """DRAM bytes per launch of ``kernel`` from the committed ncu summary of
    this workload, or None when the summary was taken on other kernel
    sources (or is missing)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                fields[k.strip()] = v.strip()
    if fields.get("kernel_rev") != kernel_rev(kernel):
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# the sources each kernel is built from (a stored ncu figure applies while
# they are unchanged)
KERNEL_SOURCES = {
    "sv_row_stats_kernel": ("sv_common.cuh", "sv_stream.cuh"),
    "sv_row_stats_compact_kernel": ("sv_common.cuh", "sv_stream.cuh"),
    "sv_draw_kernel": ("sv_common.cuh", "sv_stream.cuh", "sv_plug.cuh", "sv_sample.cuh",
                       "sv_draw.cuh", "exp2_table.inc"),
    "sv_tree_kernel": ("sv_common.cuh", "sv_stream.cuh", "sv_plug.cuh", "sv_sample.cuh",
                       "sv_tree.cuh"),
}


def code_only(text: str) -> str:
    """C/C++ source without comments and with whitespace runs collapsed: two
    sources that differ only in comments or layout give the same text."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_rev(kernel="sv_row_stats_kernel"):
    """Hash of one kernel's sources (code only, see code_only)."""
    import hashlib
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_25_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:12]


def run_tree(args):
    """Greedy tree verification (spec_verify_tree) on a tree workload: the
    streaming kernel over the N+1 target slots of every tree, then one CTA
    per tree.  Same timing rules as run_ours; the roofline is the step."""
    import torch
    import torch.distributed as dist

    from speculative_decoding_verification_25_gb300 import _native as N
    from speculative_decoding_verification_25_gb300 import api, synth
    from speculative_decoding_verification_25_gb300 import build as b

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("gloo")
    b.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = synth.make(args.workload, seed=rank_seed(args.seed, rank), workers=synth.default_workers())
    dtc = N.SV_BF16 if w.dtype == "bf16" else N.SV_F32
    B, Nn, V = w.B, w.K, w.V
    raw = torch.from_numpy(w.target.view(np.int16) if w.dtype == "bf16" else w.target)
    if w.dtype == "bf16":
        raw = raw.view(torch.bfloat16)
    host = dict(target=raw.pin_memory(), tokens=torch.from_numpy(w.draft_tokens).pin_memory(),
                parents=torch.from_numpy(w.parents).pin_memory())
    copies = [{k: v.to(dev) for k, v in host.items()} for _ in range(args.copies)]
    wsb = N.spec_verify_tree_workspace_bytes(B, Nn, V, dtc)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty(B, Nn + 1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call(c):
        st = N.spec_verify_tree_raw(c["target"].data_ptr(), dtc, c["tokens"].data_ptr(),
                                    c["parents"].data_ptr(), B, Nn, V, acc.data_ptr(),
                                    out.data_ptr(), None, ws.data_ptr(), wsb, stream.cuda_stream)
        if st != N.SV_OK:
            raise N.SpecVerifyError(st, "spec_verify_tree")

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()

    for i in range(args.warmup):
        call(copies[i % len(copies)])
    sampler = ClockSampler(local)
    sampler.start()
    clock_t0 = time.perf_counter()
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        call(copies[i % len(copies)])
    ev1.record(stream)
    barrier()
    t_ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    accepted = acc.cpu().numpy()
    if args.profile:
        sampler.stop()
        if rank == 0:
            print(json.dumps({"profile": True, "ms_per_step": t_ms / args.steps}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return
    i = 0
    while time.perf_counter() - clock_t0 < 1.5:
        call(copies[i % len(copies)])
        i += 1
        if i % 200 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()

    d_acc = torch.empty(B, dtype=torch.int32).pin_memory()
    d_out = torch.empty(B, Nn + 1, dtype=torch.int32).pin_memory()
    dst = copies[0]
    e2e_steps = max(10, min(args.steps, 100))

    def e2e_step():
        for k in host:
            dst[k].copy_(host[k], non_blocking=True)
        r = api.verify_tree(dst["target"], dst["tokens"], dst["parents"], workspace=ws)
        d_acc.copy_(r.accepted_len, non_blocking=True)
        d_out.copy_(r.out_tokens, non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world) / e2e_steps
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    ms_per_step = t_ms / args.steps
    positions = B * (Nn + 1) * world            # target slots checked
    bytes_step = B * (Nn + 1) * V * w.elt       # every slot read once, nothing re-read
    hbm, peak_src = peaks()
    gbs = bytes_step / (ms_per_step * 1e-3) / 1e9
    t1 = stored_traffic(args.workload, "sv_row_stats_kernel")
    t2 = stored_traffic(args.workload, "sv_tree_kernel")
    tree_traffic = t1 + t2 if t1 and t2 else None
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline_tree(w)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    line = {
        "metric": METRIC, "value": positions / (ms_per_step * 1e-3), "unit": "positions/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": f"{args.workload} B={B} N={Nn} nodes V={V} {w.dtype} logits",
                   "B": B, "N": Nn, "V": V, "logits": w.dtype, "T": "0 (greedy tree)",
                   "tree": "branching " + str(synth.WORKLOADS[args.workload]["tree"]),
                   "l2": f"{len(copies)} rotating input copies of {w.target.nbytes / 1e6:.2f} MB",
                   "parallelism": f"{world} independent replicas, own batch per GPU"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / hbm, "traffic": tree_traffic,
                     "kernel": "sv_row_stats_kernel + sv_tree_kernel (one step)",
                     "peak_source": peak_src, "bytes_per_launch": bytes_step,
                     "ms_per_launch": ms_per_step},
        "cpu_baseline": cpu,
        "e2e": {"value": positions / (e2e_ms * 1e-3), "unit": "positions/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d_acc.numel() * 4 + d_out.numel() * 4,
                "ms_per_step": e2e_ms},
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "extra": {"mean_accepted_depth": float(accepted.mean()),
                  "emitted_tokens_per_step": int((accepted + 1).sum())},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def _tree_job(idx):
    from oracle import oracle
    target, tokens, parents, dtype = _ORACLE_ROWS
    r = [idx % len(tokens)]
    return oracle.verify_tree_greedy(target[r], tokens[r], parents[r], dtype=dtype).accepted_len


def cpu_baseline_tree(w, budget_s=12.0, sample_rows=4):
    """The oracle's tree verification over a bounded sample, as cpu_baseline."""
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    rows = (w.target[:sample_rows], w.draft_tokens[:sample_rows], w.parents[:sample_rows], w.dtype)
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores, initializer=_oracle_init, initargs=(rows,)) as pool:
        pool.map(_tree_job, range(cores))
        t0 = time.perf_counter()
        done = 0
        for _ in pool.imap_unordered(_tree_job, range(int(budget_s * cores * 100)), chunksize=1):
            done += 1
            if time.perf_counter() - t0 > budget_s:
                break
        dt = time.perf_counter() - t0
        pool.terminate()
    return {"value": done * (w.K + 1) / dt, "unit": "positions/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} tree verifications cycling over rows 0..{sample_rows - 1} of the "
                      f"{w.name} batch (N={w.K}, V={w.V}), float64 numpy, {cores} spawn workers, "
                      f"{dt:.1f} s wall"}


def main():
    args = parse()
    from speculative_decoding_verification_25_gb300 import synth
    tree = args.workload != "all" and bool(synth.WORKLOADS[args.workload].get("tree"))
    if args.impl == "reference":
        for name in (FIVE if args.workload == "all" else (args.workload,)):
            args.workload = name
            run_reference(args)
    elif tree:
        run_tree(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
