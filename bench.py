#!/usr/bin/env python3
"""Benchmark of the ForkAttention token-mixing layer on one round.

A step is one pass of the whole layer over one synthetic round: metadata
build, full attention, sliding-window attention, GDN trunk call, GDN branch
call, options readout.  The default workload is the long-document round (4
requests, trunks of 4096-6144 tokens, 8-20 questions of 32-64 tokens each;
attention 32 q-heads / 8 kv-heads, d=128, RoPE; SWA W=1024; GDN 32 heads,
d=128, chunk 64; T_cap 32768).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.
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

WORKLOAD_ID = 3
METRIC = "ForkAttention layer tokens/s per round (attn+GDN) and % of roofline"

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one call of the full-
# attention layer on this workload, summed over the call's launches (rotary tables, key
# rotation, fp16 value copy, attention), from one ncu capture of this bench's command.  Keyed by the
# SHA-256 of the attention sources: once they change, traffic reads null until re-measured.
TRAFFIC = {"sources": ["tree_forked_hybrid_gb300/csrc/fork_attn.cu", "tree_forked_hybrid_gb300/csrc/fork_attn_tc.cu",
                       "tree_forked_hybrid_gb300/csrc/fork_attn.cuh", "tree_forked_hybrid_gb300/csrc/tc_ptx.cuh"],
           "sha256": "dc0b115b6e0d162682b32c5572ded0319d10b7c3050d872c541df3e2976163e6", "bytes": 501405440}


def _sources_sha256(paths):
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _traffic():
    if TRAFFIC["sha256"] is None or TRAFFIC["bytes"] is None:
        return None
    return TRAFFIC["bytes"] if _sources_sha256(TRAFFIC["sources"]) == TRAFFIC["sha256"] else None


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def aggregate_over_ranks(torch, dist, device, elapsed_ms: float, tokens: int):
    """Whole-job figures of one process per GPU: the slowest rank's elapsed time
    and the tokens of all ranks' rounds (each rank draws its own round)."""
    if dist is None:
        return elapsed_ms, tokens
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor([tokens], dtype=torch.int64, device=device)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None):
        self.rows = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [r for (t, r) in self.rows if t0 <= t <= t1]
        note = "timed region"
        if not rows:
            rows = [r for (_, r) in self.rows]
            note = "around the timed region (region shorter than the sampling period)"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if len(r) > 5 + i and r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "note": note}


def _gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def oracle_sample(rnd, trunk_cap=None, n_questions=1):
    """Time the CPU oracle on request 0 (trunk, optionally cut to trunk_cap
    tokens, plus its first n_questions questions).  Returns (tokens, seconds)."""
    from oracle import forkattn as orc
    from tree_forked_hybrid_gb300 import workloads as wl
    P0 = int(rnd.trunk_len[0])
    P = P0 if trunk_cap is None else min(P0, trunk_cap)
    nq = min(n_questions, int(rnd.n_q[0]))
    ql = rnd.q_len[:nq]
    # the sample as a round of its own: trunk rows [0, P) and the chosen questions' rows
    m = orc.meta_ref(rnd.desc(), rnd.R, rnd.Nq, rnd.T_cap, 32)
    rows = list(range(0, P))
    for i in range(nq):
        st, L = int(m["seg_start"][rnd.R + i]), int(m["seg_len"][rnd.R + i])
        rows.extend(range(st, st + L))
    rows = np.array(rows)
    desc = np.concatenate([[P], [nq], ql, [0], [-1]]).astype(np.int32)
    T_s = int(P + ql.sum())
    lay = {}
    for name, d in rnd.layers.items():
        lay[name] = {k: (wl.bf16_to_f32(v[rows]) if v.dtype == np.uint16 else
                         (v[rows] if k != "conv_w" else v)) for k, v in d.items()}
    view = orc.RoundView(desc, 1, nq, T_s, lay)
    t0 = time.perf_counter()
    for a in rnd.attn_shapes:
        orc.run_attention(view, a.name, window=a.window, rope_theta=a.rope_theta)
    g = orc.run_gdn(view, rnd.gdn_shape.name)
    off = np.concatenate([[0], np.cumsum(rnd.n_opt[:nq])]).astype(np.int32)
    orc.run_readout(view, g["o"].reshape(T_s, -1), rnd.w_opt_f32()[:off[-1]], off)
    return T_s, time.perf_counter() - t0


REF_TRUNK_CAP = 1024  # oracle sample: request 0, trunk cut to its first 1024 tokens, first question


def _oracle_sample_note(rnd, n):
    return (f"request 0 of the round with its trunk cut to its first {min(REF_TRUNK_CAP, int(rnd.trunk_len[0]))} "
            f"tokens plus its first question ({n} stream tokens), run through the oracle (numpy fp32)")


def run_reference(args):
    """The reference arm: the CPU oracle on the machine's host cores, each step one
    oracle sample (the same sample the cpu_baseline of the GPU arm times)."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from tree_forked_hybrid_gb300 import workloads as wl
    rnd = wl.make_round(WORKLOAD_ID)
    cores = len(os.sched_getaffinity(0))
    for _ in range(args.warmup):
        oracle_sample(rnd, REF_TRUNK_CAP)
    tok = 0
    t = 0.0
    for _ in range(args.steps):
        n, dt = oracle_sample(rnd, REF_TRUNK_CAP)
        tok += n
        t += dt
    value = tok / t
    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "impl": "reference",
           "config": _config(rnd),
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": "per step: " + _oracle_sample_note(rnd, tok // max(args.steps, 1))},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def cpu_baseline(rnd, min_seconds=10.0):
    """The oracle on the same sample as the reference arm, repeated until about
    min_seconds of CPU work have been timed."""
    tok, t, reps = 0, 0.0, 0
    while t < min_seconds and reps < 8:
        n, dt = oracle_sample(rnd, REF_TRUNK_CAP)
        tok += n
        t += dt
        reps += 1
    return {"value": tok / t, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{reps} repetitions of: " + _oracle_sample_note(rnd, tok // reps) + f"; {t:.1f} s in total"}


def _config(rnd):
    return {"workload": "long-document round: R=4, P~U[4096,6144], n~U{8..20}, |q|~U[32,64]; "
                        "attn 32q/8kv d=128 RoPE; SWA W=1024; GDN 32 heads d=128 chunk 64; readout D=4096",
            "T": rnd.T, "T_cap": rnd.T_cap, "R": rnd.R, "Nq": rnd.Nq,
            "l2": "inputs larger than L2 (about 1.2 GB of layer inputs per step)"}


def _events(torch, n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def step_times(torch, fn, stream, steps):
    """CUDA-event duration (ms) of each of `steps` back-to-back calls of fn."""
    ev = _events(torch, steps + 1)
    ev[0].record(stream)
    for i in range(steps):
        fn()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]


def latency_stats(ms):
    return {"median": float(np.median(ms)), "p10": float(np.percentile(ms, 10)),
            "p90": float(np.percentile(ms, 90)), "mean": float(np.mean(ms))}


def layer_roofline(RL, rnd, ms, peaks):
    work = RL.round_work(rnd)
    t_f = work["flops"] / (peaks["bf16_tflops"] * 1e12)
    t_b = work["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_roof = max(t_f, t_b)
    return {"t_roof_us": t_roof * 1e6, "t_meas_us": ms * 1e3, "frac": t_roof / (ms / 1e3),
            "bound": "tensor" if t_f >= t_b else "hbm", "flops": work["flops"], "bytes": work["bytes"]}


WORKLOAD_NAMES = {1: "short requests: R=32, P~U[256,512], n~U{1..4}, |q|~U[16,48]; attn 16q/4kv d=128 RoPE; "
                     "GDN 16 heads d=128; T_cap 16384",
                  2: "many questions: R=8, P~U[256,400], n=48, |q|~U[12,32]; attn 16q/4kv d=128 + SWA W=512; "
                     "GDN 16 heads; T_cap 16384",
                  3: "long documents: R=4, P~U[4096,6144], n~U{8..20}, |q|~U[32,64]; attn 32q/8kv d=128 + SWA "
                     "W=1024; GDN 32 heads; T_cap 32768",
                  "4A": "wide fork: one request, P=16384, 64 questions of U[16,64] tokens, checkpoint at 15360; "
                        "shapes as the long-document round",
                  "4B": "resume: 15360 prefix rows (K/V, GDN state and conv window from the checkpoint) + 2048 "
                        "new trunk tokens + 64 questions"}


def per_config(torch, RL, wl, DeviceRound, peaks, steps, warmup, local, main_entry):
    """Round latency (median/p10/p90), tokens/s and layer roofline fraction of the other workloads."""
    out = {"3": main_entry}
    dev = f"cuda:{local}"
    stream = torch.cuda.current_stream()

    def one(key, rnd, dr):
        for _ in range(max(warmup, 3)):
            dr.run()
        ms = step_times(torch, dr.run, stream, steps)
        if dr.status() != 0:
            raise RuntimeError(f"workload {key}: device status {dr.status():#x}")
        st = latency_stats(ms)
        out[str(key)] = {"workload": WORKLOAD_NAMES[key], "T": rnd.T, "T_cap": rnd.T_cap,
                         "tokens_per_s": rnd.T / (st["median"] / 1e3), "round_ms": st,
                         "layer_roofline": layer_roofline(RL, rnd, st["median"], peaks)}

    for wid in (1, 2):
        rnd = wl.make_round(wid)
        one(wid, rnd, DeviceRound(rnd, device=dev))
    ra = wl.make_round(4)
    dra = DeviceRound(ra, device=dev)
    one("4A", ra, dra)
    rb = wl.make_resume_round(ra)
    one("4B", rb, DeviceRound(rb, device=dev, resume_from=dra))
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads' lines")
    ap.add_argument("--no-block", action="store_true",
                    help="skip the hybrid block timing (pointwise block on the question rows vs every row)")
    ap.add_argument("--no-forest", action="store_true", help="skip the one-round token-forest line")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the short-request round timed eagerly and as one CUDA graph replay")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    ws, rank, local = _dist()
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from tree_forked_hybrid_gb300 import build as B
    B.build()
    from tree_forked_hybrid_gb300 import fork as F
    from tree_forked_hybrid_gb300 import workloads as wl
    from tree_forked_hybrid_gb300 import roofline as RL
    from tree_forked_hybrid_gb300.runner import DeviceRound

    # one round; with N GPUs it holds N times the requests and each rank runs its shard
    # (requests balanced by tokens; no exchange on the data path, the option
    # probabilities are gathered to rank 0 afterwards)
    shard = None
    if ws > 1:
        from tree_forked_hybrid_gb300 import shard as S
        shapes = wl.draw_round_shapes(WORKLOAD_ID, ws, seed=WORKLOAD_ID)
        req, P, n, ql, no, qids = S.shard_shapes(*shapes, ws, rank)
        rnd = wl.make_round(WORKLOAD_ID, seed=WORKLOAD_ID + 1000 * rank, trunk_len=P, n_q=n, q_len=ql, n_opt=no)
        shard = {"shapes": shapes, "qids": qids, "requests": req}
    else:
        rnd = wl.make_round(WORKLOAD_ID)
    dr = DeviceRound(rnd, device=f"cuda:{local}")
    stream = torch.cuda.current_stream()
    calls = [("meta", dr.step_meta)] + [(f"attn_{a.name}", (lambda n=a.name: dr.step_attn(n)))
                                        for a in rnd.attn_shapes]
    calls += [("gdn_trunk", dr.step_gdn_trunk), ("gdn_branches", dr.step_gdn_branches),
              ("readout", dr.step_readout)]
    for _ in range(max(args.warmup, 3)):
        dr.run()
    torch.cuda.synchronize()
    if dr.status() != 0:
        raise RuntimeError(f"device status {dr.status():#x}")
    if dist:
        dist.barrier()
    sampler = ClockSampler(_gpu_uuid(torch, local))
    time.sleep(0.3)
    dr.run()  # one more untimed step after the idle wait for the sampler
    ev = {name: [] for name, _ in calls}
    step_ev = _events(torch, args.steps + 1)
    torch.cuda.synchronize()
    w0 = time.time()
    step_ev[0].record(stream)
    for i in range(args.steps):
        for name, fn in calls:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ev[name].append((e0, e1))
        step_ev[i + 1].record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    sampler.stop()
    elapsed_ms, tokens_all = aggregate_over_ranks(torch, dist, f"cuda:{local}", step_ev[0].elapsed_time(step_ev[-1]),
                                                  rnd.T)
    step_ms = [step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(args.steps)]
    per_call = {name: statistics.mean(a.elapsed_time(b) for a, b in lst) for name, lst in ev.items()}
    kernel_alone = attn_kernel_alone(torch, dr, rnd, stream)
    value = tokens_all * args.steps / (elapsed_ms / 1e3)
    ms_per_step = elapsed_ms / args.steps

    peaks = _peaks()
    work = RL.round_work(rnd)
    # dominant call and its roofline; the timed region lasts well under a second, so the
    # tensor-core peak is the burst one (the sustained figure is reported beside it)
    top = max(per_call, key=per_call.get)
    if top.startswith("attn_"):
        f = work["attn"][top[5:]]["flops"]
        ach = f / (per_call[top] / 1e3) / 1e12
        traffic = _traffic() if top == "attn_attn" else None
        roof = {"kernel": f"fork_attn ({top[5:]}): rotary tables, key rotation, attn_tc_kernel",
                "bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"], "traffic": traffic,
                "traffic_unit": "bytes per call (all launches of the call)",
                "peak_note": f"bf16 dense burst ({peaks['source']}): the timed region lasts "
                             f"{elapsed_ms:.0f} ms",
                "frac_of_sustained": ach / peaks["bf16_tflops_sustained"]}
        if top == "attn_attn" and kernel_alone:
            ka = f / (kernel_alone / 1e3) / 1e12
            roof["kernel_alone"] = {"kernel": "fork_attn without the rotary embedding: fp16 values and "
                                              "attn_tc_kernel (same round: the same visible pairs and FLOPs)",
                                    "ms": kernel_alone, "achieved": ka, "peak": peaks["bf16_tflops"],
                                    "frac": ka / peaks["bf16_tflops"],
                                    "peak_note": f"bf16 dense burst ({peaks['source']}); timed alone after the "
                                                 "timed region"}
    else:
        key = "gdn" if top.startswith("gdn") else "readout"
        b = work[key]["bytes"]
        ach = b / (per_call[top] / 1e3) / 1e9
        roof = {"kernel": top, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "traffic": None, "peak_note": f"HBM copy ({peaks['source']})"}
    main_lat = latency_stats(step_ms)
    main_entry = {"workload": WORKLOAD_NAMES[3], "T": rnd.T, "T_cap": rnd.T_cap,
                  "tokens_per_s": rnd.T / (main_lat["median"] / 1e3), "round_ms": main_lat,
                  "layer_roofline": layer_roofline(RL, rnd, ms_per_step, peaks)}
    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": _config(rnd),
           "roofline": roof,
           "layer_roofline": dict(main_entry["layer_roofline"],
                                  peaks=f"{peaks['bf16_tflops']} TFLOP/s bf16 burst, {peaks['hbm_gbs']} GB/s "
                                        f"({peaks['source']})"),
           "round_ms": main_lat,
           "per_call_us": {k: v * 1e3 for k, v in per_call.items()},
           "gpu_launches": dr.launches_per_round() * args.steps,
           "clocks": sampler.summary(w0, w1)}

    # FORK_DETERMINISTIC: the same round with the flag (every kernel is composition-invariant
    # by construction, so the flag selects the same kernels)
    det = DeviceRound(rnd, device=f"cuda:{local}", flags=F.FORK_DETERMINISTIC)
    for _ in range(3):
        det.run()
    det_ms = latency_stats(step_times(torch, det.run, stream, args.steps))
    out["deterministic"] = {"round_ms": det_ms, "cost_vs_default": det_ms["median"] / main_lat["median"] - 1.0,
                            "identical_outputs": bool(torch.equal(det.gdn_out, dr.gdn_out) and
                                                      all(torch.equal(det.attn_out[n], dr.attn_out[n])
                                                          for n in dr.attn_out) and torch.equal(det.p, dr.p))}
    del det
    if not args.no_e2e:
        out["e2e"] = e2e(torch, dr, rnd, args, stream, dist, local, ws)
    if not args.no_configs and ws == 1:
        try:
            out["per_config"] = per_config(torch, RL, wl, DeviceRound, peaks, args.steps, args.warmup, local,
                                           main_entry)
        except Exception as exc:  # reported, never fatal for the main line
            out["per_config"] = {"error": f"{type(exc).__name__}: {exc}"}
    if not args.no_block and ws == 1:
        try:
            out["hybrid_block"] = hybrid_block_timing(torch, dr, rnd, stream, peaks)
        except Exception as exc:  # reported, never fatal for the main line
            out["hybrid_block"] = {"error": f"{type(exc).__name__}: {exc}"}
    if not args.no_graph and ws == 1:
        try:
            out["graph_replay"] = graph_timing(torch, args, local)
        except Exception as exc:  # reported, never fatal for the main line
            out["graph_replay"] = {"error": f"{type(exc).__name__}: {exc}"}
    if not args.no_forest and ws == 1:
        try:
            out["forest"] = forest_timing(torch, args, local, peaks)
        except Exception as exc:  # reported, never fatal for the main line
            out["forest"] = {"error": f"{type(exc).__name__}: {exc}"}
    if shard is not None:
        out["sharding"] = gather_shards(dist, dr, rnd, shard, rank, ws)
        out["config"]["sharding"] = (f"one round of {shard['shapes'][0].shape[0]} requests "
                                     f"({int(shard['shapes'][0].sum() + shard['shapes'][2].sum())} tokens) split at "
                                     f"request boundaries over {ws} GPUs; per-rank values drawn from the rank's seed")
    if rank == 0 and ws == 1 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(rnd)
    if rank == 0:
        print(json.dumps(out))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def gather_shards(dist, dr, rnd, shard, rank, ws):
    """Gather every rank's option probabilities to rank 0 in the whole round's layout and
    check each question's distribution sums to one."""
    from tree_forked_hybrid_gb300 import shard as S
    P, n, ql, no = shard["shapes"]
    p = dr.p[:int(rnd.opt_off[-1])].cpu().numpy()
    parts = [None] * ws
    dist.all_gather_object(parts, (shard["qids"], p))
    if rank != 0:
        return None
    whole = type("WholeRound", (), {})()
    whole.Nq = int(ql.shape[0])
    whole.n_opt = no
    whole.opt_off = np.concatenate([[0], np.cumsum(no)]).astype(np.int64)
    pall = S.scatter_probabilities(whole, parts)
    sums = np.add.reduceat(pall, whole.opt_off[:-1]) if whole.Nq else np.zeros(0)
    return {"requests": int(P.shape[0]), "questions": whole.Nq,
            "rank_requests": [len(x[0]) for x in parts],
            "max_abs_sum_minus_1": float(np.abs(sums - 1.0).max()) if whole.Nq else 0.0}


def hybrid_block_timing(torch, dr, rnd, stream, peaks, reps=5):
    """The last layer's pointwise block on the question rows only (fork_readout_mlp, the
    selective readout) against the same block on every stream row (fork_pointwise_rows,
    then eq. (1) from the questions' rows): CUDA-event times of the block alone and of the
    hybrid block (GDN mixer calls + block), and the readout block's HBM roofline fraction
    (its weight bytes)."""
    from tree_forked_hybrid_gb300 import fork as F
    from tree_forked_hybrid_gb300 import workloads as wl
    D = rnd.D
    Fw = 2 * D
    wts = wl.readout_block_weights(D, Fw)
    dev = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dr.device)
    W = {k: dev(v) for k, v in wts.items()}
    ws = torch.empty(F.fork_readout_mlp_workspace_bytes(dr.max_q, D, Fw), dtype=torch.uint8, device=dr.device)
    wsa = torch.empty(F.fork_pointwise_rows_workspace_bytes(rnd.T_cap, D, Fw), dtype=torch.uint8, device=dr.device)
    z = torch.empty((rnd.T_cap, D), dtype=torch.bfloat16, device=dr.device)
    p_sel = torch.empty_like(dr.p)
    p_all = torch.empty_like(dr.p)

    def selective():
        F.fork_readout_mlp(dr.meta, dr.gdn_out, D, Fw, W["g1"], W["w_gate"], W["w_up"], W["w_down"], W["g2"],
                           dr.w_opt, dr.opt_off, p_sel, ws, 0, stream)

    def all_rows():
        F.fork_pointwise_rows(dr.meta, dr.gdn_out, D, Fw, W["g1"], W["w_gate"], W["w_up"], W["w_down"], W["g2"],
                              z, wsa, 0, stream)
        F.fork_readout(dr.meta, z, D, dr.w_opt, dr.opt_off, p_all, 0, stream)

    def mixer():
        dr.step_gdn_trunk(stream)
        dr.step_gdn_branches(stream)

    def timed(fn):
        for _ in range(2):
            fn()
        return latency_stats(step_times(torch, fn, stream, reps))["median"]

    t_sel, t_all, t_mix = timed(selective), timed(all_rows), timed(mixer)
    if dr.status() != 0:
        raise RuntimeError(f"device status {dr.status():#x}")
    off = rnd.opt_off
    a, b = p_sel.cpu().numpy(), p_all.cpu().numpy()
    tv = max(0.5 * float(np.abs(a[off[i]:off[i + 1]] - b[off[i]:off[i + 1]]).sum()) for i in range(rnd.Nq)) \
        if rnd.Nq else 0.0
    nbytes = 3 * D * Fw * 2 + rnd.Nq * D * 2 + int(off[-1]) * D * 2
    gbs = nbytes / (t_sel / 1e3) / 1e9
    return {"block": f"pre-norm SwiGLU MLP + residual + final RMSNorm, D={D}, F={Fw}; Nq={rnd.Nq} question rows "
                     f"of T={rnd.T}",
            "selective_block_ms": t_sel, "all_rows_block_ms": t_all,
            "hybrid_selective_ms": t_mix + t_sel, "hybrid_all_rows_ms": t_mix + t_all,
            "saving": 1.0 - (t_mix + t_sel) / (t_mix + t_all), "tv_selective_vs_all_rows": tv,
            "selective_hbm": {"bytes": nbytes, "achieved_gbs": gbs, "frac": gbs / peaks["hbm_gbs"]}}


def graph_timing(torch, args, local, wid=1):
    """Round latency of the short-request round (32 requests, 14.9k tokens): the layer's
    calls launched one by one, and the same round replayed from the capacity-bucket graph
    pool (smallest bucket that holds it; the copy of the round's inputs into the bucket
    is not timed)."""
    from tree_forked_hybrid_gb300 import workloads as wl
    from tree_forked_hybrid_gb300.runner import DeviceRound, GraphPool
    rnd = wl.make_round(wid)
    dr = DeviceRound(rnd, device=f"cuda:{local}")
    pool = GraphPool(rnd.attn_shapes, rnd.gdn_shape, buckets=(4096, 8192, 16384, 32768), max_req=64, max_q=256,
                     max_opts=2048, device=f"cuda:{local}")
    cr, graph = pool.bucket_for(rnd)
    cr.load(rnd)
    stream = torch.cuda.current_stream()
    eager = latency_stats(step_times(torch, dr.run, stream, max(args.steps, 20)))
    for _ in range(3):
        graph.replay()
    replay = latency_stats(step_times(torch, graph.replay, stream, max(args.steps, 20)))
    if cr.status() != 0 or dr.status() != 0:
        raise RuntimeError("device status set")
    same = bool(torch.equal(cr.p[:int(rnd.opt_off[-1])], dr.p[:int(rnd.opt_off[-1])]))
    return {"workload": f"short requests: R={rnd.R}, T={rnd.T}, Nq={rnd.Nq}", "bucket_T_cap": cr.T_cap,
            "eager_ms": eager, "graph_ms": replay, "launches_per_round": dr.launches_per_round(),
            "same_probabilities": same}


def forest_timing(torch, args, local, peaks):
    """Request trees that fork twice, run as one round of one flat stream: 2 requests with
    the long-document layer shapes, each a 4096-token trunk with 4 branches of 512 tokens
    and 4 questions of 64 tokens on every branch (42 nodes, 3 depths, 14,336 tokens).
    Timed with the metadata resident (one attention call per layer, one recurrence call
    per depth, the readout) and with the host plan and its copy in every round."""
    from tree_forked_hybrid_gb300 import workloads as wl
    from tree_forked_hybrid_gb300.runner import ForestRound
    w = wl.WORKLOADS[WORKLOAD_ID]
    parent, node_len = wl.request_forest(2, (4096, 512, 64), (4, 4))
    t = wl.make_tree_round(parent, node_len, attn_shapes=w.attn, gdn_shape=w.gdn, seed=21)
    fr = ForestRound(t, device=f"cuda:{local}")
    stream = torch.cuda.current_stream()
    for _ in range(3):
        fr.run()
    steps = max(args.steps, 10)
    layers = latency_stats(step_times(torch, lambda: fr.run(meta=False), stream, steps))
    with_plan = latency_stats(step_times(torch, fr.run, stream, steps))
    if fr.status() != 0:
        raise RuntimeError(f"device status {fr.status():#x}")
    T = int(node_len.sum())
    res = {"workload": "2 request trees: trunk 4096, 4 branches x 512, 4 questions x 64 per branch",
           "nodes": t.N, "levels": fr.plan.levels, "tokens": T, "round_ms": layers,
           "round_with_plan_ms": with_plan, "tokens_per_s": T / (layers["median"] / 1e3),
           "gpu_launches_per_round": fr.launches_per_run()}
    try:
        from tree_forked_hybrid_gb300 import roofline as RL
        work = RL.forest_work(t)
        t_f = work["flops"] / (peaks["bf16_tflops"] * 1e12)
        t_b = work["bytes"] / (peaks["hbm_gbs"] * 1e9)
        t_roof = max(t_f, t_b)
        res["layer_roofline"] = {"t_roof_us": t_roof * 1e6, "frac": t_roof / (layers["median"] / 1e3),
                                 "bound": "tensor" if t_f >= t_b else "hbm", "flops": work["flops"],
                                 "bytes": work["bytes"]}
    except Exception as exc:  # the timing above stands without it
        res["layer_roofline"] = {"error": f"{type(exc).__name__}: {exc}"}
    return res


def attn_kernel_alone(torch, dr, rnd, stream, reps=10):
    """Mean duration (ms) of the full-attention layer's call without the rotary
    embedding: the value conversion to fp16 and attn_tc_kernel, which does the same
    visible-pair work as in the step.  Writes a scratch output."""
    import math
    from tree_forked_hybrid_gb300 import fork as F
    a = [x for x in rnd.attn_shapes if x.window == 0]
    if not a:
        return None
    a = a[0]
    inp = dr.inputs[a.name]
    out = torch.empty_like(dr.attn_out[a.name])
    nb = F.fork_attn_workspace_bytes(rnd.T_cap, 0, a.Hq, a.Hkv, a.d, 0.0, dr.flags)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=dr.device) if nb else None

    def call():
        F.fork_attn(dr.meta, inp["q"], inp["k"], inp["v"], out, a.Hq, a.Hkv, a.d, a.window, 0.0,
                    1.0 / math.sqrt(a.d), None, None, ws, dr.flags, stream)

    for _ in range(3):
        call()
    evs = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.mean(x.elapsed_time(y) for x, y in evs)


def e2e(torch, dr, rnd, args, stream, dist, local, ws, n_copy_streams=4):
    """Same metric through the public API with host buffers: every step copies the round's
    inputs from pinned host memory, runs the layer and reads the option probabilities back.
    Steps are pipelined as a server would run them: two device buffer sets take turns, so
    step s+1's copies (spread over several copy streams) run while step s computes; a copy
    into a buffer set waits until the step that last read it has finished."""
    from tree_forked_hybrid_gb300.runner import DeviceRound
    T = rnd.T
    rounds = [dr, DeviceRound(rnd, max_req=dr.max_req, max_q=dr.max_q, flags=dr.flags)]

    def dev_tensors(d):
        out = []
        for name, lay in d.inputs.items():
            for k, t in lay.items():
                out.append(t if k == "conv_w" else t[:T])
        return out + [d.desc, d.w_opt, d.opt_off]

    devs = [dev_tensors(d) for d in rounds]
    host = []
    for t in devs[0]:
        hp = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        hp.copy_(t.cpu())
        host.append(hp)
    h2d = sum(hp.numel() * hp.element_size() for hp in host)
    # largest copies first, each to the least loaded copy stream
    cstreams = [torch.cuda.Stream() for _ in range(n_copy_streams)]
    load = [0] * n_copy_streams
    which = [0] * len(host)
    for i in sorted(range(len(host)), key=lambda i: -host[i].numel() * host[i].element_size()):
        j = load.index(min(load))
        which[i] = j
        load[j] += host[i].numel() * host[i].element_size()
    p_host = [torch.empty(d.p.shape, dtype=d.p.dtype, pin_memory=True) for d in rounds]
    d2h = p_host[0].numel() * p_host[0].element_size()
    free = [None, None]  # per buffer set: the compute of the step that last read it is done

    def copies(b, after):
        done = []
        for j, cs in enumerate(cstreams):
            cs.wait_event(after)
            with torch.cuda.stream(cs):
                for i, hp in enumerate(host):
                    if which[i] == j:
                        devs[b][i].copy_(hp, non_blocking=True)
            e = torch.cuda.Event()
            e.record(cs)
            done.append(e)
        return done

    def step(s, start):
        b = s % 2
        ready = copies(b, free[b] if free[b] is not None else start)
        for e in ready:
            stream.wait_event(e)
        rounds[b].run(stream)
        p_host[b].copy_(rounds[b].p, non_blocking=True)
        f = torch.cuda.Event()
        f.record(stream)
        free[b] = f

    def run_steps(n):
        start = torch.cuda.Event()
        start.record(stream)
        for s in range(n):
            step(s, start)

    run_steps(max(args.warmup, 3))
    torch.cuda.synchronize()
    free[0] = free[1] = None
    if dist:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(args.steps):
        step(s, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    ms, tokens_all = aggregate_over_ranks(torch, dist, f"cuda:{local}", e0.elapsed_time(e1), T)
    for d in rounds:
        if d.status() != 0:
            raise RuntimeError(f"device status {d.status():#x}")
    # each part of one step timed alone (no overlap): copies, layer, read-back
    parts = []
    for _ in range(min(args.steps, 10)):
        e = _events(torch, 4)
        e[0].record(stream)
        for ev in copies(0, e[0]):
            stream.wait_event(ev)
        e[1].record(stream)
        rounds[0].run(stream)
        e[2].record(stream)
        p_host[0].copy_(rounds[0].p, non_blocking=True)
        e[3].record(stream)
        parts.append(e)
    torch.cuda.synchronize()
    split = [statistics.mean(e[i].elapsed_time(e[i + 1]) for e in parts) for i in range(3)]
    per_step = ms / args.steps
    return {"value": tokens_all * args.steps / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": per_step,
            "split_ms": {"h2d": split[0], "compute": split[1], "d2h": split[2],
                         "note": f"each part timed alone; in the timed steps each step's copies ({n_copy_streams} "
                                 "copy streams) overlap the previous step's layer (two device buffer sets)"}}


if __name__ == "__main__":
    main()
