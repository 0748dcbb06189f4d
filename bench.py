"""Throughput benchmark of the packed-varlen embedding encoder.

One step = one full encoder pass (embedding, 25 layers, pool + L2) over one
packed batch of the throughput sweep at the 32768-token budget, 310m shape,
bf16.  The 20 seeded batches of that size are staged on the device before
the timed region and cycled through.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the only reference this project has)
on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "encoded tokens/sec (packed varlen, bf16) at 310m shape; % of tensor peak"
UNIT = "tokens/s"
SHAPE_NAME = "310m-shape encoder (25 layers, hidden 768, 12 heads, GeGLU 3072)"
# workload name -> (tokens per batch, description); sweep32k is the headline
WORKLOADS = {
    "sweep32k": (32768, "packed sweep batches of 32768 tokens (log-uniform text lengths 8-1024)"),
    "sweep8k": (8192, "packed sweep batches of 8192 tokens (log-uniform text lengths 8-1024)"),
    "sweep2k": (2048, "packed sweep batches of 2048 tokens (log-uniform text lengths 8-1024)"),
    "long": (65536, "long documents: 8 texts of 8192 tokens"),
}
BUDGET = 32768


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-leg", type=float, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only the chosen workload (not the sweep's other sizes and the long documents)")
    ap.add_argument("--workload", default="sweep32k", choices=sorted(WORKLOADS))
    ap.add_argument("--output", default="pooled", choices=["pooled", "tokens"],
                    help="pooled: one unit vector per text (the headline); tokens: one per token")
    ap.add_argument("--proj-dim", type=int, default=128,
                    help="with --output tokens: width of the per-token projection (0 = none)")
    ap.add_argument("--norms", action="store_true", help="enable the embedding and final LayerNorms")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# DRAM bytes (read + write) per GEMM launch, the mean over the four projections,
# from one ncu capture of each projection at 32768 tokens.  Valid only for the
# kernel sources with this digest; otherwise reported as null.
GEMM_TRAFFIC_BYTES = 233.97e6
GEMM_TRAFFIC_SOURCES = ['text_embedding_encoder_gb300/csrc/k_gemm_tc.cu', 'text_embedding_encoder_gb300/csrc/tc_ptx.cuh', 'text_embedding_encoder_gb300/csrc/gemm_tc.cuh']
GEMM_TRAFFIC_DIGEST = "79dbd9b2c7257d5b"


def gemm_traffic():
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return GEMM_TRAFFIC_BYTES if h.hexdigest()[:16] == GEMM_TRAFFIC_DIGEST else None


def gemm_flops_per_token(shape, tokens_out=False):
    H, I = shape.hidden, shape.intermediate
    proj = 2.0 * H * shape.proj_dim if tokens_out else 0.0
    return 2.0 * (3 * H * H + H * H + 2 * I * H + I * H) * shape.n_layers + proj


# ---------------------------------------------------------------------------
# CPU legs (the oracle; only here and in the tests)
# ---------------------------------------------------------------------------

def cpu_oracle_sample(seconds_budget: float, threads: int):
    """Encode texts of sweep batch 0 with the oracle until the time budget is
    used; returns (tokens/s, tokens, seconds, texts)."""
    import numpy as np  # noqa: F401
    import oracle
    from text_embedding_encoder_gb300 import synth
    shape = synth.RURI_310M
    w = synth.make_weights(shape, seed=0)
    model = oracle.OracleModel(w, shape, "bf16")
    ids, cu = synth.sweep_batch(BUDGET, 0, shape.vocab)
    tokens, texts = 0, 0
    t0 = time.perf_counter()
    for j in range(len(cu) - 1):
        oracle.encode_text(ids[cu[j]:cu[j + 1]], model)
        tokens += int(cu[j + 1] - cu[j])
        texts += 1
        if time.perf_counter() - t0 >= seconds_budget:
            break
    dt = time.perf_counter() - t0
    return tokens / dt, tokens, dt, texts


def run_cpu_leg_subprocess(seconds_budget: float):
    """Run the oracle leg in a fresh interpreter with a fixed BLAS thread count."""
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    env = dict(os.environ, OPENBLAS_NUM_THREADS=str(threads), OMP_NUM_THREADS=str(threads),
               MKL_NUM_THREADS=str(threads), CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-leg", str(seconds_budget)],
                       capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(f"cpu leg failed: {r.stderr[-2000:]}")
    d = json.loads(r.stdout.strip().splitlines()[-1])
    d["cores"] = threads
    return d


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def make_batches(workload, vocab, rank=0, world=1):
    """The 20 seeded batches of a workload; rank r takes batches r, r+N, ..."""
    from text_embedding_encoder_gb300 import synth
    budget, _ = WORKLOADS[workload]
    batches = []
    for b in range(rank, synth.SWEEP_BATCHES * world, world):
        if workload == "long":
            ids, cu = synth.make_batch(synth.LONG_DOC_LENGTHS, vocab, seed=b)
        else:
            ids, cu = synth.sweep_batch(budget, b % synth.SWEEP_BATCHES + (b // synth.SWEEP_BATCHES) * 100, vocab)
        batches.append((ids, cu))
    return batches


def stage(batches, tokens_out, width):
    """Inputs resident in HBM before any timed region: (d_ids, d_cu, h_cu, d_out) per batch."""
    import torch
    out = []
    for ids, cu in batches:
        rows = len(ids) if tokens_out else len(cu) - 1
        out.append((torch.from_numpy(ids).cuda(), torch.from_numpy(cu).cuda(), cu,
                    torch.empty(rows, width, device="cuda")))
    return out


def measure(enc, d_batches, steps, warmup, tokens_out, dist=None, clocks=None):
    """W warm-up passes, then two timed regions of K passes each between CUDA
    events on the launching stream (barrier + synchronize on both sides, max
    over ranks): the first un-instrumented (the throughput; clocks sampled
    during it), the second with CUDA events around every launch (per-kernel
    split, launch count, rooflines).  Returns (ms, ms_profiled, prof, clk)."""
    import torch
    stream = torch.cuda.current_stream().cuda_stream
    encode_device = enc.encode_tokens_device if tokens_out else enc.encode_device

    def step(i):
        d_ids, d_cu, h_cu, d_out = d_batches[i % len(d_batches)]
        encode_device(d_ids, d_cu, h_cu, d_out, stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()

    def timed_region(profile: bool):
        enc.profile_enable(profile)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        ev0.record()
        for i in range(steps):
            step(i)
        ev1.record()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        t_ms = ev0.elapsed_time(ev1)
        if dist:
            t = torch.tensor([t_ms], device="cuda")
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            t_ms = float(t.item())
        return t_ms

    if clocks:
        clocks.start()
    ms = timed_region(profile=False)
    clk = clocks.stop() if clocks else None
    ms_profiled = timed_region(profile=True)
    prof = enc.profile_read()
    enc.profile_enable(False)
    return ms, ms_profiled, prof, clk


def gemm_rate(prof):
    """Algorithmic GEMM FLOPs of the profiled steps / their summed CUDA-event durations (TFLOP/s)."""
    g = prof["gemm"]
    if not g["launches"] or g["total_ms"] <= 0:
        return None
    return g["flops"] / (g["total_ms"] / 1e3) / 1e12


def hbm_rates(prof, peak_gbs):
    """Algorithmic HBM bytes / summed CUDA-event durations of the memory-bound kernel classes."""
    out = {}
    names = {"layernorm": "layernorm_kernel (both LayerNorms of every layer)",
             "embed": "embed_kernel + positions_kernel", "pool": "pool_fused_kernel (mean-pool + L2)"}
    for k, desc in names.items():
        v = prof.get(k, {})
        if v.get("launches") and v["total_ms"] > 0 and v["bytes"] > 0:
            gbs = v["bytes"] / (v["total_ms"] / 1e3) / 1e9
            out[k] = {"kernel": desc, "achieved": round(gbs, 1), "peak": peak_gbs, "unit": "GB/s",
                      "frac": round(gbs / peak_gbs, 4), "launches": v["launches"],
                      "bytes_per_launch": round(v["bytes"] / v["launches"], 1),
                      "us_per_launch": round(1e3 * v["total_ms"] / v["launches"], 2)}
    return out


def run_ours(args):
    import numpy as np
    import torch
    from text_embedding_encoder_gb300 import binding, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    tokens_out = args.output == "tokens"
    shape = synth.Shape(**{**synth.RURI_310M.as_dict(), "emb_norm": args.norms, "final_norm": args.norms,
                           "proj_dim": args.proj_dim if tokens_out else 0})

    budget, desc = WORKLOADS[args.workload]
    batches = make_batches(args.workload, shape.vocab, rank, world)
    # the other workloads of the sweep, timed in the same run (one GPU only)
    extra = [w for w in ("sweep2k", "sweep8k", "long") if w != args.workload] if world == 1 and not args.no_extra else []
    extra_batches = {w: make_batches(w, shape.vocab) for w in extra}
    max_tokens = max([budget] + [WORKLOADS[w][0] for w in extra])
    max_texts = max(len(cu) - 1 for bl in [batches] + list(extra_batches.values()) for _, cu in bl)
    weights = synth.make_weights(shape, seed=0)
    enc = binding.Encoder(shape, "bf16", max_tokens=max_tokens, max_texts=max_texts, device=local)
    enc.load_weights(weights)
    del weights

    width = enc.token_width if tokens_out else shape.hidden   # columns of one output row
    d_batches = stage(batches, tokens_out, width)
    ms, ms_profiled, prof, clk = measure(enc, d_batches, args.steps, args.warmup, tokens_out, dist,
                                         ClockSampler(local))
    tokens_per_rank = budget * args.steps
    value = tokens_per_rank * world / (ms / 1e3)

    # end to end through the public host API: pinned host inputs, H2D inside,
    # D2H of the embeddings inside, synchronous call per step
    pinned = []
    for ids, cu in batches:
        pi = torch.from_numpy(ids).pin_memory()
        pc = torch.from_numpy(cu).pin_memory()
        po = torch.empty(len(ids) if tokens_out else len(cu) - 1, width).pin_memory()
        pinned.append((pi, pc, po, len(cu) - 1))
    lib = enc.lib
    encode_host = lib.tee_encode_tokens if tokens_out else lib.tee_encode
    for i in range(2):
        pi, pc, po, n = pinned[i % len(pinned)]
        enc.check(encode_host(enc.ctx, pi.data_ptr(), pc.data_ptr(), n, po.data_ptr()))
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    h2d = d2h = 0
    for i in range(args.steps):
        pi, pc, po, n = pinned[i % len(pinned)]
        enc.check(encode_host(enc.ctx, pi.data_ptr(), pc.data_ptr(), n, po.data_ptr()))
        h2d += pi.numel() * 4 + pc.numel() * 4
        d2h += po.numel() * 4
    e2e_s = time.perf_counter() - t0
    if dist:
        t = torch.tensor([e2e_s], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_s = float(t.item())
    e2e_value = tokens_per_rank * world / e2e_s
    del pinned

    pk = peaks()
    achieved_tflops = gemm_rate(prof)
    # the GEMM rate comes from CUDA events around each single launch (a kernel
    # timed alone, tens to hundreds of microseconds), so the burst peak applies
    peak = pk["bf16_tflops"]
    launches = sum(v["launches"] for v in prof.values())

    def pct_peak(v, prof_, tokens_step):
        fpt = gemm_flops_per_token(shape, tokens_out) + prof_["attention"]["flops"] / (tokens_step * args.steps)
        return round(100.0 * v * fpt / (pk["bf16_tflops"] * 1e12), 2)

    kernel_share = {k: round(v["total_ms"] / max(1e-9, sum(x["total_ms"] for x in prof.values())), 4)
                    for k, v in prof.items() if v["launches"]}

    result = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights, uniform ids, log-uniform text lengths)",
        "config": {"workload": f"{SHAPE_NAME}, {desc}", "workload_id": args.workload,
                   "global_batch": budget * world, "tokens_per_gpu_step": budget,
                   "texts_per_batch_mean": round(float(np.mean([len(cu) - 1 for _, cu in batches])), 1),
                   "batches": len(batches), "parallelism": f"dp{world} (texts sharded, no collective)",
                   "output": (f"per-token unit vectors, projection {shape.proj_dim or 'none'}" if tokens_out
                              else "one unit vector per text (mean pool + L2)"),
                   "norms": "embedding + final LayerNorm" if args.norms else "none (the page's encoder)",
                   "l2": "inputs larger than L2 (weights 472 MB + activations per pass)"},
        "pct_tensor_peak": pct_peak(value / world, prof, budget),
        "clocks": clk,
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d // args.steps,
                "d2h_bytes_per_step": d2h // args.steps},
        "gpu_launches": launches,
        "profiled_region": {"ms_per_step": round(ms_profiled / args.steps, 4),
                            "note": "a second timed region of the same K steps with CUDA events around every "
                                    "launch; kernel_share, kernel_ms_per_step, gpu_launches and the rooflines "
                                    "come from it"},
        "roofline": {"bound": "tensor", "kernel": "gemm_tc (tcgen05 bf16 projections)",
                     "achieved": round(achieved_tflops, 1) if achieved_tflops else None,
                     "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved_tflops / peak, 4) if achieved_tflops else None,
                     "peak_source": f"{pk['source']} burst bf16 (per-launch CUDA events time each GEMM alone)",
                     "frac_of_sustained": (round(achieved_tflops / pk["bf16_tflops_sustained"], 4)
                                           if achieved_tflops else None),
                     "traffic": gemm_traffic(),
                     "traffic_unit": "bytes per launch (DRAM read + write, ncu)"},
        "roofline_hbm": hbm_rates(prof, pk["hbm_gbs"]),
        "kernel_share": kernel_share,
        "kernel_ms_per_step": {k: round(v["total_ms"] / args.steps, 4) for k, v in prof.items() if v["launches"]},
    }

    if extra:
        # the sweep's other sizes and the long documents, same protocol, same
        # context (its capacity is the largest workload's)
        sampler = ClockSampler(local)
        sampler.start()
        workloads = {}
        for w in extra:
            steps_w = args.steps if w != "long" else max(3, args.steps // 5)
            db = stage(extra_batches[w], tokens_out, width)
            ms_w, _, prof_w, _ = measure(enc, db, steps_w, max(3, args.warmup), tokens_out)
            tok = WORKLOADS[w][0]
            v_w = tok * steps_w / (ms_w / 1e3)
            r_w = gemm_rate(prof_w)
            workloads[w] = {"workload": WORKLOADS[w][1], "value": round(v_w, 1), "unit": UNIT, "steps": steps_w,
                            "ms_per_step": round(ms_w / steps_w, 4), "pct_tensor_peak": pct_peak(v_w, prof_w, tok),
                            "gemm_tflops": round(r_w, 1) if r_w else None,
                            "gemm_frac": round(r_w / peak, 4) if r_w else None,
                            "kernel_ms_per_step": {k: round(v["total_ms"] / steps_w, 4) for k, v in prof_w.items()
                                                   if v["launches"]}}
            del db
        result["workloads"] = workloads
        result["workloads_clocks"] = sampler.stop()

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            leg = run_cpu_leg_subprocess(20.0)
            result["cpu_baseline"] = {"value": round(leg["value"], 2), "unit": UNIT, "cores": leg["cores"],
                                      "kind": "oracle",
                                      "sample": f"{leg['texts']} texts / {leg['tokens']} tokens of sweep batch 0 "
                                                f"(fp64 numpy oracle, bf16-rounded weights), {leg['seconds']:.1f} s"}
        except Exception as e:  # the baseline is reported, not required
            result["cpu_baseline"] = {"value": None, "unit": UNIT, "cores": None, "kind": "oracle",
                                      "sample": f"failed: {e}"[:300]}
    enc.close()
    if dist:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    os.environ.setdefault("OPENBLAS_NUM_THREADS", str(threads))
    import numpy as np
    import oracle
    from text_embedding_encoder_gb300 import synth
    shape = synth.RURI_310M
    w = synth.make_weights(shape, seed=0)
    model = oracle.OracleModel(w, shape, "bf16")
    ids, cu = synth.sweep_batch(BUDGET, 0, shape.vocab)
    lens = np.diff(cu)
    # bounded sample per step: the texts of the batch, in order, one per step
    order = [j for j in range(len(lens)) if lens[j] <= 160] or list(range(len(lens)))

    def step(i):
        j = order[i % len(order)]
        oracle.encode_text(ids[cu[j]:cu[j + 1]], model)
        return int(lens[j])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    tokens = 0
    for i in range(args.steps):
        tokens += step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = tokens / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{SHAPE_NAME}, {WORKLOADS['sweep32k'][1]}",
                                        "workload_id": "sweep32k",
                                        "sample_per_step": "one text (<= 160 tokens) of sweep batch 0"},
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} texts, {tokens} tokens of sweep batch 0"},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse()
    if args.cpu_leg is not None:
        v, tokens, dt, texts = cpu_oracle_sample(args.cpu_leg, int(os.environ.get("OPENBLAS_NUM_THREADS", "0")))
        print(json.dumps({"value": v, "tokens": tokens, "seconds": dt, "texts": texts}))
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
