"""Time each step of the pass on its own, through the C ABI (per-step entry points).

    python profile_steps.py [--tokens 32768] [--reps 10] [--only STEP]

Builds a 310m-shape bf16 context with seeded random weights, stages one
sweep batch of the given token budget, and times every step (LayerNorm, the
four projections, global and window attention, pool) with CUDA events on the
launching stream, reporting ms per launch, TFLOP/s or GB/s.  With --only it
runs just that step (for a profiler capture: ``-k`` on the kernel name).
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
from text_embedding_encoder_gb300 import binding, synth  # noqa: E402

STEPS = ["embed", "layernorm", "qkv", "attn_global", "attn_window", "out_proj", "ffn_in", "ffn_out", "pool"]
PLAIN = ["plain_qkv", "plain_out_proj", "plain_ffn_in", "plain_ffn_out"]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--tokens", type=int, default=32768)
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--only", choices=STEPS + PLAIN, default=None)
    ap.add_argument("--long-docs", action="store_true", help="8 texts of tokens/8 each instead of a sweep batch")
    ap.add_argument("--cublas", action="store_true",
                    help="also time torch.matmul (cuBLAS) on the four projection shapes, for comparison only")
    args = ap.parse_args()

    shape = synth.RURI_310M
    H, I, T = shape.hidden, shape.intermediate, args.tokens
    if args.long_docs:
        ids, cu = synth.make_batch([T // 8] * 8, shape.vocab, seed=0)
    else:
        ids, cu = synth.sweep_batch(T, 0, shape.vocab)
    n = len(cu) - 1
    w = synth.make_weights(shape, seed=0)
    enc = binding.Encoder(shape, "bf16", max_tokens=T, max_texts=max(n, 1))
    enc.load_weights(w)
    del w
    rng = np.random.default_rng(0)
    dev = lambda a, dt=None: (torch.from_numpy(np.ascontiguousarray(a)).to(dt) if dt else  # noqa: E731
                              torch.from_numpy(np.ascontiguousarray(a))).cuda()
    x = dev(rng.standard_normal((T, H)).astype(np.float32))
    y = dev(rng.standard_normal((T, H)).astype(np.float32), torch.bfloat16)
    qkv = dev(rng.standard_normal((T, 3 * H)).astype(np.float32), torch.bfloat16)
    o = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    z = dev(rng.standard_normal((T, I)).astype(np.float32), torch.bfloat16)
    zo = torch.empty(T, I, dtype=torch.bfloat16, device="cuda")
    pos = dev(np.concatenate([np.arange(b - a) for a, b in zip(cu[:-1], cu[1:])]).astype(np.int32))
    d_cu = dev(cu)
    out = torch.empty(n, H, device="cuda")
    qkv_out = torch.empty(T, 3 * H, dtype=torch.bfloat16, device="cuda")
    lens = np.diff(cu).astype(np.float64)
    pairs_g = float((lens ** 2).sum())
    pairs_w = float(sum(sum(min(L - 1, i + 64) - max(0, i - 64) + 1 for i in range(int(L))) for L in lens))

    d_ids = dev(ids)
    steps = {
        "embed": (lambda: enc.op("tee_op_embed", d_ids, T, x, 0), None, T * H * 6.0 + T * 4.0),
        "layernorm": (lambda: enc.op("tee_op_layernorm", 0, 0, x, y, T, 0), None, T * H * 6.0),
        "qkv": (lambda: enc.op("tee_op_qkv", 0, y, pos, qkv_out, T, 0), 2.0 * T * 3 * H * H, None),
        "attn_global": (lambda: enc.op("tee_op_attention", 0, qkv, d_cu, cu, n, o, 0), 3072.0 * pairs_g, None),
        "attn_window": (lambda: enc.op("tee_op_attention", 1, qkv, d_cu, cu, n, o, 0), 3072.0 * pairs_w, None),
        "out_proj": (lambda: enc.op("tee_op_out_proj", 0, o, x, T, 0), 2.0 * T * H * H, T * H * 8.0),
        "ffn_in": (lambda: enc.op("tee_op_ffn_in", 0, y, zo, T, 0), 2.0 * T * 2 * I * H, None),
        "ffn_out": (lambda: enc.op("tee_op_ffn_out", 0, z, x, T, 0), 2.0 * T * H * I, T * H * 8.0),
        "pool": (lambda: enc.op("tee_op_pool_l2", x, d_cu, cu, n, out, 0), None, T * H * 4.0),
    }
    report = {"tokens": T, "texts": n}
    for name in STEPS:
        if args.only and name != args.only:
            continue
        fn, flops, nbytes = steps[name]
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.reps
        row = {"ms": round(ms, 4)}
        if flops:
            row["tflops"] = round(flops / ms / 1e9, 1)
        if nbytes:
            row["gbs"] = round(nbytes / ms / 1e6, 1)
        report[name] = row
    if args.cublas or (args.only or "").startswith("plain_"):
        # this library's GEMM with a plain bf16 store (no fused epilogue) on the same shapes
        for name, (n_out, k_in) in {"qkv": (3 * H, H), "out_proj": (H, H), "ffn_in": (2 * I, H),
                                    "ffn_out": (H, I)}.items():
            if args.only and args.only != "plain_" + name:
                continue
            a = torch.randn(T, k_in, device="cuda", dtype=torch.bfloat16)
            wt = torch.randn(n_out, k_in, device="cuda", dtype=torch.bfloat16)
            c = torch.empty(T, n_out, device="cuda", dtype=torch.bfloat16)
            fn = lambda: enc.op("tee_op_gemm_bf16", a, wt, c, T, n_out, k_in, 0, 0)  # noqa: E731
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.reps
            report["plain_" + name] = {"ms": round(ms, 4), "tflops": round(2.0 * T * n_out * k_in / ms / 1e9, 1)}
    if args.cublas:
        # library reference point: plain bf16 GEMMs of the same shapes (no epilogue fusion)
        for name, (n_out, k_in) in {"qkv": (3 * H, H), "out_proj": (H, H), "ffn_in": (2 * I, H),
                                    "ffn_out": (H, I)}.items():
            a = torch.randn(T, k_in, device="cuda", dtype=torch.bfloat16)
            wt = torch.randn(n_out, k_in, device="cuda", dtype=torch.bfloat16)
            for _ in range(3):
                torch.matmul(a, wt.t())
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(args.reps):
                torch.matmul(a, wt.t())
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.reps
            report["cublas_" + name] = {"ms": round(ms, 4), "tflops": round(2.0 * T * n_out * k_in / ms / 1e9, 1)}
    print(json.dumps(report))
    enc.close()


if __name__ == "__main__":
    main()
