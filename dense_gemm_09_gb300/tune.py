"""Tile-configuration sweep for the tensor-core calls.

For one problem shape and kind, times the automatic choice and every tile
configuration the library can run -- the CTA-pair kernel, the single-CTA
kernel at each tile width bn, and split-K at each (bn, S) -- and prints them
fastest first, with each result's largest difference from the automatic
choice (relative to max |C|).  This is the search over tile parameters per
problem that "如何优化一个 CUDA Matmul Kernel ... Worklog" runs in "Kernel 9:
Autotuning"; the library's automatic choice is a cost model fitted to such
sweeps.

    python -m dense_gemm_09_gb300.tune --kind f16_tn --shape 127x12288x4096

With --cublas it also times torch.matmul (cuBLAS) on the same operands and
flush, as a context line; cuBLAS is never part of the library's path.

--flush clean (the default, as in bench.py) zeroes a 512 MB buffer and then
reads another 512 MB before every timed call, so the L2 holds none of the
operands and only clean lines.  --flush write only zeroes the buffer, which
leaves the L2 full of dirty lines: the timed call then also pays for their
write-back (~5 us for a 100 MB HBM-bound call on GB300).

Operands are seeded uniform[-1, 1) values on the current GPU; the L2 cache
is flushed before every timed call, and times are means of CUDA-event
intervals (the event clock ticks in steps of about 2 us, so means resolve
finer differences than medians).
"""
from __future__ import annotations

import argparse
import statistics

import torch

import dense_gemm_09_gb300 as dg

KINDS = {
    "f32": (torch.float32, False, dg.gemm_f32, 0),  # SIMT: no tile configurations to sweep
    "tf32": (torch.float32, False, dg.gemm_tf32, 32),
    "f16_tn": (torch.float16, True, dg.gemm_f16_tn, 32),
    "f16_nn": (torch.float16, False, dg.gemm_f16_nn, 64),
    "bf16_tn": (torch.bfloat16, True, dg.gemm_bf16_tn, 32),
    "bf16_nn": (torch.bfloat16, False, dg.gemm_bf16_nn, 64),
}


def configs(step: int, sms: int, M: int, N: int):
    if step == 0:
        return [(dg.TUNE_AUTO, 256, 1)]
    """Every (variant, bn, split) worth timing: the pair kernels (256 x 256
    and 256 x 512 tiles, each round-robin and with the stream-K tail, with
    the ordinary and the finer stage ring; 128 x bn tiles of the small-M
    pair), and for each tile width bn the single-CTA kernel
    and the splits that fit one wave (step 0: the FP32 SIMT call, automatic
    only)."""
    out = [(dg.TUNE_AUTO, 256, 1), (dg.TUNE_PAIR, 256, dg.SK_OFF), (dg.TUNE_PAIR, 256, dg.SK_ON),
           (dg.TUNE_PAIR_WIDE, 256, dg.SK_OFF),
           (dg.TUNE_PAIR_WIDE, 256, dg.SK_ON),
           (dg.TUNE_PAIR_FINE, 256, dg.SK_OFF), (dg.TUNE_PAIR_FINE, 256, dg.SK_ON),
           (dg.TUNE_PAIR_WIDE_FINE, 256, dg.SK_OFF), (dg.TUNE_PAIR_WIDE_FINE, 256, dg.SK_ON),
           (dg.TUNE_PAIR128, 256, 1), (dg.TUNE_PAIR128, 192, 1), (dg.TUNE_PAIR128, 128, 1)]
    tiles_m = (M + 127) // 128
    for bn in range(256, 31, -step):
        out.append((dg.TUNE_SINGLE, bn, 1))
        tiles = tiles_m * ((N + bn - 1) // bn)
        for S in range(2, 9):
            if tiles * S <= sms:
                out.append((dg.TUNE_SPLIT, bn, S))
    return out


def cublas_call(kind: str, A, B, out):
    """The same product through torch.matmul (cuBLAS), for context only: FP32
    with TF32 disabled, TF32 with it enabled, the TN kinds as A @ B^T."""
    tn = KINDS[kind][1]
    torch.backends.cuda.matmul.allow_tf32 = kind == "tf32"
    torch.mm(A, B.t() if tn else B, out=out)


def sweep(kind: str, M: int, N: int, K: int, reps: int = 30, warmup: int = 3, seed: int = 0,
          cublas: bool = False, cublas_only: bool = False, profile_range: bool = False,
          flush_mode: str = "clean"):
    dtype, tn, fn, step = KINDS[kind]
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(seed)
    A = (torch.rand((M, K), generator=g) * 2 - 1).to(dtype).to(dev)
    Bshape = (N, K) if tn else (K, N)
    B = (torch.rand(Bshape, generator=g) * 2 - 1).to(dtype).to(dev)
    C = torch.empty((M, N), dtype=dtype, device=dev)
    flush = torch.empty(512 * 2**20 // 4, device=dev)
    flush_read = torch.ones(512 * 2**20 // 4, device=dev) if flush_mode == "clean" else None
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ref = None
    rows = []
    cases = [] if cublas_only else [(v, bn, sp, None) for v, bn, sp in configs(step, sms, M, N)]
    if cublas or cublas_only:
        cases.append((None, 0, 0, "cublas (torch.matmul, context only)"))
    tf32_flag = torch.backends.cuda.matmul.allow_tf32
    for variant, bn, split, label in cases:
        def call():
            if label:
                cublas_call(kind, A, B, C)
                return
            if variant != dg.TUNE_AUTO:
                dg.tune_next(variant, bn, split)
            fn(A, B, C, 1.0, 0.0)
        for _ in range(warmup):
            call()
        times = []
        for _ in range(reps):
            flush.zero_()
            if flush_read is not None:
                flush_read.sum()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            if profile_range:  # only the timed calls, for `ncu --profile-from-start off`
                torch.cuda.profiler.start()
            call()
            if profile_range:
                torch.cuda.profiler.stop()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        name = label or dg.last_kernel()
        out = C.float()
        if ref is None:
            ref = out.clone()
            scale = max(ref.abs().max().item(), 1e-30)
        diff = (out - ref).abs().max().item() / scale
        ms = statistics.mean(times)
        rows.append((ms, name, variant == dg.TUNE_AUTO, diff))
    torch.backends.cuda.matmul.allow_tf32 = tf32_flag
    assert dg.device_status() == dg.OK
    auto_name = rows[0][1] if not cublas_only else ""
    best = {}  # one line per kernel actually run (a request the call cannot take runs the automatic one)
    for ms, name, _, diff in rows:
        if name not in best or ms < best[name][0]:
            best[name] = (ms, diff)
    return sorted((ms, name, name == auto_name, diff) for name, (ms, diff) in best.items())


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--kind", choices=sorted(KINDS), default="f16_tn")
    ap.add_argument("--shape", required=True, help="MxNxK")
    ap.add_argument("--reps", type=int, default=30)
    ap.add_argument("--cublas", action="store_true",
                    help="also time torch.matmul (cuBLAS) on the same operands, for context")
    ap.add_argument("--cublas-only", action="store_true", help="time only the torch.matmul line")
    ap.add_argument("--profile-range", action="store_true",
                    help="bracket each timed call with the profiler start/stop API, so that "
                         "ncu --profile-from-start off captures those launches and nothing else")
    ap.add_argument("--flush", choices=("clean", "write"), default="clean",
                    help="clean: zero 512 MB, then read another 512 MB before each call (as the bench); "
                         "write: only zero it, leaving dirty lines in L2")
    a = ap.parse_args()
    M, N, K = (int(v) for v in a.shape.lower().split("x"))
    table = sweep(a.kind, M, N, K, reps=a.reps, cublas=a.cublas, cublas_only=a.cublas_only,
                  profile_range=a.profile_range, flush_mode=a.flush)
    flops = 2.0 * M * N * K
    print("%s %dx%dx%d (flush: %s)" % (a.kind, M, N, K, a.flush))
    for ms, name, auto, diff in table:
        print("  %-44s %9.4f ms %9.2f TFLOP/s  max rel diff %.1e%s"
              % (name, ms, flops / ms / 1e9, diff, "   <- automatic" if auto else ""))


if __name__ == "__main__":
    main()
