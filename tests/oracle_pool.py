"""Full-size oracle comparisons spread over host processes (test helper).

The fp64 oracle is plain numpy and its query rows are independent, so a
full-size workload is cut into (head, block of query rows) tasks and run on a
``spawn`` process pool, one single-threaded BLAS per worker.  Each task gets
the seeded bf16 inputs of its head (bit patterns), computes the oracle's
result for its rows, compares it with the CUDA path's output for the same
rows, and returns only error statistics; the caller combines them into the
maximum and the mean over every element of the output.

Nothing here touches the GPU or torch: the caller hands over host arrays.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

import synth
from oracle import attention as oatt
from oracle import fp8 as ofp8
from oracle import prologue as opro

_BLAS_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _stats(o_ref, lse_ref, o_gpu, lse_gpu, tol=None):
    """Error statistics of one task's rows against the oracle."""
    err = np.abs(o_gpu - o_ref)
    out = {"max": float(err.max()), "sum": float(err.sum()), "n": int(err.size),
           "finite": bool(np.all(np.isfinite(o_gpu))),
           "lse_max": float(np.abs(lse_gpu - lse_ref).max())}
    if tol is not None:
        out["ratio_max"] = float((err / tol).max())
    return out


def _exact_task(t):
    """Exact attention: from raw q/k through the oracle prologue ("e2e"), or
    from the CUDA prologue's own q-hat/k-hat ("attn")."""
    rows = np.arange(t["r0"], t["r1"])
    cu, pos = t["cu"], t["pos"]
    if t["kind"] == "e2e":
        q = opro.qk_prologue(synth.bf16_bits_to_f64(t["q"]), t["gain_q"], pos[rows], t["eps"])
        k = opro.qk_prologue(synth.bf16_bits_to_f64(t["k"]), t["gain_k"], pos, t["eps"])
    else:
        q = synth.bf16_bits_to_f64(t["q"])
        k = synth.bf16_bits_to_f64(t["k"])
    v = synth.bf16_bits_to_f64(t["v"])
    o, lse = oatt.attention_rows(q, k, v, cu, t["scale"], [0], rows)
    return _stats(o, lse[0], synth.bf16_bits_to_f64(t["o"]), t["lse"])


def _fp8_task(t):
    """FP8 variant: exact attention on the dequantised codes, and the
    per-element bound of the kernel's P rounding."""
    rows = np.arange(t["r0"], t["r1"])
    cu = t["cu"]
    qd, kd, vd = ofp8.dequantize(t["q8"], t["sq"], t["k8"], t["sk"], t["v8"], t["sv"])
    o, lse = oatt.attention_rows(qd, kd, vd, cu, t["scale"], [0], rows)
    qfull = np.zeros_like(kd)
    qfull[rows] = qd
    bound = ofp8.error_bound(qfull, kd, vd, cu, t["scale"], [0], rows)
    tol = bound + 2.0 ** -8 * np.abs(o) + 1e-4
    return _stats(o, lse[0], synth.bf16_bits_to_f64(t["o"]), t["lse"], tol=tol)


def _run_task(t):
    return _fp8_task(t) if t["kind"] == "fp8" else _exact_task(t)


def row_blocks(S: int, rows_per_task: int):
    return [(r0, min(S, r0 + rows_per_task)) for r0 in range(0, S, rows_per_task)]


def run(tasks, workers: int | None = None):
    """Runs the tasks on a spawn pool; returns the combined statistics:
    max and mean absolute error over every compared element, max lse error,
    all outputs finite, and (FP8) the largest error / bound ratio."""
    workers = workers or min(len(tasks), os.cpu_count() or 1)
    saved = {k: os.environ.get(k) for k in _BLAS_VARS}
    for k in _BLAS_VARS:
        os.environ[k] = "1"
    try:
        with mp.get_context("spawn").Pool(workers) as pool:
            parts = pool.map(_run_task, tasks, chunksize=1)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    total = {"max": max(p["max"] for p in parts),
             "mean": sum(p["sum"] for p in parts) / sum(p["n"] for p in parts),
             "n": sum(p["n"] for p in parts),
             "lse_max": max(p["lse_max"] for p in parts),
             "finite": all(p["finite"] for p in parts)}
    if all("ratio_max" in p for p in parts):
        total["ratio_max"] = max(p["ratio_max"] for p in parts)
    return total


def exact_tasks(kind, cu, pos, q_bits, k_bits, v_bits, o_bits, lse, gain_q, gain_k, eps, scale,
                rows_per_task=4096):
    """Tasks over every (head, row block).  q_bits/k_bits/v_bits/o_bits: uint16
    [S, H, 128] bf16 patterns (q/k raw for "e2e", the CUDA prologue's outputs
    for "attn"); lse: fp32 [H, S] from the CUDA path."""
    S, Hh, _ = q_bits.shape
    tasks = []
    for h in range(Hh):
        k_h = np.ascontiguousarray(k_bits[:, h:h + 1])
        v_h = np.ascontiguousarray(v_bits[:, h:h + 1])
        for r0, r1 in row_blocks(S, rows_per_task):
            tasks.append({"kind": kind, "r0": r0, "r1": r1, "cu": cu, "pos": pos,
                          "q": np.ascontiguousarray(q_bits[r0:r1, h:h + 1]), "k": k_h, "v": v_h,
                          "o": np.ascontiguousarray(o_bits[r0:r1, h:h + 1]),
                          "lse": np.asarray(lse[h, r0:r1], dtype=np.float64),
                          "gain_q": np.asarray(gain_q, dtype=np.float64),
                          "gain_k": np.asarray(gain_k, dtype=np.float64), "eps": eps, "scale": scale})
    return tasks


def fp8_tasks(cu, q8, sq, k8, sk, v8, sv, o_bits, lse, scale, rows_per_task=4096):
    """Tasks for the FP8 variant: codes [S, H, 128] uint8 (v8 token-major),
    scales sq, sk [H, S] and sv [H, 128] fp32, the CUDA output o_bits and lse."""
    S, Hh, _ = q8.shape
    tasks = []
    for h in range(Hh):
        for r0, r1 in row_blocks(S, rows_per_task):
            tasks.append({"kind": "fp8", "r0": r0, "r1": r1, "cu": cu,
                          "q8": np.ascontiguousarray(q8[r0:r1, h:h + 1]),
                          "sq": np.ascontiguousarray(sq[h:h + 1, r0:r1]),
                          "k8": np.ascontiguousarray(k8[:, h:h + 1]), "sk": np.ascontiguousarray(sk[h:h + 1]),
                          "v8": np.ascontiguousarray(v8[:, h:h + 1]), "sv": np.ascontiguousarray(sv[h:h + 1]),
                          "o": np.ascontiguousarray(o_bits[r0:r1, h:h + 1]),
                          "lse": np.asarray(lse[h, r0:r1], dtype=np.float64), "scale": scale})
    return tasks
