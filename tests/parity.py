"""Comparison helpers shared by the GPU parity tests, the smoke check and the
bench's parity line.  Tolerances for bfloat16 outputs: max-abs <= 2e-2 and
mean-abs <= 2e-3 against the fp64 oracle; additionally relative RMS <= 1e-2
and LSE max-abs <= 1e-3.  The extra two matter at large N: with N(0,1)
inputs the output's own standard deviation is about sqrt(e/N) (0.006 at
72,576 tokens), so max-abs 2e-2 alone would pass a badly wrong result, while
LSE pins the softmax denominator independently of the averaging over V."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import workloads as W

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
REL_RMS = 1e-2
LSE_ABS = 1e-3
MODULATE_REL = 1e-5


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def ordered(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers ordered like the values they encode."""
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    return np.abs(ordered(a_bits) - ordered(b_bits))


def attention_errors(q, k, v, o_gpu: torch.Tensor, heads: int, rows_per_head: int, scale: float,
                     lse_gpu: torch.Tensor | None = None, head_list=None) -> dict:
    """Compare GPU attention (o_gpu [N, H*128] bf16, lse_gpu [H, N]) with the
    oracle on sampled rows of every head (all rows when rows_per_head is 0)."""
    n = q.shape[0]
    o_cpu = o_gpu.detach().cpu()
    lse_cpu = lse_gpu.detach().cpu().numpy() if lse_gpu is not None else None
    worst, total_abs, count, se, sref, lse_worst = 0.0, 0.0, 0, 0.0, 0.0, 0.0
    for h in (head_list if head_list is not None else range(heads)):
        rows = W.sampled_rows(n, h, rows_per_head).numpy()
        o_ref, lse_ref = oracle.attn_rows(q, k, v, h, rows, scale)
        got = o_cpu[rows, h * 128:(h + 1) * 128].to(torch.float64).numpy()
        d = np.abs(got - o_ref)
        worst = max(worst, float(d.max()))
        total_abs += float(d.sum())
        count += d.size
        se += float((d * d).sum())
        sref += float((o_ref * o_ref).sum())
        if lse_cpu is not None:
            lse_worst = max(lse_worst, float(np.abs(lse_cpu[h, rows] - lse_ref).max()))
    return {"max_abs": worst, "mean_abs": total_abs / count, "rel_rms": math.sqrt(se / max(sref, 1e-300)),
            "lse_max_abs": lse_worst if lse_cpu is not None else None}


def assert_attention_ok(err: dict):
    assert err["max_abs"] <= MAX_ABS, err
    assert err["mean_abs"] <= MEAN_ABS, err
    assert err["rel_rms"] <= REL_RMS, err
    if err["lse_max_abs"] is not None:
        assert err["lse_max_abs"] <= LSE_ABS, err
