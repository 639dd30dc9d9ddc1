"""Shared helpers for the GPU parity tests: move a seeded case to the GPU (the pools are
filled by the library's own reshape_and_cache), build the oracle's pools on the CPU (by
the oracle's own scatter), and compare against the stated tolerances."""

from __future__ import annotations

import functools

import torch

import oracle
import paged_kv_attention_gb300 as pa
import workloads

# Tolerances of the hot path: fp32 caches max abs <= 1e-5; bf16 caches (fp32 accumulation)
# max abs <= 2e-2 and mean abs <= 4e-3, against the float64 oracle.
TOL = {torch.float32: dict(max_abs=1e-5, mean_abs=1e-5),
       torch.bfloat16: dict(max_abs=2e-2, mean_abs=4e-3)}


def gpu_pools(case: workloads.PagedCase, dev="cuda"):
    kc, vc = (t.to(dev) for t in case.empty_pools())
    pa.reshape_and_cache(case.key.to(dev), case.value.to(dev), kc, vc, case.slot_mapping.to(dev))
    return kc, vc


def oracle_pools(case: workloads.PagedCase):
    kc, vc = case.empty_pools()
    oracle.reshape_and_cache(case.key, case.value, kc, vc, case.slot_mapping)
    return kc, vc


@functools.lru_cache(maxsize=4)
def named_case(name: str):
    case = workloads.NAMED[name]()
    return case, oracle_pools(case)


def check_close(got: torch.Tensor, want: torch.Tensor, dtype: torch.dtype, rows=None, label=""):
    g = got.detach().double().cpu()
    w = want
    if rows is not None:
        g, w = g[rows], w[rows]
    assert torch.isfinite(g).all(), f"{label}: non-finite output"
    diff = (g - w).abs()
    tol = TOL[dtype]
    mx, mean = diff.max().item(), diff.mean().item()
    assert mx <= tol["max_abs"], f"{label}: max abs {mx:.3e} > {tol['max_abs']}"
    assert mean <= tol["mean_abs"], f"{label}: mean abs {mean:.3e} > {tol['mean_abs']}"
    return mx, mean
