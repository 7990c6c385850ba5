"""Comparison rules between the CUDA path and the oracle.

Floating-point values: |gpu - ref| <= ATOL + RTOL * |ref| (bf16 inputs, fp32 accumulation
against fp64).  Ids are bit-exact, except where the decision is a near-tie that fp32 cannot
settle the way fp64 does:
  - top-k: a differing cluster is excused if its oracle score is within TIE of the k-th;
  - greedy / Gumbel argmax: excused if the oracle keys of the two tokens differ by < TIE;
  - accept / reject: excused if |ln u - (ln p - ln q)| < TIE;
  - inverse-CDF draws: excused if u * R lies within ICDF_TOL * R of the oracle's cumulative
    boundary at the GPU's token.
An excused id ends the comparison of everything downstream of it in that sequence.
"""
from __future__ import annotations

import math

import numpy as np

import oracle

ATOL, RTOL = 1e-2, 1e-3
TIE = 1e-3
ICDF_TOL = 1e-5


def assert_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    err = np.abs(gpu - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance; max err {err.max():.3g}"


def topk_same_or_excused(gpu_ids, scores, k) -> bool:
    """True if identical; False if they differ only at excused near-ties; raises otherwise."""
    g = set(int(x) for x in gpu_ids)
    ref = oracle.topk(scores, k)[0]
    r = set(int(x) for x in ref)
    if g == r:
        return True
    kth = np.sort(np.asarray(scores, np.float64))[::-1][k - 1]
    for c in g ^ r:
        assert abs(scores[c] - kth) < TIE, f"top-k differs at cluster {c} (score {scores[c]}, k-th {kth})"
    return False


def draft_key(l, S, j, T, seed, pos, row):
    if T == 0.0:
        return float(l[j])
    return float(l[j]) / T - math.log(-math.log(oracle.gumbel_uniform(seed, int(j), pos, row)))


def token_same_or_excused(gpu_idx, ref_idx, l, S, T, seed, pos, row) -> bool:
    if gpu_idx == ref_idx:
        return True
    assert 0 <= gpu_idx < len(S), f"GPU token index {gpu_idx} outside the list"
    kg = draft_key(l, S, gpu_idx, T, seed, pos, row)
    kr = draft_key(l, S, ref_idx, T, seed, pos, row)
    assert abs(kg - kr) < TIE, f"draft token differs: gpu idx {gpu_idx} key {kg}, oracle idx {ref_idx} key {kr}"
    return False


def softmax_full(z, T):
    x = np.asarray(z, np.float64) / T
    x = np.exp(x - x.max())
    return x / x.sum()


def q_dense(l, S, T, V):
    x = np.asarray(l, np.float64) / T
    q = np.exp(x - x.max())
    q /= q.sum()
    out = np.zeros(V)
    out[np.asarray(S)] = q
    return out


def icdf_acceptable(w, u, v) -> bool:
    """Is v an inverse-CDF draw of weights w at uniform u, up to ICDF_TOL?"""
    w = np.asarray(w, np.float64)
    R = w.sum()
    c = np.cumsum(w)
    lo = c[v - 1] if v > 0 else 0.0
    return w[v] >= 0 and lo - ICDF_TOL * R <= u * R < c[v] + ICDF_TOL * R


def accept_margin(p, q, u):
    """|ln u - (ln p - ln q)|; inf when p or q is 0 (no near-tie possible)."""
    if p <= 0 or q <= 0:
        return math.inf
    return abs(math.log(u) - (math.log(p) - math.log(q)))
