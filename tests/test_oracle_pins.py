"""Pins of the CPU oracle against things other than itself.

Each test checks one oracle function against an independent route to the same answer:
a library primitive (numpy fp64 matmul, Python's sort, scipy's chi-square), brute force on
tiny inputs, exact rational arithmetic (``fractions``) for the verification rule, or
cuRAND's host-side Philox4x32-10 generator.  They are chosen so that a plausible slip in the
oracle (a dropped bias, the wrong activation, a transposed weight, a wrong tie rule, a wrong
sign in the residual, a temperature applied to one side only) fails at least one of them.
"""
import ctypes
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wl

scipy_stats = pytest.importorskip("scipy.stats")


def _bf16(rng, shape, std):
    return wl.to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(std))


def _f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------------------------------
# Philox4x32-10 against cuRAND's host generator (library routine, runs without a GPU)
# ---------------------------------------------------------------------------------------
def _curand_host_philox(seed: int, n: int, offset: int = 0):
    path = None
    for cand in ("/usr/local/cuda/lib64/libcurand.so", "libcurand.so", "libcurand.so.10"):
        try:
            lib = ctypes.CDLL(cand)
            path = cand
            break
        except OSError:
            continue
    if path is None:
        pytest.skip("libcurand not available")
    gen = ctypes.c_void_p()
    if lib.curandCreateGeneratorHost(ctypes.byref(gen), 161):   # CURAND_RNG_PSEUDO_PHILOX4_32_10
        pytest.skip("cuRAND host generator unavailable")
    assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
    assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
    buf = (ctypes.c_uint32 * n)()
    assert lib.curandGenerate(gen, buf, ctypes.c_size_t(n)) == 0
    lib.curandDestroyGenerator(gen)
    return np.array(buf[:], dtype=np.uint32)


@pytest.mark.parametrize("seed", [0, 1, 0x0123456789ABCDEF, 0xFFFFFFFFFFFFFFFF])
def test_philox_matches_curand_host(seed):
    # cuRAND's host Philox stream for a seed is subsequence-major: block j is
    # Philox(counter (0, 0, j, 0), key (seed_lo, seed_hi)), four words per block.  This
    # exercises all four counter words' paths (words 0 and 2 are multiplied, 1 and 3 xored).
    n = 4 * 256
    ref = _curand_host_philox(seed, n)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    mine = np.concatenate([oracle.philox4x32_10([0, 0, j, 0], key) for j in range(n // 4)])
    assert np.array_equal(mine, ref)


@pytest.mark.parametrize("start", [1 << 16, 77 << 16, 1 << 48, (3 << 48) + (2 << 16) + 5])
def test_philox_counter_words_0_1_match_curand_host(start):
    # Far into the host stream the block index spills into counter words 0 and 1: block j
    # sits at counter ((j >> 16) mod 2^32, j >> 48, j & 0xFFFF, 0).  Starting there with a
    # generator offset of 4 * j words pins the oracle's use of words 0 and 1 as well.
    seed = 0x9E3779B97F4A7C15
    ref = _curand_host_philox(seed, 4 * 32, offset=4 * start)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    blocks = []
    for j in range(start, start + 32):
        blocks.append(oracle.philox4x32_10([(j >> 16) & 0xFFFFFFFF, j >> 48, j & 0xFFFF, 0], key))
    assert np.array_equal(np.concatenate(blocks), ref)


def test_philox_high_counter_words_change_output():
    key = [7, 9]
    base = oracle.philox4x32_10([5, 0, 0, 0], key)
    for w in range(1, 4):
        ctr = [5, 0, 0, 0]
        ctr[w] = 1
        assert not np.array_equal(oracle.philox4x32_10(ctr, key), base)


def test_gumbel_uniform_range_and_uniformity():
    seed = 0xDEADBEEF12345678
    us = np.array([oracle.gumbel_uniform(seed, v, 3, 1) for v in range(40000)])
    assert us.min() > 0.0 and us.max() < 1.0
    # exactly representable in fp32 (odd multiples of 2^-24)
    assert np.all(us.astype(np.float32).astype(np.float64) == us)
    hist, _ = np.histogram(us, bins=40, range=(0, 1))
    _, pval = scipy_stats.chisquare(hist)
    assert pval > 1e-4
    # the list index, position and row all move the draw
    a = oracle.gumbel_uniform(seed, 11, 3, 1)
    assert a != oracle.gumbel_uniform(seed, 11, 4, 1)
    assert a != oracle.gumbel_uniform(seed, 11, 3, 2)
    assert a != oracle.gumbel_uniform(seed ^ 1, 11, 3, 1)


# ---------------------------------------------------------------------------------------
# Router: numpy fp64 matmul + activation (GELU through math.erf)
# ---------------------------------------------------------------------------------------
@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_router_matches_numpy(act):
    rng = np.random.default_rng(11)
    B, d, Hr, M = 3, 96, 40, 17
    H = _bf16(rng, (B, d), 1.0)
    W1, b1 = _bf16(rng, (Hr, d), 0.1), _bf16(rng, (Hr,), 0.5)
    W2, b2 = _bf16(rng, (M, Hr), 0.1), _bf16(rng, (M,), 0.5)
    s, u = oracle.router(H, W1, b1, W2, b2, act)
    pre = _f64(H) @ _f64(W1).T + _f64(b1)
    if act == "relu":
        u_ref = np.maximum(pre, 0.0)
    else:
        u_ref = np.vectorize(lambda x: 0.5 * x * (1.0 + math.erf(x / math.sqrt(2.0))))(pre)
    s_ref = u_ref @ _f64(W2).T + _f64(b2)
    np.testing.assert_allclose(u, u_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s, s_ref, rtol=1e-12, atol=1e-12)
    # the activation matters on these inputs (some pre-activations are negative)
    assert (pre < 0).any()


# ---------------------------------------------------------------------------------------
# Top-k: Python's sort with the (score desc, id asc) rule; ties planted on purpose
# ---------------------------------------------------------------------------------------
def test_topk_matches_sort_with_ties():
    rng = np.random.default_rng(5)
    for trial in range(200):
        M = int(rng.integers(1, 70))
        k = int(rng.integers(1, M + 1))
        s = np.round(rng.standard_normal(M) * 2) / 2.0     # coarse grid -> many exact ties
        ids = oracle.topk(s, k)[0]
        ref = sorted(range(M), key=lambda c: (-s[c], c))[:k]
        assert ids.tolist() == sorted(ref), (trial, M, k)


def test_topk_decides_on_fp32_scores():
    # two fp64 scores that round to the same fp32 value tie, and the lower id wins
    s = np.array([1.0, 1.0 + 1e-12, 0.5])
    assert oracle.topk(s, 1)[0].tolist() == [0]


# ---------------------------------------------------------------------------------------
# Shortlist: brute-force union (v in S <=> cluster_of[v] selected), canonical order
# ---------------------------------------------------------------------------------------
def test_shortlist_is_union_of_clusters():
    cfg = wl.config("tiny")
    off, tok = wl.cluster_partition(cfg, 3)
    cluster_of = np.empty(cfg.V, dtype=np.int64)
    for c in range(cfg.M):
        cluster_of[tok[off[c]:off[c + 1]]] = c
    rng = np.random.default_rng(2)
    for k in (1, 5, cfg.M):
        ids = np.sort(rng.choice(cfg.M, size=k, replace=False)).astype(np.int32)
        S = oracle.shortlist(off, tok, ids)
        members = set(np.nonzero(np.isin(cluster_of, ids))[0].tolist())
        assert set(S.tolist()) == members and len(S) == len(members)
        assert len(S) == int(sum(off[c + 1] - off[c] for c in ids))
        # canonical order: clusters ascending, CSR order inside each
        cl = cluster_of[S]
        assert np.all(np.diff(cl) >= 0)
        for c in ids:
            assert S[cl == c].tolist() == tok[off[c]:off[c + 1]].tolist()


# ---------------------------------------------------------------------------------------
# Head: with every cluster selected the shortlist head is the dense head, permuted by S
# ---------------------------------------------------------------------------------------
def test_head_all_clusters_equals_dense_projection():
    cfg = wl.config("tiny")
    inp = wl.chain_inputs(cfg, 1)
    S = oracle.shortlist(inp["csr_off"], inp["csr_tok"], np.arange(cfg.M, dtype=np.int32))
    assert sorted(S.tolist()) == list(range(cfg.V))
    H = inp["H"][0, :2]
    L = oracle.head(H, inp["W"], S)
    dense = _f64(H) @ _f64(inp["W"]).T                     # [2, V]
    np.testing.assert_allclose(L, dense[:, S], rtol=1e-12, atol=1e-12)


def test_head_rows_follow_shortlist_order():
    rng = np.random.default_rng(8)
    W = _bf16(rng, (50, 24), 1.0)
    h = _bf16(rng, (1, 24), 1.0)
    S = np.array([7, 3, 49, 0], dtype=np.int32)
    L = oracle.head(h, W, S)[0]
    np.testing.assert_allclose(L, (_f64(W)[S] @ _f64(h)[0]), rtol=1e-12)


# ---------------------------------------------------------------------------------------
# Draft sampling: softmax statistics, greedy brute force, Gumbel-max chi-square
# ---------------------------------------------------------------------------------------
def test_softmax_stats_and_shift_invariance():
    rng = np.random.default_rng(4)
    l = rng.standard_normal(300) * 3
    S = rng.permutation(1000)[:300].astype(np.int32)
    for T in (1.0, 0.7, 2.5):
        _, _, m, s = oracle.draft_sample(l, S, T, 1, 1, 0)
        assert m == pytest.approx(l.max() / T, rel=1e-15)
        q = np.exp(l / T - m) / s
        assert q.sum() == pytest.approx(1.0, rel=1e-12)
        _, _, m2, s2 = oracle.draft_sample(l + 5.0, S, T, 1, 1, 0)
        np.testing.assert_allclose(np.exp((l + 5.0) / T - m2) / s2, q, rtol=1e-12)


def test_greedy_is_argmax_with_lower_id_tie():
    l = np.array([0.5, 2.0, -1.0, 2.0])
    S = np.array([40, 17, 3, 9], dtype=np.int32)
    tok, idx, _, _ = oracle.draft_sample(l, S, 0.0, 0, 1, 0)
    assert (tok, idx) == (9, 3)            # 17 and 9 tie; the lower vocabulary id wins
    rng = np.random.default_rng(0)
    for _ in range(50):
        l = rng.standard_normal(40)
        S = rng.permutation(200)[:40].astype(np.int32)
        tok, idx, _, _ = oracle.draft_sample(l, S, 0.0, 0, 1, 0)
        assert idx == int(np.argmax(l)) and tok == S[idx]


def _sample_many(l, S, T, seed, n, pos=1):
    L = oracle.lib()
    la = np.ascontiguousarray(l, np.float64)
    Sa = np.ascontiguousarray(S, np.int32)
    idx = np.zeros(1, np.int64)
    m = np.zeros(1)
    s = np.zeros(1)
    pl, pS, pi, pm, ps = (a.ctypes.data_as(ctypes.c_void_p) for a in (la, Sa, idx, m, s))
    out = np.empty(n, dtype=np.int64)
    for r in range(n):
        L.orc_draft_sample(pl, pS, Sa.size, float(T), seed, pos, r, pi, pm, ps)
        out[r] = idx[0]
    return out


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_gumbel_draws_follow_softmax(T):
    l = np.array([0.3, -1.2, 1.1, 0.0, 2.0, -0.4, 0.9])
    S = np.array([5, 1, 12, 7, 3, 30, 8], dtype=np.int32)
    n = 300_000
    draws = _sample_many(l, S, T, 0xABCDEF, n)
    q = np.exp(l / T - (l / T).max())
    q /= q.sum()
    obs = np.bincount(draws, minlength=len(l))
    _, pval = scipy_stats.chisquare(obs, q * n)
    assert pval > 1e-4
    # the same counts fail against the distribution at another temperature
    q_wrong = np.exp(l / (T * 1.3))
    q_wrong /= q_wrong.sum()
    _, pbad = scipy_stats.chisquare(obs, q_wrong * n)
    assert pbad < 1e-6


# ---------------------------------------------------------------------------------------
# Chain verification
# ---------------------------------------------------------------------------------------
def _P(a):
    return np.ascontiguousarray(a).ctypes.data_as(ctypes.c_void_p)


def _verify_chain_flat(z, ql, qoff, S, didx, u, T):
    """Direct call for large batches: z [B, g+1, V] f32, ql / S flat, qoff [B*g+1]."""
    B, g1, V = z.shape
    z, ql, qoff, S, didx, u = (np.ascontiguousarray(a) for a in (
        z.astype(np.float32), ql.astype(np.float64), qoff.astype(np.int64),
        S.astype(np.int32), didx.astype(np.int64), u.astype(np.float32)))
    acc = np.zeros(B, np.int32)
    corr = np.zeros(B, np.int32)
    rc = oracle.lib().orc_verify_chain(B, g1 - 1, V, float(T), _P(z), _P(ql), _P(qoff), _P(S),
                                       _P(didx), _P(u), _P(acc), _P(corr))
    assert rc == 0
    return acc, corr


def _rule_chain(p_rows, q_rows, xs, us):
    """Speculative-sampling rule in exact rationals. p_rows: gamma+1 dicts v -> Fraction over
    the full vocabulary; q_rows: gamma dicts over the shortlists; xs drafts; us uniforms.
    Returns (accepted, correction, min margin of every comparison taken)."""
    gamma = len(xs)
    margin = Fraction(1)
    V = len(p_rows[0])

    def icdf(w, u):
        nonlocal margin
        tot = sum(w)
        c = Fraction(0)
        for v in range(V):
            c += w[v]
            margin = min(margin, abs(c - u * tot))
            if c > u * tot:
                return v
        raise AssertionError

    for t in range(gamma):
        p, q, x, u = p_rows[t], q_rows[t], xs[t], us[t]
        margin = min(margin, abs(u * q.get(x, 0) - p[x]))
        if u * q.get(x, 0) < p[x]:
            continue
        r = [max(Fraction(0), p[v] - q.get(v, Fraction(0))) for v in range(V)]
        return t, icdf(r, us[gamma]), margin
    return gamma, icdf([p_rows[gamma][v] for v in range(V)], us[gamma]), margin


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_verify_chain_matches_exact_rule_enumeration(T):
    F = Fraction
    V = 4
    p = [[F(1, 8), F(3, 8), F(1, 4), F(1, 4)],
         [F(1, 2), F(1, 8), F(1, 8), F(1, 4)],
         [F(1, 16), F(7, 16), F(5, 16), F(3, 16)]]
    S = [np.array([3, 0, 1], np.int32), np.array([2, 3], np.int32)]
    q = [{3: F(1, 4), 0: F(1, 2), 1: F(1, 4)}, {2: F(3, 4), 3: F(1, 4)}]
    # logits that give these distributions at temperature T: z = T * log p
    z = np.array([[T * math.log(float(x)) for x in row] for row in p], np.float32)
    ql = [np.array([T * math.log(float(q[t][int(v)])) for v in S[t]]) for t in range(2)]
    G = 9
    grid = [F(2 * i + 1, 2 * G) for i in range(G)]
    cases = []
    for j1 in range(len(S[0])):
        for j2 in range(len(S[1])):
            for u1 in grid:
                for u2 in grid:
                    for u3 in grid:
                        cases.append((j1, j2, u1, u2, u3))
    B = len(cases)
    zz = np.broadcast_to(z, (B, 3, V))
    qoff = np.arange(0, 2 * B + 1) // 2 * 5 + (np.arange(0, 2 * B + 1) % 2) * 3
    flat_ql = np.tile(np.concatenate(ql), B)
    flat_S = np.tile(np.concatenate(S), B)
    didx = np.array([[c[0], c[1]] for c in cases])
    uu = np.array([[float(c[2]), float(c[3]), float(c[4])] for c in cases], np.float32)
    acc, corr = _verify_chain_flat(zz, flat_ql, qoff, flat_S, didx, uu, T)
    checked = 0
    for i, (j1, j2, u1, u2, u3) in enumerate(cases):
        xs = [int(S[0][j1]), int(S[1][j2])]
        a, c, margin = _rule_chain(p, q, xs, [u1, u2, u3])
        if margin < F(1, 10**5):          # too close to a boundary for fp32 inputs
            continue
        assert (acc[i], corr[i]) == (a, c), (i, xs, u1, u2, u3)
        checked += 1
    assert checked > 0.9 * B


def test_speculative_rule_is_exact_in_rationals():
    # The rule the oracle follows emits the first token with the target distribution:
    # P(v) = q(v) min(1, p/q) + P(reject) * norm(max(0, p - q))(v) = p(v), exactly.
    F = Fraction
    p = [F(1, 10), F(2, 5), F(3, 10), F(1, 5)]
    q = [F(1, 2), F(0), F(1, 4), F(1, 4)]
    acc_v = [q[v] * min(F(1), p[v] / q[v]) if q[v] else F(0) for v in range(4)]
    rej = 1 - sum(acc_v)
    r = [max(F(0), p[v] - q[v]) for v in range(4)]
    emit = [acc_v[v] + rej * r[v] / sum(r) for v in range(4)]
    assert emit == p


def _chain_trials(l1, S1, z, T, n, seed):
    """n independent single-draft trials: x ~ q via the oracle's Gumbel draw, then verify."""
    rng = np.random.default_rng(seed)
    V = z.shape[1]
    draws = _sample_many(l1, S1, T, 0x5EED ^ seed, n)
    zz = np.broadcast_to(z[None], (n, 2, V))
    qoff = np.arange(n + 1) * len(S1)
    uu = wl.open_uniforms(rng, (n, 2))
    acc, corr = _verify_chain_flat(zz, np.tile(l1, n), qoff, np.tile(S1, n), draws[:, None], uu, T)
    first = np.where(acc >= 1, S1[draws], corr)
    return first, draws, uu, acc


@pytest.mark.slow
@pytest.mark.parametrize("T", [1.0, 0.7])
def test_verify_chain_output_follows_target_chi_square(T):
    V = 8
    rng = np.random.default_rng(21)
    z = (rng.standard_normal((2, V)) * 1.5).astype(np.float32)
    S1 = np.array([6, 1, 2, 4, 0], np.int32)
    l1 = rng.standard_normal(5) * 1.5
    n = 1_000_000
    first, draws, uu, acc = _chain_trials(l1, S1, z, T, n, 3)
    p = np.exp(z[0].astype(np.float64) / T)
    p /= p.sum()
    obs = np.bincount(first, minlength=V)
    _, pval = scipy_stats.chisquare(obs, p * n)
    assert pval > 1e-4
    assert 0 < acc.mean() < 1          # both branches are taken
    # Negative control: a verifier that draws the correction from p instead of the
    # residual max(0, p - q) over-weights the drafted tokens and must fail the same test.
    cdf = np.cumsum(p)
    wrong_corr = np.searchsorted(cdf, uu[:, 1] * cdf[-1], side="right")
    wrong = np.where(acc >= 1, S1[draws], wrong_corr)
    _, pbad = scipy_stats.chisquare(np.bincount(wrong, minlength=V), p * n)
    assert pbad < 1e-6


def test_verify_chain_greedy_brute_force():
    rng = np.random.default_rng(9)
    V, gamma, B = 30, 4, 300
    z = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    am = z.argmax(axis=2)
    S = np.arange(V, dtype=np.int32)
    # drafts that agree with the target argmax for a random prefix, then disagree
    didx = np.empty((B, gamma), np.int64)
    agree = rng.integers(0, gamma + 1, size=B)
    for b in range(B):
        for t in range(gamma):
            didx[b, t] = am[b, t] if t < agree[b] else (am[b, t] + 1 + rng.integers(0, V - 1)) % V
    qoff = np.arange(B * gamma + 1) * V
    acc, corr = _verify_chain_flat(z, np.zeros(B * gamma * V), qoff, np.tile(S, B * gamma),
                                   didx, np.full((B, gamma + 1), 0.5, np.float32), 0.0)
    for b in range(B):
        A = int(agree[b])
        assert acc[b] == A
        assert corr[b] == am[b, A]


# ---------------------------------------------------------------------------------------
# Tree verification
# ---------------------------------------------------------------------------------------
def _verify_tree_flat(z, parent, D, ql, qoff, S, soff, didx, u_node, u_res, T):
    B, n1, V = z.shape
    N = n1 - 1
    arrs = [np.ascontiguousarray(a) for a in (
        z.astype(np.float32), parent.astype(np.int32), ql.astype(np.float64),
        qoff.astype(np.int64), S.astype(np.int32), soff.astype(np.int64),
        didx.astype(np.int64), u_node.astype(np.float32), u_res.astype(np.float32))]
    acc = np.zeros(B, np.int32)
    corr = np.zeros(B, np.int32)
    path = np.zeros((B, D), np.int32)
    rc = oracle.lib().orc_verify_tree(B, D, N // D, V, float(T), *[_P(a) for a in arrs],
                                      _P(acc), _P(corr), _P(path))
    assert rc == 0
    return acc, corr, path


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_chain_shaped_tree_equals_chain_verify(T):
    rng = np.random.default_rng(31)
    V, D, B = 40, 4, 200
    parent = np.array([-1, 0, 1, 2], np.int32)           # one node per depth
    lists = [rng.permutation(V)[:int(rng.integers(5, 20))].astype(np.int32) for _ in range(D)]
    z = (rng.standard_normal((B, D + 1, V)) * 2).astype(np.float32)
    l = [rng.standard_normal((B, len(S))) for S in lists]
    didx = np.stack([rng.integers(0, len(S), size=B) for S in lists], axis=1)
    if T == 0.0:     # make some drafts agree with the target argmax
        for b in range(0, B, 2):
            for t in range(D):
                hit = np.nonzero(lists[t] == z[b, t].argmax())[0]
                if hit.size:
                    didx[b, t] = hit[0]
    u = wl.open_uniforms(rng, (B, D + 1))
    # chain layout
    qoff = np.zeros(B * D + 1, np.int64)
    qoff[1:] = np.cumsum([len(lists[t]) for b in range(B) for t in range(D)])
    ql = np.concatenate([l[t][b] for b in range(B) for t in range(D)])
    Sf = np.concatenate([lists[t] for b in range(B) for t in range(D)])
    acc_c, corr_c = _verify_chain_flat(z, ql, qoff, Sf, didx, u, T)
    # tree layout: node n = depth n+1; same shortlists; u_res all equal to the chain's last u
    acc_t, corr_t, path = _verify_tree_flat(
        z, parent, D, ql, qoff, Sf, qoff, didx, u[:, :D], np.repeat(u[:, D:], D + 1, axis=1), T)
    assert np.array_equal(acc_c, acc_t)
    assert np.array_equal(corr_c, corr_t)
    for b in range(B):
        assert path[b, :acc_t[b]].tolist() == list(range(acc_t[b]))
    assert 0 < acc_c.mean() < D or T == 0.0


def _rule_tree_two_siblings(p, q1, q2, x1, x2, u1, u2, ur):
    """Sibling-sequential rejection at the root in exact rationals (one depth, 2 children)."""
    V = len(p)
    margin = Fraction(1)

    def icdf(w, u):
        nonlocal margin
        tot = sum(w)
        c = Fraction(0)
        for v in range(V):
            c += w[v]
            margin = min(margin, abs(c - u * tot))
            if c > u * tot:
                return v

    margin = min(margin, abs(u1 * q1[x1] - p[x1]))
    if u1 * q1[x1] < p[x1]:
        return 1, None, margin, 0
    r = [max(Fraction(0), p[v] - q1[v]) for v in range(V)]
    R = sum(r)
    p2 = [x / R for x in r]
    margin = min(margin, abs(u2 * q2[x2] - p2[x2]))
    if u2 * q2[x2] < p2[x2]:
        return 1, None, margin, 1
    r2 = [max(Fraction(0), p2[v] - q2[v]) for v in range(V)]
    return 0, icdf(r2, ur), margin, -1


def test_verify_tree_matches_exact_rule_and_is_exact():
    F = Fraction
    V = 3
    p = [F(1, 2), F(1, 3), F(1, 6)]
    q1 = [F(1, 4), F(3, 4), F(0)]        # shortlist {0, 1}
    q2 = [F(2, 3), F(1, 3), F(0)]
    S = np.array([0, 1], np.int32)
    z = np.array([[math.log(float(x)) for x in p]] + [[0.0] * V] * 2, np.float32)
    ql = np.array([math.log(float(q1[0])), math.log(float(q1[1])),
                   math.log(float(q2[0])), math.log(float(q2[1]))])
    G = 12
    grid = [F(2 * i + 1, 2 * G) for i in range(G)]
    cases = [(a, b, u1, u2, ur) for a in range(2) for b in range(2)
             for u1 in grid for u2 in grid for ur in grid]
    B = len(cases)
    parent = np.array([-1, -1], np.int32)
    qoff = np.arange(2 * B + 1) * 2
    soff = np.arange(B + 1) * 2
    acc, corr, path = _verify_tree_flat(
        np.broadcast_to(z, (B, 3, V)), parent, 1, np.tile(ql, B), qoff, np.tile(S, B), soff,
        np.array([[c[0], c[1]] for c in cases]),
        np.array([[float(c[2]), float(c[3])] for c in cases]),
        np.array([[float(c[4]), float(c[4])] for c in cases]), 1.0)
    emit = [F(0)] * V
    checked = 0
    for i, (a, b, u1, u2, ur) in enumerate(cases):
        A, c, margin, node = _rule_tree_two_siblings(p, q1, q2, a, b, u1, u2, ur)
        tok = [a, b][node] if A else c
        if margin >= F(1, 10**5):
            assert acc[i] == A and path[i, 0] == node
            if not A:
                assert corr[i] == c
            checked += 1
        emit[tok] += q1[a] * q2[b] / G ** 3
    assert checked > 0.9 * B
    # exactness of the rule itself, with the uniforms integrated exactly: the emitted-token
    # law at the root is p.  (The grid above approximates the integral; here we integrate.)
    exact = [F(0)] * V
    for a in range(2):
        for b in range(2):
            w = q1[a] * q2[b]
            pa1 = min(F(1), p[a] / q1[a])
            exact[a] += w * pa1
            r = [max(F(0), p[v] - q1[v]) for v in range(V)]
            p2 = [x / sum(r) for x in r]
            pa2 = min(F(1), p2[b] / q2[b])
            exact[b] += w * (1 - pa1) * pa2
            r2 = [max(F(0), p2[v] - q2[v]) for v in range(V)]
            for v in range(V):
                exact[v] += w * (1 - pa1) * (1 - pa2) * r2[v] / sum(r2)
    assert exact == p
    # and the grid-integrated oracle law is within the grid resolution of it
    assert max(abs(float(emit[v] - p[v])) for v in range(V)) < 3.0 / G


@pytest.mark.slow
def test_verify_tree_output_follows_target_chi_square():
    V, n = 8, 600_000
    rng = np.random.default_rng(77)
    z = np.zeros((4, V), np.float32)
    z[0] = rng.standard_normal(V) * 1.5
    S = np.array([7, 2, 3, 0, 5], np.int32)
    ls = [rng.standard_normal(5) * 1.5 for _ in range(3)]
    draws = np.stack([_sample_many(ls[i], S, 1.0, 0xBEEF + i, n) for i in range(3)], axis=1)
    parent = np.array([-1, -1, -1], np.int32)
    u_node = wl.open_uniforms(rng, (n, 3))
    u_res = wl.open_uniforms(rng, (n, 2))
    acc, corr, path = _verify_tree_flat(
        np.broadcast_to(z, (n, 4, V)), parent, 1, np.tile(np.concatenate(ls), n),
        np.arange(3 * n + 1) * 5, np.tile(S, n), np.arange(n + 1) * 5, draws, u_node, u_res, 1.0)
    node = path[:, 0]
    first = np.where(acc >= 1, S[draws[np.arange(n), np.maximum(node, 0)]], corr)
    p = np.exp(z[0].astype(np.float64))
    p /= p.sum()
    _, pval = scipy_stats.chisquare(np.bincount(first, minlength=V), p * n)
    assert pval > 1e-4
    assert (node == 1).any() and (node == 2).any() and (acc == 0).any()


# ---------------------------------------------------------------------------------------
# Spherical k-means over the LM-head rows (the offline clustering step)
# ---------------------------------------------------------------------------------------
def _bf16_rows(x):
    return wl.to_bf16_bits(np.asarray(x, np.float32))


def test_kmeans_recovers_a_planted_partition():
    # Six orthonormal directions, 100 rows around each (cosine to their direction > 0.9), rows
    # of different lengths, ids shuffled: seeded with one row of each group, one step must
    # return exactly the planted groups, listed in ascending token id.
    rng = np.random.default_rng(31)
    M, per, d = 6, 100, 64
    Q, _ = np.linalg.qr(rng.standard_normal((d, d)))
    dirs = Q[:M]
    labels = np.repeat(np.arange(M), per)
    perm = rng.permutation(M * per)
    labels = labels[perm]
    X = dirs[labels] + 0.02 * rng.standard_normal((M * per, d))
    X *= rng.uniform(0.5, 3.0, size=(M * per, 1))
    W = _bf16_rows(X)
    init = np.array([np.nonzero(labels == c)[0][0] for c in range(M)], np.int32)
    cent = oracle.kmeans_init(W, init)
    cent, assign, off, tok, _ = oracle.kmeans_step(W, cent)
    assert np.array_equal(assign, labels)
    for c in range(M):
        assert np.array_equal(tok[off[c]:off[c + 1]], np.nonzero(labels == c)[0])


def test_kmeans_assignment_is_the_nearest_centroid_by_cosine():
    # The assignment against scipy's cosine distance (an independent library routine): with
    # exact centroids it is argmin_c cosdist(W_v, mu_c); with bf16 centroids, against the
    # centroids rounded to bf16, up to fp32 near-ties.
    from scipy.spatial.distance import cdist
    rng = np.random.default_rng(5)
    V, d, M = 700, 48, 9
    W = _bf16_rows(rng.standard_normal((V, d)))
    Wf = wl.bf16_bits_to_f32(W).astype(np.float64)
    mu = rng.standard_normal((M, d))
    mu /= np.linalg.norm(mu, axis=1, keepdims=True)
    _, assign, _, _, _ = oracle.kmeans_step(W, mu, round_bf16=False)
    assert np.array_equal(assign, np.argmin(cdist(Wf, mu, "cosine"), axis=1))
    mub = wl.bf16_bits_to_f32(wl.to_bf16_bits(mu.astype(np.float32))).astype(np.float64)
    _, assign_b, _, _, _ = oracle.kmeans_step(W, mu, round_bf16=True)
    ref = np.argmin(cdist(Wf, mub, "cosine"), axis=1)
    s = Wf @ mub.T
    for v in np.nonzero(assign_b != ref)[0]:
        assert abs(s[v, assign_b[v]] - s[v, ref[v]]) < 1e-6 * np.linalg.norm(Wf[v])


def test_kmeans_update_and_csr():
    # The update against numpy: each centroid is the normalised sum of its tokens' unit rows; a
    # cluster no token picks keeps its centroid; the CSR lists every token once, by cluster,
    # ascending inside a cluster, and agrees with the assignment.
    rng = np.random.default_rng(6)
    V, d, M = 500, 40, 8
    X = rng.standard_normal((V, d))
    X[:, 0] = np.abs(X[:, 0]) + 0.5                     # every row has a positive first coordinate
    W = _bf16_rows(X)
    Wf = wl.bf16_bits_to_f32(W).astype(np.float64)
    mu = rng.standard_normal((M, d)) * 0.3
    mu[:, 0] = 3.0                                      # near the rows' common direction ...
    mu[M - 1] = 0.0
    mu[M - 1, 0] = -1.0                                 # ... except one, away from every row: stays empty
    mu /= np.linalg.norm(mu, axis=1, keepdims=True)
    new, assign, off, tok, _ = oracle.kmeans_step(W, mu, round_bf16=False)
    assert off[0] == 0 and off[M] == V and np.all(np.diff(off) >= 0)
    assert np.array_equal(np.sort(tok), np.arange(V))
    for c in range(M):
        part = tok[off[c]:off[c + 1]]
        assert np.all(np.diff(part) > 0) and np.all(assign[part] == c)
        if part.size == 0:
            assert np.array_equal(new[c], mu[c])
        else:
            s = (Wf[part] / np.linalg.norm(Wf[part], axis=1, keepdims=True)).sum(axis=0)
            np.testing.assert_allclose(new[c], s / np.linalg.norm(s), rtol=1e-12, atol=1e-14)
    assert off[M] - off[M - 1] == 0


def test_kmeans_objective_never_decreases():
    # Lloyd's property for the cosine objective with exact centroids: J of the assignment made
    # from the updated centroids is at least J of the previous one.
    cfg = wl.config("tiny")
    W = wl.lm_head(cfg, 0)
    init = np.random.default_rng(2).permutation(cfg.V)[:cfg.M]
    cent = oracle.kmeans_init(W, init)
    prev = -np.inf
    for _ in range(5):
        cent, _, _, _, J = oracle.kmeans_step(W, cent, round_bf16=False)
        assert J >= prev - 1e-9 * abs(J)
        prev = J
