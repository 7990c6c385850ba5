"""CPU oracle for the DynaSpec draft head and speculative-sampling verifier.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it.  The product package never imports it and shares no code with it.

The arithmetic lives in ``dynaspec_oracle.c`` (plain C, fp64 accumulation, one plain loop
per definition); this module builds it with gcc, loads it with ctypes and strings its
steps together in the order of the DynaSpec pipeline (summary "DynaSpec: Context-aware
Dynamic Speculative Sampling for Large-Vocabulary Language Models", Technical Details >
Pipeline Flow): router -> top-k clusters -> shortlist -> gathered projection -> draft
sampling, then rejection-sampling verification over the full vocabulary.

Every function here is pinned by ``tests/test_oracle_pins.py`` against something other
than itself (numpy fp64 matmul, brute-force sorts and set unions, exact rational
enumeration, chi-square tests, cuRAND's host Philox generator).  One output has no pin:
the end-to-end quality figures of the pages (mean accepted length, speed-up), which need
trained models; parity unpinned for those.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dynaspec_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_dynaspec_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O2, IEEE math, OpenMP) next to its source."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_D = ctypes.c_double
_U64 = ctypes.c_uint64


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        L.orc_set_threads.argtypes = [_I]
        L.orc_get_threads.restype = _I
        L.orc_philox4x32_10.argtypes = [_P, _P, _P]
        L.orc_gumbel_uniform.argtypes = [_U64, _I64, _I, _I]
        L.orc_gumbel_uniform.restype = _D
        L.orc_router.argtypes = [_P, _I, _I, _P, _P, _I, _P, _P, _I, _I, _P, _P]
        L.orc_router.restype = _I
        L.orc_topk.argtypes = [_P, _I, _I, _I, _P]
        L.orc_topk.restype = _I
        L.orc_shortlist.argtypes = [_P, _P, _I, _P, _I, _P]
        L.orc_shortlist.restype = _I64
        L.orc_head.argtypes = [_P, _I, _I, _P, _P, _I64, _P]
        L.orc_draft_sample.argtypes = [_P, _P, _I64, _D, _U64, _I, _I, _P, _P, _P]
        L.orc_draft_sample.restype = ctypes.c_int32
        L.orc_verify_chain.argtypes = [_I, _I, _I, _D, _P, _P, _P, _P, _P, _P, _P, _P]
        L.orc_verify_chain.restype = _I
        L.orc_verify_tree.argtypes = [_I, _I, _I, _I, _D, _P, _P, _P, _P, _P, _P, _P,
                                      _P, _P, _P, _P, _P]
        L.orc_verify_tree.restype = _I
        L.orc_kmeans_init.argtypes = [_P, _I, _I, _P, _I, _P]
        L.orc_kmeans_init.restype = _I
        L.orc_kmeans_step.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P]
        L.orc_kmeans_step.restype = _I
        _lib = L
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


# ---------------------------------------------------------------------------------------
# Single steps
# ---------------------------------------------------------------------------------------
def philox4x32_10(ctr, key) -> np.ndarray:
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def gumbel_uniform(seed: int, j: int, pos: int, row: int) -> float:
    """The draft draw's uniform for entry j of a shortlist (its index in list order)."""
    return float(lib().orc_gumbel_uniform(seed, j, pos, row))


_ACT = {"relu": 0, "gelu": 1}


def router(H, W1, b1, W2, b2, act: str):
    """Cluster scores s [B, M] (fp64) and the hidden layer u [B, Hr] for hidden states H [B, d]."""
    H = _c(H, np.uint16)
    B, d = H.shape
    Hr, M = W1.shape[0], W2.shape[0]
    W1, b1, W2, b2 = (_c(a, np.uint16) for a in (W1, b1, W2, b2))
    u = np.zeros((B, Hr), dtype=np.float64)
    s = np.zeros((B, M), dtype=np.float64)
    rc = lib().orc_router(_ptr(H), B, d, _ptr(W1), _ptr(b1), Hr, _ptr(W2), _ptr(b2), M,
                          _ACT[act], _ptr(u), _ptr(s))
    if rc:
        raise ValueError(f"orc_router failed ({rc})")
    return s, u


def topk(scores, k: int) -> np.ndarray:
    """Top-k cluster ids per row of scores [B, M], ascending id, ties to the lower id."""
    s = _c(np.atleast_2d(scores), np.float64)
    B, M = s.shape
    ids = np.zeros((B, k), dtype=np.int32)
    if lib().orc_topk(_ptr(s), B, M, k, _ptr(ids)):
        raise ValueError("orc_topk: bad k")
    return ids


def shortlist(csr_off, csr_tok, ids) -> np.ndarray:
    off = _c(csr_off, np.int32)
    tok = _c(csr_tok, np.int32)
    ids = _c(ids, np.int32).ravel()
    M = off.shape[0] - 1
    cap = int(sum(int(off[c + 1]) - int(off[c]) for c in ids)) if ids.size else 0
    S = np.zeros(max(cap, 1), dtype=np.int32)
    n = lib().orc_shortlist(_ptr(off), _ptr(tok), M, _ptr(ids), ids.size, _ptr(S))
    if n < 0:
        raise ValueError("orc_shortlist: cluster id out of range")
    return S[:n].copy()


def head(H, W, S) -> np.ndarray:
    """Gathered-head logits l [R, |S|] (fp64) for hidden rows H [R, d] sharing shortlist S."""
    H = _c(np.atleast_2d(H), np.uint16)
    W = _c(W, np.uint16)
    S = _c(S, np.int32)
    R, d = H.shape
    out = np.zeros((R, S.size), dtype=np.float64)
    lib().orc_head(_ptr(H), R, d, _ptr(W), _ptr(S), S.size, _ptr(out))
    return out


def draft_sample(l, S, T: float, seed: int, pos: int, row: int):
    """(token, index in S, m, s) of the draft draw over one shortlist row of logits l."""
    l = _c(l, np.float64)
    S = _c(S, np.int32)
    idx = np.zeros(1, dtype=np.int64)
    m = np.zeros(1)
    s = np.zeros(1)
    tok = lib().orc_draft_sample(_ptr(l), _ptr(S), S.size, float(T), seed, pos, row,
                                 _ptr(idx), _ptr(m), _ptr(s))
    return int(tok), int(idx[0]), float(m[0]), float(s[0])


def verify_chain(z, q_logits, shortlists, draft_idx, u, T: float):
    """Chain verification for B sequences.

    z [B, gamma+1, V] fp32; q_logits[b][t] and shortlists[b][t] (t = 0..gamma-1) the draft
    logits and shortlist of draft position t+1; draft_idx [B, gamma] index of x_t in its
    shortlist; u [B, gamma+1].  Returns (accepted_len [B], correction [B]).
    """
    z = _c(z, np.float32)
    B, g1, V = z.shape
    gamma = g1 - 1
    lens = [len(shortlists[b][t]) for b in range(B) for t in range(gamma)]
    qoff = np.zeros(B * gamma + 1, dtype=np.int64)
    qoff[1:] = np.cumsum(lens)
    ql = _c(np.concatenate([np.asarray(q_logits[b][t], np.float64).ravel()
                            for b in range(B) for t in range(gamma)]), np.float64)
    S = _c(np.concatenate([np.asarray(shortlists[b][t]).ravel()
                           for b in range(B) for t in range(gamma)]), np.int32)
    di = _c(draft_idx, np.int64).ravel()
    uu = _c(u, np.float32)
    acc = np.zeros(B, dtype=np.int32)
    corr = np.zeros(B, dtype=np.int32)
    rc = lib().orc_verify_chain(B, gamma, V, float(T), _ptr(z), _ptr(ql), _ptr(qoff), _ptr(S),
                                _ptr(di), _ptr(uu), _ptr(acc), _ptr(corr))
    if rc:
        raise RuntimeError(f"orc_verify_chain failed ({rc})")
    return acc, corr


def verify_tree(z, parent, shortlists, node_logits, draft_idx, u_node, u_res, T: float):
    """Tree verification for B sequences.

    z [B, 1+N, V]; parent [N]; shortlists[b][dep-1] the shortlist of depth dep;
    node_logits[b][n] node n's draft logits over its depth's shortlist; draft_idx [B, N];
    u_node [B, N]; u_res [B, D+1].  Returns (accepted_len [B], correction [B], path [B, D]).
    """
    z = _c(z, np.float32)
    B, n1, V = z.shape
    N = n1 - 1
    parent = _c(parent, np.int32)
    D = len(shortlists[0])
    Wd = N // D
    slen = [len(shortlists[b][k]) for b in range(B) for k in range(D)]
    soff = np.zeros(B * D + 1, dtype=np.int64)
    soff[1:] = np.cumsum(slen)
    S = _c(np.concatenate([np.asarray(shortlists[b][k]).ravel()
                           for b in range(B) for k in range(D)]), np.int32)
    qlen = [len(node_logits[b][n]) for b in range(B) for n in range(N)]
    qoff = np.zeros(B * N + 1, dtype=np.int64)
    qoff[1:] = np.cumsum(qlen)
    ql = _c(np.concatenate([np.asarray(node_logits[b][n], np.float64).ravel()
                            for b in range(B) for n in range(N)]), np.float64)
    di = _c(draft_idx, np.int64).ravel()
    un = _c(u_node, np.float32)
    ur = _c(u_res, np.float32)
    acc = np.zeros(B, dtype=np.int32)
    corr = np.zeros(B, dtype=np.int32)
    path = np.zeros((B, D), dtype=np.int32)
    rc = lib().orc_verify_tree(B, D, Wd, V, float(T), _ptr(z), _ptr(parent), _ptr(ql),
                               _ptr(qoff), _ptr(S), _ptr(soff), _ptr(di), _ptr(un), _ptr(ur),
                               _ptr(acc), _ptr(corr), _ptr(path))
    if rc:
        raise RuntimeError(f"orc_verify_tree failed ({rc})")
    return acc, corr, path


# ---------------------------------------------------------------------------------------
# Whole speculation steps, in pipeline order
# ---------------------------------------------------------------------------------------
def chain_step(inp: dict, T: float | None = None, seqs=None, positions=None, verify=True):
    """Run the whole chain step for the sequences `seqs` (default: all).

    Returns per sequence b and position t (0-based, draft position t+1): scores, cluster
    ids, shortlist, logits, (token, index, m, s); and the verification outputs.
    The router at position t+1 reads H[b, t]; the head reads H[b, t+1]; the Gumbel counter
    uses pos = t+1 and row = b.
    """
    cfg = inp["cfg"]
    T = cfg.T if T is None else T
    B = cfg.B
    seqs = range(B) if seqs is None else seqs
    gamma = cfg.gamma
    positions = range(gamma) if positions is None else positions
    out = {}
    for b in seqs:
        rows = []
        for t in positions:
            s, _ = router(inp["H"][b, t][None], inp["W1"], inp["b1"], inp["W2"], inp["b2"], cfg.act)
            ids = topk(s, cfg.budget[t])[0]
            S = shortlist(inp["csr_off"], inp["csr_tok"], ids)
            l = head(inp["H"][b, t + 1][None], inp["W"], S)[0]
            tok, idx, m, ssum = draft_sample(l, S, T, inp["gumbel_seed"], t + 1, b)
            rows.append(dict(scores=s[0], ids=ids, S=S, logits=l, token=tok, idx=idx, m=m, s=ssum))
        out[b] = rows
    if verify and list(positions) == list(range(gamma)):
        seq_list = list(seqs)
        acc, corr = verify_chain(
            inp["z"][seq_list],
            [[out[b][t]["logits"] for t in range(gamma)] for b in seq_list],
            [[out[b][t]["S"] for t in range(gamma)] for b in seq_list],
            np.array([[out[b][t]["idx"] for t in range(gamma)] for b in seq_list]),
            inp["u"][seq_list], T)
        for i, b in enumerate(seq_list):
            out[b] = dict(positions=out[b], accepted=int(acc[i]), correction=int(corr[i]))
    else:
        for b in list(out):
            out[b] = dict(positions=out[b])
    return out


def tree_step(inp: dict, T: float | None = None, seqs=None, verify=True):
    """Run the whole tree step (router per (sequence, depth), shared per-depth shortlist,
    one draft row per node, tree verification).  Gumbel counter: pos = depth, row = the
    node's head row b*width + i."""
    cfg = inp["cfg"]
    T = cfg.T if T is None else T
    D, Wd = cfg.gamma, cfg.width
    seqs = range(cfg.B) if seqs is None else seqs
    out = {}
    for b in seqs:
        depths = []
        for dep in range(1, D + 1):
            s, _ = router(inp["Hr_h"][b, dep - 1][None], inp["W1"], inp["b1"], inp["W2"],
                          inp["b2"], cfg.act)
            ids = topk(s, cfg.budget[dep - 1])[0]
            S = shortlist(inp["csr_off"], inp["csr_tok"], ids)
            Hrows = inp["Hn"][dep - 1, b * Wd:(b + 1) * Wd]
            L = head(Hrows, inp["W"], S)
            nodes = []
            for i in range(Wd):
                tok, idx, m, ssum = draft_sample(L[i], S, T, inp["gumbel_seed"], dep, b * Wd + i)
                nodes.append(dict(logits=L[i], token=tok, idx=idx, m=m, s=ssum))
            depths.append(dict(scores=s[0], ids=ids, S=S, nodes=nodes))
        out[b] = dict(depths=depths)
    if verify:
        seq_list = list(seqs)
        acc, corr, path = verify_tree(
            inp["z"][seq_list], inp["parent"],
            [[out[b]["depths"][k]["S"] for k in range(D)] for b in seq_list],
            [[out[b]["depths"][n // Wd]["nodes"][n % Wd]["logits"] for n in range(D * Wd)]
             for b in seq_list],
            np.array([[out[b]["depths"][n // Wd]["nodes"][n % Wd]["idx"] for n in range(D * Wd)]
                      for b in seq_list]),
            inp["u_node"][seq_list], inp["u_res"][seq_list], T)
        for i, b in enumerate(seq_list):
            out[b].update(accepted=int(acc[i]), correction=int(corr[i]), path=path[i].tolist())
    return out


def static_chain_step(inp: dict, T: float | None = None, seqs=None, verify=True):
    """The static-shortlist baseline's chain step: the fixed list inp["static_ids"] at every
    position (no router), then the same head, draft sampling and verification as chain_step
    (DynaSpec abstract and summary, Comparison to Prior Work: the fixed-shortlist drafters the
    pages compare against).  Same return layout as chain_step (without scores and ids)."""
    cfg = inp["cfg"]
    T = cfg.T if T is None else T
    seqs = list(range(cfg.B) if seqs is None else seqs)
    S = np.asarray(inp["static_ids"], dtype=np.int32)
    out = {}
    for b in seqs:
        rows = []
        for t in range(cfg.gamma):
            l = head(inp["H"][b, t + 1][None], inp["W"], S)[0]
            tok, idx, m, ssum = draft_sample(l, S, T, inp["gumbel_seed"], t + 1, b)
            rows.append(dict(S=S, logits=l, token=tok, idx=idx, m=m, s=ssum))
        out[b] = dict(positions=rows)
    if verify:
        acc, corr = verify_chain(
            inp["z"][seqs], [[p["logits"] for p in out[b]["positions"]] for b in seqs],
            [[S] * cfg.gamma for _ in seqs],
            np.array([[p["idx"] for p in out[b]["positions"]] for b in seqs]), inp["u"][seqs], T)
        for i, b in enumerate(seqs):
            out[b].update(accepted=int(acc[i]), correction=int(corr[i]))
    return out


# ---------------------------------------------------------------------------------------
# Spherical k-means over the LM-head rows (the offline clustering step before the path)
# ---------------------------------------------------------------------------------------
def kmeans_init(W, init_rows) -> np.ndarray:
    """Centroids [M, d] (fp64): the rows init_rows of W scaled to unit length."""
    W = _c(W, np.uint16)
    V, d = W.shape
    init = _c(init_rows, np.int32)
    cent = np.zeros((init.size, d), dtype=np.float64)
    if lib().orc_kmeans_init(_ptr(W), V, d, _ptr(init), init.size, _ptr(cent)):
        raise ValueError("kmeans_init: a row index outside W")
    return cent


def kmeans_step(W, cent, round_bf16=True):
    """One Lloyd step of spherical k-means (see dynaspec_oracle.c).  Returns (new centroids,
    assignment [V], csr_off [M+1], csr_tok [V], objective of the assignment)."""
    W = _c(W, np.uint16)
    V, d = W.shape
    cent = np.array(cent, dtype=np.float64, order="C", copy=True)
    M = cent.shape[0]
    assign = np.zeros(V, dtype=np.int32)
    off = np.zeros(M + 1, dtype=np.int32)
    tok = np.zeros(V, dtype=np.int32)
    obj = np.zeros(1)
    rc = lib().orc_kmeans_step(_ptr(W), V, d, M, int(bool(round_bf16)), _ptr(cent), _ptr(assign),
                               _ptr(off), _ptr(tok), _ptr(obj))
    if rc:
        raise RuntimeError(f"orc_kmeans_step failed ({rc})")
    return cent, assign, off, tok, float(obj[0])
