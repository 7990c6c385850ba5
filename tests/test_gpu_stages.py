"""Stage-by-stage parity of the CUDA path (through the C ABI) against the CPU oracle.

Each stage is fed the oracle's own upstream result, so a stage is checked on its own: the
shortlist builder gets the oracle's cluster ids, the head gets the oracle's shortlist, the
verifier gets the oracle's draft logits (rounded to fp32) and tokens.  Tolerances and
near-tie excuses are the ones in tests/parity.py.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle                          # noqa: E402
import workloads as wl                 # noqa: E402
from parity import (ICDF_TOL, assert_close, topk_same_or_excused, token_same_or_excused,  # noqa: E402
                    softmax_full, q_dense, icdf_acceptable, accept_margin, TIE)
import gpu_util as gu                  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ds():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from dynamic_vocab_draft_gb300 import build
    build.build()
    import dynamic_vocab_draft_gb300 as pkg
    pkg.load_library()
    return pkg.api


# ---------------------------------------------------------------------------------------
def test_device_philox_matches_oracle(ds):
    rng = np.random.default_rng(0)
    ctr = rng.integers(0, 1 << 32, size=(2048, 4), dtype=np.uint64).astype(np.uint32)
    for seed in (0, 0x0123456789ABCDEF, 0xFFFFFFFF00000001):
        out = torch.zeros(2048, 4, dtype=torch.int32, device=gu.dev())
        ds.philox4x32_10(gu.i32(ctr.view(np.int32)), seed, out)
        got = out.cpu().numpy().view(np.uint32)
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for i in range(0, 2048, 37):
            assert np.array_equal(got[i], oracle.philox4x32_10(ctr[i], key)), i


@pytest.mark.parametrize("name", ["tiny", "llama_b1"])
def test_vocab_index(ds, name):
    inp = gu.chain_inputs(name)
    off, tok = inp["csr_off"], inp["csr_tok"]
    V = tok.size
    cof = torch.empty(V, dtype=torch.int32, device=gu.dev())
    rk = torch.empty(V, dtype=torch.int32, device=gu.dev())
    st = gu.status()
    ds.vocab_index(gu.i32(off), gu.i32(tok), cof, rk, st)
    ref_c = np.empty(V, np.int32)
    ref_r = np.empty(V, np.int32)
    for c in range(off.size - 1):
        ref_c[tok[off[c]:off[c + 1]]] = c
        ref_r[tok[off[c]:off[c + 1]]] = np.arange(off[c + 1] - off[c])
    assert np.array_equal(cof.cpu().numpy(), ref_c)
    assert np.array_equal(rk.cpu().numpy(), ref_r)
    assert st.item() == 0


# ---------------------------------------------------------------------------------------
@pytest.mark.parametrize("name,B,sms", [("tiny", 1, -1), ("small_batched", 5, -1), ("llama_b1", 1, -1),
                                        ("batched", 32, -1), ("large_b1_f5", 1, -1), ("large_b8_f10", 8, -1),
                                        ("large_b64_f100", 64, -1), ("large_b64_f100", 2, -1),
                                        ("large_b64_f100", 100, -1), ("large_b64_f100", 20, -1),
                                        ("large_b64_f100", 40, -1), ("llama_b1", 1, 40), ("large_b1_f5", 1, 3),
                                        ("batched", 32, 16), ("small_batched", 5, 3), ("large_b64_f100", 64, 152)])
def test_router_topk(ds, name, B, sms):
    # B = 1: CUDA-core GEMV; 2 <= B <= 64: tensor-core layers; B > 64: CUDA-core batched GEMV.
    # B larger than the configuration's batch stacks the hidden states of several positions.
    # sms: the SMs the launches are sized for (-1: the library's default).
    inp = gu.chain_inputs(name)
    cfg = inp["cfg"]
    H = inp["H"]
    Hrows = np.concatenate([H[:, t] for t in range(H.shape[1])])[:B]
    B = Hrows.shape[0]
    scores_ref, _ = oracle.router(Hrows, inp["W1"], inp["b1"], inp["W2"], inp["b2"], cfg.act)
    scores = torch.empty(B, cfg.M, dtype=torch.float32, device=gu.dev())
    st = gu.status()
    ws = ds.workspace(ds.router_workspace_bytes(B, cfg.Hr), gu.dev())
    for pos in range(1, cfg.gamma + 1):
        k = cfg.budget[pos - 1]
        ids = torch.empty(B, k, dtype=torch.int32, device=gu.dev())
        ds.router_topk(gu.bf16(Hrows), gu.bf16(inp["W1"]), gu.bf16(inp["b1"]), gu.bf16(inp["W2"]),
                       gu.bf16(inp["b2"]), cfg.act, cfg.budget, pos, scores, ids, ws, st, sms=sms)
        torch.cuda.synchronize()
        assert_close(scores.cpu().numpy(), scores_ref, f"{name} router scores")
        g = ids.cpu().numpy()
        for b in range(B):
            assert np.all(np.diff(g[b]) > 0)
            topk_same_or_excused(g[b], scores_ref[b], k)
    assert st.item() == 0


def test_topk_exact_ties_and_edges(ds):
    # scores with exact ties: the GPU must break them to the lower id, like the oracle.
    M, B = 300, 3
    rng = np.random.default_rng(1)
    s = (np.round(rng.standard_normal((B, M)) * 4) / 4).astype(np.float32)
    s[1] = 0.0
    s[2, ::2] = -0.0                   # -0 and +0 tie
    d = 8
    # a router whose output equals the bias: W2 = 0, b2 = scores (exactly representable)
    b2 = wl.to_bf16_bits(s[0])
    for b in range(B):
        b2 = wl.to_bf16_bits(s[b])
        assert np.array_equal(wl.bf16_bits_to_f32(b2), s[b])
        for k in (1, 7, 150, M):
            scores = torch.empty(1, M, dtype=torch.float32, device=gu.dev())
            ids = torch.empty(1, k, dtype=torch.int32, device=gu.dev())
            ws = ds.workspace(ds.router_workspace_bytes(1, 8), gu.dev())
            ds.router_topk(gu.bf16(np.zeros((1, d), np.uint16)), gu.bf16(np.zeros((8, d), np.uint16)),
                           gu.bf16(np.zeros(8, np.uint16)), gu.bf16(np.zeros((M, 8), np.uint16)),
                           gu.bf16(b2), "relu", [k], 1, scores, ids, ws, gu.status())
            ref = oracle.topk(s[b].astype(np.float64), k)[0]
            assert np.array_equal(ids.cpu().numpy()[0], ref), (b, k)


# ---------------------------------------------------------------------------------------
def _oracle_lists(inp, B, pos):
    cfg = inp["cfg"]
    s, _ = oracle.router(inp["H"][:B, pos - 1], inp["W1"], inp["b1"], inp["W2"], inp["b2"], cfg.act)
    ids = oracle.topk(s, cfg.budget[pos - 1])
    lists = [oracle.shortlist(inp["csr_off"], inp["csr_tok"], ids[b]) for b in range(B)]
    return ids, lists


def _gpu_shortlist(ds, inp, ids, union=True, cap=None):
    cfg = inp["cfg"]
    B, k = ids.shape
    V, M = cfg.V, cfg.M
    cap = B * V if cap is None else cap
    vs_off = torch.zeros(B + 1, dtype=torch.int32, device=gu.dev())
    vs_ids = torch.full((cap + 64,), -7, dtype=torch.int32, device=gu.dev())
    cpos = torch.empty(B * M, dtype=torch.int32, device=gu.dev())
    un = (torch.empty(V, dtype=torch.int32, device=gu.dev()), torch.empty(V, dtype=torch.int32, device=gu.dev()),
          torch.zeros(1, dtype=torch.int32, device=gu.dev())) if union else (None, None, None)
    st = gu.status()
    ws = ds.workspace(ds.shortlist_workspace_bytes(B, M), gu.dev())
    ds.build_shortlist(gu.i32(inp["csr_off"]), gu.i32(inp["csr_tok"]), gu.i32(ids), vs_off, vs_ids[:cap],
                       cpos, ws, st, *un)
    torch.cuda.synchronize()
    return vs_off, vs_ids, cpos, un, st


@pytest.mark.parametrize("name,B", [("tiny", 1), ("small_batched", 5), ("llama_b1", 1), ("batched", 32)])
def test_shortlist_matches_oracle(ds, name, B):
    inp = gu.chain_inputs(name)
    cfg = inp["cfg"]
    B = min(B, inp["H"].shape[0])
    ids, lists = _oracle_lists(inp, B, 1)
    vs_off, vs_ids, cpos, un, st = _gpu_shortlist(ds, inp, ids)
    assert st.item() == 0
    off = vs_off.cpu().numpy()
    got = vs_ids.cpu().numpy()
    cp = cpos.cpu().numpy().reshape(B, cfg.M)
    sizes = np.diff(inp["csr_off"])
    for b in range(B):
        assert np.array_equal(got[off[b]:off[b + 1]], lists[b])
        ref_cpos = np.full(cfg.M, -1)
        run = 0
        for c in ids[b]:
            ref_cpos[c] = run
            run += sizes[c]
        assert np.array_equal(cp[b], ref_cpos)
    assert (got[off[B]:] == -7).all()
    # batch union: clusters selected by any list, ascending, CSR order inside
    sel = np.unique(ids.ravel())
    ref_union = oracle.shortlist(inp["csr_off"], inp["csr_tok"], sel.astype(np.int32))
    n = int(un[2].item())
    assert n == ref_union.size
    assert np.array_equal(un[0].cpu().numpy()[:n], ref_union)
    ucl = un[1].cpu().numpy()[:n]
    assert np.array_equal(ucl, np.repeat(sel, sizes[sel]))


def test_shortlist_all_and_one_cluster(ds):
    inp = gu.chain_inputs("tiny")
    M = inp["cfg"].M
    for k in (M, 1):
        ids = np.arange(k, dtype=np.int32)[None] + (0 if k == M else 17)
        vs_off, vs_ids, _, un, st = _gpu_shortlist(ds, inp, ids)
        ref = oracle.shortlist(inp["csr_off"], inp["csr_tok"], ids[0])
        assert np.array_equal(vs_ids.cpu().numpy()[:vs_off[1].item()], ref)
        assert st.item() == 0


def test_shortlist_device_errors(ds):
    inp = gu.chain_inputs("tiny")
    ids, lists = _oracle_lists(inp, 1, 1)
    cap = len(lists[0]) - 10
    vs_off, vs_ids, _, _, st = _gpu_shortlist(ds, inp, ids, union=False, cap=cap)
    assert st.item() & 0x20                                    # capacity bit
    assert (vs_ids.cpu().numpy()[cap:] == -7).all()            # nothing written past the capacity
    bad = ids.copy()
    bad[0, -1] = inp["cfg"].M + 3
    _, _, _, _, st = _gpu_shortlist(ds, inp, bad, union=False)
    assert st.item() & 0x10                                    # bad-index bit


# ---------------------------------------------------------------------------------------
# Batch 1 through a table of the selected clusters (no copied ids)
# ---------------------------------------------------------------------------------------
def _merged_empty_csr(csr_off):
    """The same token order with every odd cluster emptied into the even one before it."""
    off = csr_off.copy()
    M = off.size - 1
    for i in range(1, M, 2):
        off[i] = csr_off[i + 1]
    return off


def _table_step(ds, inp, pos, csr_off, cap=None, T=1.0, copy=True):
    """Router with the list table for position pos, then the table head; also the copy-path
    head on the same cluster ids.  Returns host arrays."""
    cfg = inp["cfg"]
    dev = gu.dev()
    k = cfg.budget[pos - 1]
    V, M = cfg.V, cfg.M
    cap = V if cap is None else cap
    r = ds.Router(gu.bf16(inp["W1"]), gu.bf16(inp["b1"]), gu.bf16(inp["W2"]), gu.bf16(inp["b2"]), cfg.act,
                  cfg.budget)
    H = gu.bf16(inp["H"][:1, pos - 1])
    scores = torch.empty(1, M, dtype=torch.float32, device=dev)
    ids = torch.empty(1, k, dtype=torch.int32, device=dev)
    cpos = torch.full((M,), -9, dtype=torch.int32, device=dev)
    vs_off = torch.full((2,), -9, dtype=torch.int32, device=dev)
    table = torch.full((2 * (k + 1),), -9, dtype=torch.int32, device=dev)
    st = gu.status()
    ws = ds.workspace(r.workspace_bytes(1), dev)
    off_d, tok_d = gu.i32(csr_off), gu.i32(inp["csr_tok"])
    r.topk_list_b1(H, pos, off_d, V, scores, ids, cpos, vs_off, table, cap, ws, st)
    Hh = gu.bf16(inp["H"][:1, pos])
    W = gu.device_head(inp)
    outs = []
    for mode in ("table", "copy") if copy else ("table",):
        logits = torch.full((cap + 64,), float("nan"), dtype=torch.float32, device=dev)
        tok, tix = (torch.full((1,), -5, dtype=torch.int32, device=dev) for _ in range(2))
        rmax, rsum = (torch.empty(1, dtype=torch.float32, device=dev) for _ in range(2))
        wsh = ds.workspace(ds.head_workspace_bytes(1), dev)
        if mode == "table":
            ds.gathered_head_b1_table(Hh, W, table, k, tok_d, T, inp["gumbel_seed"], pos, logits[:cap], tok, tix,
                                      wsh, st, row_max=rmax, row_sumexp=rsum)
        else:
            ids_h = ids.cpu().numpy()
            S = oracle.shortlist(csr_off, inp["csr_tok"], ids_h[0])
            if S.size > cap:
                break
            so = torch.tensor([0, S.size], dtype=torch.int32, device=dev)
            ds.gathered_head(Hh, 1, W, so, gu.i32(S) if S.size else torch.zeros(1, dtype=torch.int32, device=dev),
                             T, inp["gumbel_seed"], pos, logits[:cap], tok, tix, wsh, st, row_max=rmax,
                             row_sumexp=rsum)
        torch.cuda.synchronize()
        outs.append(tuple(x.cpu().numpy() for x in (logits, tok, tix, rmax, rsum)))
    r.close()
    return dict(scores=scores.cpu().numpy()[0], ids=ids.cpu().numpy()[0], cpos=cpos.cpu().numpy(),
                vs_off=vs_off.cpu().numpy(), table=table.cpu().numpy().reshape(k + 1, 2), st=st.item(), outs=outs)


@pytest.mark.parametrize("name,T,empty", [("tiny", 1.0, False), ("tiny", 0.0, True), ("llama_b1", 1.0, False),
                                          ("llama_b1", 0.0, True), ("large_b1_f5", 1.0, False),
                                          ("large_b1_f100", 1.0, False)])
def test_list_table_path_matches_oracle(ds, name, T, empty):
    # The router writes {list start, CSR start} per selected cluster (ascending id) and the list
    # size; the head reads each entry's token through it.  Against the oracle's shortlist of the
    # same clusters, and bit for bit against the head on the copied list.  `empty`: a CSR in
    # which every odd cluster is empty (selected empty clusters must not shift the lookup).
    inp = gu.chain_inputs(name)
    cfg = inp["cfg"]
    csr_off = _merged_empty_csr(inp["csr_off"]) if empty else inp["csr_off"]
    sizes = np.diff(csr_off)
    for pos in sorted({1, 2, cfg.gamma}):
        k = cfg.budget[pos - 1]
        o = _table_step(ds, inp, pos, csr_off, T=T)
        assert o["st"] == 0
        s_ref, _ = oracle.router(inp["H"][:1, pos - 1], inp["W1"], inp["b1"], inp["W2"], inp["b2"], cfg.act)
        assert_close(o["scores"], s_ref[0], "router scores")
        ids = o["ids"]
        assert np.all(np.diff(ids) > 0)
        topk_same_or_excused(ids, s_ref[0], k)
        starts = np.concatenate([[0], np.cumsum(sizes[ids])])
        assert np.array_equal(o["table"][:k, 0], starts[:k])
        assert np.array_equal(o["table"][:k, 1], csr_off[ids])
        assert tuple(o["table"][k]) == (starts[k], 0)
        assert tuple(o["vs_off"]) == (0, starts[k])
        cp = np.full(cfg.M, -1)
        cp[ids] = starts[:k]
        assert np.array_equal(o["cpos"], cp)
        S = oracle.shortlist(csr_off, inp["csr_tok"], ids)
        n = S.size
        logits, tok, tix, rmax, rsum = o["outs"][0]
        l_ref = oracle.head(inp["H"][:1, pos], inp["W"], S)[0]
        assert_close(logits[:n], l_ref, "table head logits")
        assert np.isnan(logits[n:]).all()
        rtok, ridx, m, s = oracle.draft_sample(l_ref, S, T, inp["gumbel_seed"], pos, 0)
        assert_close([rmax[0]], [m], "row max")
        np.testing.assert_allclose(rsum[0], s, rtol=2e-3)
        if token_same_or_excused(int(tix[0]), ridx, l_ref, S, T, inp["gumbel_seed"], pos, 0):
            assert tok[0] == rtok
        assert S[tix[0]] == tok[0]
        for a, b in zip(o["outs"][0], o["outs"][1]):       # same rows, same grid: same bits
            assert np.array_equal(a, b, equal_nan=True)


def test_list_table_capacity_and_bad_csr(ds):
    inp = gu.chain_inputs("tiny")
    cfg = inp["cfg"]
    # a list longer than the caller's logits: reported, and read as empty (nothing written)
    o = _table_step(ds, inp, 1, inp["csr_off"], cap=5)
    assert o["st"] & 0x20
    k = cfg.budget[0]
    assert tuple(o["table"][k]) == (0, 0) and tuple(o["vs_off"]) == (0, 0)
    assert np.isnan(o["outs"][0][0]).all()
    # a CSR slice past V: reported, read as empty
    bad = inp["csr_off"].copy()
    bad[1:] = np.minimum(bad[1:] + cfg.V, 2 * cfg.V)
    bad[-1] = 2 * cfg.V
    o = _table_step(ds, inp, 1, bad, copy=False)
    assert o["st"] & 0x10


# ---------------------------------------------------------------------------------------
# Gathered head
# ---------------------------------------------------------------------------------------
def _run_head(ds, inp, Hrows, G, ids, T, pos, union, free_sms=-1):
    """Head on the GPU for lists built from the oracle's cluster ids; returns host arrays."""
    cfg = inp["cfg"]
    B = ids.shape[0]
    vs_off, vs_ids, cpos, un, st = _gpu_shortlist(ds, inp, ids, union=union)
    cof = torch.empty(cfg.V, dtype=torch.int32, device=gu.dev())
    rk = torch.empty(cfg.V, dtype=torch.int32, device=gu.dev())
    ds.vocab_index(gu.i32(inp["csr_off"]), gu.i32(inp["csr_tok"]), cof, rk, st)
    R = B * G
    logits = torch.full((B * cfg.V * G,), float("nan"), dtype=torch.float32, device=gu.dev())
    tok = torch.empty(R, dtype=torch.int32, device=gu.dev())
    tix = torch.empty(R, dtype=torch.int32, device=gu.dev())
    rmax = torch.empty(R, dtype=torch.float32, device=gu.dev())
    rsum = torch.empty(R, dtype=torch.float32, device=gu.dev())
    ws = ds.workspace(ds.head_workspace_bytes(R), gu.dev())
    ds.gathered_head(gu.bf16(Hrows), G, gu.device_head(inp), vs_off, vs_ids, T, inp["gumbel_seed"], pos,
                     logits, tok, tix, ws, st, cpos=cpos, rank_in_cluster=rk,
                     union=un if union else None, row_max=rmax, row_sumexp=rsum, free_sms=free_sms)
    torch.cuda.synchronize()
    assert st.item() == 0
    return (vs_off.cpu().numpy(), logits.cpu().numpy(), tok.cpu().numpy(), tix.cpu().numpy(),
            rmax.cpu().numpy(), rsum.cpu().numpy())


def _check_head(inp, Hrows, G, ids, T, pos, out, rows_to_check=None):
    vs_off, logits, tok, tix, rmax, rsum = out
    B = ids.shape[0]
    R = B * G
    for r in (range(R) if rows_to_check is None else rows_to_check):
        b, g = divmod(r, G)
        S = oracle.shortlist(inp["csr_off"], inp["csr_tok"], ids[b])
        n = S.size
        l_ref = oracle.head(Hrows[r][None], inp["W"], S)[0]
        base = vs_off[b] * G + g * n
        assert_close(logits[base:base + n], l_ref, f"head logits row {r}")
        rtok, ridx, m, s = oracle.draft_sample(l_ref, S, T, inp["gumbel_seed"], pos, r)
        assert_close([rmax[r]], [m], "row max")
        np.testing.assert_allclose(rsum[r], s, rtol=2e-3)
        if token_same_or_excused(int(tix[r]), ridx, l_ref, S, T, inp["gumbel_seed"], pos, r):
            assert tok[r] == rtok


@pytest.mark.parametrize("name,T", [("tiny", 1.0), ("tiny", 0.0), ("small_batched", 0.8),
                                    ("llama_b1", 1.0), ("llama_b1", 0.0), ("large_b1_f5", 1.0)])
def test_head_per_row_path(ds, name, T):
    inp = gu.chain_inputs(name)
    cfg = inp["cfg"]
    for pos in (1, cfg.gamma):
        ids, _ = _oracle_lists(inp, 1, pos)
        Hrows = inp["H"][:1, pos]
        out = _run_head(ds, inp, Hrows, 1, ids, T, pos, union=False)
        _check_head(inp, Hrows, 1, ids, T, pos, out)


@pytest.mark.parametrize("union", [False, True])
def test_head_free_sms(ds, union):
    # The SMs a head leaves free change only its grid: every SM (0), the default (-1), and more
    # than the GPU has (one SM is still used) each match the oracle.  The per-row path computes
    # every logit in one warp whatever the grid, so its logits, draws and maxima are the same
    # bits; the union GEMM splits its work by the grid (the fp32 parts of a tile add in another
    # grouping), so there the logits agree to rounding.
    inp = gu.chain_inputs("small_batched")
    cfg = inp["cfg"]
    B = 1 if not union else 3
    ids, _ = _oracle_lists(inp, B, 1)
    Hrows = inp["H"][:B, 1]
    outs = [_run_head(ds, inp, Hrows, 1, ids, cfg.T, 1, union, free_sms=f) for f in (-1, 0, 1 << 20)]
    for o in outs:
        _check_head(inp, Hrows, 1, ids, cfg.T, 1, o)
    for o in outs[1:]:
        assert np.array_equal(outs[0][0], o[0])     # list offsets
        if union:
            np.testing.assert_allclose(o[1], outs[0][1], rtol=1e-5, atol=1e-5)
        else:
            for i in (1, 2, 3, 4):                  # logits, tokens, indices, maxima
                assert np.array_equal(outs[0][i], o[i], equal_nan=True)
            np.testing.assert_allclose(o[5], outs[0][5], rtol=1e-5)


def test_head_all_clusters_is_dense_head(ds):
    inp = gu.chain_inputs("small_batched")
    cfg = inp["cfg"]
    ids = np.arange(cfg.M, dtype=np.int32)[None]
    Hrows = inp["H"][:1, 1]
    vs_off, logits, *_ = _run_head(ds, inp, Hrows, 1, ids, 1.0, 1, union=False)
    S = oracle.shortlist(inp["csr_off"], inp["csr_tok"], ids[0])
    dense = wl.bf16_bits_to_f32(Hrows).astype(np.float64) @ wl.bf16_bits_to_f32(inp["W"]).astype(np.float64).T
    assert_close(logits[:cfg.V], dense[0, S], "dense equivalence")


@pytest.mark.parametrize("union", [False, True])
def test_head_rows_longer_than_one_load_round(ds, union):
    # d = 10248: the batch-1 head takes three rounds of loads per row (4096, 4096 and a ragged
    # 2056 columns; the first row's first round is issued before h is staged), the union GEMM
    # 81 k-stages of 128 columns with a ragged last one
    cfg = wl.config("small_batched").with_(name="small_batched_wide", d=10248)
    inp = wl.chain_inputs(cfg, 0, with_head=False)
    inp["W"] = gu._lm_head(cfg.V, cfg.d, inp["seed"])[0]
    B = 3 if union else 1
    for pos in (1, cfg.gamma):
        ids, _ = _oracle_lists(inp, B, pos)
        Hrows = inp["H"][:B, pos]
        out = _run_head(ds, inp, Hrows, 1, ids, cfg.T, pos, union=union)
        _check_head(inp, Hrows, 1, ids, cfg.T, pos, out)


@pytest.mark.parametrize("name,B,G,T", [("small_batched", 5, 1, 0.8), ("small_batched", 5, 1, 0.0),
                                        ("tiny", 1, 3, 1.0), ("small_batched", 3, 7, 1.0),
                                        # 40, 60 and 128 head rows: N = 48, 64 and 128 columns (128
                                        # is the most the union path takes; its stages hold one
                                        # 64-column atom instead of two)
                                        ("small_batched", 5, 8, 1.0), ("small_batched", 5, 12, 0.0),
                                        ("small_batched", 4, 32, 0.8)])
def test_head_union_path(ds, name, B, G, T):
    inp = gu.chain_inputs(name)
    cfg = inp["cfg"]
    rng = np.random.default_rng(3)
    for pos in (1, cfg.gamma):
        ids, _ = _oracle_lists(inp, min(B, inp["H"].shape[0]), pos)
        if ids.shape[0] < B:
            ids = np.concatenate([ids, ids[:B - ids.shape[0]]])
        Hrows = wl.to_bf16_bits(rng.standard_normal((B * G, cfg.d)).astype(np.float32))
        out = _run_head(ds, inp, Hrows, G, ids, T, pos, union=True)
        _check_head(inp, Hrows, G, ids, T, pos, out)


@pytest.mark.parametrize("union", [False, True])
def test_head_empty_lists(ds, union):
    # An empty list gives token = token_idx = -1 and touches no logit; the other lists of the
    # same call are unaffected.  Batch 1 with an empty list; two lists with the first empty;
    # and (union path) an empty union.
    inp = gu.chain_inputs("tiny")
    cfg = inp["cfg"]
    V, M, d = cfg.V, cfg.M, cfg.d
    cof = torch.empty(V, dtype=torch.int32, device=gu.dev())
    rk = torch.empty(V, dtype=torch.int32, device=gu.dev())
    ds.vocab_index(gu.i32(inp["csr_off"]), gu.i32(inp["csr_tok"]), cof, rk, gu.status())
    S1 = oracle.shortlist(inp["csr_off"], inp["csr_tok"], np.array([3, 7], np.int32))
    sizes = np.diff(inp["csr_off"])
    cases = [(1, [np.zeros(0, np.int32)], [[]])]
    if union:
        cases += [(2, [np.zeros(0, np.int32), S1], [[], [3, 7]]), (2, [np.zeros(0, np.int32)] * 2, [[], []])]
    else:
        cases += [(2, [np.zeros(0, np.int32), S1], [[], [3, 7]])]
    rng = np.random.default_rng(11)
    for B, lists, clus in cases:
        offs = np.concatenate([[0], np.cumsum([len(x) for x in lists])]).astype(np.int32)
        ids = np.concatenate(lists + [np.zeros(1, np.int32)]).astype(np.int32)
        cpos = np.full((B, M), -1, np.int32)
        for b, cl in enumerate(clus):
            run = 0
            for c in cl:
                cpos[b, c] = run
                run += sizes[c]
        H = wl.to_bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
        cap = max(int(offs[-1]), 1)
        logits = torch.full((cap,), float("nan"), dtype=torch.float32, device=gu.dev())
        tok = torch.full((B,), 7, dtype=torch.int32, device=gu.dev())
        tix = torch.full((B,), 7, dtype=torch.int32, device=gu.dev())
        st = gu.status()
        ws = ds.workspace(ds.head_workspace_bytes(B), gu.dev())
        un = None
        if union:
            uids = np.concatenate([S1] if any(len(x) for x in lists) else [np.zeros(0, np.int32)]).astype(np.int32)
            ucl = np.concatenate([[c] * sizes[c] for c in (3, 7)]).astype(np.int32) if len(uids) else np.zeros(0, np.int32)
            un = (gu.i32(np.concatenate([uids, [0]])), gu.i32(np.concatenate([ucl, [0]])),
                  gu.i32(np.array([len(uids)], np.int32)))
        ds.gathered_head(gu.bf16(H), 1, gu.device_head(inp), gu.i32(offs), gu.i32(ids), 1.0, inp["gumbel_seed"], 1,
                         logits, tok, tix, ws, st, cpos=gu.i32(cpos.ravel()), rank_in_cluster=rk, union=un)
        torch.cuda.synchronize()
        assert st.item() == 0
        t, j = tok.cpu().numpy(), tix.cpu().numpy()
        for b in range(B):
            if len(lists[b]) == 0:
                assert t[b] == -1 and j[b] == -1, (B, b, t, j)
            else:
                l_ref = oracle.head(H[b:b + 1], inp["W"], lists[b])[0]
                lg = logits.cpu().numpy()[offs[b]:offs[b + 1]]
                assert_close(lg, l_ref, "head logits next to an empty list")
                rtok, ridx, _, _ = oracle.draft_sample(l_ref, lists[b], 1.0, inp["gumbel_seed"], 1, b)
                if token_same_or_excused(int(j[b]), ridx, l_ref, lists[b], 1.0, inp["gumbel_seed"], 1, b):
                    assert t[b] == rtok


@pytest.mark.parametrize("G", [1, 10])
def test_head_union_full_size_sampled(ds, G):
    # Llama-3-8B shape, 32 lists (G=1, batched chain) or 8 lists x 10 nodes (tree): every
    # token / statistic row is checked for a sample of rows, logits of those rows in full.
    inp = gu.chain_inputs("batched")
    B = 32 if G == 1 else 8
    ids, _ = _oracle_lists(inp, B, 1)
    rng = np.random.default_rng(5)
    Hrows = inp["H"][:B, 1] if G == 1 else wl.to_bf16_bits(rng.standard_normal((B * G, 4096)).astype(np.float32))
    out = _run_head(ds, inp, Hrows, G, ids, 0.7, 1, union=True)
    # every row of the first and the last list
    _check_head(inp, Hrows, G, ids, 0.7, 1, out, rows_to_check=list(range(G)) + list(range((B - 1) * G, B * G)))


# ---------------------------------------------------------------------------------------
# Verification
# ---------------------------------------------------------------------------------------
def _host_cpos(inp, ids):
    sizes = np.diff(inp["csr_off"])
    M = inp["cfg"].M
    out = np.full((ids.shape[0], M), -1, np.int32)
    for b in range(ids.shape[0]):
        run = 0
        for c in ids[b]:
            out[b, c] = run
            run += sizes[c]
    return out


def _vocab_index_dev(ds, inp):
    V = inp["cfg"].V
    cof = torch.empty(V, dtype=torch.int32, device=gu.dev())
    rk = torch.empty(V, dtype=torch.int32, device=gu.dev())
    ds.vocab_index(gu.i32(inp["csr_off"]), gu.i32(inp["csr_tok"]), cof, rk, gu.status())
    return cof, rk


def _chain_oracle(inp, B, T):
    ref = oracle.chain_step(inp, T=T, seqs=range(B), verify=False)
    return [ref[b]["positions"] for b in range(B)]


def _check_chain_verify(ds, inp, pos_rows, z, u, T, with_stats=False):
    """pos_rows[b][t]: oracle per-position dicts. Runs GPU verify on the oracle's draft data
    and compares with the oracle's verification of the same data.  with_stats: hand the
    verifier the draft rows' softmax statistics (as the head gives them) instead of letting it
    reduce the draft rows itself."""
    cfg = inp["cfg"]
    B, gamma, V, M = len(pos_rows), cfg.gamma, cfg.V, cfg.M
    cap = B * V
    q = np.zeros((gamma, cap), np.float32)
    offs = np.zeros((gamma, B + 1), np.int32)
    cpos = np.zeros((gamma, B * M), np.int32)
    draft = np.zeros((gamma, B), np.int32)
    for t in range(gamma):
        run = 0
        ids = np.stack([pos_rows[b][t]["ids"] for b in range(B)])
        cpos[t] = _host_cpos(inp, ids).ravel()
        for b in range(B):
            l = pos_rows[b][t]["logits"]
            offs[t, b] = run
            q[t, run:run + l.size] = l.astype(np.float32)
            run += l.size
            draft[t, b] = pos_rows[b][t]["token"]
        offs[t, B] = run
    # the oracle verifies the same fp32-rounded draft logits
    acc_ref, corr_ref = oracle.verify_chain(
        z, [[q[t, offs[t, b]:offs[t, b + 1]].astype(np.float64) for t in range(gamma)] for b in range(B)],
        [[pos_rows[b][t]["S"] for t in range(gamma)] for b in range(B)],
        np.array([[pos_rows[b][t]["idx"] for t in range(gamma)] for b in range(B)]), u, T)
    cof, rk = _vocab_index_dev(ds, inp)
    acc = torch.empty(B, dtype=torch.int32, device=gu.dev())
    corr = torch.empty(B, dtype=torch.int32, device=gu.dev())
    st = gu.status()
    ws = ds.workspace(ds.verify_workspace_bytes(B, gamma, V), gu.dev())
    stats = {}
    if with_stats:
        te = T if T > 0 else 1.0
        qm = np.zeros((gamma, B), np.float32)
        qs = np.zeros((gamma, B), np.float32)
        for t in range(gamma):
            for b in range(B):
                x = q[t, offs[t, b]:offs[t, b + 1]].astype(np.float64) / te
                qm[t, b] = x.max()
                qs[t, b] = np.exp(x - x.max()).sum()
        stats = dict(q_max=gu.f32(qm), q_sumexp=gu.f32(qs))
    ds.verify(gu.f32(z), T, gu.f32(q), gu.i32(offs), gu.i32(cpos), cof, rk, gu.i32(draft), gu.f32(u),
              acc, corr, ws, st, **stats)
    torch.cuda.synchronize()
    assert st.item() == 0
    acc, corr = acc.cpu().numpy(), corr.cpu().numpy()
    n_exact = 0
    for b in range(B):
        if acc[b] != acc_ref[b]:
            t = min(acc[b], acc_ref[b])
            S = pos_rows[b][t]["S"]
            lq = q[t, offs[t, b]:offs[t, b + 1]]
            x = draft[t, b]
            p = softmax_full(z[b, t], T)[x]
            qq = q_dense(lq, S, T, V)[x]
            assert T > 0 and accept_margin(p, qq, u[b, t]) < TIE, (b, acc[b], acc_ref[b])
            continue
        if corr[b] == corr_ref[b]:
            n_exact += 1
            continue
        assert T > 0, (b, corr[b], corr_ref[b])
        t = acc[b]
        p = softmax_full(z[b, t], T)
        if t < gamma:
            S = pos_rows[b][t]["S"]
            w = np.maximum(p - q_dense(q[t, offs[t, b]:offs[t, b + 1]], S, T, V), 0.0)
            if w.sum() <= 0:
                w = p
        else:
            w = p
        assert icdf_acceptable(w, float(u[b, gamma]), int(corr[b])), (b, corr[b], corr_ref[b])
    return acc, acc_ref, n_exact


@pytest.mark.parametrize("name,B,T", [("tiny", 1, 1.0), ("small_batched", 5, 0.8), ("small_batched", 5, 0.0),
                                      ("llama_b1", 1, 1.0)])
@pytest.mark.parametrize("mode", ["independent", "aligned", "half"])
def test_verify_chain(ds, name, B, T, mode):
    inp = gu.chain_inputs(name)
    cfg = inp["cfg"]
    rows = _chain_oracle(inp, B, T)
    z = inp["z"][:B].copy()
    rng = np.random.default_rng(11)
    if mode != "independent":
        # target rows that agree with the draft on the first positions: p ~ q there
        upto = cfg.gamma if mode == "aligned" else cfg.gamma // 2
        for b in range(B):
            for t in range(upto):
                S, l = rows[b][t]["S"], rows[b][t]["logits"]
                z[b, t] = -60.0
                z[b, t, S] = l.astype(np.float32)
                if T == 0.0:
                    z[b, t, rows[b][t]["token"]] += 1.0
    u = inp["u"][:B].copy()
    if mode == "half":
        u[:, :] = wl.open_uniforms(rng, u.shape)
    for trial in range(3):
        acc, acc_ref, n_exact = _check_chain_verify(ds, inp, rows, z, u, T)
        u = wl.open_uniforms(rng, u.shape)
    if mode == "aligned" and T > 0:
        assert acc_ref.mean() > 0.5 * cfg.gamma           # the accept path is exercised


def _synthetic_chain_rows(inp, B, T, rng):
    """Seeded draft data at a workload's sizes without running the drafter: per (sequence,
    position) a random set of budget[t] clusters, its shortlist, N(0, 2^2) draft logits and a
    token drawn from them."""
    cfg = inp["cfg"]
    rows = []
    for b in range(B):
        r = []
        for t in range(cfg.gamma):
            ids = np.sort(rng.choice(cfg.M, cfg.budget[t], replace=False)).astype(np.int32)
            S = oracle.shortlist(inp["csr_off"], inp["csr_tok"], ids)
            l = rng.standard_normal(S.size) * 2.0
            idx = int(np.argmax(l / T + rng.gumbel(size=S.size))) if T > 0 else int(np.argmax(l))
            r.append(dict(ids=ids, S=S, logits=l, token=int(S[idx]), idx=idx))
        rows.append(r)
    return rows


@pytest.mark.parametrize("T", [0.7, 0.0])
@pytest.mark.parametrize("mode", ["independent", "aligned", "half"])
@pytest.mark.parametrize("with_stats", [False, True])
def test_verify_chain_wide_grid(ds, T, mode, with_stats):
    # The batched workload's sizes (B = 32, gamma = 6, V = 128,256): the verifier takes its wide
    # grid here (8192-element statistics chunks, or with the draft rows' statistics given the
    # pipelined statistics kernel; 2048-element residual chunks without staging), and with
    # target rows that agree with the draft the accept walk runs past t = 1 and, in "aligned",
    # to the bonus draw from row gamma + 1.
    inp = gu.chain_inputs("batched")
    cfg = inp["cfg"]
    B = cfg.B
    rng = np.random.default_rng(23)
    rows = _synthetic_chain_rows(inp, B, T, rng)           # T = 0: greedy drafts (the argmax)
    z = inp["z"][:B].copy()
    if mode != "independent":
        upto = cfg.gamma if mode == "aligned" else cfg.gamma // 2
        for b in range(B):
            for t in range(upto):
                S, l = rows[b][t]["S"], rows[b][t]["logits"]
                z[b, t] = -60.0
                z[b, t, S] = l.astype(np.float32)
                if T == 0.0:
                    z[b, t, rows[b][t]["token"]] += 1.0
    u = inp["u"][:B].copy()
    longest = 0
    for trial in range(2):
        acc, acc_ref, n_exact = _check_chain_verify(ds, inp, rows, z, u, T, with_stats)
        longest = max(longest, int(acc_ref.max()))
        assert n_exact >= B // 2
        u = wl.open_uniforms(rng, u.shape)
    if mode == "aligned":
        assert longest == cfg.gamma                        # a bonus draw was compared
    if mode == "half":
        assert longest >= cfg.gamma // 2


@pytest.mark.parametrize("gamma", [1, 32])
def test_verify_chain_gamma_limits(ds, gamma):
    # the fewest and the most draft positions the chain verifier takes; with target rows that
    # agree with the draft the accept path runs to the end (bonus draw from row gamma + 1)
    cfg = wl.config("tiny").with_(name=f"tiny_gamma{gamma}", gamma=gamma, budget=tuple([8] * gamma))
    inp = wl.chain_inputs(cfg, 0, with_head=False)
    inp["W"] = gu._lm_head(cfg.V, cfg.d, inp["seed"])[0]
    rows = _chain_oracle(inp, 1, cfg.T)
    aligned = inp["z"][:1].copy()
    for t in range(gamma):
        aligned[0, t] = -60.0
        aligned[0, t, rows[0][t]["S"]] = rows[0][t]["logits"].astype(np.float32)
    rng = np.random.default_rng(gamma)
    longest = 0
    for z in (inp["z"][:1].copy(), aligned):
        u = inp["u"][:1].copy()
        for trial in range(4):
            acc, acc_ref, _ = _check_chain_verify(ds, inp, rows, z, u, cfg.T)
            longest = max(longest, int(acc_ref.max()))
            u = wl.open_uniforms(rng, u.shape)
    assert longest >= min(gamma, 8)


def test_verify_tree_size_limits(ds):
    # the widest and deepest tree the walk takes: 32 depths of 64 nodes (64 children at the root)
    cfg = wl.config("tiny_tree")
    B, D, Wd, V, M = 1, 32, 64, cfg.V, cfg.M
    N = D * Wd
    csr_off, csr_tok = wl.cluster_partition(cfg, 0)
    parent = wl.tree_parents(D, Wd)
    rng = np.random.default_rng(13)
    ids = [np.sort(np.stack([rng.choice(M, 6, replace=False) for _ in range(B)]), axis=1) for k in range(D)]
    S = [[oracle.shortlist(csr_off, csr_tok, ids[k][b]) for k in range(D)] for b in range(B)]
    qfp = [[(rng.standard_normal(S[b][n // Wd].size) * 2.0).astype(np.float32) for n in range(N)]
           for b in range(B)]
    didx = np.array([[int(np.argmax(qfp[b][n])) for n in range(N)] for b in range(B)])
    u_node = rng.random((B, N)).astype(np.float32)
    u_res = rng.random((B, D + 1)).astype(np.float32)
    z0 = (rng.standard_normal((B, 1 + N, V)) * 2.0).astype(np.float32)
    for mode in ("independent", "aligned"):
        z = z0 if mode == "independent" else _align_targets(z0, parent, S, qfp, D, Wd)
        acc_ref = _run_tree_verify(ds, V, M, csr_off, csr_tok, parent, D, Wd, ids, S, qfp, didx, z,
                                   u_node, u_res, cfg.T, with_stats=True)
        if mode == "aligned":
            assert acc_ref.sum() >= 4


def _run_tree_verify(ds, V, M, csr_off, csr_tok, parent, D, Wd, ids, S, qfp, didx, z, u_node, u_res, T,
                     with_stats):
    """GPU tree verification on host-built draft data against the oracle's.  ids[k] [B, k_c]
    cluster ids of depth k+1; S[b][k] the lists; qfp[b][n] node n's fp32 draft logits;
    didx [B, N] each node's token index in its list."""
    B = z.shape[0]
    acc_ref, corr_ref, path_ref = oracle.verify_tree(
        z, parent, S, [[q.astype(np.float64) for q in qfp[b]] for b in range(B)], didx, u_node, u_res, T)
    cap = max(sum(S[b][k].size for b in range(B)) for k in range(D))
    q = np.zeros((D, cap * Wd), np.float32)
    ids_dev = np.zeros((D, cap), np.int32)
    offs = np.zeros((D, B + 1), np.int32)
    cpos = np.zeros((D, B * M), np.int32)
    ntok = np.zeros((D, B * Wd), np.int32)
    qmax = np.zeros((D, B * Wd), np.float32)
    qsum = np.zeros((D, B * Wd), np.float32)
    sizes = np.diff(csr_off)
    for k in range(D):
        run = 0
        for b in range(B):
            n_b = S[b][k].size
            offs[k, b] = run
            ids_dev[k, run:run + n_b] = S[b][k]
            row = np.full(M, -1, np.int32)
            pos = 0
            for c in ids[k][b]:
                row[c] = pos
                pos += sizes[c]
            cpos[k, b * M:(b + 1) * M] = row
            for i in range(Wd):
                l = qfp[b][k * Wd + i]
                q[k, run * Wd + i * n_b: run * Wd + (i + 1) * n_b] = l
                ntok[k, b * Wd + i] = S[b][k][didx[b, k * Wd + i]]
                if T > 0:
                    x = l.astype(np.float64) / T
                    qmax[k, b * Wd + i] = np.float32(x.max())
                    qsum[k, b * Wd + i] = np.float32(np.exp(x - x.max()).sum())
            run += n_b
        offs[k, B] = run
    cof = torch.empty(V, dtype=torch.int32, device=gu.dev())
    rk = torch.empty(V, dtype=torch.int32, device=gu.dev())
    ds.vocab_index(gu.i32(csr_off), gu.i32(csr_tok), cof, rk, gu.status())
    acc = torch.empty(B, dtype=torch.int32, device=gu.dev())
    corr = torch.empty(B, dtype=torch.int32, device=gu.dev())
    path = torch.empty(B, D, dtype=torch.int32, device=gu.dev())
    st = gu.status()
    ws = ds.workspace(ds.verify_tree_workspace_bytes(B, D, Wd, V), gu.dev())
    stats = dict(q_max=gu.f32(qmax), q_sumexp=gu.f32(qsum)) if with_stats and T > 0 else {}
    ds.verify_tree(gu.f32(z), D, Wd, T, gu.i32(parent), gu.f32(q), gu.i32(offs), gu.i32(ids_dev), gu.i32(cpos),
                   cof, rk, gu.i32(ntok), gu.f32(u_node), gu.f32(u_res), acc, corr, path, ws, st, **stats)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(acc.cpu().numpy(), acc_ref), (acc.cpu().numpy(), acc_ref)
    assert np.array_equal(path.cpu().numpy(), path_ref)
    corr_gpu = corr.cpu().numpy()
    if not np.array_equal(corr_gpu, corr_ref):
        # inverse-CDF near-tie (fp32 vs fp64 cumulative sums): the GPU's token must lie between
        # the oracle's draws at u_res -/+ ICDF_TOL (the draw is monotone in u)
        assert T > 0
        qd = [[q.astype(np.float64) for q in qfp[b]] for b in range(B)]
        lo = oracle.verify_tree(z, parent, S, qd, didx, u_node, np.clip(u_res - ICDF_TOL, 0, 1).astype(np.float32), T)
        hi = oracle.verify_tree(z, parent, S, qd, didx, u_node, np.clip(u_res + ICDF_TOL, 0, 1).astype(np.float32), T)
        for b in np.nonzero(corr_gpu != corr_ref)[0]:
            assert lo[0][b] == acc_ref[b] and hi[0][b] == acc_ref[b]
            assert lo[1][b] <= corr_gpu[b] <= hi[1][b], (b, corr_gpu[b], corr_ref[b], lo[1][b], hi[1][b])
    return acc_ref


def _align_targets(z, parent, S, qfp, D, Wd, upto=None):
    """Make each node's target row look like its first child's draft row (the accept path),
    for nodes above depth `upto` (all by default)."""
    z = z.copy()
    upto = D if upto is None else upto
    for b in range(z.shape[0]):
        for n in range(-1, D * Wd):
            dep = n // Wd + 1 if n >= 0 else 0
            if dep >= upto:
                continue
            kids = [c for c in range(D * Wd) if parent[c] == n]
            if not kids:
                continue
            z[b, n + 1] = -60.0
            z[b, n + 1, S[b][dep]] = qfp[b][kids[0]]
    return z


@pytest.mark.parametrize("with_stats", [False, True])
def test_verify_tree(ds, with_stats):
    inp = gu.tree_inputs("tiny_tree")
    cfg = inp["cfg"]
    B, D, Wd, V, M = cfg.B, cfg.gamma, cfg.width, cfg.V, cfg.M
    N = D * Wd
    ref = oracle.tree_step(inp, verify=False)
    S = [[ref[b]["depths"][k]["S"] for k in range(D)] for b in range(B)]
    ids = [np.stack([ref[b]["depths"][k]["ids"] for b in range(B)]) for k in range(D)]
    qfp = [[ref[b]["depths"][n // Wd]["nodes"][n % Wd]["logits"].astype(np.float32) for n in range(N)]
           for b in range(B)]
    didx = np.array([[ref[b]["depths"][n // Wd]["nodes"][n % Wd]["idx"] for n in range(N)] for b in range(B)])
    for mode in ("independent", "aligned"):
        z = inp["z"] if mode == "independent" else _align_targets(inp["z"], inp["parent"], S, qfp, D, Wd)
        acc_ref = _run_tree_verify(ds, V, M, inp["csr_off"], inp["csr_tok"], inp["parent"], D, Wd, ids, S, qfp,
                                   didx, z, inp["u_node"], inp["u_res"], cfg.T, with_stats)
        if mode == "aligned":
            assert acc_ref.sum() > 0


@pytest.mark.parametrize("T", [0.8, 0.0])
def test_verify_tree_full_size(ds, T):
    # The tree workload's sizes (V = 128256, M = 1024, B = 8, 6 depths x 10 nodes) with seeded
    # host-built lists and draft rows; the aligned variant walks deep.
    cfg = wl.config("tree")
    B, D, Wd, V, M = cfg.B, cfg.gamma, cfg.width, cfg.V, cfg.M
    N = D * Wd
    csr_off, csr_tok = wl.cluster_partition(cfg, 0)
    parent = wl.tree_parents(D, Wd)
    rng = np.random.default_rng(7)
    ids = [np.sort(np.stack([rng.choice(M, cfg.budget[k], replace=False) for _ in range(B)]), axis=1)
           for k in range(D)]
    S = [[oracle.shortlist(csr_off, csr_tok, ids[k][b]) for k in range(D)] for b in range(B)]
    qfp = [[(rng.standard_normal(S[b][n // Wd].size) * 2.0).astype(np.float32) for n in range(N)]
           for b in range(B)]
    didx = np.array([[int(np.argmax(qfp[b][n])) for n in range(N)] for b in range(B)])
    u_node = rng.random((B, N)).astype(np.float32)
    u_res = rng.random((B, D + 1)).astype(np.float32)
    z0 = (rng.standard_normal((B, 1 + N, V)) * 3.0).astype(np.float32)
    for mode in ("independent", "aligned", "partial"):
        z = z0 if mode == "independent" else _align_targets(z0, parent, S, qfp, D, Wd,
                                                            upto=3 if mode == "partial" else None)
        acc_ref = _run_tree_verify(ds, V, M, csr_off, csr_tok, parent, D, Wd, ids, S, qfp, didx, z,
                                   u_node, u_res, T, with_stats=True)
        if mode == "aligned":
            assert acc_ref.sum() >= B
        if mode == "partial":
            assert (acc_ref >= 1).all() and (acc_ref < D).all()


@pytest.mark.parametrize("B,budget,cap", [(40, (400, 262), 32768), (80, (200, 131), 16384)])
def test_verify_tree_long_lists(ds, B, budget, cap):
    # 40 sequences (clusters of two CTAs: the walk keeps a list of up to 32,768 entries in the
    # cluster's shared memory) or 80 (one CTA each: 16,384) with lists around and above that
    # size, so both the shared-memory residual and the global one are walked, in the same call,
    # against the oracle.
    cfg = wl.config("tree")
    D, Wd, V, M = 2, 4, cfg.V, cfg.M
    N = D * Wd
    csr_off, csr_tok = wl.cluster_partition(cfg, 0)
    parent = wl.tree_parents(D, Wd)
    rng = np.random.default_rng(11)
    ids = [np.sort(np.stack([rng.choice(M, budget[k], replace=False) for _ in range(B)]), axis=1)
           for k in range(D)]
    S = [[oracle.shortlist(csr_off, csr_tok, ids[k][b]) for k in range(D)] for b in range(B)]
    sizes = np.array([[S[b][k].size for k in range(D)] for b in range(B)])
    assert (sizes > cap).any() and (sizes <= cap).any()
    qfp = [[(rng.standard_normal(S[b][n // Wd].size) * 2.0).astype(np.float32) for n in range(N)]
           for b in range(B)]
    didx = np.array([[int(np.argmax(qfp[b][n])) for n in range(N)] for b in range(B)])
    u_node = rng.random((B, N)).astype(np.float32)
    u_res = rng.random((B, D + 1)).astype(np.float32)
    z0 = (rng.standard_normal((B, 1 + N, V)) * 3.0).astype(np.float32)
    for mode in ("independent", "aligned"):
        z = z0 if mode == "independent" else _align_targets(z0, parent, S, qfp, D, Wd)
        acc_ref = _run_tree_verify(ds, V, M, csr_off, csr_tok, parent, D, Wd, ids, S, qfp, didx, z,
                                   u_node, u_res, 0.8, with_stats=True)
        if mode == "aligned":
            assert acc_ref.sum() >= B


# ---------------------------------------------------------------------------------------
# Device-side errors: an id the kernels cannot use sets DS_DEV_BAD_INDEX (0x10) in the status
# word; nothing faults and the other rows of the call are still computed.
# ---------------------------------------------------------------------------------------
BAD_INDEX = 0x10


@pytest.mark.parametrize("union", [False, True])
def test_head_bad_token_id_sets_status(ds, union):
    inp = gu.chain_inputs("tiny")
    cfg = inp["cfg"]
    V, M, d = cfg.V, cfg.M, cfg.d
    cof = torch.empty(V, dtype=torch.int32, device=gu.dev())
    rk = torch.empty(V, dtype=torch.int32, device=gu.dev())
    ds.vocab_index(gu.i32(inp["csr_off"]), gu.i32(inp["csr_tok"]), cof, rk, gu.status())
    ids = np.array([[3, 7]], np.int32)
    S = oracle.shortlist(inp["csr_off"], inp["csr_tok"], ids[0]).copy()
    S[5] = V + 17                                       # not a token id
    cpos = _host_cpos(inp, ids)
    H = wl.to_bf16_bits(np.random.default_rng(2).standard_normal((1, d)).astype(np.float32))
    logits = torch.full((S.size,), float("nan"), dtype=torch.float32, device=gu.dev())
    tok = torch.empty(1, dtype=torch.int32, device=gu.dev())
    tix = torch.empty(1, dtype=torch.int32, device=gu.dev())
    st = gu.status()
    ws = ds.workspace(ds.head_workspace_bytes(1), gu.dev())
    un = None
    if union:
        sizes = np.diff(inp["csr_off"])
        ucl = np.concatenate([[c] * sizes[c] for c in ids[0]]).astype(np.int32)
        un = (gu.i32(S), gu.i32(ucl), gu.i32(np.array([S.size], np.int32)))
    ds.gathered_head(gu.bf16(H), 1, gu.device_head(inp), gu.i32(np.array([0, S.size], np.int32)), gu.i32(S),
                     1.0, inp["gumbel_seed"], 1, logits, tok, tix, ws, st, cpos=gu.i32(cpos.ravel()),
                     rank_in_cluster=rk, union=un)
    torch.cuda.synchronize()
    assert st.item() & BAD_INDEX
    good = np.delete(np.arange(S.size), 5)
    l_ref = oracle.head(H, inp["W"], S[good])[0]
    assert_close(logits.cpu().numpy()[good], l_ref, "head logits beside a bad id")


def test_verify_draft_token_outside_its_list_sets_status(ds):
    inp = gu.chain_inputs("tiny")
    cfg = inp["cfg"]
    rows = _chain_oracle(inp, 1, 1.0)
    V, M, gamma = cfg.V, cfg.M, cfg.gamma
    q = np.zeros((gamma, V), np.float32)
    offs = np.zeros((gamma, 2), np.int32)
    cpos = np.zeros((gamma, M), np.int32)
    draft = np.zeros((gamma, 1), np.int32)
    for t in range(gamma):
        l = rows[0][t]["logits"]
        q[t, :l.size] = l
        offs[t] = [0, l.size]
        cpos[t] = _host_cpos(inp, rows[0][t]["ids"][None]).ravel()
        draft[t, 0] = rows[0][t]["token"]
    # a token whose cluster the first position's list does not select
    outside = np.setdiff1d(np.arange(V), rows[0][0]["S"])[0]
    draft[0, 0] = outside
    cof, rk = _vocab_index_dev(ds, inp)
    acc = torch.empty(1, dtype=torch.int32, device=gu.dev())
    corr = torch.empty(1, dtype=torch.int32, device=gu.dev())
    st = gu.status()
    ws = ds.workspace(ds.verify_workspace_bytes(1, gamma, V), gu.dev())
    ds.verify(gu.f32(inp["z"][:1]), 1.0, gu.f32(q), gu.i32(offs), gu.i32(cpos), cof, rk, gu.i32(draft),
              gu.f32(inp["u"][:1]), acc, corr, ws, st)
    torch.cuda.synchronize()
    assert st.item() & BAD_INDEX
    assert acc.item() == 0                              # the bad draft is rejected


# ---------------------------------------------------------------------------------------
# Bounded waits: a pipeline wait that runs out of budget gives up, reports DS_DEV_TIMEOUT
# (0x40) in the status word and lets the call return; nothing hangs or faults, and the
# context stays usable.
# ---------------------------------------------------------------------------------------
TIMEOUT = 0x40


def test_bounded_wait_gives_up_and_reports_timeout(ds):
    # The union head (tensor-core GEMM) with a pipeline-wait budget of one cycle: the MMA
    # thread's wait for the first stage cannot be met that fast, so it gives up and the other
    # roles stop after it (the MMA thread still drains its own work before the tensor memory is
    # freed).  Then, with the default budget back and a fresh workspace, the same call is exact.
    inp = gu.chain_inputs("small_batched")
    cfg = inp["cfg"]
    B = 5
    ids, _ = _oracle_lists(inp, B, 1)
    Hrows = inp["H"][:B, 1]
    vs_off, vs_ids, cpos, un, st = _gpu_shortlist(ds, inp, ids, union=True)
    assert st.item() == 0
    cof, rk = _vocab_index_dev(ds, inp)
    R = B
    logits = torch.zeros(B * cfg.V, dtype=torch.float32, device=gu.dev())
    tok = torch.empty(R, dtype=torch.int32, device=gu.dev())
    tix = torch.empty(R, dtype=torch.int32, device=gu.dev())
    statuses = []
    try:
        ds.set_wait_budget(1)
        for trial in range(2):
            st = gu.status()
            ws = ds.workspace(ds.head_workspace_bytes(R), gu.dev())     # a timed-out call's counters stay behind
            ds.gathered_head(gu.bf16(Hrows), 1, gu.device_head(inp), vs_off, vs_ids, 0.8, inp["gumbel_seed"], 1,
                             logits, tok, tix, ws, st, cpos=cpos, rank_in_cluster=rk, union=un)
            torch.cuda.synchronize()
            statuses.append(int(st.item()))
    finally:
        ds.set_wait_budget(0)
    assert all(x & TIMEOUT for x in statuses), statuses
    out = _run_head(ds, inp, Hrows, 1, ids, 0.8, 1, union=True)
    _check_head(inp, Hrows, 1, ids, 0.8, 1, out)
