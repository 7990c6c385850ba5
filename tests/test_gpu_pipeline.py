"""Whole speculation steps on the GPU (the launch sequence the benchmark times, including the
side-stream router and CUDA-graph replay) against the oracle's whole step on the same seeded
inputs.  Per sequence, positions are compared in order; an excused near-tie ends the
comparison of that sequence (everything after it depends on the tie's outcome).
"""
import functools

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle                          # noqa: E402
from parity import (assert_close, topk_same_or_excused, token_same_or_excused, TIE, ICDF_TOL,  # noqa: E402
                    softmax_full, q_dense, icdf_acceptable, accept_margin)
import gpu_util as gu                  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from dynamic_vocab_draft_gb300 import build
    build.build()
    import dynamic_vocab_draft_gb300 as p
    p.load_library()
    return p


def make_chain(pkg, inp, T, **kw):
    cfg = inp["cfg"]
    d = pkg.pipeline.ChainDrafter(
        gu.device_head(inp), gu.bf16(inp["W1"]), gu.bf16(inp["b1"]), gu.bf16(inp["W2"]), gu.bf16(inp["b2"]),
        torch.as_tensor(inp["csr_off"]), torch.as_tensor(inp["csr_tok"]),
        B=cfg.B, gamma=cfg.gamma, budget=cfg.budget, act=cfg.act, T=T, seed=inp["gumbel_seed"], **kw)
    d.H.copy_(gu.bf16(np.ascontiguousarray(inp["H"].transpose(1, 0, 2))))
    d.z.copy_(gu.f32(inp["z"]))
    d.u.copy_(gu.f32(inp["u"]))
    return d


def compare_chain(inp, d, T, seqs, ref=None, z=None):
    """Compare the drafter's step with the oracle's (`ref`, default: the oracle's whole step on
    the same inputs); z: the target logits the step verified against (default inp["z"])."""
    cfg = inp["cfg"]
    z = inp["z"] if z is None else z
    ref = oracle.chain_step(inp, T=T, seqs=seqs) if ref is None else ref
    scores = d.scores.cpu().numpy()
    offs = d.vs_offsets.cpu().numpy()
    logits = d.logits.cpu().numpy()
    toks = d.tokens.cpu().numpy()
    tix = d.token_idx.cpu().numpy()
    acc = d.accepted.cpu().numpy()
    corr = d.correction.cpu().numpy()
    full = 0
    for b in seqs:
        r = ref[b]
        ok = True
        for t in range(cfg.gamma):
            p = r["positions"][t]
            assert_close(scores[t, b], p["scores"], "router scores")
            cids = d.cluster_ids[t][b].cpu().numpy()
            if not topk_same_or_excused(cids, p["scores"], cfg.budget[t]):
                ok = False
                break
            assert np.array_equal(d.list_ids(t, b), p["S"])
            assert_close(logits[t, offs[t, b]:offs[t, b + 1]], p["logits"], "head logits")
            if not token_same_or_excused(int(tix[t, b]), p["idx"], p["logits"], p["S"], T,
                                         inp["gumbel_seed"], t + 1, b):
                ok = False
                break
            assert toks[t, b] == p["token"]
        if not ok:
            continue
        if acc[b] != r["accepted"]:
            t = min(acc[b], r["accepted"])
            p = r["positions"][t]
            pz = softmax_full(z[b, t], T)[p["token"]]
            qx = q_dense(p["logits"], p["S"], T, cfg.V)[p["token"]]
            assert T > 0 and accept_margin(pz, qx, inp["u"][b, t]) < TIE
            continue
        if corr[b] != r["correction"]:
            assert T > 0
            t = acc[b]
            pz = softmax_full(z[b, t], T)
            if t < cfg.gamma:
                p = r["positions"][t]
                w = np.maximum(pz - q_dense(p["logits"], p["S"], T, cfg.V), 0)
                w = w if w.sum() > 0 else pz
            else:
                w = pz
            assert icdf_acceptable(w, float(inp["u"][b, cfg.gamma]), int(corr[b]))
        full += 1
    return full


@pytest.mark.parametrize("name,T,seqs", [
    ("tiny", None, None), ("small_batched", None, None), ("small_batched", 0.0, None),
    ("llama_b1", 1.0, None), ("llama_b1", 0.0, None),
    ("batched", None, [0, 13, 31]),
    ("large_b1_f5", None, None), ("large_b1_f100", None, None), ("large_b8_f10", None, [0, 7]),
    ("large_b64_f10", None, [0, 21, 42, 63]),
    ("large_b8_f40", None, [0, 5]),          # lists of 40% of a 262,144-token vocabulary
])
def test_chain_step_matches_oracle(pkg, name, T, seqs):
    inp = gu.chain_inputs(name)
    cfg = inp["cfg"]
    T = cfg.T if T is None else T
    seqs = list(range(cfg.B)) if seqs is None else seqs
    d = make_chain(pkg, inp, T)
    d.step()
    torch.cuda.synchronize()
    d.check_status()
    full = compare_chain(inp, d, T, seqs)
    assert full >= max(1, len(seqs) // 2)
    # the same step replayed from a CUDA graph gives the same results, bit for bit
    snap = [x.clone() for x in (d.logits, d.tokens, d.accepted, d.correction)]
    d.capture()
    for _ in range(2):
        d.replay()
    torch.cuda.synchronize()
    for a, b in zip(snap, (d.logits, d.tokens, d.accepted, d.correction)):
        assert torch.equal(a, b)
    # the step with its host transfers (inputs from pinned host memory, the target logits and
    # uniforms on the copy stream, results back in one block): the same results, bit for bit,
    # with the device inputs and outputs wiped before the replay
    out_h = _replay_io(d, early=(d.H,), late=(d.z, d.u))
    assert torch.equal(out_h, torch.cat([snap[2], snap[3], snap[1].flatten()]).cpu())


@pytest.mark.parametrize("name,T", [("tiny", 1.0), ("llama_b1", 1.0), ("llama_b1", 0.0), ("large_b1_f100", 1.0)])
def test_chain_b1_list_table_and_copied_list_agree(pkg, name, T):
    # Batch 1 through the list table, through copied lists (a shortlist launch per position),
    # and with the table at the first position only: the same step, bit for bit, and each
    # matches the oracle.
    inp = gu.chain_inputs(name)
    gamma = inp["cfg"].gamma
    outs = []
    for table in (True, False, [True] + [False] * (gamma - 1)):
        d = make_chain(pkg, inp, T, list_table=table)
        assert d.table_pos == (table if isinstance(table, list) else [table] * gamma)
        d.step()
        torch.cuda.synchronize()
        d.check_status()
        compare_chain(inp, d, T, [0])
        outs.append((d.out.clone(), d.logits.clone(), d.vs_offsets.clone(), d.cpos.clone(), d.token_idx.clone()))
        del d
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["llama_b1", "large_b1_f5"])
def test_chain_b1_side_sms_agree(pkg, name):
    # Batch 1 with the heads leaving 16, 40 or the modelled number of SMs to the routers beside
    # them (and the routers sized for them): the same lists, logits, draws and verification bit
    # for bit (per-row GEMV and top-k do not depend on the grid); the heads' row statistics fold
    # a different number of block partials, so they agree to rounding.  The default matches the
    # oracle.
    inp = gu.chain_inputs(name)
    gamma = inp["cfg"].gamma
    outs = []
    for side in (None, 16, 40):
        d = make_chain(pkg, inp, 1.0, side_sms=side)
        assert d.head_free[-1] == 0 and len(d.head_free) == gamma
        assert d.router_sms == [-1] + d.head_free[:-1]
        if side is not None:
            assert d.head_free[:-1] == [side] * (gamma - 1)
        d.step()
        torch.cuda.synchronize()
        d.check_status()
        if side is None:
            compare_chain(inp, d, 1.0, [0])
        outs.append((d.out.clone(), d.logits.clone(), d.vs_offsets.clone(), d.scores.clone(), d.token_idx.clone(),
                     d.row_max.clone(), d.row_sumexp.clone()))
        del d
    for other in outs[1:]:
        for a, b in zip(outs[0][:5], other[:5]):
            assert torch.equal(a, b)
        assert torch.equal(outs[0][5], other[5])                  # the maximum is exact
        torch.testing.assert_close(outs[0][6], other[6], rtol=1e-5, atol=0)


def _aligned_chain_ref(inp, T, seqs, upto):
    """Target rows that agree with the oracle's draft rows at positions t < upto for the
    sequences `seqs` (z = draft logits on the list, -60 elsewhere), and the oracle's whole step
    verified against them: the accept walk runs past t = 1 (to the bonus draw when upto =
    gamma)."""
    cfg = inp["cfg"]
    dr = oracle.chain_step(inp, T=T, seqs=seqs, verify=False)
    z = inp["z"].copy()
    for b in seqs:
        for t in range(upto):
            p = dr[b]["positions"][t]
            z[b, t] = -60.0
            z[b, t, p["S"]] = p["logits"].astype(np.float32)
    acc, corr = oracle.verify_chain(
        z[seqs], [[p["logits"] for p in dr[b]["positions"]] for b in seqs],
        [[p["S"] for p in dr[b]["positions"]] for b in seqs],
        np.array([[p["idx"] for p in dr[b]["positions"]] for b in seqs]), inp["u"][seqs], T)
    ref = {b: dict(positions=dr[b]["positions"], accepted=int(acc[i]), correction=int(corr[i]))
           for i, b in enumerate(seqs)}
    return z, ref


@pytest.mark.parametrize("name,seqs,upto", [
    ("large_b64_f10", [0, 21, 42, 63], 6), ("large_b64_f10", [5, 50], 3),
    ("batched", [0, 13, 31], 6), ("batched", [4, 20], 3),
])
def test_chain_step_aligned_targets(pkg, name, seqs, upto):
    # Whole steps on the wide verification grid (B = 32 at V = 128,256; B = 64 at V = 262,144)
    # where the sampled sequences' target rows agree with their draft rows, so acceptances,
    # the residual draw after a later rejection and the bonus draw are compared end to end.
    inp = gu.chain_inputs(name)
    cfg = inp["cfg"]
    T = cfg.T
    z, ref = _aligned_chain_ref(inp, T, seqs, upto)
    d = make_chain(pkg, inp, T)
    d.z.copy_(gu.f32(z))
    d.step()
    torch.cuda.synchronize()
    d.check_status()
    full = compare_chain(inp, d, T, seqs, ref=ref, z=z)
    assert full >= max(1, len(seqs) // 2)
    acc = [ref[b]["accepted"] for b in seqs]
    assert max(acc) >= min(upto, cfg.gamma - 1)


@pytest.mark.parametrize("name,T", [("tiny_static", None), ("tiny_static", 0.0), ("small_batched_static", None),
                                    ("llama_b1_static32k", None)])
def test_static_chain_step_matches_oracle(pkg, name, T):
    # The static-shortlist baseline: one fixed list at every position (per-row head at batch 1,
    # the union head at batch 5), the same verification, against the oracle's composition of
    # its head, draw and verification steps on that list.
    inp = gu.chain_inputs(name)
    cfg = inp["cfg"]
    T = cfg.T if T is None else T
    d = pkg.pipeline.StaticChainDrafter(gu.device_head(inp), inp["static_ids"], B=cfg.B, gamma=cfg.gamma, T=T,
                                        seed=inp["gumbel_seed"])
    d.H.copy_(gu.bf16(np.ascontiguousarray(inp["H"].transpose(1, 0, 2))))
    d.z.copy_(gu.f32(inp["z"]))
    d.u.copy_(gu.f32(inp["u"]))
    d.step()
    torch.cuda.synchronize()
    d.check_status()
    ref = oracle.static_chain_step(inp, T=T)
    offs = d.vs_offsets.cpu().numpy()
    ids = d.vs_ids.cpu().numpy()
    logits = d.logits.cpu().numpy()
    tix = d.token_idx.cpu().numpy()
    toks = d.tokens.cpu().numpy()
    full = 0
    for b in range(cfg.B):
        ok = True
        for t in range(cfg.gamma):
            p = ref[b]["positions"][t]
            assert np.array_equal(ids[offs[t, b]:offs[t, b + 1]], p["S"])      # list order kept
            assert_close(logits[t, offs[t, b]:offs[t, b + 1]], p["logits"], "static head logits")
            if not token_same_or_excused(int(tix[t, b]), p["idx"], p["logits"], p["S"], T, inp["gumbel_seed"],
                                         t + 1, b):
                ok = False
                break
            assert toks[t, b] == p["token"]
        if not ok:
            continue
        if d.accepted[b].item() != ref[b]["accepted"]:
            t = min(d.accepted[b].item(), ref[b]["accepted"])
            p = ref[b]["positions"][t]
            pz = softmax_full(inp["z"][b, t], T)[p["token"]]
            qx = q_dense(p["logits"], p["S"], T, cfg.V)[p["token"]]
            assert T > 0 and accept_margin(pz, qx, inp["u"][b, t]) < TIE
            continue
        if d.correction[b].item() != ref[b]["correction"]:
            assert T > 0
            t = ref[b]["accepted"]
            pz = softmax_full(inp["z"][b, t], T)
            if t < cfg.gamma:
                p = ref[b]["positions"][t]
                w = np.maximum(pz - q_dense(p["logits"], p["S"], T, cfg.V), 0)
                w = w if w.sum() > 0 else pz
            else:
                w = pz
            assert icdf_acceptable(w, float(inp["u"][b, cfg.gamma]), int(d.correction[b].item()))
        full += 1
    assert full >= max(1, cfg.B // 2)
    # graph replay gives the same results
    snap = d.out.clone()
    d.capture()
    d.replay()
    torch.cuda.synchronize()
    assert torch.equal(snap, d.out)


def _standin_weights(d, F, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    mk = lambda *shape: (torch.randn(*shape, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    return mk(d, 2 * d), mk(d, d), mk(2 * F, d), mk(d, F)


def test_drafter_standin_numerics(pkg):
    # The drafter stand-in (a measurement helper with the weight volume of an EAGLE step) against
    # the same chain in numpy fp64: h_out = bf16(h_base + scale * Wdn (silu(Wg y2) * (Wu y2))),
    # y2 = Wmix Wfc [h_prev; E[x]].  scale = 0 returns h_base bit for bit; a token outside the
    # vocabulary sets DS_DEV_BAD_INDEX.
    d, F, V = 264, 520, 777
    Wfc, Wmix, Wug, Wdn = _standin_weights(d, F, 3)
    g = torch.Generator(device="cuda").manual_seed(4)
    E = (torch.randn(V, d, generator=g, device="cuda") * 0.5).to(torch.bfloat16)
    h_prev = torch.randn(d, generator=g, device="cuda").to(torch.bfloat16)
    h_base = (torch.randn(d, generator=g, device="cuda") * 0.1).to(torch.bfloat16)
    ws = pkg.api.workspace(pkg.api.drafter_standin_workspace_bytes(d, F), gu.dev())
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)
    # scale 1000 makes the chain's term (~0.4) dominate the base (~0.1), so an error in any layer shows
    for x, scale in ((5, 1000.0), (776, 1000.0), (5, 0.0)):
        x_prev = torch.tensor([x], dtype=torch.int32, device="cuda")
        out = torch.empty(d, dtype=torch.bfloat16, device="cuda")
        st = gu.status()
        pkg.api.drafter_standin(h_prev, x_prev, E, Wfc, Wmix, Wug, Wdn, h_base, scale, out, ws, st)
        torch.cuda.synchronize()
        assert st.item() == 0
        if scale == 0.0:
            assert torch.equal(out, h_base)
            continue
        u = np.concatenate([f64(h_prev), f64(E[x])])
        y2 = f64(Wmix) @ (f64(Wfc) @ u)
        gg, uu = f64(Wug)[:F] @ y2, f64(Wug)[F:] @ y2
        ref = f64(h_base) + scale * (f64(Wdn) @ (gg / (1.0 + np.exp(-gg)) * uu))
        got = f64(out)
        # one bf16 rounding of the result (8 significant bits) plus fp32 accumulation
        assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-3), np.abs(got - ref).max()
    st = gu.status()
    pkg.api.drafter_standin(h_prev, torch.tensor([V], dtype=torch.int32, device="cuda"), E, Wfc, Wmix, Wug, Wdn,
                            h_base, 1.0, out, ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0x10


@pytest.mark.parametrize("serial", [False, True])
def test_chain_step_with_drafter_standin(pkg, serial):
    # The step with a drafter stand-in before every head (router t+1 waiting for the drafter
    # step that computes the hidden state it reads; or, serial, the routers on the main stream)
    # and scale 0: the hidden states are the workload's, so every result equals the plain
    # step's, bit for bit, eagerly and from a CUDA graph.
    inp = gu.chain_inputs("tiny")
    cfg = inp["cfg"]
    ref = make_chain(pkg, inp, cfg.T)
    ref.step()
    torch.cuda.synchronize()
    d = make_chain(pkg, inp, cfg.T)
    d.attach_drafter(*_standin_weights(cfg.d, 512, 9), scale=0.0)
    d.serial_router = serial
    d.H_base.copy_(d.H)
    d.H[1:].zero_()                                     # computed by the drafter step
    d.x0.fill_(17)
    d.step()
    torch.cuda.synchronize()
    d.check_status()
    assert ref.table_pos == d.table_pos
    for a, b in ((ref.out, d.out), (ref.logits, d.logits), (ref.vs_offsets, d.vs_offsets), (ref.cpos, d.cpos)):
        assert torch.equal(a, b)
    for t in range(cfg.gamma):
        assert np.array_equal(ref.list_ids(t), d.list_ids(t))
    d.enable_head_timing()
    d.enable_overlap_timing()
    d.capture()
    d.out.zero_()
    d.replay(timed=True)
    torch.cuda.synchronize()
    assert torch.equal(ref.out, d.out)
    if not serial:
        ov = d.overlap_times_ms()
        for t in range(1, cfg.gamma):
            # router t starts after the drafter step that produced its input, head t after router t
            assert ov[t][0] >= ov[t - 1][3] - 1e-3 and ov[t][4] >= ov[t][1] - 1e-3


def test_prefetch_rows_changes_no_result(pkg):
    # The side stream's L2 prefetch of the next head's first rows (ds_prefetch_rows) is a hint:
    # the step's outputs are bit for bit those of the step without it, eagerly and from a graph.
    inp = gu.chain_inputs("llama_b1")
    cfg = inp["cfg"]
    outs = []
    for rows in (0, 2176):
        d = pkg.pipeline.ChainDrafter(
            gu.device_head(inp), gu.bf16(inp["W1"]), gu.bf16(inp["b1"]), gu.bf16(inp["W2"]), gu.bf16(inp["b2"]),
            torch.as_tensor(inp["csr_off"]), torch.as_tensor(inp["csr_tok"]),
            B=1, gamma=cfg.gamma, budget=cfg.budget, act=cfg.act, T=cfg.T, seed=inp["gumbel_seed"], prefetch_rows=rows)
        d.H.copy_(gu.bf16(np.ascontiguousarray(inp["H"].transpose(1, 0, 2))))
        d.z.copy_(gu.f32(inp["z"]))
        d.u.copy_(gu.f32(inp["u"]))
        d.capture()
        d.replay()
        torch.cuda.synchronize()
        d.check_status()
        outs.append((d.out.clone(), d.logits.clone()))
        del d
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def _replay_io(d, early, late):
    pin = lambda x: (x.cpu().pin_memory(), x)
    out_h = torch.empty(d.out.shape, dtype=d.out.dtype).pin_memory()
    d.capture_io([pin(x) for x in early], [pin(x) for x in late], out_h)
    for x in tuple(early) + tuple(late) + (d.out,):
        x.zero_()
    out_h.fill_(-7)
    d.replay_io()
    torch.cuda.synchronize()
    d.check_status()
    return out_h


@functools.lru_cache(maxsize=2)
def _tree_draft(name, seqs):
    """The oracle's drafting part of a tree step (routers, lists, node logits and tokens)."""
    return oracle.tree_step(gu.tree_inputs(name), seqs=list(seqs), verify=False)


def _tree_targets(inp, dr, seqs, aligned):
    """Target logits: the workload's, or, for the sampled sequences, rows that agree with the
    first child's draft row at every node (z = that row on the depth's list, -60 elsewhere), so
    the walk accepts deep into the tree."""
    if not aligned:
        return inp["z"]
    cfg = inp["cfg"]
    D, Wd = cfg.gamma, cfg.width
    parent = np.asarray(inp["parent"])
    z = inp["z"].copy()
    for b in seqs:
        for n in range(-1, D * Wd):
            dep = n // Wd + 1 if n >= 0 else 0          # 0-based depth of n's children
            if dep >= D:
                continue
            kids = np.nonzero(parent == n)[0]
            if kids.size == 0:
                continue
            dd = dr[b]["depths"][dep]
            z[b, n + 1] = -60.0
            z[b, n + 1, dd["S"]] = dd["nodes"][int(kids[0]) % Wd]["logits"].astype(np.float32)
    return z


@pytest.mark.parametrize("name,seqs,aligned", [
    ("tiny_tree", (0, 1), False), ("tiny_tree", (0, 1), True),
    ("tree", (0, 5), False), ("tree", (0, 5), True),
])
def test_tree_step_matches_oracle(pkg, name, seqs, aligned):
    # The whole tree step (routers, per-depth lists, node rows on the union head, draws, tree
    # verification) against the oracle, on the tiny tree and at the tree workload's full size
    # (B = 8, 6 depths x 10 nodes, V = 128,256) on sampled sequences, with the workload's
    # target rows and with rows that make the walk accept deep into the tree.
    inp = gu.tree_inputs(name)
    cfg = inp["cfg"]
    D, Wd, T = cfg.gamma, cfg.width, cfg.T
    seqs = list(seqs)
    dr = _tree_draft(name, tuple(seqs))
    z = _tree_targets(inp, dr, seqs, aligned)
    d = pkg.pipeline.TreeDrafter(
        gu.device_head(inp), gu.bf16(inp["W1"]), gu.bf16(inp["b1"]), gu.bf16(inp["W2"]), gu.bf16(inp["b2"]),
        torch.as_tensor(inp["csr_off"]), torch.as_tensor(inp["csr_tok"]), inp["parent"],
        B=cfg.B, D=D, Wd=Wd, budget=cfg.budget, act=cfg.act, T=T, seed=inp["gumbel_seed"])
    d.Hr_h.copy_(gu.bf16(np.ascontiguousarray(inp["Hr_h"].transpose(1, 0, 2))))
    d.Hn.copy_(gu.bf16(inp["Hn"]))
    d.z.copy_(gu.f32(z))
    d.u_node.copy_(gu.f32(inp["u_node"]))
    d.u_res.copy_(gu.f32(inp["u_res"]))
    d.step()
    torch.cuda.synchronize()
    d.check_status()
    N = D * Wd
    Sx = [[dr[b]["depths"][k]["S"] for k in range(D)] for b in seqs]
    Lx = [[dr[b]["depths"][n // Wd]["nodes"][n % Wd]["logits"] for n in range(N)] for b in seqs]
    Ix = np.array([[dr[b]["depths"][n // Wd]["nodes"][n % Wd]["idx"] for n in range(N)] for b in seqs])
    acc_ref, corr_ref, path_ref = oracle.verify_tree(z[seqs], inp["parent"], Sx, Lx, Ix, inp["u_node"][seqs],
                                                     inp["u_res"][seqs], T)
    offs = d.vs_offsets.cpu().numpy()
    logits = d.logits.cpu().numpy()
    toks = d.tokens.cpu().numpy()
    tix = d.token_idx.cpu().numpy()
    full = 0
    for i, b in enumerate(seqs):
        ok = True
        for k in range(D):
            dp = dr[b]["depths"][k]
            if not topk_same_or_excused(d.cluster_ids[k][b].cpu().numpy(), dp["scores"], cfg.budget[k]):
                ok = False
                break
            n_b = dp["S"].size
            assert offs[k, b + 1] - offs[k, b] == n_b
            for j in range(Wd):
                base = offs[k, b] * Wd + j * n_b
                nd = dp["nodes"][j]
                assert_close(logits[k, base:base + n_b], nd["logits"], "tree head logits")
                if not token_same_or_excused(int(tix[k, b * Wd + j]), nd["idx"], nd["logits"], dp["S"],
                                             T, inp["gumbel_seed"], k + 1, b * Wd + j):
                    ok = False
                else:
                    assert toks[k, b * Wd + j] == nd["token"]
            if not ok:
                break
        if not ok:
            continue
        assert d.accepted[b].item() == acc_ref[i], (b, d.accepted[b].item(), acc_ref[i])
        assert d.path[b].tolist() == path_ref[i].tolist()
        cg = d.correction[b].item()
        if cg != corr_ref[i]:
            # inverse-CDF near-tie: the GPU's token lies between the oracle's draws at
            # u_res -/+ ICDF_TOL with the same accepted path
            assert T > 0
            ur = inp["u_res"][seqs]
            lo = oracle.verify_tree(z[seqs], inp["parent"], Sx, Lx, Ix, inp["u_node"][seqs],
                                    np.clip(ur - ICDF_TOL, 0, 1).astype(np.float32), T)
            hi = oracle.verify_tree(z[seqs], inp["parent"], Sx, Lx, Ix, inp["u_node"][seqs],
                                    np.clip(ur + ICDF_TOL, 0, 1).astype(np.float32), T)
            assert lo[0][i] == acc_ref[i] and hi[0][i] == acc_ref[i]
            assert lo[1][i] <= cg <= hi[1][i], (b, cg, corr_ref[i], lo[1][i], hi[1][i])
        full += 1
    assert full >= 1
    if aligned:
        assert max(acc_ref) >= 2                         # the walk went past the first depths
    if name == "tiny_tree" and not aligned:
        # the step with its host transfers gives the same results block
        snap = d.out.clone()
        out_h = _replay_io(d, early=(d.Hr_h, d.Hn), late=(d.z, d.u_node, d.u_res))
        assert torch.equal(out_h, snap.cpu())


@pytest.mark.parametrize("nbytes", [16, 48, 57344, 1 << 20, 7, 1001])
def test_copy_between_pinned_host_and_device(pkg, nbytes):
    # ds_copy in both directions (16-byte vectors when aligned, bytes otherwise), and device to
    # device, against the source bytes
    rng = np.random.default_rng(nbytes)
    src = torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8)).pin_memory()
    dev_buf = torch.full((nbytes,), 7, dtype=torch.uint8, device=gu.dev())
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    dev2 = torch.zeros(nbytes, dtype=torch.uint8, device=gu.dev())
    pkg.api.copy(dev_buf, src)
    pkg.api.copy(dev2, dev_buf)
    pkg.api.copy(back, dev2)
    torch.cuda.synchronize()
    assert torch.equal(dev_buf.cpu(), src)
    assert torch.equal(back, src)
    with pytest.raises(ValueError):
        pkg.api.copy(dev_buf, torch.zeros(nbytes, dtype=torch.uint8))     # pageable host memory
