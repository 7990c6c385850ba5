"""Whole speculation steps on the GPU (the launch sequence the benchmark times, including the
side-stream router and CUDA-graph replay) against the oracle's whole step on the same seeded
inputs.  Per sequence, positions are compared in order; an excused near-tie ends the
comparison of that sequence (everything after it depends on the tie's outcome).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle                          # noqa: E402
from parity import (assert_close, topk_same_or_excused, token_same_or_excused, TIE,  # noqa: E402
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


def make_chain(pkg, inp, T):
    cfg = inp["cfg"]
    d = pkg.pipeline.ChainDrafter(
        gu.device_head(inp), gu.bf16(inp["W1"]), gu.bf16(inp["b1"]), gu.bf16(inp["W2"]), gu.bf16(inp["b2"]),
        torch.as_tensor(inp["csr_off"]), torch.as_tensor(inp["csr_tok"]),
        B=cfg.B, gamma=cfg.gamma, budget=cfg.budget, act=cfg.act, T=T, seed=inp["gumbel_seed"])
    d.H.copy_(gu.bf16(np.ascontiguousarray(inp["H"].transpose(1, 0, 2))))
    d.z.copy_(gu.f32(inp["z"]))
    d.u.copy_(gu.f32(inp["u"]))
    return d


def compare_chain(inp, d, T, seqs):
    cfg = inp["cfg"]
    ref = oracle.chain_step(inp, T=T, seqs=seqs)
    scores = d.scores.cpu().numpy()
    offs = d.vs_offsets.cpu().numpy()
    ids_all = d.vs_ids.cpu().numpy()
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
            S = ids_all[t, offs[t, b]:offs[t, b + 1]]
            assert np.array_equal(S, p["S"])
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
            pz = softmax_full(inp["z"][b, t], T)[p["token"]]
            qx = q_dense(p["logits"], p["S"], T, cfg.V)[p["token"]]
            assert T > 0 and accept_margin(pz, qx, inp["u"][b, t]) < TIE
            continue
        if corr[b] != r["correction"]:
            assert T > 0
            t = acc[b]
            pz = softmax_full(inp["z"][b, t], T)
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


def test_tree_step_matches_oracle(pkg):
    for name, seqs in (("tiny_tree", None),):
        inp = gu.tree_inputs(name)
        cfg = inp["cfg"]
        d = pkg.pipeline.TreeDrafter(
            gu.device_head(inp), gu.bf16(inp["W1"]), gu.bf16(inp["b1"]), gu.bf16(inp["W2"]), gu.bf16(inp["b2"]),
            torch.as_tensor(inp["csr_off"]), torch.as_tensor(inp["csr_tok"]), inp["parent"],
            B=cfg.B, D=cfg.gamma, Wd=cfg.width, budget=cfg.budget, act=cfg.act, T=cfg.T, seed=inp["gumbel_seed"])
        d.Hr_h.copy_(gu.bf16(np.ascontiguousarray(inp["Hr_h"].transpose(1, 0, 2))))
        d.Hn.copy_(gu.bf16(inp["Hn"]))
        d.z.copy_(gu.f32(inp["z"]))
        d.u_node.copy_(gu.f32(inp["u_node"]))
        d.u_res.copy_(gu.f32(inp["u_res"]))
        d.step()
        torch.cuda.synchronize()
        d.check_status()
        ref = oracle.tree_step(inp)
        Wd, D = cfg.width, cfg.gamma
        offs = d.vs_offsets.cpu().numpy()
        logits = d.logits.cpu().numpy()
        toks = d.tokens.cpu().numpy()
        tix = d.token_idx.cpu().numpy()
        for b in (range(cfg.B) if seqs is None else seqs):
            ok = True
            for k in range(D):
                dp = ref[b]["depths"][k]
                if not topk_same_or_excused(d.cluster_ids[k][b].cpu().numpy(), dp["scores"], cfg.budget[k]):
                    ok = False
                    break
                n_b = dp["S"].size
                for i in range(Wd):
                    base = offs[k, b] * Wd + i * n_b
                    nd = dp["nodes"][i]
                    assert_close(logits[k, base:base + n_b], nd["logits"], "tree head logits")
                    if not token_same_or_excused(int(tix[k, b * Wd + i]), nd["idx"], nd["logits"], dp["S"],
                                                 cfg.T, inp["gumbel_seed"], k + 1, b * Wd + i):
                        ok = False
                    else:
                        assert toks[k, b * Wd + i] == nd["token"]
            if ok:
                assert d.accepted[b].item() == ref[b]["accepted"]
                assert d.path[b].tolist() == ref[b]["path"]
                assert d.correction[b].item() == ref[b]["correction"]
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
