"""ds_gathered_head_noalloc: the gathered head for callers that cannot give the library scratch
memory (their device memory belongs to a pool or framework that cannot grow mid-step, or their
plugin interface passes only inputs and outputs).  It must give the same logits, statistics
and draft tokens as ds_gathered_head with a caller workspace, on consecutive calls that reuse
its one fixed scratch array, on both the per-row and the union path.

Kept in a file of its own, collected last; it also runs alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle                          # noqa: E402
from parity import assert_close        # noqa: E402
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


def _lists(inp, B, pos):
    cfg = inp["cfg"]
    s, _ = oracle.router(inp["H"][:B, pos - 1], inp["W1"], inp["b1"], inp["W2"], inp["b2"], cfg.act)
    return oracle.topk(s, cfg.budget[pos - 1])


def _setup(pkg, inp, ids, union):
    api = pkg.api
    cfg = inp["cfg"]
    B = ids.shape[0]
    dev = gu.dev()
    st = gu.status()
    vs_off = torch.zeros(B + 1, dtype=torch.int32, device=dev)
    vs_ids = torch.zeros(B * cfg.V, dtype=torch.int32, device=dev)
    cpos = torch.empty(B * cfg.M, dtype=torch.int32, device=dev)
    un = tuple(torch.zeros(n, dtype=torch.int32, device=dev) for n in (cfg.V, cfg.V, 1)) if union else None
    ws = api.workspace(api.shortlist_workspace_bytes(B, cfg.M), dev)
    api.build_shortlist(gu.i32(inp["csr_off"]), gu.i32(inp["csr_tok"]), gu.i32(ids), vs_off, vs_ids, cpos, ws, st,
                        *(un if union else (None, None, None)))
    cof = torch.empty(cfg.V, dtype=torch.int32, device=dev)
    rk = torch.empty(cfg.V, dtype=torch.int32, device=dev)
    api.vocab_index(gu.i32(inp["csr_off"]), gu.i32(inp["csr_tok"]), cof, rk, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return vs_off, vs_ids, cpos, rk, un


def _outputs(R, cap, dev):
    return dict(logits=torch.full((cap,), float("nan"), device=dev),
                rmax=torch.empty(R, device=dev), rsum=torch.empty(R, device=dev),
                tok=torch.full((R,), -5, dtype=torch.int32, device=dev),
                tix=torch.full((R,), -5, dtype=torch.int32, device=dev))


def _call_noalloc(pkg, H, B, G, W, cfg, vs_off, vs_ids, cpos, rk, un, T, seed, pos, out, st):
    lib = pkg._lib.load()
    P = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None   # noqa: E731
    u = un if un is not None else (None, None, None)
    return lib.ds_gathered_head_noalloc(
        P(H), B, G, P(W), cfg.V, cfg.d, P(vs_off), P(vs_ids), P(cpos), cfg.M, P(rk),
        P(u[0]), P(u[1]), P(u[2]), float(T), seed, pos,
        P(out["logits"]), P(out["rmax"]), P(out["rsum"]), P(out["tok"]), P(out["tix"]), -1,
        P(st), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("name,B,G,T,union", [("tiny", 1, 1, 1.0, False), ("small_batched", 5, 1, 0.0, False),
                                              ("small_batched", 5, 2, 0.8, True), ("tiny", 1, 32, 1.0, True)])
def test_noalloc_head_matches_workspace_head(pkg, name, B, G, T, union):
    inp = gu.chain_inputs(name)
    cfg = inp["cfg"]
    dev = gu.dev()
    rng = np.random.default_rng(17)
    for pos in (1, cfg.gamma):
        ids = _lists(inp, min(B, inp["H"].shape[0]), pos)
        vs_off, vs_ids, cpos, rk, un = _setup(pkg, inp, ids, union)
        R = B * G
        Hrows = gu.bf16(inp["H"][:B, pos] if G == 1 else
                        gu.wl.to_bf16_bits(rng.standard_normal((R, cfg.d)).astype(np.float32)))
        W = gu.device_head(inp)
        cap = B * cfg.V * G
        ref = _outputs(R, cap, dev)
        st = gu.status()
        ws = pkg.api.workspace(pkg.api.head_workspace_bytes(R), dev)
        pkg.api.gathered_head(Hrows, G, W, vs_off, vs_ids, T, inp["gumbel_seed"], pos, ref["logits"], ref["tok"],
                              ref["tix"], ws, st, cpos=cpos, rank_in_cluster=rk, union=un,
                              row_max=ref["rmax"], row_sumexp=ref["rsum"])
        n = int(vs_off[-1].item()) * G
        for call in range(2):                  # two calls in a row share the scratch array
            out = _outputs(R, cap, dev)
            rc = _call_noalloc(pkg, Hrows, B, G, W, cfg, vs_off, vs_ids, cpos, rk, un, T, inp["gumbel_seed"],
                               pos, out, st)
            assert rc == 0, pkg._lib.load().ds_status_string(rc)
            torch.cuda.synchronize()
            assert st.item() == 0
            assert_close(out["logits"][:n].cpu().numpy(), ref["logits"][:n].cpu().numpy(), f"logits call {call}")
            assert_close(out["rmax"].cpu().numpy(), ref["rmax"].cpu().numpy(), "row max")
            np.testing.assert_allclose(out["rsum"].cpu().numpy(), ref["rsum"].cpu().numpy(), rtol=1e-5)
            assert torch.equal(out["tok"], ref["tok"]) and torch.equal(out["tix"], ref["tix"])


def test_noalloc_head_rejects_more_rows_than_its_scratch_holds(pkg):
    inp = gu.chain_inputs("tiny")
    cfg = inp["cfg"]
    ids = _lists(inp, 1, 1)
    vs_off, vs_ids, cpos, rk, un = _setup(pkg, inp, ids, True)
    R = 33
    out = _outputs(R, cfg.V * R, gu.dev())
    H = torch.zeros(R, cfg.d, dtype=torch.bfloat16, device=gu.dev())
    rc = _call_noalloc(pkg, H, 1, R, gu.device_head(inp), cfg, vs_off, vs_ids, cpos, rk, un, 1.0, 1, 1, out,
                       gu.status())
    assert rc == 2                             # DS_ERR_UNSUPPORTED, nothing launched
    torch.cuda.synchronize()
    assert (out["tok"] == -5).all()
