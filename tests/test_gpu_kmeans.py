"""Spherical k-means over the LM-head rows on the GPU (ds_kmeans_init, ds_kmeans_step: the
offline clustering step before the path) against the oracle's, on the same seeded rows and the
same initial centroids.  One step is compared element by element (assignments bit-exact up to
fp32 near-ties of the scores, the CSR exactly, centroids within fp32 rounding); several steps
run on each side on their own and must end in the same clusters for nearly every token.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle                          # noqa: E402
import workloads as wl                 # noqa: E402
import gpu_util as gu                  # noqa: E402

pytestmark = pytest.mark.gpu

# V, d, M: the Tiny shape; ragged rows (d = 392: a short last k-stage) with 300 centroids (three
# tensor-core launches of 128, 128 and 44 centroids) over several row tiles with a ragged tail
CASES = [(4096, 256, 32), (9001, 392, 300)]
TIE = 1e-4                             # near-tie of two scores, relative to |W_v|


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from dynamic_vocab_draft_gb300 import build
    build.build()
    import dynamic_vocab_draft_gb300 as pkg
    pkg.load_library()
    return pkg.api


def _rows(V, d):
    W = wl.lm_head(wl.config("tiny").with_(V=V, d=d), 3)
    init = np.random.default_rng([V, d]).permutation(V)[:0]
    return W, init


def _gpu_setup(api, W, init_rows, M):
    V, d = W.shape
    Wd = gu.bf16(W)
    cent = torch.empty(M, d, dtype=torch.float32, device=gu.dev())
    inv = torch.empty(V, dtype=torch.float32, device=gu.dev())
    st = gu.status()
    api.kmeans_init(Wd, gu.i32(init_rows), cent, inv, st)
    ws = api.workspace(api.kmeans_workspace_bytes(V, d, M), gu.dev())
    out = dict(assign=torch.empty(V, dtype=torch.int32, device=gu.dev()),
               off=torch.empty(M + 1, dtype=torch.int32, device=gu.dev()),
               tok=torch.empty(V, dtype=torch.int32, device=gu.dev()))
    return Wd, cent, inv, ws, st, out


def _check_csr(assign, off, tok, M):
    V = assign.size
    assert off[0] == 0 and off[M] == V and np.all(np.diff(off) >= 0)
    assert np.array_equal(np.sort(tok), np.arange(V))
    for c in range(M):
        part = tok[off[c]:off[c + 1]]
        assert np.all(np.diff(part) > 0) and np.all(assign[part] == c)


@pytest.mark.parametrize("V,d,M", CASES)
def test_kmeans_init_matches_oracle(api, V, d, M):
    W, _ = _rows(V, d)
    init = np.random.default_rng(M).permutation(V)[:M].astype(np.int32)
    _, cent, inv, _, st, _ = _gpu_setup(api, W, init, M)
    torch.cuda.synchronize()
    assert st.item() == 0
    np.testing.assert_allclose(cent.cpu().numpy(), oracle.kmeans_init(W, init), rtol=0, atol=2e-6)
    Wf = wl.bf16_bits_to_f32(W).astype(np.float64)
    np.testing.assert_allclose(inv.cpu().numpy(), 1.0 / np.linalg.norm(Wf, axis=1), rtol=2e-6)


@pytest.mark.parametrize("V,d,M", CASES)
def test_kmeans_step_matches_oracle(api, V, d, M):
    # both sides start from the oracle's centroids (the GPU takes them rounded to fp32; both
    # score against the same bf16 copy of those)
    W, _ = _rows(V, d)
    init = np.random.default_rng(M + 1).permutation(V)[:M].astype(np.int32)
    cent0 = oracle.kmeans_init(W, init)
    Wd, cent, inv, ws, st, out = _gpu_setup(api, W, init, M)
    cent.copy_(torch.from_numpy(cent0.astype(np.float32)))
    api.kmeans_step(Wd, inv, cent, out["assign"], out["off"], out["tok"], ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    new_ref, a_ref, off_ref, tok_ref, _ = oracle.kmeans_step(W, cent0.astype(np.float32).astype(np.float64))
    a = out["assign"].cpu().numpy()
    off, tok = out["off"].cpu().numpy(), out["tok"].cpu().numpy()
    _check_csr(a, off, tok, M)
    diff = np.nonzero(a != a_ref)[0]
    if diff.size:
        Wf = wl.bf16_bits_to_f32(W).astype(np.float64)
        mub = wl.bf16_bits_to_f32(wl.to_bf16_bits(cent0.astype(np.float32))).astype(np.float64)
        for v in diff:
            s = Wf[v] @ mub.T
            assert abs(s[a[v]] - s[a_ref[v]]) < TIE * np.linalg.norm(Wf[v]), (v, a[v], a_ref[v])
        assert diff.size <= max(2, V // 1000)
    else:
        assert np.array_equal(off, off_ref) and np.array_equal(tok, tok_ref)
        np.testing.assert_allclose(cent.cpu().numpy(), new_ref, rtol=1e-4, atol=2e-5)


@pytest.mark.parametrize("V,d,M", CASES)
def test_kmeans_iterations_agree_and_feed_the_path(api, V, d, M):
    # five steps on each side on their own: the same clusters for nearly every token; the GPU's
    # CSR is a valid vocabulary partition for the path (ds_vocab_index inverts it exactly)
    W, _ = _rows(V, d)
    init = np.random.default_rng(M + 2).permutation(V)[:M].astype(np.int32)
    cent_ref = oracle.kmeans_init(W, init)
    Wd, cent, inv, ws, st, out = _gpu_setup(api, W, init, M)
    for _ in range(5):
        cent_ref, a_ref, _, _, _ = oracle.kmeans_step(W, cent_ref)
        api.kmeans_step(Wd, inv, cent, out["assign"], out["off"], out["tok"], ws, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    a = out["assign"].cpu().numpy()
    assert np.mean(a == a_ref) >= 0.99
    off, tok = out["off"].cpu().numpy(), out["tok"].cpu().numpy()
    _check_csr(a, off, tok, M)
    cof = torch.empty(V, dtype=torch.int32, device=gu.dev())
    rk = torch.empty(V, dtype=torch.int32, device=gu.dev())
    api.vocab_index(out["off"], out["tok"], cof, rk, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(cof.cpu().numpy(), a)
    r = rk.cpu().numpy()
    assert np.array_equal(tok[off[a] + r], np.arange(V))
