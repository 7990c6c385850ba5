"""Seeded synthetic inputs for the DynaSpec draft head and its verifier.

This module draws inputs and nothing else: LM-head and router weights, drafter hidden
states, the vocabulary-cluster partition, target logits and the verification uniforms.
It holds none of the method's arithmetic (no router, top-k, shortlist, projection,
softmax, sampling or verification), so both the CUDA path and the CPU oracle can be fed
from it without sharing any of the computation under test.

Shapes follow the workloads the DynaSpec pages describe (Llama-3-8B drafter head,
V = 128,256; DynaSpec summary, "Experiments & Results" and "Key Results"), which need
trained weights and datasets that are not available; every array here is an i.i.d.
synthetic stand-in with the stated shape and distribution.

All randomness comes from numpy's PCG64 (``np.random.default_rng``), which gives the
same stream on x86-64 and aarch64, so a (config, seed) pair names one input set on every
machine.
"""
from __future__ import annotations

import dataclasses
import numpy as np

__all__ = [
    "Config", "CONFIGS", "config", "to_bf16_bits", "bf16_bits_to_f32",
    "cluster_partition", "chain_inputs", "tree_inputs", "open_uniforms",
    "tree_parents", "static_shortlist",
]


@dataclasses.dataclass(frozen=True)
class Config:
    """One synthetic workload.

    V: vocabulary size; d: drafter hidden size; M: number of vocabulary clusters;
    Hr: router hidden width; act: router activation ("relu" or "gelu");
    sizes: cluster-size law, ("uniform", lo, hi) or ("lognormal", sigma_log);
    B: sequences; gamma: draft positions (chain) or tree depth (tree);
    budget: clusters kept per position, length gamma;
    T: temperature (0 = greedy); sigma_p: std of the target logits;
    width: tree nodes per depth (tree workloads only);
    static: size of a fixed shortlist used at every position instead of the router's
    (0: the dynamic shortlist).
    """
    name: str
    V: int
    d: int
    M: int
    Hr: int
    act: str
    sizes: tuple
    B: int
    gamma: int
    budget: tuple
    T: float
    sigma_p: float
    mode: str = "chain"
    width: int = 0
    static: int = 0

    def with_(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


LLAMA_BUDGET = (320, 272, 224, 192, 160, 128)


def _large_budget(frac: float) -> tuple:
    k = int(round(frac * 2048))
    return (k,) * 6


CONFIGS = {
    # V=4096, d=256, 32 clusters of U{64..192} tokens, router 256->512->32 GELU.
    "tiny": Config("tiny", V=4096, d=256, M=32, Hr=512, act="gelu",
                   sizes=("uniform", 64, 192), B=1, gamma=4, budget=(8, 6, 4, 2),
                   T=1.0, sigma_p=2.0),
    # Llama-3-8B-shaped drafter head, one sequence, 6-position chain.
    "llama_b1": Config("llama_b1", V=128256, d=4096, M=1024, Hr=1024, act="relu",
                       sizes=("lognormal", 0.5), B=1, gamma=6, budget=LLAMA_BUDGET,
                       T=1.0, sigma_p=3.0),
    "llama_b1_greedy": Config("llama_b1_greedy", V=128256, d=4096, M=1024, Hr=1024,
                              act="relu", sizes=("lognormal", 0.5), B=1, gamma=6,
                              budget=LLAMA_BUDGET, T=0.0, sigma_p=3.0),
    # 32 sequences, each with its own router output and shortlist.
    "batched": Config("batched", V=128256, d=4096, M=1024, Hr=1024, act="relu",
                      sizes=("lognormal", 0.5), B=32, gamma=6, budget=LLAMA_BUDGET,
                      T=0.7, sigma_p=3.0),
    # 8 sequences, tree of depth 6 with 10 nodes per depth sharing the depth's shortlist.
    "tree": Config("tree", V=128256, d=4096, M=1024, Hr=1024, act="relu",
                   sizes=("lognormal", 0.5), B=8, gamma=6, budget=LLAMA_BUDGET,
                   T=1.0, sigma_p=3.0, mode="tree", width=10),
}
# The static-shortlist baseline on the Llama shape: one fixed list of 32,768 tokens at every
# position (the pages compare DynaSpec's ~28K dynamic lists with 32K static ones), with the
# same hidden states, target logits and uniforms as llama_b1.
CONFIGS["llama_b1_static32k"] = CONFIGS["llama_b1"].with_(name="llama_b1_static32k", static=32768)
CONFIGS["tiny_static"] = CONFIGS["tiny"].with_(name="tiny_static", static=1000)
# Small parity cases the oracle finishes in seconds: several tiles, ragged tails (V, d and
# the router width are not multiples of the kernels' tile sizes).
CONFIGS["small_batched"] = Config("small_batched", V=9001, d=392, M=70, Hr=328, act="relu",
                                  sizes=("lognormal", 0.5), B=5, gamma=3, budget=(20, 12, 7),
                                  T=0.8, sigma_p=2.0)
CONFIGS["tiny_tree"] = Config("tiny_tree", V=4096, d=256, M=32, Hr=512, act="gelu",
                              sizes=("uniform", 64, 192), B=2, gamma=3, budget=(8, 6, 4),
                              T=1.0, sigma_p=2.0, mode="tree", width=4)
CONFIGS["small_batched_static"] = CONFIGS["small_batched"].with_(name="small_batched_static", static=2500)
for _b in (1, 8, 64):
    for _f in (5, 10, 20, 40, 100):
        CONFIGS[f"large_b{_b}_f{_f}"] = Config(
            f"large_b{_b}_f{_f}", V=262144, d=2560, M=2048, Hr=1024, act="relu",
            sizes=("lognormal", 0.5), B=_b, gamma=6, budget=_large_budget(_f / 100.0),
            T=1.0, sigma_p=3.0)


def config(name: str, **overrides) -> Config:
    cfg = CONFIGS[name]
    return cfg.with_(**overrides) if overrides else cfg


# --------------------------------------------------------------------------------------
# bf16 storage.  Weights and hidden states are stored as raw bf16 bit patterns (uint16);
# both consumers widen them exactly (bf16 -> f32 -> f64 is exact).
# --------------------------------------------------------------------------------------
def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    step = 1 << 26                      # bounded float32 temporaries for the 1 GB heads
    for i in range(0, n, step):
        m = min(step, n - i)
        x = rng.standard_normal(m, dtype=np.float32)
        x *= np.float32(std)
        out[i:i + m] = to_bf16_bits(x)
    return out.reshape(shape)


def open_uniforms(rng: np.random.Generator, shape) -> np.ndarray:
    """float32 uniforms strictly inside (0, 1): (2*(w >> 9) + 1) * 2^-24 from 32 random bits."""
    w = rng.integers(0, 1 << 32, size=shape, dtype=np.uint64).astype(np.uint32)
    return ((2.0 * (w >> np.uint32(9)).astype(np.float64) + 1.0) * 2.0 ** -24).astype(np.float32)


# --------------------------------------------------------------------------------------
# Vocabulary-cluster partition (stand-in for the offline spherical k-means over LM-head
# rows, DynaSpec summary "Key Novelty"): a seeded random permutation of V cut into M
# clusters, stored as CSR (offsets[M+1], tokens[V]).
# --------------------------------------------------------------------------------------
def cluster_partition(cfg: Config, seed: int):
    rng = np.random.default_rng([seed, 1])
    V, M = cfg.V, cfg.M
    if cfg.sizes[0] == "uniform":
        raw = rng.integers(cfg.sizes[1], cfg.sizes[2] + 1, size=M).astype(np.float64)
    elif cfg.sizes[0] == "lognormal":
        sigma = float(cfg.sizes[1])
        mean = V / M
        mu = np.log(mean) - sigma * sigma / 2.0
        raw = rng.lognormal(mu, sigma, size=M)
    else:
        raise ValueError(cfg.sizes)
    raw = np.maximum(raw, 1.0)
    sizes = np.maximum(np.floor(raw * (V / raw.sum())).astype(np.int64), 1)
    # Rescale to sum exactly V: hand the remainder out one token at a time from cluster 0,
    # or take the excess back from the largest clusters (never below one token).
    rem = V - int(sizes.sum())
    if rem > 0:
        sizes[np.arange(rem) % M] += 1
    while rem < 0:
        i = int(np.argmax(sizes))
        sizes[i] -= 1
        rem += 1
    assert int(sizes.sum()) == V and sizes.min() >= 1
    offsets = np.zeros(M + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(sizes)
    tokens = rng.permutation(V).astype(np.int32)
    return offsets, tokens


def static_shortlist(cfg: Config, seed: int) -> np.ndarray:
    """A fixed shortlist of cfg.static token ids, in list order: the first cfg.static entries of
    a seeded permutation of V.  It stands in for a frequency-ranked list (the most frequent
    tokens of a corpus, highest first), which would need a corpus; like such a list, its ids
    are in no particular order."""
    return np.random.default_rng([seed, 8]).permutation(cfg.V)[:cfg.static].astype(np.int32)


def _router_weights(cfg: Config, seed: int):
    rng = np.random.default_rng([seed, 2])
    return dict(
        W1=_normal_bf16(rng, (cfg.Hr, cfg.d), 0.02),
        b1=_normal_bf16(rng, (cfg.Hr,), 0.02),
        W2=_normal_bf16(rng, (cfg.M, cfg.Hr), 0.02),
        b2=_normal_bf16(rng, (cfg.M,), 0.02),
    )


def lm_head(cfg: Config, seed: int) -> np.ndarray:
    """The drafter LM head W [V, d] as bf16 bits, N(0, 0.02)."""
    return _normal_bf16(np.random.default_rng([seed, 3]), (cfg.V, cfg.d), 0.02)


def _gumbel_seed(seed: int) -> int:
    """The 64-bit key of the counter-based generator that draws the drafter's Gumbel noise."""
    return int(np.random.default_rng([seed, 4]).integers(0, 1 << 63, dtype=np.int64)) | (1 << 63)


def chain_inputs(cfg: Config, seed: int = 0, with_head: bool = True) -> dict:
    """Inputs of one chain speculation step (configs Tiny, Llama, Batched, Large).

    H[b, t] for t = 0..gamma is the drafter hidden state: the router at draft position
    t (1-based) reads H[b, t-1] and the head reads H[b, t].  z[b, t-1] (t = 1..gamma+1)
    are the target model's logits for draft position t over the full vocabulary;
    row gamma+1 serves the bonus token.  u[b, t-1] are the verification uniforms; u[b,
    gamma] drives the correction / bonus draw.
    """
    assert cfg.mode == "chain"
    off, tok = cluster_partition(cfg, seed)
    out = dict(cfg=cfg, seed=seed, csr_off=off, csr_tok=tok, gumbel_seed=_gumbel_seed(seed))
    out.update(_router_weights(cfg, seed))
    rng = np.random.default_rng([seed, 5])
    out["H"] = _normal_bf16(rng, (cfg.B, cfg.gamma + 1, cfg.d), 1.0)
    rng = np.random.default_rng([seed, 6])
    z = rng.standard_normal((cfg.B, cfg.gamma + 1, cfg.V), dtype=np.float32)
    z *= np.float32(cfg.sigma_p)
    out["z"] = z
    out["u"] = open_uniforms(np.random.default_rng([seed, 7]), (cfg.B, cfg.gamma + 1))
    if cfg.static:
        out["static_ids"] = static_shortlist(cfg, seed)
    if with_head:
        out["W"] = lm_head(cfg, seed)
    return out


def tree_parents(depth: int, width: int) -> np.ndarray:
    """Parent of every tree node, nodes numbered depth-major: n = (dep-1)*width + i.

    All depth-1 nodes hang off the root (parent -1); node i at depth dep >= 2 hangs off
    node i // 2 of depth dep-1.  Only the node count (60), the depth (6) and the width (10)
    of this EAGLE-style tree are fixed by the workload; this wiring is one plain choice.
    """
    par = np.empty(depth * width, dtype=np.int32)
    par[:width] = -1
    for dep in range(2, depth + 1):
        for i in range(width):
            par[(dep - 1) * width + i] = (dep - 2) * width + i // 2
    return par


def tree_inputs(cfg: Config, seed: int = 0, with_head: bool = True) -> dict:
    """Inputs of one tree speculation step (config Tree).

    Hr_h[b, dep-1]: hidden state the router reads for depth dep of sequence b.
    Hn[dep-1, b*width + i]: hidden state of node i at depth dep of sequence b (the head row
    that proposes that node's token).  z[b, 0] is the target row at the root, z[b, 1 + n]
    the target row after node n.  u_node[b, n] is node n's acceptance uniform; u_res[b,
    dep] draws the correction when the walk stops at depth dep (0 = root).
    """
    assert cfg.mode == "tree"
    D, Wd = cfg.gamma, cfg.width
    off, tok = cluster_partition(cfg, seed)
    out = dict(cfg=cfg, seed=seed, csr_off=off, csr_tok=tok, gumbel_seed=_gumbel_seed(seed),
               parent=tree_parents(D, Wd))
    out.update(_router_weights(cfg, seed))
    rng = np.random.default_rng([seed, 5])
    out["Hr_h"] = _normal_bf16(rng, (cfg.B, D, cfg.d), 1.0)
    out["Hn"] = _normal_bf16(rng, (D, cfg.B * Wd, cfg.d), 1.0)
    rng = np.random.default_rng([seed, 6])
    z = rng.standard_normal((cfg.B, 1 + D * Wd, cfg.V), dtype=np.float32)
    z *= np.float32(cfg.sigma_p)
    out["z"] = z
    urng = np.random.default_rng([seed, 7])
    out["u_node"] = open_uniforms(urng, (cfg.B, D * Wd))
    out["u_res"] = open_uniforms(urng, (cfg.B, D + 1))
    if with_head:
        out["W"] = lm_head(cfg, seed)
    return out
