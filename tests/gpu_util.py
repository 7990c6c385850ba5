"""Shared helpers of the GPU tests: device upload and cached seeded inputs."""
from __future__ import annotations

import functools

import numpy as np
import torch

import workloads as wl


def dev():
    return torch.device("cuda:0")


def bf16(a: np.ndarray) -> torch.Tensor:
    """bf16 bit patterns (uint16 numpy) -> bf16 CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev()).view(torch.bfloat16)


def i32(a) -> torch.Tensor:
    return torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32)).to(dev())


def f32(a) -> torch.Tensor:
    return torch.as_tensor(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


@functools.lru_cache(maxsize=2)
def _lm_head(V: int, d: int, seed: int):
    W = wl.lm_head(wl.config("tiny").with_(V=V, d=d), seed)
    return W, bf16(W)


@functools.lru_cache(maxsize=3)
def chain_inputs(name: str, seed: int = 0):
    cfg = wl.config(name)
    inp = wl.chain_inputs(cfg, seed, with_head=False)
    inp["W"] = _lm_head(cfg.V, cfg.d, seed)[0]
    return inp


@functools.lru_cache(maxsize=1)
def tree_inputs(name: str, seed: int = 0):
    cfg = wl.config(name)
    inp = wl.tree_inputs(cfg, seed, with_head=False)
    inp["W"] = _lm_head(cfg.V, cfg.d, seed)[0]
    return inp


def device_head(inp) -> torch.Tensor:
    cfg = inp["cfg"]
    return _lm_head(cfg.V, cfg.d, inp["seed"])[1]


def status() -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=dev())
