"""Thin torch-facing binding of the DynaSpec C ABI: argument marshalling only.

Every function takes CUDA tensors (device memory owned by the caller), checks dtype, device
and contiguity, and calls the library function of the same name on the current (or given)
CUDA stream.  bf16 tensors may be ``torch.bfloat16`` or raw ``torch.int16``/``uint16`` bits.
All computation happens in the library's kernels.
"""
from __future__ import annotations

import torch

from . import _lib

ACT = {"relu": 0, "gelu": 1}


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t, dtypes, name, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtypes and t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


BF16 = (torch.bfloat16, torch.int16, torch.uint16)
I32 = (torch.int32,)
F32 = (torch.float32,)


def workspace(nbytes: int, device) -> torch.Tensor:
    """Zero-filled scratch of at least `nbytes` (the counters it may hold start at zero)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def router_workspace_bytes(B, Hr):
    return int(_lib.load().ds_router_workspace_bytes(B, Hr))


def shortlist_workspace_bytes(B, M):
    return int(_lib.load().ds_shortlist_workspace_bytes(B, M))


def head_workspace_bytes(rows):
    return int(_lib.load().ds_head_workspace_bytes(rows))


def verify_workspace_bytes(B, gamma, V):
    return int(_lib.load().ds_verify_workspace_bytes(B, gamma, V))


def verify_tree_workspace_bytes(B, D, Wd, V):
    return int(_lib.load().ds_verify_tree_workspace_bytes(B, D, Wd, V))


OP = {"router": 1, "shortlist": 2, "head": 3, "verify": 4, "verify_tree": 5}


def workspace_bytes(op, B, V=0, M=0, gamma=0, hidden=0, width=0):
    """ds_workspace_bytes: the workspace of call `op` (a name of OP) for the given sizes."""
    return int(_lib.load().ds_workspace_bytes(OP[op], B, V, M, gamma, hidden, width))


def set_wait_budget(cycles: int) -> None:
    """ds_set_wait_budget: cycles a kernel's bounded pipeline wait may take (0 = default)."""
    _lib.check(_lib.load().ds_set_wait_budget(int(cycles)), "ds_set_wait_budget")


class Router:
    """A router handle (ds_router_create): W1 [Hr, d], b1 [Hr], W2 [M, Hr], b2 [M] (CUDA
    tensors that must outlive the handle), the activation and the per-position budget table."""

    def __init__(self, W1, b1, W2, b2, act, budget):
        import ctypes
        self.Hr, self.d = W1.shape
        self.M = W2.shape[0]
        self._keep = (W1, b1, W2, b2)
        bud = torch.as_tensor(list(budget), dtype=torch.int32).contiguous()
        h = ctypes.c_void_p()
        _lib.check(_lib.load().ds_router_create(
            ctypes.byref(h), _ptr(W1, BF16, "W1"), _ptr(b1, BF16, "b1"), _ptr(W2, BF16, "W2"),
            _ptr(b2, BF16, "b2"), self.d, self.Hr, self.M, ACT.get(act, act), bud.data_ptr(),
            bud.numel()), "ds_router_create")
        self.handle = h

    def workspace_bytes(self, B):
        return int(_lib.load().ds_router_workspace_bytes_h(self.handle, B))

    def topk(self, H, pos, scores, cluster_ids, ws, status, stream=None, sms=-1):
        """ds_router_topk_h for draft position `pos` (1-based); scores may be None; sms: SMs to
        size the launches for (-1: the library's default)."""
        B = H.shape[0]
        _lib.check(_lib.load().ds_router_topk_h(
            self.handle, _ptr(H, BF16, "H"), B, int(pos), _ptr(scores, F32, "scores", True),
            _ptr(cluster_ids, I32, "cluster_ids"), int(sms), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
            _ptr(status, I32, "status"), _stream(stream)), "ds_router_topk_h")

    def topk_list_b1(self, H, pos, csr_off, V, scores, cluster_ids, cpos, vs_offsets, list_table, capacity,
                     ws, status, stream=None, sms=-1):
        """ds_router_topk_list_b1: batch 1, the router and top-k of position `pos` with the list's
        table (list_table [2 (k+1)] int32), cpos [M] and vs_offsets [2] instead of copied ids."""
        _lib.check(_lib.load().ds_router_topk_list_b1(
            self.handle, _ptr(H, BF16, "H"), int(pos), _ptr(csr_off, I32, "csr_off"), int(V),
            _ptr(scores, F32, "scores"), _ptr(cluster_ids, I32, "cluster_ids"), _ptr(cpos, I32, "cpos"),
            _ptr(vs_offsets, I32, "vs_offsets"), _ptr(list_table, I32, "list_table"), int(capacity),
            int(sms), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _ptr(status, I32, "status"),
            _stream(stream)), "ds_router_topk_list_b1")

    def close(self):
        if getattr(self, "handle", None):
            _lib.load().ds_router_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def vocab_index(csr_off, csr_tok, cluster_of, rank_in_cluster, status, stream=None):
    M = csr_off.numel() - 1
    V = csr_tok.numel()
    _lib.check(_lib.load().ds_vocab_index(
        _ptr(csr_off, I32, "csr_off"), _ptr(csr_tok, I32, "csr_tok"), M, V,
        _ptr(cluster_of, I32, "cluster_of"), _ptr(rank_in_cluster, I32, "rank_in_cluster"),
        _ptr(status, I32, "status"), _stream(stream)), "ds_vocab_index")


def router_topk(H, W1, b1, W2, b2, act, budget, pos, scores, cluster_ids, ws, status, stream=None, sms=-1):
    """budget: host int32 tensor / sequence of clusters kept per draft position; sms: SMs to size
    the launches for (-1: the library's default)."""
    B, d = H.shape
    Hr = W1.shape[0]
    M = W2.shape[0]
    bud = torch.as_tensor(budget, dtype=torch.int32).contiguous()
    _lib.check(_lib.load().ds_router_topk(
        _ptr(H, BF16, "H"), B, d, _ptr(W1, BF16, "W1"), _ptr(b1, BF16, "b1"), Hr,
        _ptr(W2, BF16, "W2"), _ptr(b2, BF16, "b2"), M, ACT.get(act, act),
        bud.data_ptr(), bud.numel(), int(pos),
        _ptr(scores, F32, "scores"), _ptr(cluster_ids, I32, "cluster_ids"), int(sms),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _ptr(status, I32, "status"),
        _stream(stream)), "ds_router_topk")


def build_shortlist(csr_off, csr_tok, cluster_ids, vs_offsets, vs_ids, cpos, ws, status,
                    union_ids=None, union_cluster=None, union_count=None, stream=None):
    M = csr_off.numel() - 1
    V = csr_tok.numel()
    B, k = cluster_ids.shape
    _lib.check(_lib.load().ds_build_shortlist(
        _ptr(csr_off, I32, "csr_off"), _ptr(csr_tok, I32, "csr_tok"), M, V,
        _ptr(cluster_ids, I32, "cluster_ids"), B, k,
        _ptr(vs_offsets, I32, "vs_offsets"), _ptr(vs_ids, I32, "vs_ids"), vs_ids.numel(),
        _ptr(cpos, I32, "cpos"),
        _ptr(union_ids, I32, "union_ids", True), _ptr(union_cluster, I32, "union_cluster", True),
        _ptr(union_count, I32, "union_count", True),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _ptr(status, I32, "status"),
        _stream(stream)), "ds_build_shortlist")


def gathered_head(H, G, W, vs_offsets, vs_ids, T, seed, pos, logits, token, token_idx, ws, status,
                  cpos=None, rank_in_cluster=None, union=None, row_max=None, row_sumexp=None,
                  stream=None, free_sms=-1):
    """H [B*G, d]; union = (union_ids, union_cluster, union_count) or None (per-row path);
    free_sms: SMs left free for other streams (-1: the library's default, 0: none)."""
    R, d = H.shape
    B = vs_offsets.numel() - 1
    if R != B * G:
        raise ValueError(f"H has {R} rows, expected B*G = {B}*{G}")
    V = W.shape[0]
    M = cpos.numel() // B if cpos is not None else 0
    uids, ucl, ucnt = union if union is not None else (None, None, None)
    _lib.check(_lib.load().ds_gathered_head(
        _ptr(H, BF16, "H"), B, G, _ptr(W, BF16, "W"), V, d,
        _ptr(vs_offsets, I32, "vs_offsets"), _ptr(vs_ids, I32, "vs_ids"),
        _ptr(cpos, I32, "cpos", True), M, _ptr(rank_in_cluster, I32, "rank_in_cluster", True),
        _ptr(uids, I32, "union_ids", True), _ptr(ucl, I32, "union_cluster", True),
        _ptr(ucnt, I32, "union_count", True),
        float(T), int(seed) & 0xFFFFFFFFFFFFFFFF, int(pos),
        _ptr(logits, F32, "logits"), _ptr(row_max, F32, "row_max", True),
        _ptr(row_sumexp, F32, "row_sumexp", True),
        _ptr(token, I32, "token"), _ptr(token_idx, I32, "token_idx"), int(free_sms),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _ptr(status, I32, "status"),
        _stream(stream)), "ds_gathered_head")


def prefetch_rows(W, vs_ids, offsets, first_rows, blocks=0, stream=None):
    """ds_prefetch_rows: L2 prefetch of the W rows of a list's first `first_rows` entries."""
    V, d = W.shape
    _lib.check(_lib.load().ds_prefetch_rows(
        _ptr(W, BF16, "W"), V, d, _ptr(vs_ids, I32, "vs_ids"), _ptr(offsets, I32, "offsets"), int(first_rows),
        int(blocks), _stream(stream)), "ds_prefetch_rows")


def gathered_head_b1_table(H, W, list_table, k, csr_tok, T, seed, pos, logits, token, token_idx, ws, status,
                           row_max=None, row_sumexp=None, stream=None, free_sms=-1):
    """ds_gathered_head_b1_table: the batch-1 head over the list a table describes (H [d] or [1, d])."""
    V, d = W.shape
    _lib.check(_lib.load().ds_gathered_head_b1_table(
        _ptr(H, BF16, "H"), _ptr(W, BF16, "W"), V, d, _ptr(list_table, I32, "list_table"), int(k),
        _ptr(csr_tok, I32, "csr_tok"), float(T), int(seed) & 0xFFFFFFFFFFFFFFFF, int(pos),
        _ptr(logits, F32, "logits"), _ptr(row_max, F32, "row_max", True), _ptr(row_sumexp, F32, "row_sumexp", True),
        _ptr(token, I32, "token"), _ptr(token_idx, I32, "token_idx"), int(free_sms),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _ptr(status, I32, "status"),
        _stream(stream)), "ds_gathered_head_b1_table")


def verify(p_logits, T, q_logits, vs_offsets, cpos, cluster_of, rank_in_cluster, draft_ids,
           uniforms, accepted_len, correction, ws, status, q_max=None, q_sumexp=None, stream=None):
    """p_logits [B, gamma+1, V]; q_logits [gamma, q_stride]; vs_offsets [gamma, B+1];
    cpos [gamma, B*M]; draft_ids [gamma, B]; uniforms [B, gamma+1]; q_max / q_sumexp
    [gamma, B] optional (the head's row statistics)."""
    B, g1, V = p_logits.shape
    gamma = g1 - 1
    M = cpos.shape[-1] // B
    _lib.check(_lib.load().ds_verify(
        _ptr(p_logits, F32, "p_logits"), B, gamma, V, float(T),
        _ptr(q_logits, F32, "q_logits"), q_logits.stride(0),
        _ptr(q_max, F32, "q_max", True), _ptr(q_sumexp, F32, "q_sumexp", True),
        _ptr(vs_offsets, I32, "vs_offsets"), _ptr(cpos, I32, "cpos"), M,
        _ptr(cluster_of, I32, "cluster_of"), _ptr(rank_in_cluster, I32, "rank_in_cluster"),
        _ptr(draft_ids, I32, "draft_ids"), _ptr(uniforms, F32, "uniforms"),
        _ptr(accepted_len, I32, "accepted_len"), _ptr(correction, I32, "correction"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _ptr(status, I32, "status"),
        _stream(stream)), "ds_verify")


def verify_tree(p_logits, D, Wd, T, parent, q_logits, vs_offsets, vs_ids, cpos, cluster_of,
                rank_in_cluster, node_tokens, u_node, u_res, accepted_len, correction, path,
                ws, status, q_max=None, q_sumexp=None, stream=None):
    """p_logits [B, 1+D*Wd, V]; q_logits [D, q_stride]; vs_offsets [D, B+1]; vs_ids [D, vs_stride];
    cpos [D, B*M]; node_tokens [D, B*Wd]; q_max / q_sumexp [D, B*Wd] optional (the head's row
    statistics)."""
    B, n1, V = p_logits.shape
    M = cpos.shape[-1] // B
    _lib.check(_lib.load().ds_verify_tree(
        _ptr(p_logits, F32, "p_logits"), B, D, Wd, V, float(T), _ptr(parent, I32, "parent"),
        _ptr(q_logits, F32, "q_logits"), q_logits.stride(0),
        _ptr(q_max, F32, "q_max", True), _ptr(q_sumexp, F32, "q_sumexp", True),
        _ptr(vs_offsets, I32, "vs_offsets"), _ptr(vs_ids, I32, "vs_ids"), vs_ids.stride(0),
        _ptr(cpos, I32, "cpos"), M,
        _ptr(cluster_of, I32, "cluster_of"), _ptr(rank_in_cluster, I32, "rank_in_cluster"),
        _ptr(node_tokens, I32, "node_tokens"), _ptr(u_node, F32, "u_node"),
        _ptr(u_res, F32, "u_res"),
        _ptr(accepted_len, I32, "accepted_len"), _ptr(correction, I32, "correction"),
        _ptr(path, I32, "path"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _ptr(status, I32, "status"),
        _stream(stream)), "ds_verify_tree")


def kmeans_workspace_bytes(V, d, M):
    return int(_lib.load().ds_kmeans_workspace_bytes(V, d, M))


def kmeans_init(W, init_rows, cent, inv_norm, status, stream=None):
    """ds_kmeans_init: W [V, d] bf16; init_rows [M] int32; cent [M, d], inv_norm [V] fp32 (out)."""
    V, d = W.shape
    M = init_rows.numel()
    _lib.check(_lib.load().ds_kmeans_init(
        _ptr(W, BF16, "W"), V, d, _ptr(init_rows, I32, "init_rows"), M, _ptr(cent, F32, "cent"),
        _ptr(inv_norm, F32, "inv_norm"), _ptr(status, I32, "status"), _stream(stream)), "ds_kmeans_init")


def kmeans_step(W, inv_norm, cent, assign, csr_off, csr_tok, ws, status, stream=None):
    """ds_kmeans_step: one Lloyd iteration; cent [M, d] fp32 in/out."""
    V, d = W.shape
    M = cent.shape[0]
    _lib.check(_lib.load().ds_kmeans_step(
        _ptr(W, BF16, "W"), V, d, M, _ptr(inv_norm, F32, "inv_norm"), _ptr(cent, F32, "cent"),
        _ptr(assign, I32, "assign"), _ptr(csr_off, I32, "csr_off"), _ptr(csr_tok, I32, "csr_tok"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _ptr(status, I32, "status"),
        _stream(stream)), "ds_kmeans_step")


def drafter_standin_workspace_bytes(d, F):
    return int(_lib.load().ds_drafter_standin_workspace_bytes(d, F))


def drafter_standin(h_prev, x_prev, E, Wfc, Wmix, Wug, Wdn, h_base, scale, h_out, ws, status, stream=None):
    """ds_drafter_standin: h_prev, h_base, h_out [d] bf16; x_prev a one-element int32 CUDA tensor;
    E [V, d]; Wfc [d, 2d]; Wmix [d, d]; Wug [2F, d]; Wdn [d, F]."""
    d = h_prev.numel()
    F = Wdn.shape[1]
    _lib.check(_lib.load().ds_drafter_standin(
        _ptr(h_prev, BF16, "h_prev"), _ptr(x_prev, I32, "x_prev"), E.shape[0], _ptr(E, BF16, "E"),
        _ptr(Wfc, BF16, "Wfc"), _ptr(Wmix, BF16, "Wmix"), _ptr(Wug, BF16, "Wug"), _ptr(Wdn, BF16, "Wdn"),
        d, F, _ptr(h_base, BF16, "h_base"), float(scale), _ptr(h_out, BF16, "h_out"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _ptr(status, I32, "status"),
        _stream(stream)), "ds_drafter_standin")


def philox4x32_10(ctr, seed, out, stream=None):
    n = ctr.shape[0]
    _lib.check(_lib.load().ds_philox4x32_10(
        _ptr(ctr, (torch.int32, torch.uint32), "ctr"), int(seed) & 0xFFFFFFFFFFFFFFFF,
        _ptr(out, (torch.int32, torch.uint32), "out"), n, _stream(stream)), "ds_philox4x32_10")


def copy(dst, src, stream=None):
    """dst <- src (same byte size, both contiguous) by a kernel on `stream`; each side is a CUDA
    tensor or a pinned CPU tensor (see ds_copy)."""
    for t, name in ((dst, "dst"), (src, "src")):
        if not isinstance(t, torch.Tensor) or not t.is_contiguous():
            raise ValueError(f"copy: {name} must be a contiguous tensor")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"copy: {name} must be a CUDA tensor or pinned host memory")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("copy: dst and src differ in size")
    _lib.check(_lib.load().ds_copy(dst.data_ptr(), src.data_ptr(), nbytes, _stream(stream)), "ds_copy")


def event_record(event, stream=None):
    """Record a torch.cuda.Event so that it is timeable inside a captured CUDA graph.  The
    event must already exist (torch creates it on its first ordinary record())."""
    if not event.cuda_event:
        raise ValueError("event_record: record the event once outside capture first")
    _lib.check(_lib.load().ds_event_record(event.cuda_event, _stream(stream)), "ds_event_record")
