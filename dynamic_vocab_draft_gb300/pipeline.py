"""One DynaSpec speculation step on one GPU, stage by stage through the C ABI.

Pipeline order (DynaSpec summary, Technical Details > Pipeline Flow): router on a parallel
stream, draft computation on the main stream, a synchronisation, the gathered projection,
then rejection-sampling verification.  Per draft position t the router and shortlist build
(at batch 1 with small budgets: the router and the list's cluster table) run on a side stream (Novel Architectural Elements: the router runs concurrently, on a CUDA
stream of its own), an event marks the shortlist ready, and the main stream waits on that
event before the gathered head.

Dependencies are the method's.  The router of position t reads H_{t-1}, which the drafter
computes from the token drawn at position t-2, so router t waits for head t-2 (routers 1 and 2
read hidden states that exist when the step starts); it then runs beside head t-1 (and, in a
full drafter, beside the drafter computation of H_t).  The head of position t waits for its
shortlist.

Buffers are allocated once per drafter; a step launches kernels only.  ``capture()`` records
one whole step (both streams) into a CUDA graph that ``replay()`` launches in one call.
``capture_io()`` records a step together with the copies of its inputs from pinned host
memory and of its results back to the host: the inputs the drafting stages read are copied
first (up to 2 MB each by a kernel, ds_copy, which skips the copy engine's start-up; larger
ones by the copy engine), then the ones only verification reads (target logits, uniforms) by
the copy engine on a copy stream while the drafting stages run, and the
results (one contiguous block per drafter, ``self.out``) by one ds_copy.  Host-to-device copies
on several streams were measured to take turns on one copy engine, so one copy stream is the
default.
"""
from __future__ import annotations

import numpy as np
import torch

from . import api


def router_launches(B: int) -> int:
    """Kernels one ds_router_topk call launches: two GEMVs at B = 1 or B > 64; two tensor-core
    layers and a top-k in between."""
    return 2 if B == 1 or B > 64 else 3


class _Common:
    def _setup_vocab(self, csr_off, csr_tok, dev):
        self.csr_off = csr_off.to(dev, torch.int32).contiguous()
        self.csr_tok = csr_tok.to(dev, torch.int32).contiguous()
        self.M = self.csr_off.numel() - 1
        self.V = self.csr_tok.numel()
        self.cluster_of = torch.empty(self.V, dtype=torch.int32, device=dev)
        self.rank = torch.empty(self.V, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        api.vocab_index(self.csr_off, self.csr_tok, self.cluster_of, self.rank, self.status)

    def check_status(self):
        s = int(self.status.item())
        if s:
            from . import _lib
            raise _lib.DynaSpecError(f"device status {s:#x}: {_lib.load().ds_status_string(s).decode()}")

    def capture(self):
        """Record one step into a CUDA graph (the step's inputs are the drafter's buffers).  With
        head timing enabled a second graph, with the timing events, is recorded as well."""
        events, self.head_events = self.head_events, None
        self.step()                              # warm up: lazy attributes, library state
        torch.cuda.synchronize()
        self.graph = self._record()
        self.head_events = events
        self.graph_timed = self._record() if events else None
        return self.graph

    def _record(self):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step()
        return g

    def replay(self, timed=False):
        """Launch the captured step; timed=True launches the graph that also records the
        per-head timing events."""
        (self.graph_timed if timed else self.graph).replay()

    def capture_io(self, early, late, out_host, copy_streams=1, kernel_copy_max=2 << 20):
        """Record a step with its host transfers into a CUDA graph (see the module docstring).
        early, late: [(pinned host tensor, device buffer)] copied before the step (by ds_copy up
        to `kernel_copy_max` bytes each, else by the copy engine), and beside the drafting stages
        (each split into `copy_streams` contiguous parts, one per copy stream), respectively;
        out_host: a pinned host tensor shaped like ``self.out`` that receives the results."""
        assert out_host.shape == self.out.shape and out_host.dtype == self.out.dtype
        events, self.head_events = self.head_events, None
        self.step()                              # warm up outside the capture
        torch.cuda.synchronize()
        copies = [torch.cuda.Stream(device=self.dev) for _ in range(max(1, copy_streams))]
        done = [torch.cuda.Event() for _ in copies]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            main = torch.cuda.current_stream(self.dev)
            for h, dv in early:
                if h.numel() * h.element_size() <= kernel_copy_max:
                    api.copy(dv, h)
                else:
                    dv.copy_(h, non_blocking=True)
            # the late copies fork after the early ones: copy-engine transfers queue in the order
            # they become ready, and the drafting stages must not wait behind the target logits
            k = len(copies)
            for i, c in enumerate(copies):
                c.wait_stream(main)
                with torch.cuda.stream(c):
                    for h, dv in late:
                        hf, df = h.view(-1), dv.view(-1)
                        lo, hi = hf.numel() * i // k, hf.numel() * (i + 1) // k
                        if hi > lo:
                            df[lo:hi].copy_(hf[lo:hi], non_blocking=True)
                    done[i].record(c)
            self.step(before_verify=done)
            api.copy(out_host, self.out)
        self.head_events = events
        self.graph_io, self._io_keep = g, (copies, done)
        return g

    def replay_io(self):
        """Launch the step recorded by capture_io() (inputs in, step, results out)."""
        self.graph_io.replay()

    def enable_head_timing(self):
        """Time every position's head launch with CUDA events (also inside a captured graph).
        Call before capture(); read with head_times_ms() after a step or replay."""
        self.head_events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                            for _ in range(self.n_heads())]
        for a, b in self.head_events:          # torch creates the CUDA event on its first record
            a.record()
            b.record()
        torch.cuda.synchronize()

    def head_times_ms(self):
        return [a.elapsed_time(b) for a, b in self.head_events]

    def _run(self, n, before_verify):
        """Enqueue one step of n positions (see the module docstring for the dependencies).
        Events are recorded before anything waits on them, in host order, so the same code
        serves eager execution and graph capture.

        With a drafter stand-in attached (ChainDrafter.attach_drafter) position t first runs the
        drafter step that computes H[t+1] from H[t] and the previous token on the main stream;
        the router of position t+1 reads H[t+1] and so waits for that step; with
        ``serial_router`` the routers run on the main stream right before their heads instead
        (the schedule without overlap, for comparison)."""
        main = torch.cuda.current_stream(self.dev)
        self.side.wait_stream(main)                # the step's inputs are in place
        drafter = getattr(self, "drafter", None)
        serial = getattr(self, "serial_router", False)
        timing = self.head_events is not None and getattr(self, "route_events", None) is not None

        def route(t, after):
            if serial:
                self.route(t)
                self.ready[t].record(main)
                return
            with torch.cuda.stream(self.side):
                if after is not None:
                    self.side.wait_event(after)
                if timing:
                    api.event_record(self.route_events[t][0])
                self.route(t)
                if timing:
                    api.event_record(self.route_events[t][1])
                self.ready[t].record(self.side)

        if drafter is None:
            for t in range(min(2, n)):
                route(t, None)
        elif not serial:
            route(0, None)
        for t in range(n):
            if drafter is not None:
                if timing:
                    api.event_record(self.draft_events[t][0])
                self.draft(t)
                if timing:
                    api.event_record(self.draft_events[t][1])
                self.drafted[t].record(main)
                if serial:
                    route(t, None)
                elif t + 1 < n:
                    route(t + 1, self.drafted[t])
            main.wait_event(self.ready[t])
            if self.head_events:
                api.event_record(self.head_events[t][0])
            self.head(t)
            if self.head_events:
                api.event_record(self.head_events[t][1])
            self.head_done[t].record(main)
            if drafter is None and t + 2 < n:
                route(t + 2, self.head_done[t])
        for ev in before_verify or ():
            main.wait_event(ev)
        self.verify()



# Batch 1: SMs a head leaves to the side stream, where the next position's router runs beside
# it.  Fitted to measurements on GB300 (N SMs, HBM at about 6.7 TB/s): a head over L bytes of W
# rows on n SMs takes about 9 us + L / (n / N x 6.7 TB/s); the router beside it, reading R bytes
# of weights on s SMs at their share of the same HBM, about 21 us + R / (s / N x 6.7 TB/s).  The
# choice is the s in 16, 24, 32, 40 that makes the slower of the two the fastest (the smaller s
# on a tie): 16 beside Llama-size lists, more beside short lists, where the router would
# otherwise hold up the next head (beyond 40 the head itself slows more than the router gains).
SIDE_SMS_CHOICES = (16, 24, 32, 40)


def side_sms_b1(list_bytes, router_bytes, sms):
    bw = 6.7e6                                     # bytes per microsecond
    def span(s):
        head = 9.0 + list_bytes / ((sms - s) / sms * bw)
        router = 21.0 + router_bytes / (s / sms * bw)
        return max(head, router)
    return min(SIDE_SMS_CHOICES, key=lambda s: (span(s), s))


class ChainDrafter(_Common):
    """Chain drafting: B sequences, gamma draft positions, one shortlist per (sequence, position).

    Weights (device tensors, bf16 bits): W [V, d], W1 [Hr, d], b1 [Hr], W2 [M, Hr], b2 [M].
    Per-step inputs are written into ``self.H`` [gamma+1, B, d] (hidden states; the router at
    position t reads H[t-1], the head H[t]), ``self.z`` [B, gamma+1, V] (target logits) and
    ``self.u`` [B, gamma+1] (verification uniforms).

    At batch 1 a list can be named by a table of its selected clusters instead of a copy of its
    token ids (``list_table``): the router's top-k block writes the table and the head reads
    each token through it and the CSR, one launch fewer on the side stream.  The head stages the
    table in shared memory and searches it once per row, which costs it a little, so the default
    (None) takes the table where the launch it saves is on the critical path: at the first
    position (nothing runs before it) and where the previous position's head is too short to
    hide the side stream (it moves less than ``TABLE_PREV_BYTES`` of W on average), and only
    for budgets up to ``TABLE_MAX_K`` clusters.  ``list_table`` may also be a bool (every
    position) or a sequence of gamma bools.
    """

    TABLE_MAX_K = 512
    TABLE_PREV_BYTES = 100e6

    def __init__(self, W, W1, b1, W2, b2, csr_off, csr_tok, *, B, gamma, budget, act, T, seed,
                 union=None, prefetch_rows=0, list_table=None, side_sms=None):
        dev = W.device
        self.dev = dev
        self.W, self.W1, self.b1, self.W2, self.b2 = W, W1, b1, W2, b2
        self._setup_vocab(csr_off, csr_tok, dev)
        self.d = W.shape[1]
        self.Hr = W1.shape[0]
        self.B, self.gamma = B, gamma
        self.budget = torch.tensor(list(budget), dtype=torch.int32)
        self.act, self.T, self.seed = act, float(T), int(seed)
        self.union = (B > 1) if union is None else bool(union)
        # batch 1: the side stream fetches this many of the next head's first W rows into L2
        self.prefetch_rows = int(prefetch_rows) if B == 1 and not self.union else 0
        # batch 1: the list as a table of its selected clusters (no copy of its ids)
        if list_table is None:
            row_bytes = 2.0 * W.shape[1] * W.shape[0] / max(1, int(csr_off.numel()) - 1)   # per cluster
            list_table = [int(budget[t]) <= self.TABLE_MAX_K
                          and (t == 0 or int(budget[t - 1]) * row_bytes < self.TABLE_PREV_BYTES)
                          for t in range(gamma)]
        per_pos = list(list_table) if isinstance(list_table, (list, tuple)) else [bool(list_table)] * gamma
        assert len(per_pos) == gamma
        ok = B == 1 and not self.union and not self.prefetch_rows
        self.table_pos = [bool(x) and ok for x in per_pos]
        self.table_mode = any(self.table_pos)
        # SMs head t leaves free for the router of position t+1 beside it (the last head: none),
        # and the SMs that router sizes its launches for (-1: the library's defaults)
        self.head_free = [-1] * (gamma - 1) + [0]
        if B == 1 and not self.union:
            if side_sms is None:
                nsm = torch.cuda.get_device_properties(dev).multi_processor_count
                cl = W.shape[0] / max(1, int(csr_off.numel()) - 1)           # mean cluster size
                rb = 2.0 * (W1.shape[0] * W1.shape[1] + W2.shape[0] * W2.shape[1])
                side_sms = [side_sms_b1(int(budget[t]) * cl * (2 * self.d + 8), rb, nsm) for t in range(gamma - 1)]
            elif isinstance(side_sms, int):
                side_sms = [side_sms] * (gamma - 1)
            self.head_free = [int(x) for x in side_sms][:gamma - 1] + [0]
        self.router_sms = [-1] + self.head_free[:gamma - 1]
        V, M = self.V, self.M
        cap = B * V
        i32 = dict(dtype=torch.int32, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        self.H = torch.zeros(gamma + 1, B, self.d, dtype=torch.bfloat16, device=dev)
        self.z = torch.zeros(B, gamma + 1, V, **f32)
        self.u = torch.full((B, gamma + 1), 0.5, **f32)
        self.scores = torch.empty(gamma, B, M, **f32)
        self.cluster_ids = [torch.empty(B, int(self.budget[t]), **i32) for t in range(gamma)]
        self.vs_offsets = torch.zeros(gamma, B + 1, **i32)
        self.vs_ids = torch.zeros(gamma, cap, **i32)
        self.cpos = torch.empty(gamma, B * M, **i32)
        if self.table_mode:
            self.list_table = torch.zeros(gamma, 2 * (max(int(x) for x in budget) + 1), **i32)
        if self.union:
            self.union_ids = torch.empty(gamma, V, **i32)
            self.union_cluster = torch.empty(gamma, V, **i32)
            self.union_count = torch.zeros(gamma, 1, **i32)
        self.logits = torch.zeros(gamma, cap, **f32)
        self.row_max = torch.empty(gamma, B, **f32)
        self.row_sumexp = torch.empty(gamma, B, **f32)
        # results in one block: accepted [B], correction [B], draft tokens [gamma, B]
        self.out = torch.empty((2 + gamma) * B, **i32)
        self.accepted = self.out[:B]
        self.correction = self.out[B:2 * B]
        self.tokens = self.out[2 * B:].view(gamma, B)
        self.token_idx = torch.empty(gamma, B, **i32)
        self.router = api.Router(W1, b1, W2, b2, act, budget)
        self.ws_router = [api.workspace(self.router.workspace_bytes(B), dev) for _ in range(gamma)]
        self.ws_short = [api.workspace(api.shortlist_workspace_bytes(B, M), dev) for _ in range(gamma)]
        self.ws_head = api.workspace(api.head_workspace_bytes(B), dev)
        self.ws_verify = api.workspace(api.verify_workspace_bytes(B, gamma, V), dev)
        self.side = torch.cuda.Stream(device=dev)
        self.ready = [torch.cuda.Event() for _ in range(gamma)]
        self.head_done = [torch.cuda.Event() for _ in range(gamma)]
        self.graph = None
        # optional [(start, end)] timing events around each position's head launch
        self.head_events = None

    def route(self, t, stream=None):
        """Router + top-k + shortlist of draft position t (0-based) for all sequences."""
        if self.table_pos[t]:
            self.router.topk_list_b1(self.H[t], t + 1, self.csr_off, self.V, self.scores[t], self.cluster_ids[t],
                                     self.cpos[t], self.vs_offsets[t], self.list_table[t], self.logits.shape[1],
                                     self.ws_router[t], self.status, stream, sms=self.router_sms[t])
            return
        self.router.topk(self.H[t], t + 1, self.scores[t], self.cluster_ids[t], self.ws_router[t], self.status,
                         stream, sms=self.router_sms[t])
        un = (self.union_ids[t], self.union_cluster[t], self.union_count[t]) if self.union else (None,) * 3
        api.build_shortlist(self.csr_off, self.csr_tok, self.cluster_ids[t], self.vs_offsets[t],
                            self.vs_ids[t], self.cpos[t], self.ws_short[t], self.status,
                            un[0], un[1], un[2], stream)
        if self.prefetch_rows and t > 0:
            api.prefetch_rows(self.W, self.vs_ids[t], self.vs_offsets[t], self.prefetch_rows, stream=stream)

    def head(self, t, stream=None):
        # the last position's head has the GPU to itself (no router runs beside it)
        free = self.head_free[t]
        if self.table_pos[t]:
            api.gathered_head_b1_table(self.H[t + 1], self.W, self.list_table[t], int(self.budget[t]), self.csr_tok,
                                       self.T, self.seed, t + 1, self.logits[t], self.tokens[t], self.token_idx[t],
                                       self.ws_head, self.status, row_max=self.row_max[t],
                                       row_sumexp=self.row_sumexp[t], stream=stream, free_sms=free)
            return
        api.gathered_head(self.H[t + 1], 1, self.W, self.vs_offsets[t], self.vs_ids[t], self.T,
                          self.seed, t + 1, self.logits[t], self.tokens[t], self.token_idx[t],
                          self.ws_head, self.status, cpos=self.cpos[t], rank_in_cluster=self.rank,
                          union=(self.union_ids[t], self.union_cluster[t], self.union_count[t])
                          if self.union else None,
                          row_max=self.row_max[t], row_sumexp=self.row_sumexp[t], stream=stream, free_sms=free)

    def verify(self, stream=None):
        api.verify(self.z, self.T, self.logits, self.vs_offsets, self.cpos, self.cluster_of, self.rank,
                   self.tokens, self.u, self.accepted, self.correction, self.ws_verify, self.status,
                   q_max=self.row_max, q_sumexp=self.row_sumexp, stream=stream)

    def step(self, before_verify=None):
        """One speculation step; verification first waits for the events in `before_verify`, if
        given (inputs that only verification reads may still be arriving)."""
        self._run(self.gamma, before_verify)

    def list_ids(self, t, b=0):
        """The token ids of list (t, b) as a host array: copied ids, or (batch 1 with a table) the
        CSR slices of the selected clusters the table names."""
        if not self.table_pos[t]:
            o = self.vs_offsets[t].cpu().numpy()
            return self.vs_ids[t, o[b]:o[b + 1]].cpu().numpy()
        k = int(self.budget[t])
        tab = self.list_table[t, :2 * (k + 1)].cpu().numpy().reshape(k + 1, 2)
        tok = self.csr_tok.cpu().numpy()
        parts = [tok[tab[s, 1]:tab[s, 1] + (tab[s + 1, 0] - tab[s, 0])] for s in range(k)]
        return np.concatenate(parts) if parts else np.zeros(0, np.int32)

    def attach_drafter(self, Wfc, Wmix, Wug, Wdn, scale=0.0, E=None):
        """Put a drafter stand-in (ds_drafter_standin) before every head, batch 1 only.  The step
        then reads H[0] (the hidden state before the first position) and ``self.x0`` (the last
        accepted token) and computes H[t+1] = bf16(H_base[t+1] + scale * f(H[t], x_t)) for
        t = 0..gamma-1, x_t being the token drawn at position t (x0 for t = 0); ``self.H_base``
        [gamma+1, 1, d] holds the base hidden states.  With scale = 0, H[t+1] = H_base[t+1]
        exactly, so results equal those of the plain step on those hidden states.  E: token
        embeddings (default: the LM head, tied)."""
        if self.B != 1:
            raise ValueError("the drafter stand-in runs at batch 1")
        dev = self.dev
        self.drafter = dict(E=self.W if E is None else E, Wfc=Wfc, Wmix=Wmix, Wug=Wug, Wdn=Wdn, scale=float(scale))
        self.H_base = torch.zeros_like(self.H)
        self.x0 = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws_draft = api.workspace(api.drafter_standin_workspace_bytes(self.d, Wdn.shape[1]), dev)
        self.drafted = [torch.cuda.Event() for _ in range(self.gamma)]
        self.serial_router = False

    def draft(self, t, stream=None):
        """The drafter stand-in of position t: H[t+1] from H[t] and the previous token."""
        dr = self.drafter
        x_prev = self.x0 if t == 0 else self.tokens[t - 1]
        api.drafter_standin(self.H[t, 0], x_prev, dr["E"], dr["Wfc"], dr["Wmix"], dr["Wug"], dr["Wdn"],
                            self.H_base[t + 1, 0], dr["scale"], self.H[t + 1, 0], self.ws_draft, self.status,
                            stream=stream)

    def enable_overlap_timing(self):
        """With a drafter attached: also time each position's router + shortlist (side stream)
        and drafter step (main stream) inside the instrumented graph.  Call after
        enable_head_timing() and before capture()."""
        mk = lambda: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                      for _ in range(self.gamma)]
        self.route_events, self.draft_events = mk(), mk()
        for a, b in self.route_events + self.draft_events:
            a.record()
            b.record()
        torch.cuda.synchronize()

    def overlap_times_ms(self):
        """Per position: (router start, router end, drafter start, drafter end, head start, head
        end), in ms from the first drafter step's start (from the last instrumented replay)."""
        t0 = self.draft_events[0][0]
        out = []
        for t in range(self.gamma):
            r0, r1 = self.route_events[t]
            d0, d1 = self.draft_events[t]
            h0, h1 = self.head_events[t]
            out.append(tuple(t0.elapsed_time(e) for e in (r0, r1, d0, d1, h0, h1)))
        return out

    def n_heads(self) -> int:
        return self.gamma

    def launches_per_step(self) -> int:
        n_router = router_launches(self.B)
        n_short = 1 if self.B == 1 and not self.union else 2
        n_head = 2 if self.union else 1
        n_draft = 5 if getattr(self, "drafter", None) is not None else 0
        n_pref = self.gamma - 1 if self.prefetch_rows else 0
        return self.gamma * (n_router + n_short + n_head + n_draft) - n_short * sum(self.table_pos) + n_pref + 2


class TreeDrafter(_Common):
    """Tree drafting: B sequences, D depths of Wd nodes; the Wd nodes of one depth of one
    sequence share that depth's shortlist, so the head is a dense contraction of B*Wd rows
    against the union of the B shortlists.

    Per-step inputs: ``self.Hr_h`` [D, B, d] (router hidden state per depth), ``self.Hn``
    [D, B*Wd, d] (node hidden states), ``self.z`` [B, 1+D*Wd, V], ``self.u_node`` [B, D*Wd],
    ``self.u_res`` [B, D+1]; ``self.parent`` [D*Wd] the tree's wiring.
    """

    def __init__(self, W, W1, b1, W2, b2, csr_off, csr_tok, parent, *, B, D, Wd, budget, act, T, seed):
        dev = W.device
        self.dev = dev
        self.W, self.W1, self.b1, self.W2, self.b2 = W, W1, b1, W2, b2
        self._setup_vocab(csr_off, csr_tok, dev)
        self.d = W.shape[1]
        self.Hr = W1.shape[0]
        self.B, self.D, self.Wd = B, D, Wd
        self.budget = torch.tensor(list(budget), dtype=torch.int32)
        self.act, self.T, self.seed = act, float(T), int(seed)
        V, M, N = self.V, self.M, D * Wd
        cap = B * V
        i32 = dict(dtype=torch.int32, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        self.parent = torch.as_tensor(parent, dtype=torch.int32).to(dev)
        self.Hr_h = torch.zeros(D, B, self.d, dtype=torch.bfloat16, device=dev)
        self.Hn = torch.zeros(D, B * Wd, self.d, dtype=torch.bfloat16, device=dev)
        self.z = torch.zeros(B, 1 + N, V, **f32)
        self.u_node = torch.full((B, N), 0.5, **f32)
        self.u_res = torch.full((B, D + 1), 0.5, **f32)
        self.scores = torch.empty(D, B, M, **f32)
        self.cluster_ids = [torch.empty(B, int(self.budget[t]), **i32) for t in range(D)]
        self.vs_offsets = torch.zeros(D, B + 1, **i32)
        self.vs_ids = torch.zeros(D, cap, **i32)
        self.cpos = torch.empty(D, B * M, **i32)
        self.union_ids = torch.empty(D, V, **i32)
        self.union_cluster = torch.empty(D, V, **i32)
        self.union_count = torch.zeros(D, 1, **i32)
        self.logits = torch.zeros(D, cap * Wd, **f32)
        self.row_max = torch.empty(D, B * Wd, **f32)
        self.row_sumexp = torch.empty(D, B * Wd, **f32)
        # results in one block: accepted [B], correction [B], path [B, D], node tokens [D, B*Wd]
        self.out = torch.empty(2 * B + B * D + D * B * Wd, **i32)
        self.accepted = self.out[:B]
        self.correction = self.out[B:2 * B]
        self.path = self.out[2 * B:2 * B + B * D].view(B, D)
        self.tokens = self.out[2 * B + B * D:].view(D, B * Wd)
        self.token_idx = torch.empty(D, B * Wd, **i32)
        self.router = api.Router(W1, b1, W2, b2, act, budget)
        self.ws_router = [api.workspace(self.router.workspace_bytes(B), dev) for _ in range(D)]
        self.ws_short = [api.workspace(api.shortlist_workspace_bytes(B, M), dev) for _ in range(D)]
        self.ws_head = api.workspace(api.head_workspace_bytes(B * Wd), dev)
        self.ws_verify = api.workspace(api.verify_tree_workspace_bytes(B, D, Wd, V), dev)
        self.side = torch.cuda.Stream(device=dev)
        self.ready = [torch.cuda.Event() for _ in range(D)]
        self.head_done = [torch.cuda.Event() for _ in range(D)]
        self.graph = None
        self.head_events = None

    def route(self, t, stream=None):
        self.router.topk(self.Hr_h[t], t + 1, self.scores[t], self.cluster_ids[t], self.ws_router[t],
                         self.status, stream)
        api.build_shortlist(self.csr_off, self.csr_tok, self.cluster_ids[t], self.vs_offsets[t],
                            self.vs_ids[t], self.cpos[t], self.ws_short[t], self.status,
                            self.union_ids[t], self.union_cluster[t], self.union_count[t], stream)

    def head(self, t, stream=None):
        # the last depth's head has the GPU to itself (no router runs beside it)
        api.gathered_head(self.Hn[t], self.Wd, self.W, self.vs_offsets[t], self.vs_ids[t], self.T,
                          self.seed, t + 1, self.logits[t], self.tokens[t], self.token_idx[t],
                          self.ws_head, self.status, cpos=self.cpos[t], rank_in_cluster=self.rank,
                          union=(self.union_ids[t], self.union_cluster[t], self.union_count[t]),
                          row_max=self.row_max[t], row_sumexp=self.row_sumexp[t], stream=stream,
                          free_sms=0 if t == self.D - 1 else -1)

    def verify(self, stream=None):
        api.verify_tree(self.z, self.D, self.Wd, self.T, self.parent, self.logits, self.vs_offsets,
                        self.vs_ids, self.cpos, self.cluster_of, self.rank, self.tokens, self.u_node,
                        self.u_res, self.accepted, self.correction, self.path, self.ws_verify,
                        self.status, q_max=self.row_max, q_sumexp=self.row_sumexp, stream=stream)

    def step(self, before_verify=None):
        """One speculation step; verification first waits for the events in `before_verify`, if
        given."""
        self._run(self.D, before_verify)

    def n_heads(self) -> int:
        return self.D

    def launches_per_step(self) -> int:
        return self.D * (router_launches(self.B) + 2 + 2) + 2


class StaticChainDrafter(_Common):
    """The static-shortlist baseline: chain drafting with one fixed token list at every draft
    position and for every sequence, through the same head and verification kernels, with no
    router and no per-position shortlist build.  The pages compare DynaSpec's context-dependent
    lists (about 28K tokens on average) with a fixed 32K-token list (DynaSpec abstract; summary,
    Key Results and Comparison to Prior Work).

    The list enters the library as a two-cluster partition of the vocabulary: cluster 0 holds
    the list's tokens in list order, cluster 1 the rest, and every sequence selects cluster 0.
    The head and the verifier then find a token's list position through the same cluster
    inverse as for dynamic lists.  Inputs as for ChainDrafter (``self.H``: the heads read
    H[t+1]; ``self.z``, ``self.u``).
    """

    def __init__(self, W, static_ids, *, B, gamma, T, seed, union=None):
        dev = W.device
        self.dev = dev
        self.W = W
        V = W.shape[0]
        ids = torch.as_tensor(static_ids, dtype=torch.int32).flatten().cpu()
        n = ids.numel()
        if n < 1 or n > V:
            raise ValueError("the static list needs 1..V tokens")
        member = torch.zeros(V, dtype=torch.bool)
        member[ids.long()] = True
        if int(member.sum()) != n:
            raise ValueError("the static list repeats a token")
        rest = torch.nonzero(~member).flatten().to(torch.int32)
        self._setup_vocab(torch.tensor([0, n, V], dtype=torch.int32), torch.cat([ids, rest]), dev)
        self.d = W.shape[1]
        self.B, self.gamma, self.n_static = B, gamma, n
        self.T, self.seed = float(T), int(seed)
        self.union = (B > 1) if union is None else bool(union)
        M = self.M                                         # 2
        i32 = dict(dtype=torch.int32, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        cap = B * n
        # the lists, built once: every sequence selects cluster 0
        offs1 = torch.zeros(B + 1, **i32)
        vs1 = torch.zeros(cap, **i32)
        cpos1 = torch.empty(B * M, **i32)
        un = (torch.empty(V, **i32), torch.empty(V, **i32), torch.zeros(1, **i32)) if self.union else (None,) * 3
        ws = api.workspace(api.shortlist_workspace_bytes(B, M), dev)
        api.build_shortlist(self.csr_off, self.csr_tok, torch.zeros(B, 1, **i32), offs1, vs1, cpos1, ws,
                            self.status, *un)
        self.vs_offsets = offs1.repeat(gamma, 1).contiguous()
        self.vs_ids = vs1
        self.cpos = cpos1.repeat(gamma, 1).contiguous()
        self.union_ids, self.union_cluster, self.union_count = un
        self.H = torch.zeros(gamma + 1, B, self.d, dtype=torch.bfloat16, device=dev)
        self.z = torch.zeros(B, gamma + 1, V, **f32)
        self.u = torch.full((B, gamma + 1), 0.5, **f32)
        self.logits = torch.zeros(gamma, cap, **f32)
        self.row_max = torch.empty(gamma, B, **f32)
        self.row_sumexp = torch.empty(gamma, B, **f32)
        self.out = torch.empty((2 + gamma) * B, **i32)
        self.accepted = self.out[:B]
        self.correction = self.out[B:2 * B]
        self.tokens = self.out[2 * B:].view(gamma, B)
        self.token_idx = torch.empty(gamma, B, **i32)
        self.ws_head = api.workspace(api.head_workspace_bytes(B), dev)
        self.ws_verify = api.workspace(api.verify_workspace_bytes(B, gamma, V), dev)
        self.graph = None
        self.head_events = None
        torch.cuda.synchronize()
        self.check_status()

    def head(self, t, stream=None):
        # nothing runs beside the static list's heads: every SM
        api.gathered_head(self.H[t + 1], 1, self.W, self.vs_offsets[t], self.vs_ids, self.T,
                          self.seed, t + 1, self.logits[t], self.tokens[t], self.token_idx[t],
                          self.ws_head, self.status, cpos=self.cpos[t], rank_in_cluster=self.rank,
                          union=(self.union_ids, self.union_cluster, self.union_count) if self.union else None,
                          row_max=self.row_max[t], row_sumexp=self.row_sumexp[t], stream=stream, free_sms=0)

    def verify(self, stream=None):
        api.verify(self.z, self.T, self.logits, self.vs_offsets, self.cpos, self.cluster_of, self.rank,
                   self.tokens, self.u, self.accepted, self.correction, self.ws_verify, self.status,
                   q_max=self.row_max, q_sumexp=self.row_sumexp, stream=stream)

    def step(self, before_verify=None):
        """One speculation step: the gamma heads on the current stream, then verification
        (which first waits for the events in `before_verify`, if given)."""
        main = torch.cuda.current_stream(self.dev)
        for t in range(self.gamma):
            if self.head_events:
                api.event_record(self.head_events[t][0])
            self.head(t)
            if self.head_events:
                api.event_record(self.head_events[t][1])
        for ev in before_verify or ():
            main.wait_event(ev)
        self.verify()

    def n_heads(self) -> int:
        return self.gamma

    def launches_per_step(self) -> int:
        return self.gamma * (2 if self.union else 1) + 2
