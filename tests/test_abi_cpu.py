"""The C-ABI library loads on a machine without a GPU, exports every symbol the header
declares, answers workspace queries, and rejects bad host-side arguments before it launches
anything (no compute call reaches a device here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dynaspec.h")


@pytest.fixture(scope="module")
def lib():
    from dynamic_vocab_draft_gb300 import build
    build.build()
    from dynamic_vocab_draft_gb300 import _lib
    return _lib.load()


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ds_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    from dynamic_vocab_draft_gb300 import _lib
    assert set(_lib.SIGNATURES) == set(names)


def test_status_strings(lib):
    for code in (0, 1, 2, 3, 4, 0x10, 0x20, 0x40, 0x30, 12345):
        s = lib.ds_status_string(code)
        assert isinstance(s, bytes) and s
    assert lib.ds_version() == 4


def test_workspace_queries(lib):
    assert lib.ds_router_workspace_bytes(1, 1024) >= 4096
    assert lib.ds_router_workspace_bytes(0, 1024) == 0
    assert lib.ds_shortlist_workspace_bytes(32, 1024) >= 32 * 4 + 1024 * 4
    assert lib.ds_head_workspace_bytes(80) > lib.ds_head_workspace_bytes(1)
    assert lib.ds_verify_workspace_bytes(1, 6, 128256) > 0
    assert lib.ds_verify_tree_workspace_bytes(8, 6, 10, 128256) >= 8 * 128256 * 4
    for q in (lib.ds_router_workspace_bytes(3, 40), lib.ds_head_workspace_bytes(7)):
        assert q % 256 == 0


FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: every call below fails its host checks


def test_host_argument_checks(lib):
    budget = (ctypes.c_int32 * 2)(4, 4)
    bptr = ctypes.cast(budget, ctypes.c_void_p)
    # router: NULL H; d not a multiple of 8; pos out of the budget table; k > M; no workspace
    assert lib.ds_router_topk(None, 1, 64, FAKE, FAKE, 64, FAKE, FAKE, 32, 0, bptr, 2, 1,
                              FAKE, FAKE, -1, FAKE, 1 << 20, None, None) == 1
    assert lib.ds_router_topk(FAKE, 1, 60, FAKE, FAKE, 64, FAKE, FAKE, 32, 0, bptr, 2, 1,
                              FAKE, FAKE, -1, FAKE, 1 << 20, None, None) == 1
    assert lib.ds_router_topk(FAKE, 1, 64, FAKE, FAKE, 64, FAKE, FAKE, 32, 0, bptr, 2, 3,
                              FAKE, FAKE, -1, FAKE, 1 << 20, None, None) == 1
    assert lib.ds_router_topk(FAKE, 1, 64, FAKE, FAKE, 64, FAKE, FAKE, 3, 0, bptr, 2, 1,
                              FAKE, FAKE, -1, FAKE, 1 << 20, None, None) == 1
    assert lib.ds_router_topk(FAKE, 1, 64, FAKE, FAKE, 64, FAKE, FAKE, 32, 7, bptr, 2, 1,
                              FAKE, FAKE, -1, FAKE, 1 << 20, None, None) == 1
    assert lib.ds_router_topk(FAKE, 1, 64, FAKE, FAKE, 64, FAKE, FAKE, 32, 0, bptr, 2, 1,
                              FAKE, FAKE, -1, None, 0, None, None) == 4
    # shortlist: only some of the union outputs; k > M
    assert lib.ds_build_shortlist(FAKE, FAKE, 32, 4096, FAKE, 1, 4, FAKE, FAKE, 4096, FAKE,
                                  FAKE, None, None, FAKE, 1 << 20, None, None) == 1
    assert lib.ds_build_shortlist(FAKE, FAKE, 32, 4096, FAKE, 1, 40, FAKE, FAKE, 4096, FAKE,
                                  None, None, None, FAKE, 1 << 20, None, None) == 1
    # head: negative temperature; d % 8; union path needs cpos; per-row path needs G == 1
    args = [FAKE, 1, 1, FAKE, 4096, 256, FAKE, FAKE, None, 0, None, None, None, None,
            1.0, 0, 1, FAKE, None, None, FAKE, FAKE, -1, FAKE, 1 << 24, None, None]
    a = list(args); a[14] = -1.0
    assert lib.ds_gathered_head(*a) == 1
    a = list(args); a[5] = 250
    assert lib.ds_gathered_head(*a) == 1
    a = list(args); a[11] = FAKE; a[12] = FAKE; a[13] = FAKE
    assert lib.ds_gathered_head(*a) == 1
    a = list(args); a[2] = 4
    assert lib.ds_gathered_head(*a) == 2
    a = list(args); a[24] = 16
    assert lib.ds_gathered_head(*a) == 4
    # union path: more than 128 head rows, or a vocabulary above 2^20, is unsupported
    union = list(args); union[8] = FAKE; union[9] = 32; union[10] = FAKE
    union[11] = FAKE; union[12] = FAKE; union[13] = FAKE; union[24] = 1 << 30
    a = list(union); a[1] = 8; a[2] = 17
    assert lib.ds_gathered_head(*a) == 2
    a = list(union); a[4] = (1 << 20) + 1
    assert lib.ds_gathered_head(*a) == 2
    # verify: gamma beyond the limit; NULL uniforms
    assert lib.ds_verify(FAKE, 1, 40, 4096, 1.0, FAKE, 4096, None, None, FAKE, FAKE, 32, FAKE, FAKE, FAKE, FAKE,
                         FAKE, FAKE, FAKE, 1 << 24, None, None) == 1
    assert lib.ds_verify(FAKE, 1, 4, 4096, 1.0, FAKE, 4096, None, None, FAKE, FAKE, 32, FAKE, FAKE, FAKE, None,
                         FAKE, FAKE, FAKE, 1 << 24, None, None) == 1
    # tree verify: Wd beyond the limit; only one of q_max / q_sumexp; NULL vs_ids
    tree = [FAKE, 1, 3, 4, 4096, 1.0, FAKE, FAKE, 4096, None, None, FAKE, FAKE, 4096, FAKE, 32, FAKE, FAKE,
            FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 26, None, None]
    t = list(tree); t[3] = 65
    assert lib.ds_verify_tree(*t) == 1
    t = list(tree); t[9] = FAKE
    assert lib.ds_verify_tree(*t) == 1
    t = list(tree); t[12] = None
    assert lib.ds_verify_tree(*t) == 1
    t = list(tree); t[25] = 16
    assert lib.ds_verify_tree(*t) == 4
    assert lib.ds_philox4x32_10(None, 0, FAKE, 4, None) == 1
    # copy: NULL ends and overlapping ranges are refused before any launch; zero bytes is a no-op
    assert lib.ds_copy(None, FAKE, 16, None) == 1
    assert lib.ds_copy(FAKE, None, 16, None) == 1
    assert lib.ds_copy(FAKE, ctypes.c_void_p(0x10008), 16, None) == 1
    assert lib.ds_copy(ctypes.c_void_p(0x10008), FAKE, 16, None) == 1
    assert lib.ds_copy(FAKE, FAKE, 0, None) == 0


def test_copy_refuses_memory_the_device_cannot_reach(lib):
    # two ordinary (pageable) host buffers, as a C caller would pass them: the library looks
    # both ends up before launching and refuses them (here, without a GPU, the lookup itself
    # fails, which is refused the same way)
    a = ctypes.create_string_buffer(64)
    b = ctypes.create_string_buffer(64)
    assert lib.ds_copy(ctypes.cast(a, ctypes.c_void_p), ctypes.cast(b, ctypes.c_void_p), 64, None) == 1


def test_copy_binding_refuses_pageable_host_memory():
    # ds_copy reaches host memory from a kernel, so the binding takes CUDA tensors or pinned
    # host tensors only; a pageable tensor is refused before the library is called
    torch = pytest.importorskip("torch")
    from dynamic_vocab_draft_gb300 import api
    with pytest.raises(ValueError):
        api.copy(torch.zeros(16, dtype=torch.uint8), torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(ValueError):
        api.copy(torch.zeros(16, dtype=torch.uint8)[::2], torch.zeros(8, dtype=torch.uint8))


def test_unified_workspace_query_matches_the_per_call_queries(lib):
    # ds_workspace_bytes(op, B, V, M, gamma, hidden, width) dispatches to the per-call queries
    for B in (1, 5, 32):
        assert lib.ds_workspace_bytes(1, B, 0, 0, 0, 1024, 0) == lib.ds_router_workspace_bytes(B, 1024)
        assert lib.ds_workspace_bytes(2, B, 0, 1024, 0, 0, 0) == lib.ds_shortlist_workspace_bytes(B, 1024)
        assert lib.ds_workspace_bytes(3, B, 0, 0, 0, 0, 10) == lib.ds_head_workspace_bytes(B * 10)
        assert lib.ds_workspace_bytes(4, B, 128256, 0, 6, 0, 0) == lib.ds_verify_workspace_bytes(B, 6, 128256)
        assert lib.ds_workspace_bytes(5, B, 128256, 0, 6, 0, 10) == lib.ds_verify_tree_workspace_bytes(B, 6, 10, 128256)
    assert lib.ds_workspace_bytes(9, 1, 1, 1, 1, 1, 1) == 0
    assert lib.ds_workspace_bytes(3, 0, 0, 0, 0, 0, 1) == 0


def test_router_handle_host_side(lib):
    # the handle is host memory: create / query / destroy need no device
    budget = (ctypes.c_int32 * 3)(8, 6, 4)
    bptr = ctypes.cast(budget, ctypes.c_void_p)
    h = ctypes.c_void_p()
    # bad arguments: NULL out, NULL weight, d % 8, act, a budget entry beyond M
    assert lib.ds_router_create(None, FAKE, FAKE, FAKE, FAKE, 256, 512, 32, 1, bptr, 3) == 1
    assert lib.ds_router_create(ctypes.byref(h), None, FAKE, FAKE, FAKE, 256, 512, 32, 1, bptr, 3) == 1
    assert h.value is None
    assert lib.ds_router_create(ctypes.byref(h), FAKE, FAKE, FAKE, FAKE, 250, 512, 32, 1, bptr, 3) == 1
    assert lib.ds_router_create(ctypes.byref(h), FAKE, FAKE, FAKE, FAKE, 256, 512, 32, 5, bptr, 3) == 1
    assert lib.ds_router_create(ctypes.byref(h), FAKE, FAKE, FAKE, FAKE, 256, 512, 5, 1, bptr, 3) == 1
    assert lib.ds_router_create(ctypes.byref(h), FAKE, FAKE, FAKE, FAKE, 256, 512, 32, 1, bptr, 3) == 0
    assert h.value
    # workspace: the router call's plus the scores (B x M fp32), 256-byte aligned parts
    for B in (1, 5):
        base = lib.ds_router_workspace_bytes(B, 512)
        assert lib.ds_router_workspace_bytes_h(h, B) == ((base + 255) // 256) * 256 + ((B * 32 * 4 + 255) // 256) * 256
    # NULL handle, too small a workspace, position outside the table: refused before any launch
    assert lib.ds_router_topk_h(None, FAKE, 1, 1, None, FAKE, -1, FAKE, 1 << 20, None, None) == 1
    assert lib.ds_router_topk_h(h, FAKE, 1, 1, None, FAKE, -1, FAKE, 16, None, None) == 4
    assert lib.ds_router_topk_h(h, FAKE, 1, 4, None, FAKE, -1, FAKE, 1 << 20, None, None) == 1
    assert lib.ds_router_destroy(h) == 0
    assert lib.ds_router_destroy(None) == 0


def test_wait_budget_arguments(lib):
    assert lib.ds_set_wait_budget(-1) == 1
    assert lib.ds_set_wait_budget(1000) == 0
    assert lib.ds_set_wait_budget(0) == 0          # back to the default


def test_batch1_side_sms_rule():
    # The side-stream share at batch 1: 16 SMs beside Llama-size heads (every position of the
    # 6-position budget), more beside the short lists of a 262,144-token vocabulary (5% and 10%
    # of its 2,048 clusters), none of it beyond the largest choice.
    from dynamic_vocab_draft_gb300.pipeline import SIDE_SMS_CHOICES, side_sms_b1
    llama_router = 2.0 * (1024 * 4096 + 1024 * 1024)
    for k in (320, 272, 224, 192, 160):
        assert side_sms_b1(k * (128256 / 1024) * (2 * 4096 + 8), llama_router, 152) == 16
    large_router = 2.0 * (1024 * 2560 + 2048 * 1024)
    row = (262144 / 2048) * (2 * 2560 + 8)
    assert side_sms_b1(102 * row, large_router, 152) == 40
    assert side_sms_b1(205 * row, large_router, 152) == 24
    assert side_sms_b1(410 * row, large_router, 152) == 16
    assert side_sms_b1(1.0, 1e12, 152) == max(SIDE_SMS_CHOICES)
    # a router with nothing to read never needs more than the smallest share
    assert side_sms_b1(1e9, 0.0, 152) == 16
