"""The C-ABI library loads without a GPU and exports every entry point that
include/gdnspec.h declares (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdnspec.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_hybrid_gb300 import build
    build.build()
    return ctypes.CDLL(os.path.join(ROOT, "speculative_decoding_hybrid_gb300", "libgdnspec.so"))


def test_header_declares_the_six_calls():
    names = declared_functions()
    for n in ("gdn_decode_step", "gdn_verify", "mtp_greedy_accept", "gdn_commit", "gdn_chunked_prefill",
              "plan_transaction"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_binding_covers_every_export(lib):
    from speculative_decoding_hybrid_gb300 import binding
    assert sorted(binding.EXPORTS) == declared_functions()


def test_host_checks_need_no_gpu(lib):
    from speculative_decoding_hybrid_gb300 import binding as gs
    d = gs.dims(16, 32, 128, 128)
    # NULL pointers are refused before anything is launched.
    st = gs.lib.gdn_verify(ctypes.byref(d), 1, 4, None, None, None, None, None, None, None, 0, 1, None, None, None,
                           0, None, None, None)
    assert st == gs.GDN_ERR_NULL
    bad = gs.dims(16, 30, 128, 128)          # h_v not a multiple of h_qk
    assert gs.lib.gdn_decode_step(ctypes.byref(bad), 1, *([None] * 6), 0, 1, None, None, None, None, None) \
        == gs.GDN_ERR_SHAPE
    odd = gs.dims(16, 32, 96, 96)            # unsupported head size
    assert gs.lib.gdn_decode_step(ctypes.byref(odd), 1, *([None] * 6), 0, 1, None, None, None, None, None) \
        == gs.GDN_ERR_SHAPE
    assert gs.status_string(gs.GDN_ERR_DUP_SLOT) == "duplicate destination slot"
    assert gs.mtp_accept_workspace_bytes(1024, 151936) >= 1024 * 8


def test_multi_layer_calls_check_arguments_before_launching(lib):
    from speculative_decoding_hybrid_gb300 import binding as gs
    d = gs.dims(16, 32, 128, 128)
    verify = lambda n, rows: gs.lib.gdn_verify_layers(ctypes.byref(d), n, 1, 4, None, rows, None, 0, 0, 1, None,
                                                      None, 0, None, 0, None, 0, None, None)
    assert verify(-1, None) == gs.GDN_ERR_ARG
    assert verify(0, None) == gs.GDN_OK          # nothing to issue
    assert verify(2, None) == gs.GDN_ERR_NULL
    at = gs.lib.gdn_verify_at_layers(ctypes.byref(d), 3, 1, 4, None, None, None, 0, None, None, 0, None, 0, None,
                                     0, None, None)
    assert at == gs.GDN_ERR_NULL
    rp = gs.lib.gdn_verify_replay_layers(ctypes.byref(d), -2, 1, 4, None, None, 4, None, None, None, None, 0, 0, 1,
                                         None, None, None, 0, None, None)
    assert rp == gs.GDN_ERR_ARG


def test_decode_transaction_checks_arguments_before_planning(lib):
    """gdn_decode_transaction refuses missing buffers and request lists that
    hold a prefill before it plans anything (the pool stays as it was)."""
    from speculative_decoding_hybrid_gb300 import binding as gs
    d = gs.dims(2, 4, 16, 16)
    pool = gs.Pool(4)
    held = pool.alloc()
    plan = gs.Plan(2)
    reqs = (gs.gdn_req * 2)()
    reqs[0] = gs.gdn_req(gs.REQ_DECODE, 3, 0, 1, 1 << 20, held)
    reqs[1] = gs.gdn_req(gs.REQ_PREFILL, 0, 5, 0, 1 << 20, -1)
    lim = gs.gdn_plan_limits(64, 2, 3)
    txn = ctypes.c_uint32(7)
    io = gs.gdn_decode_io()
    before = (pool.refcount.copy(), pool.free_list())
    # no device buffers in io
    st = gs.lib.gdn_decode_transaction(ctypes.byref(d), 1, 8, reqs, 2, ctypes.byref(lim), ctypes.byref(pool.c),
                                       ctypes.byref(plan.c), ctypes.byref(txn), ctypes.byref(io), None, None)
    assert st == gs.GDN_ERR_NULL
    # every pointer set (never dereferenced on this path): the prefill is refused before planning
    for name, _ in gs.gdn_decode_io._fields_:
        if name not in ("slot_stride", "layer_stride", "num_slots", "ckpt_layer_stride", "o_layer_stride", "vocab",
                        "logit_row_stride", "workspace_bytes"):
            setattr(io, name, 16)
    st = gs.lib.gdn_decode_transaction(ctypes.byref(d), 1, 8, reqs, 2, ctypes.byref(lim), ctypes.byref(pool.c),
                                       ctypes.byref(plan.c), ctypes.byref(txn), ctypes.byref(io), None, None)
    assert st == gs.GDN_ERR_ARG
    assert (pool.refcount == before[0]).all() and pool.free_list() == before[1] and txn.value == 7
    assert reqs[0].slot == held and reqs[0].cur_len == 1


def test_arena_transaction_needs_every_request(lib):
    """gdn_decode_transaction_at keeps one location per request and layer:
    a plan that leaves a request out (row budget too small) is undone before
    anything is launched, and the pool keeps its slots."""
    from speculative_decoding_hybrid_gb300 import binding as gs
    d = gs.dims(2, 4, 16, 16)
    pool = gs.Pool(4)
    held = [pool.alloc(), pool.alloc()]
    plan = gs.Plan(2)
    reqs = (gs.gdn_req * 2)()
    for i in range(2):
        reqs[i] = gs.gdn_req(gs.REQ_DECODE, 3, 0, 1, 1 << 20, held[i])
    lim = gs.gdn_plan_limits(4, 2, 3)        # room for one request of 4 rows only
    txn = ctypes.c_uint32(3)
    io = gs.gdn_decode_io()
    for name, _ in gs.gdn_decode_io._fields_:
        if name not in ("slot_stride", "layer_stride", "num_slots", "ckpt_layer_stride", "o_layer_stride", "vocab",
                        "logit_row_stride", "workspace_bytes"):
            setattr(io, name, 16)
    ar = gs.gdn_arena_io()
    ar.arena, ar.loc, ar.elems_total = 16, 16, 1 << 20
    before = (pool.refcount.copy(), pool.free_list())
    st = gs.lib.gdn_decode_transaction_at(ctypes.byref(d), 1, 8, reqs, 2, ctypes.byref(lim), ctypes.byref(pool.c),
                                          ctypes.byref(plan.c), ctypes.byref(txn), ctypes.byref(io), ctypes.byref(ar),
                                          None, None)
    assert st == gs.GDN_ERR_ARG
    assert (pool.refcount == before[0]).all() and sorted(pool.free_list()) == sorted(before[1])
    assert txn.value == 3 and [reqs[i].slot for i in range(2)] == held
