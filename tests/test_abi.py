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
