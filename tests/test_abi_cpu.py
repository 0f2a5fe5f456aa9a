"""CPU-side checks of the C ABI: the library builds, loads without a GPU,
exports every function include/gnnagg.h declares, and the binding's ctypes
prototypes cover exactly that set.  No compute call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(gnn_[a-z0-9_]+)\s*\(", src))
    return names


def test_header_declares_the_boundary_calls():
    need = {"gnn_csr_build", "gnn_boundary_index", "gnn_quant_pack", "gnn_dequant_unpack",
            "gnn_spmm_fwd", "gnn_spmm_bwd", "gnn_last_error", "gnn_sync_check"}
    assert need <= _declared()


def test_library_exports_every_declared_symbol():
    from sparse_aggregation_message_gb300 import builder as b
    path = b.build()
    lib = ctypes.CDLL(path)
    missing = [n for n in sorted(_declared()) if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_prototypes_match_header():
    from sparse_aggregation_message_gb300 import _abi
    assert set(_abi.PROTOTYPES) == _declared()


def test_version_and_error_text_without_gpu():
    from sparse_aggregation_message_gb300 import _abi
    lib = _abi.load()
    assert lib.gnn_version() >= 10000
    assert isinstance(lib.gnn_last_error(), bytes)


def test_host_validation_rejects_bad_arguments_before_launch():
    """Argument errors come back from the host without touching a GPU."""
    from sparse_aggregation_message_gb300 import _abi
    lib = _abi.load()
    # NULL inputs, F out of range, misaligned strides
    assert lib.gnn_quant_pack(None, 4, 0, None, 1, None, None, 0, None, None, None) == 1
    assert lib.gnn_quant_pack(ctypes.c_void_p(16), 4, 2000, None, 1, ctypes.c_void_p(16),
                              ctypes.c_void_p(16), 0, ctypes.c_void_p(16), ctypes.c_void_p(16),
                              None) == 2
    assert lib.gnn_quant_pack(ctypes.c_void_p(16), 6, 5, None, 1, ctypes.c_void_p(16),
                              ctypes.c_void_p(16), 0, ctypes.c_void_p(16), ctypes.c_void_p(16),
                              None) == 1
    assert b"ldx" in lib.gnn_last_error()
    csr = _abi.GnnCsr(4, 0, 4, 16, 16, 16)
    # the backward needs a symmetric matrix
    assert lib.gnn_spmm_bwd(ctypes.byref(csr), None, ctypes.c_void_p(16), 4, 4, 0, None, None,
                            ctypes.c_void_p(16), 4, None, 0, None) == 2
    # a split plan needs its workspace
    csr2 = _abi.GnnCsr(4, 1, 4, 16, 16, 16, 64, 1, 3, 16, 16, 16, 16)
    assert lib.gnn_spmm_fwd(ctypes.byref(csr2), None, ctypes.c_void_p(16), 4, 4, None, None,
                            ctypes.c_void_p(16), 4, None, 0, None, 0, None) == 1
    assert b"workspace" in lib.gnn_last_error()
    rule = _abi.GnnBitRule()
    rule.n_levels = 2
    rule.pct[0] = 90
    rule.bits[0], rule.bits[1] = 3, 8  # 3 bits is not a width
    b = _abi.GnnBoundary()
    b.P = 2
    assert lib.gnn_boundary_index(ctypes.byref(csr), ctypes.byref(rule), 1, 4, ctypes.byref(b),
                                  ctypes.c_void_p(16), 0, None) == 1
