"""ctypes front of the oracle's C routines (coracle.c).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle``: the same definitions
as oracle.py (quantise + pack, fixed-order halo partials, forward and
backward aggregation in fp64), written as plain C loops so that full-size
message buffers can be compared and the oracle can run on every host core.
The library is compiled in-tree with gcc (``-O2 -ffp-contract=off
-fopenmp``) on first use."""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "coracle.c")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libcoracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile coracle.c into oracle/_build/libcoracle.so (with OpenMP when
    the compiler has it, else single-threaded)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    tmp = LIB + f".{os.getpid()}.tmp"
    base = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-shared", "-fPIC",
            SRC, "-o", tmp, "-lm"]
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if r.returncode != 0:
        r = subprocess.run(base, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"gcc failed on coracle.c:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
        L.orc_max_threads.restype = ctypes.c_int
        L.orc_set_threads.argtypes = [ctypes.c_int]
        L.orc_fmix32.restype = u32
        L.orc_fmix32.argtypes = [u32]
        L.orc_hash32.restype = u32
        L.orc_hash32.argtypes = [u32, u32, u32]
        L.orc_rowbytes.restype = i64
        L.orc_rowbytes.argtypes = [i32, i32]
        L.orc_quant_pack.argtypes = [vp, i64, i32, vp, i64, vp, vp, u32, i64, vp, vp]
        L.orc_halo_quant_pack.argtypes = [i64, vp, vp, vp, vp, i64, i32, vp, vp, u32, i64, vp, vp]
        L.orc_spmm_fwd_rows.argtypes = [vp, vp, vp, vp, i64, i32, vp, vp, vp, vp, vp, i64, vp, vp]
        L.orc_spmm_bwd_rows.argtypes = [vp, vp, vp, vp, i64, i32, vp, vp, vp, vp, vp, vp, vp, i64,
                                        vp, vp]
        _lib = L
    return _lib


def _c(a, dtype):
    """A C-contiguous array of this dtype (copied only when needed)."""
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def max_threads() -> int:
    return int(lib().orc_max_threads())


def set_threads(t: int) -> None:
    lib().orc_set_threads(int(t))


def fmix32(h: int) -> int:
    return int(lib().orc_fmix32(h & 0xFFFFFFFF))


def hash32(seed: int, s: int, j: int) -> int:
    return int(lib().orc_hash32(seed & 0xFFFFFFFF, s & 0xFFFFFFFF, j & 0xFFFFFFFF))


def quant_pack(X, F, row_idx, bits, off, seed, total=None, key0=0):
    """Rows X[row_idx[r], :F] (row_idx None: X[r]) quantised with width
    bits[r] and row key key0 + r, packed at off[r] (off[R], when given, is
    the buffer size).  Returns (packed uint8 buffer, meta fp32 [R, 2] =
    (min, scale))."""
    X, px = _c(X, np.float32)
    bits, pb = _c(bits, np.uint8)
    off, po = _c(off, np.int64)
    R = bits.size
    if total is None:
        if off.size > R:
            total = int(off[R])
        else:
            total = max((int(off[r]) + int(lib().orc_rowbytes(int(bits[r]), F)) for r in range(R)),
                        default=0)
    packed = np.zeros(max(total, 1), np.uint8)
    meta = np.zeros((R, 2), np.float32)
    ri, pr = (None, None) if row_idx is None else _c(row_idx, np.int32)
    lib().orc_quant_pack(px, X.shape[1], F, pr, R, pb, po, seed & 0xFFFFFFFF, int(key0),
                         packed.ctypes.data, meta.ctypes.data)
    return packed[:total], meta


def halo_quant_pack(bnd, G, F, slot_bits, slot_off, seed, s0=0, s1=None):
    """Backward messages of slots [s0, s1) (default all): the fixed-order fp32
    halo partial of G, quantised with key s and packed at
    slot_off[s] - slot_off[s0]."""
    S = int(bnd["n_slots"])
    s1 = S if s1 is None else s1
    G, pg = _c(G, np.float32)
    srp, p1 = _c(bnd["slot_rowptr"][s0:s1 + 1], np.int64)
    scol, p2 = _c(bnd["slot_col"], np.int32)
    sval, p3 = _c(bnd["slot_val"], np.float32)
    bits, pb = _c(slot_bits[s0:s1], np.uint8)
    off, po = _c(np.asarray(slot_off[s0:s1 + 1], np.int64) - int(slot_off[s0]), np.int64)
    total = int(off[-1])
    packed = np.zeros(max(total, 1), np.uint8)
    meta = np.zeros((s1 - s0, 2), np.float32)
    lib().orc_halo_quant_pack(s1 - s0, p1, p2, p3, pg, G.shape[1], F, pb, po, seed & 0xFFFFFFFF,
                              int(s0), packed.ctypes.data, meta.ctypes.data)
    return packed[:total], meta


def spmm_fwd_rows(rowptr, bnd, H, F, packed, meta, slot_bits, slot_off, rows):
    """fp64 forward aggregation (M, T) of the given rows from the oracle's
    own message buffer packed/meta."""
    rows, prw = _c(rows, np.int64)
    rp, p1 = _c(rowptr, np.int64)
    cr, p2 = _c(bnd["col_remap"], np.int32)
    vr, p3 = _c(bnd["val_remap"], np.float32)
    H, ph = _c(H, np.float32)
    pk, p4 = _c(packed, np.uint8)
    mt, p5 = _c(meta, np.float32)
    sb, p6 = _c(slot_bits, np.uint8)
    so, p7 = _c(slot_off, np.int64)
    M = np.zeros((rows.size, F), np.float64)
    T = np.zeros((rows.size, F), np.float64)
    lib().orc_spmm_fwd_rows(p1, p2, p3, ph, H.shape[1], F, p4, p5, p6, p7, prw, rows.size,
                            M.ctypes.data, T.ctypes.data)
    return M, T


def spmm_bwd_rows(rowptr, bnd, G, F, packed, meta, slot_bits, slot_off, rows):
    """fp64 backward aggregation (dH, T) of the given rows: local A^T
    entries plus the dequantised backward messages each row owns."""
    rows, prw = _c(rows, np.int64)
    rp, p1 = _c(rowptr, np.int64)
    cr, p2 = _c(bnd["col_remap"], np.int32)
    wt, p3 = _c(bnd["val_remap_t"] if "val_remap_t" in bnd else bnd["val_remap"], np.float32)
    G, pg = _c(G, np.float32)
    op, p4 = _c(bnd["own_ptr"], np.int64)
    os_, p5 = _c(bnd["own_slot"], np.int32)
    pk, p6 = _c(packed, np.uint8)
    mt, p7 = _c(meta, np.float32)
    sb, p8 = _c(slot_bits, np.uint8)
    so, p9 = _c(slot_off, np.int64)
    dH = np.zeros((rows.size, F), np.float64)
    T = np.zeros((rows.size, F), np.float64)
    lib().orc_spmm_bwd_rows(p1, p2, p3, pg, G.shape[1], F, p4, p5, p6, p7, p8, p9, prw, rows.size,
                            dH.ctypes.data, T.ctypes.data)
    return dH, T
