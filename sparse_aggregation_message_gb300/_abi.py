"""ctypes view of libgnnagg.so: struct layouts and function prototypes that
mirror include/gnnagg.h one to one."""
from __future__ import annotations

import ctypes
import os

from . import builder as _build

c_i32, c_i64, c_u8, c_u16, c_u32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint8, ctypes.c_uint16, ctypes.c_uint32
c_size, c_vp, c_char_p = ctypes.c_size_t, ctypes.c_void_p, ctypes.c_char_p
P_i64 = ctypes.POINTER(c_i64)
P_size = ctypes.POINTER(c_size)

STATUS = {0: "GNN_OK", 1: "GNN_ERR_INVALID_ARG", 2: "GNN_ERR_UNSUPPORTED", 3: "GNN_ERR_CUDA",
          4: "GNN_ERR_DEVICE_CHECK", 5: "GNN_ERR_TIMEOUT", 6: "GNN_ERR_CAPACITY"}

CSR_SYMMETRIZE, CSR_DEDUP, CSR_SELF_LOOPS, CSR_MEAN = 1, 2, 4, 8
CSR_GCN = CSR_SYMMETRIZE | CSR_DEDUP | CSR_SELF_LOOPS


class GnnCsr(ctypes.Structure):
    _fields_ = [("n", c_i32), ("symmetric", c_i32), ("nnz", c_i64), ("rowptr", c_vp),
                ("col", c_vp), ("val", c_vp), ("split_len", c_i32), ("n_long", c_i32),
                ("n_pieces", c_i64), ("long_rows", c_vp), ("piece_ptr", c_vp),
                ("piece_row", c_vp), ("piece_beg", c_vp), ("val_t", c_vp)]


class GnnBitRule(ctypes.Structure):
    _fields_ = [("n_levels", c_i32), ("pct", c_i32 * 3), ("bits", c_u8 * 4)]


class GnnBoundary(ctypes.Structure):
    _fields_ = [("P", c_i32), ("n", c_i32), ("n_slots", c_i64), ("nnz_cut", c_i64), ("F", c_i32),
                ("reserved", c_i32), ("part_start", c_vp), ("send_start", c_vp),
                ("slot_node", c_vp), ("col_remap", c_vp), ("val_remap", c_vp), ("local_cnt", c_vp),
                ("slot_rowptr", c_vp),
                ("slot_col", c_vp), ("slot_val", c_vp), ("own_ptr", c_vp), ("own_slot", c_vp),
                ("node_bits", c_vp), ("slot_bits", c_vp), ("slot_off", c_vp),
                ("long_slot_len", c_i32), ("n_long_slots", c_i32), ("long_slots", c_vp),
                ("val_remap_t", c_vp), ("halo_order", c_vp)]


class GnnBlocked(ctypes.Structure):
    _fields_ = [("T", c_i32), ("n_rb", c_i32), ("n_tiles", c_i64), ("n_entries", c_i64),
                ("rb_tile_ptr", c_vp), ("tile_cb", c_vp), ("tile_ptr", c_vp), ("tile_rowptr", c_vp),
                ("ent_col", c_vp), ("ent_val", c_vp), ("residual", GnnCsr), ("res_local_cnt", c_vp)]


GNN_LDR_MAX_DELTA = 64


class GnnLdrState(ctypes.Structure):
    _fields_ = [("lambda_", ctypes.c_double), ("delta", c_i32), ("b_min", c_i32), ("b_max", c_i32),
                ("t", c_i32), ("base_bits", c_i32), ("async_next", c_i32), ("F", ctypes.c_double),
                ("ldr", ctypes.c_double * (GNN_LDR_MAX_DELTA + 1))]


P_csr = ctypes.POINTER(GnnCsr)
P_bnd = ctypes.POINTER(GnnBoundary)
P_rule = ctypes.POINTER(GnnBitRule)
P_blk = ctypes.POINTER(GnnBlocked)

# name -> (restype, argtypes)
PROTOTYPES = {
    "gnn_last_error": (c_char_p, []),
    "gnn_version": (ctypes.c_int, []),
    "gnn_kernel_launches": (ctypes.c_ulonglong, []),
    "gnn_csr_build_workspace": (ctypes.c_int, [c_i32, c_i64, c_u32, P_size]),
    "gnn_csr_build": (ctypes.c_int, [c_i32, c_i64, c_vp, c_vp, c_u32, c_i64, P_csr, c_vp, c_size, c_vp]),
    "gnn_csr_split_workspace": (ctypes.c_int, [P_csr, P_size]),
    "gnn_csr_split_count": (ctypes.c_int, [P_csr, c_i32, ctypes.POINTER(c_i32), P_i64, c_vp, c_size, c_vp]),
    "gnn_csr_split": (ctypes.c_int, [P_csr, c_vp, c_size, c_vp]),
    "gnn_boundary_workspace": (ctypes.c_int, [P_csr, c_i32, P_size]),
    "gnn_boundary_count": (ctypes.c_int, [P_csr, c_i32, P_i64, P_i64, c_vp, c_size, c_vp]),
    "gnn_boundary_index": (ctypes.c_int, [P_csr, P_rule, c_u8, c_i32, P_bnd, c_vp, c_size, c_vp]),
    "gnn_boundary_set_bits": (ctypes.c_int, [P_csr, P_rule, c_u8, c_i32, P_bnd, c_vp, c_size, c_vp]),
    "gnn_boundary_long_slots_count": (ctypes.c_int, [P_bnd, c_i32, ctypes.POINTER(c_i32), c_vp, c_size, c_vp]),
    "gnn_boundary_long_slots": (ctypes.c_int, [P_bnd, c_vp, c_size, c_vp]),
    "gnn_slot_offsets_workspace": (ctypes.c_int, [c_i64, P_size]),
    "gnn_slot_offsets": (ctypes.c_int, [c_vp, c_i64, c_i32, c_vp, c_vp, c_size, c_vp]),
    "gnn_quant_pack": (ctypes.c_int, [c_vp, c_i64, c_i32, c_vp, c_i64, c_vp, c_vp, c_u32, c_vp, c_vp, c_vp]),
    "gnn_quant_pack_owned": (ctypes.c_int, [P_bnd, c_vp, c_i64, c_i32, c_u32, c_vp, c_vp, c_vp]),
    "gnn_dequant_unpack": (ctypes.c_int, [c_vp, c_vp, c_vp, c_vp, c_i64, c_i32, c_vp, c_i64, c_vp]),
    "gnn_spmm_workspace": (ctypes.c_int, [P_csr, c_i32, P_size]),
    "gnn_spmm_fwd": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_i64, c_i32, c_vp, c_vp, c_vp, c_i64, c_vp, c_i64,
                                    c_vp, c_size, c_vp]),
    "gnn_spmm_fwd_noalloc": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_i64, c_i32, c_vp, c_vp, c_vp, c_i64,
                                            c_vp, c_i64, c_vp]),
    "gnn_spmm_bwd": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_i64, c_i32, c_u32, c_vp, c_vp, c_vp, c_i64,
                                    c_vp, c_size, c_vp]),
    "gnn_dense_workspace": (ctypes.c_int, [c_i64, c_i32, c_i32, P_size]),
    "gnn_dense_fwd": (ctypes.c_int, [c_vp, c_i64, c_i64, c_i32, c_vp, c_i32, c_i32, c_vp, c_i64, c_vp,
                                     c_size, c_vp]),
    "gnn_dense_bwd": (ctypes.c_int, [c_vp, c_i64, c_i64, c_i32, c_vp, c_i32, c_vp, c_i64, c_vp, c_i64,
                                     c_i32, c_vp, c_i64, c_vp, c_vp, c_size, c_vp]),
    "gnn_layer_workspace": (ctypes.c_int, [P_csr, c_i32, c_i32, P_size]),
    "gnn_layer_fwd": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_i64, c_i32, c_vp, c_i32, c_i32, c_u32, c_vp,
                                     c_vp, c_vp, c_i64, c_vp, c_i64, c_vp, c_size, c_vp]),
    "gnn_layer_bwd": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_i64, c_vp, c_i64, c_i32, c_vp, c_i64, c_vp,
                                     c_i32, c_i32, c_u32, c_vp, c_vp, c_vp, c_vp, c_i64, c_vp, c_size,
                                     c_vp]),
    "gnn_halo_quant_pack": (ctypes.c_int, [P_bnd, c_vp, c_i64, c_i32, c_u32, c_vp, c_vp, c_vp]),
    "gnn_quant_pack_slots": (ctypes.c_int, [c_vp, c_i64, c_i32, c_vp, c_i64, c_i64, c_vp, c_vp, c_u32,
                                            c_vp, c_vp, c_vp]),
    "gnn_halo_quant_pack_slots": (ctypes.c_int, [P_bnd, c_vp, c_i64, c_i32, c_i64, c_i64, c_u32, c_vp,
                                                 c_vp, c_vp]),
    "gnn_spmm_bwd_local": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_i64, c_i32, c_vp, c_vp, c_vp, c_i64, c_vp,
                                          c_size, c_vp]),
    "gnn_layer_fwd_async": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_i64, c_i32, c_vp, c_i32, c_i32, c_u32,
                                           c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_vp, c_i64, c_vp, c_size,
                                           c_vp, c_vp]),
    "gnn_layer_bwd_async": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_i64, c_vp, c_i64, c_i32, c_vp, c_i64,
                                           c_vp, c_i32, c_i32, c_u32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp,
                                           c_i64, c_vp, c_size, c_vp, c_vp]),
    "gnn_layer_tf_workspace": (ctypes.c_int, [P_csr, c_i32, c_i32, P_size]),
    "gnn_layer_fwd_tf": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_i64, c_i32, c_vp, c_i32, c_i32, c_u32,
                                        c_vp, c_vp, c_vp, c_i64, c_vp, c_i64, c_vp, c_i64, c_vp, c_size,
                                        c_vp]),
    "gnn_layer_bwd_tf": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_i64, c_vp, c_i64, c_i32, c_vp, c_i64,
                                        c_vp, c_i32, c_i32, c_u32, c_vp, c_vp, c_vp, c_vp, c_i64,
                                        c_vp, c_size, c_vp]),
    "gnn_gat_index": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_vp, c_vp]),
    "gnn_gat_workspace": (ctypes.c_int, [P_csr, P_bnd, c_i32, c_i32, P_size]),
    "gnn_gat_layer_fwd": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_i64, c_i32, c_vp, c_i32, c_vp, c_vp, c_i32,
                                         c_u32, c_vp, c_vp, c_vp, c_i64, c_vp, c_i64, c_vp, c_vp, c_i64,
                                         c_vp, c_size, c_vp]),
    "gnn_gat_layer_bwd": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_vp, c_vp, c_i64, c_vp, c_i64, c_i32, c_vp,
                                         c_i64, c_vp, c_i64, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32,
                                         c_i32, c_u32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i64, c_vp,
                                         c_vp, c_size, c_vp]),
    "gnn_spmm_bwd_masked": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_i64, c_i32, c_u32, c_vp, c_vp, c_vp, c_i64,
                                           c_vp, c_i64, c_vp, c_size, c_vp]),
    "gnn_spmm_bwd_local_masked": (ctypes.c_int, [P_csr, P_bnd, c_vp, c_i64, c_i32, c_vp, c_vp, c_vp,
                                                 c_i64, c_vp, c_i64, c_vp, c_size, c_vp]),
    "gnn_dense_bwd_z": (ctypes.c_int, [c_vp, c_i64, c_i64, c_i32, c_vp, c_i32, c_vp, c_i64, c_vp, c_i64, c_vp,
                                       c_vp, c_size, c_vp]),
    "gnn_blocked_workspace": (ctypes.c_int, [P_csr, P_bnd, c_i32, c_i32, P_size]),
    "gnn_blocked_count": (ctypes.c_int, [P_csr, P_bnd, c_i32, c_i32, P_i64, P_i64, P_i64, c_vp, c_size, c_vp]),
    "gnn_blocked_build": (ctypes.c_int, [P_csr, P_bnd, c_i32, c_i32, P_blk, c_vp, c_size, c_vp]),
    "gnn_blocked_spmm_workspace": (ctypes.c_int, [P_blk, c_i32, P_size]),
    "gnn_spmm_fwd_blocked": (ctypes.c_int, [P_csr, P_bnd, P_blk, c_vp, c_i64, c_i32, c_vp, c_vp, c_vp, c_i64,
                                            c_vp, c_i64, c_vp, c_size, c_vp]),
    "gnn_spmm_bwd_blocked": (ctypes.c_int, [P_csr, P_bnd, P_blk, c_vp, c_i64, c_i32, c_u32, c_vp, c_vp, c_vp,
                                            c_i64, c_vp, c_i64, c_vp, c_i64, c_vp, c_size, c_vp]),
    "gnn_ldr_init": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_double, c_i32, c_i32, c_i32]),
    "gnn_ldr_update": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(ctypes.c_double), c_i32,
                                      ctypes.c_double]),
    "gnn_quant_divide": (ctypes.c_int, [c_vp, c_vp, c_vp, c_i64, c_vp]),
    "gnn_sync_check": (ctypes.c_int, [c_vp]),
}

_LIB = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libgnnagg.so (building it first if it is missing or stale)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if build_if_missing:
        _build.build()
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"libgnnagg.so not found at {_build.LIB}; run build() first")
    _LIB = open_lib(_build.LIB)
    return _LIB


def open_lib(path: str):
    """A library handle for `path` with the C prototypes attached."""
    lib = ctypes.CDLL(path)
    for name, (res, args) in PROTOTYPES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def use_lib(lib):
    """Route every binding call through `lib` (a handle from open_lib);
    returns the handle used before.  For tests of build variants."""
    global _LIB
    old, _LIB = _LIB, lib
    return old


class GnnError(RuntimeError):
    def __init__(self, name, status, msg):
        super().__init__(f"{name} -> {STATUS.get(status, status)}: {msg}")
        self.status = status


def call(name, *args):
    lib = load()
    st = getattr(lib, name)(*args)
    if st != 0:
        raise GnnError(name, st, lib.gnn_last_error().decode(errors="replace"))
    return st
