"""Python binding of libgnnagg.so (boundary-quantised GCN aggregation on
GB300).  Functions carry the C entry points' names and only marshal torch
tensors (device memory) and the current CUDA stream into the C ABI; every
step of the computation runs in the library's CUDA kernels.  There is no CPU
path: without the library or a CUDA device the calls raise."""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field
from typing import Optional, Sequence

from . import _abi
from ._abi import (CSR_DEDUP, CSR_GCN, CSR_MEAN, CSR_SELF_LOOPS, CSR_SYMMETRIZE,  # noqa: F401
                   GnnBitRule, GnnBlocked,
                   GnnBoundary, GnnCsr, GnnError, GnnLdrState, call, load)

LdrState = GnnLdrState

__all__ = [
    "Csr", "Boundary", "BitRule", "GnnError", "load", "build",
    "gnn_csr_build", "gnn_csr_split", "gnn_spmm_workspace", "spmm_ws", "gnn_spmm_fwd_noalloc", "gnn_boundary_index", "gnn_boundary_long_slots", "gnn_boundary_set_bits", "gnn_slot_offsets",
    "gnn_quant_pack", "gnn_quant_pack_owned", "gnn_dequant_unpack", "gnn_spmm_fwd", "gnn_spmm_bwd", "gnn_sync_check", "gnn_kernel_launches",
    "rowbytes", "ld_for", "ldb_for", "gnn_dense_workspace", "gnn_dense_fwd", "gnn_dense_bwd",
    "gnn_layer_workspace", "gnn_layer_fwd", "gnn_layer_bwd",
    "gnn_halo_quant_pack", "gnn_spmm_bwd_local", "gnn_quant_pack_slots", "gnn_halo_quant_pack_slots", "gnn_layer_fwd_async", "gnn_layer_bwd_async",
    "LdrState", "gnn_ldr_init", "gnn_ldr_update", "gnn_quant_divide",
    "gnn_layer_tf_workspace", "gnn_layer_fwd_tf", "gnn_layer_bwd_tf",
    "gnn_gat_index", "gnn_gat_workspace", "gnn_gat_layer_fwd", "gnn_gat_layer_bwd",
    "gnn_spmm_bwd_masked", "gnn_spmm_bwd_local_masked", "gnn_dense_bwd_z", "ldz_for",
    "Blocked", "gnn_blocked_build", "gnn_spmm_fwd_blocked", "gnn_spmm_bwd_blocked",
]


def build(force: bool = False) -> str:
    from . import builder as _b
    return _b.build(force=force)


def _torch():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("sparse_aggregation_message_gb300 needs a CUDA device")
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def ld_for(F: int) -> int:
    """fp32 row stride: F rounded up to a multiple of 4."""
    return (F + 3) // 4 * 4


def ldb_for(F: int) -> int:
    """bf16 row stride for dense-transform inputs: F rounded up to 16."""
    return (F + 15) // 16 * 16


def ldz_for(F: int) -> int:
    """bf16 row stride of a pre-activation gradient dZ: F rounded up to 64."""
    return (F + 63) // 64 * 64


def rowbytes(b: int, F: int) -> int:
    return 16 * ((4 * F + 15) // 16) if b == 32 else 16 * ((F * b + 127) // 128)


@dataclass
class BitRule:
    """Boundary-pool width rule: level = #{i : 100*c > pct[i]*n}, mask =
    bits[level], width = min(8, mask * base)."""
    pct: Sequence[int]
    bits: Sequence[int]

    def to_c(self) -> GnnBitRule:
        r = GnnBitRule()
        r.n_levels = len(self.bits)
        assert len(self.pct) == len(self.bits) - 1
        for i, p in enumerate(self.pct):
            r.pct[i] = int(p)
        for i, b in enumerate(self.bits):
            r.bits[i] = int(b)
        return r


@dataclass
class Csr:
    n: int
    nnz: int
    symmetric: bool
    rowptr: object
    col: object
    val: object
    split_len: int = 0
    n_long: int = 0
    n_pieces: int = 0
    split: dict = field(default_factory=dict)
    val_t: object = None  # A^T weights (mean aggregation); None when A is symmetric

    def c(self) -> GnnCsr:
        s = self.split
        return GnnCsr(self.n, int(self.symmetric), self.nnz, _ptr(self.rowptr), _ptr(self.col),
                      _ptr(self.val), self.split_len, self.n_long, self.n_pieces,
                      _ptr(s.get("long_rows")), _ptr(s.get("piece_ptr")), _ptr(s.get("piece_row")),
                      _ptr(s.get("piece_beg")), _ptr(self.val_t))


@dataclass
class Boundary:
    P: int
    n: int
    n_slots: int
    nnz_cut: int
    F: int
    arrays: dict = field(default_factory=dict)
    long_slot_len: int = 0
    n_long_slots: int = 0

    def __getattr__(self, k):
        arrays = self.__dict__.get("arrays", {})
        if k in arrays:
            return arrays[k]
        raise AttributeError(k)

    def c(self, slot_off=None, F=None) -> GnnBoundary:
        a = self.arrays
        b = GnnBoundary()
        b.P, b.n, b.n_slots, b.nnz_cut = self.P, self.n, self.n_slots, self.nnz_cut
        b.F = self.F if F is None else F
        for k in ("part_start", "send_start", "slot_node", "col_remap", "val_remap", "local_cnt",
                  "slot_rowptr", "slot_col", "slot_val", "own_ptr", "own_slot", "node_bits",
                  "slot_bits"):
            setattr(b, k, _ptr(a[k]))
        b.slot_off = _ptr(a["slot_off"] if slot_off is None else slot_off)
        b.long_slot_len, b.n_long_slots = self.long_slot_len, self.n_long_slots
        b.long_slots = _ptr(a.get("long_slots"))
        b.val_remap_t = _ptr(a.get("val_remap_t"))
        b.halo_order = _ptr(a.get("halo_order"))
        return b


def _workspace(nbytes: int, device):
    torch = _torch()
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def gnn_csr_build(n: int, src, dst, flags: int = CSR_GCN, stream=None) -> Csr:
    """Edge list (int32 device tensors) -> Csr with GCN weights (or mean
    weights with CSR_MEAN, plus the A^T weights when symmetrised)."""
    torch = _torch()
    dev = src.device
    m = int(src.numel())
    ws_bytes = ctypes.c_size_t()
    call("gnn_csr_build_workspace", n, m, flags, ctypes.byref(ws_bytes))
    ws = _workspace(ws_bytes.value, dev)
    cap = (2 * m if flags & CSR_SYMMETRIZE else m) + (n if flags & CSR_SELF_LOOPS else 0)
    rowptr = torch.empty(n + 1, dtype=torch.int64, device=dev)
    col = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    val = torch.empty(max(cap, 1), dtype=torch.float32, device=dev)
    want_t = bool(flags & CSR_MEAN) and bool(flags & CSR_SYMMETRIZE)
    val_t = torch.empty(max(cap, 1), dtype=torch.float32, device=dev) if want_t else None
    out = GnnCsr(n, 0, 0, rowptr.data_ptr(), col.data_ptr(), val.data_ptr())
    out.val_t = _ptr(val_t)
    call("gnn_csr_build", n, m, _ptr(src), _ptr(dst), flags, cap, ctypes.byref(out), _ptr(ws),
         ws.numel(), _stream(stream))
    nnz = int(out.nnz)
    return Csr(n=n, nnz=nnz, symmetric=bool(out.symmetric), rowptr=rowptr, col=col[:nnz],
               val=val[:nnz], val_t=val_t[:nnz] if (val_t is not None and out.val_t) else None)


def gnn_csr_split(csr: Csr, split_len: int = 512, stream=None) -> Csr:
    """Attach a row-split plan: rows longer than split_len are cut into pieces
    of split_len entries (load balance for high-degree rows)."""
    torch = _torch()
    dev = csr.rowptr.device
    c = csr.c()
    ws_bytes = ctypes.c_size_t()
    call("gnn_csr_split_workspace", ctypes.byref(c), ctypes.byref(ws_bytes))
    ws = _workspace(ws_bytes.value, dev)
    nl, npc = ctypes.c_int32(), ctypes.c_int64()
    st = _stream(stream)
    call("gnn_csr_split_count", ctypes.byref(c), split_len, ctypes.byref(nl), ctypes.byref(npc),
         _ptr(ws), ws.numel(), st)
    nl, npc = nl.value, npc.value
    split = dict(long_rows=torch.empty(max(nl, 1), dtype=torch.int32, device=dev),
                 piece_ptr=torch.empty(nl + 1, dtype=torch.int64, device=dev),
                 piece_row=torch.empty(max(npc, 1), dtype=torch.int32, device=dev),
                 piece_beg=torch.empty(max(npc, 1), dtype=torch.int64, device=dev))
    out = Csr(csr.n, csr.nnz, csr.symmetric, csr.rowptr, csr.col, csr.val, split_len, nl, npc, split,
              csr.val_t)
    c2 = out.c()
    call("gnn_csr_split", ctypes.byref(c2), _ptr(ws), ws.numel(), st)
    return out


def gnn_spmm_workspace(csr: Csr, F: int) -> int:
    nb = ctypes.c_size_t()
    c = csr.c()
    call("gnn_spmm_workspace", ctypes.byref(c), F, ctypes.byref(nb))
    return nb.value


def spmm_ws(csr: Csr, F: int, device="cuda"):
    """A workspace tensor sized for the aggregation calls (or None)."""
    nb = gnn_spmm_workspace(csr, F)
    return _workspace(nb, device) if nb else None


def gnn_boundary_index(csr: Csr, P: int, rule: BitRule, base_bits: int, F: int,
                       stream=None) -> Boundary:
    torch = _torch()
    dev = csr.rowptr.device
    c = csr.c()
    ws_bytes = ctypes.c_size_t()
    call("gnn_boundary_workspace", ctypes.byref(c), P, ctypes.byref(ws_bytes))
    ws = _workspace(ws_bytes.value, dev)
    S, nc = ctypes.c_int64(), ctypes.c_int64()
    st = _stream(stream)
    call("gnn_boundary_count", ctypes.byref(c), P, ctypes.byref(S), ctypes.byref(nc), _ptr(ws),
         ws.numel(), st)
    S, nc, n = S.value, nc.value, csr.n
    i32, i64, u8, f32 = torch.int32, torch.int64, torch.uint8, torch.float32

    def e(k, dt):
        return torch.empty(max(k, 1), dtype=dt, device=dev)

    a = dict(part_start=e(P + 1, i64), send_start=e(P + 1, i64), slot_node=e(S, i32),
             col_remap=e(csr.nnz, i32), val_remap=e(csr.nnz, f32), local_cnt=e(n, i32),
             slot_rowptr=e(S + 1, i64), slot_col=e(nc, i32),
             slot_val=e(nc, f32), own_ptr=e(n + 1, i64), own_slot=e(S, i32), node_bits=e(n, u8),
             slot_bits=e(S, u8), slot_off=e(S + 1, i64))
    if csr.val_t is not None:
        a["val_remap_t"] = e(csr.nnz, f32)
    b = Boundary(P=P, n=n, n_slots=S, nnz_cut=nc, F=F, arrays=a)
    cb = b.c()
    call("gnn_boundary_index", ctypes.byref(c), ctypes.byref(rule.to_c()), base_bits, F,
         ctypes.byref(cb), _ptr(ws), ws.numel(), st)
    sizes = dict(part_start=P + 1, send_start=P + 1, slot_node=S, col_remap=csr.nnz,
                 val_remap=csr.nnz, local_cnt=n, slot_rowptr=S + 1, slot_col=nc, slot_val=nc, own_ptr=n + 1, own_slot=S,
                 node_bits=n, slot_bits=S, slot_off=S + 1, val_remap_t=csr.nnz)
    b.arrays = {k: v[:sizes[k]] for k, v in a.items()}
    return b


def gnn_boundary_long_slots(csr: Csr, bnd: Boundary, long_slot_len: int = 128, stream=None,
                            halo_order: bool = True) -> None:
    """Attach the list of slots with more than long_slot_len backward entries
    (their halo partials are then summed by a whole thread block each) and,
    with halo_order, the halo kernel's visiting order (slots by first
    backward entry)."""
    torch = _torch()
    dev = csr.rowptr.device
    c = csr.c()
    ws_bytes = ctypes.c_size_t()
    call("gnn_boundary_workspace", ctypes.byref(c), bnd.P, ctypes.byref(ws_bytes))
    ws = _workspace(ws_bytes.value, dev)
    cb = bnd.c()
    nl = ctypes.c_int32()
    st = _stream(stream)
    call("gnn_boundary_long_slots_count", ctypes.byref(cb), long_slot_len, ctypes.byref(nl), _ptr(ws),
         ws.numel(), st)
    bnd.arrays["long_slots"] = torch.empty(max(nl.value, 1), dtype=torch.int32, device=dev)
    bnd.long_slot_len, bnd.n_long_slots = long_slot_len, nl.value
    if halo_order:
        bnd.arrays["halo_order"] = torch.empty(max(bnd.n_slots, 1), dtype=torch.int32, device=dev)
    else:
        bnd.arrays.pop("halo_order", None)
    cb = bnd.c()
    call("gnn_boundary_long_slots", ctypes.byref(cb), _ptr(ws), ws.numel(), st)


def gnn_boundary_set_bits(csr: Csr, bnd: Boundary, rule: BitRule, base_bits: int, F: int,
                          stream=None) -> None:
    dev = csr.rowptr.device
    c = csr.c()
    ws_bytes = ctypes.c_size_t()
    call("gnn_boundary_workspace", ctypes.byref(c), bnd.P, ctypes.byref(ws_bytes))
    ws = _workspace(ws_bytes.value, dev)
    cb = bnd.c()
    call("gnn_boundary_set_bits", ctypes.byref(c), ctypes.byref(rule.to_c()), base_bits, F,
         ctypes.byref(cb), _ptr(ws), ws.numel(), _stream(stream))
    bnd.F = F


def gnn_slot_offsets(slot_bits, n_slots: int, F: int, stream=None):
    """Byte offsets [S+1] of each slot's packed row for feature width F."""
    torch = _torch()
    dev = slot_bits.device
    ws_bytes = ctypes.c_size_t()
    call("gnn_slot_offsets_workspace", n_slots, ctypes.byref(ws_bytes))
    ws = _workspace(ws_bytes.value, dev)
    off = torch.empty(n_slots + 1, dtype=torch.int64, device=dev)
    call("gnn_slot_offsets", _ptr(slot_bits), n_slots, F, _ptr(off), _ptr(ws), ws.numel(),
         _stream(stream))
    return off


def gnn_quant_pack(X, F: int, row_idx, n_rows: int, row_bits, row_off, seed: int, packed, meta,
                   stream=None) -> None:
    call("gnn_quant_pack", _ptr(X), X.stride(0), F, _ptr(row_idx), n_rows, _ptr(row_bits),
         _ptr(row_off), seed & 0xFFFFFFFF, _ptr(packed), _ptr(meta), _stream(stream))


def gnn_quant_pack_owned(bnd: Boundary, X, F: int, seed: int, packed, meta, slot_off=None,
                         stream=None) -> None:
    """Every slot's forward message (the bytes gnn_quant_pack writes for the
    slot rows), formed node by node: each boundary node's row is prepared once
    for all the partitions it is sent to."""
    cb = bnd.c(slot_off, F if slot_off is not None else None)
    call("gnn_quant_pack_owned", ctypes.byref(cb), _ptr(X), X.stride(0), F, seed & 0xFFFFFFFF,
         _ptr(packed), _ptr(meta), _stream(stream))


def gnn_quant_divide(a, b, q, stream=None) -> None:
    """q = a / b as the quantiser divides (fp32 tensors of equal size)."""
    call("gnn_quant_divide", _ptr(a), _ptr(b), _ptr(q), a.numel(), _stream(stream))


def gnn_dequant_unpack(packed, meta, row_off, row_bits, n_rows: int, F: int, out,
                       stream=None) -> None:
    call("gnn_dequant_unpack", _ptr(packed), _ptr(meta), _ptr(row_off), _ptr(row_bits), n_rows, F,
         _ptr(out), out.stride(0), _stream(stream))


def gnn_spmm_fwd_noalloc(csr: Csr, bnd: Optional[Boundary], H, F: int, packed=None, meta=None,
                         M=None, Mb=None, slot_off=None, stream=None) -> None:
    """gnn_spmm_fwd for callers that cannot allocate: scratch comes from a
    fixed device array inside the library (see the C header)."""
    c = csr.c()
    cb = bnd.c(slot_off, F if slot_off is not None else None) if bnd is not None else None
    call("gnn_spmm_fwd_noalloc", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None,
         _ptr(H), H.stride(0), F, _ptr(packed), _ptr(meta), _ptr(M),
         M.stride(0) if M is not None else 0, _ptr(Mb), Mb.stride(0) if Mb is not None else 0,
         _stream(stream))


def _ws_args(csr: Csr, F: int, ws, device):
    if ws is None and csr.split_len:
        ws = spmm_ws(csr, F, device)
    return _ptr(ws), (ws.numel() * ws.element_size() if ws is not None else 0)


def gnn_spmm_fwd(csr: Csr, bnd: Optional[Boundary], H, F: int, packed=None, meta=None, M=None,
                 Mb=None, slot_off=None, ws=None, stream=None) -> None:
    c = csr.c()
    cb = bnd.c(slot_off, F if slot_off is not None else None) if bnd is not None else None
    wp, wn = _ws_args(csr, F, ws, H.device)
    call("gnn_spmm_fwd", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None, _ptr(H),
         H.stride(0), F, _ptr(packed), _ptr(meta), _ptr(M), M.stride(0) if M is not None else 0,
         _ptr(Mb), Mb.stride(0) if Mb is not None else 0, wp, wn, _stream(stream))


def gnn_spmm_bwd(csr: Csr, bnd: Optional[Boundary], G, F: int, seed: int, packed_ws, meta_ws, dH,
                 slot_off=None, ws=None, stream=None) -> None:
    c = csr.c()
    cb = bnd.c(slot_off, F if slot_off is not None else None) if bnd is not None else None
    wp, wn = _ws_args(csr, F, ws, G.device)
    call("gnn_spmm_bwd", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None, _ptr(G),
         G.stride(0), F, seed & 0xFFFFFFFF, _ptr(packed_ws), _ptr(meta_ws), _ptr(dH), dH.stride(0),
         wp, wn, _stream(stream))


def gnn_halo_quant_pack(bnd: Boundary, G, F: int, seed: int, packed, meta, slot_off=None,
                        stream=None) -> None:
    """Backward messages only: each slot's halo partial of G, quantised and
    packed."""
    cb = bnd.c(slot_off, F if slot_off is not None else None)
    call("gnn_halo_quant_pack", ctypes.byref(cb), _ptr(G), G.stride(0), F, seed & 0xFFFFFFFF,
         _ptr(packed), _ptr(meta), _stream(stream))


def gnn_quant_pack_slots(X, F: int, slot_node, s0: int, s1: int, slot_bits, slot_off, seed: int,
                         packed, meta, stream=None) -> None:
    """Forward messages of slots s0..s1-1 only (row key s), at their places in
    the slot-ordered buffer."""
    call("gnn_quant_pack_slots", _ptr(X), X.stride(0), F, _ptr(slot_node), int(s0), int(s1),
         _ptr(slot_bits), _ptr(slot_off), seed & 0xFFFFFFFF, _ptr(packed), _ptr(meta),
         _stream(stream))


def gnn_halo_quant_pack_slots(bnd: Boundary, G, F: int, s0: int, s1: int, seed: int, packed, meta,
                              slot_off=None, stream=None) -> None:
    """Backward messages of slots s0..s1-1 only."""
    cb = bnd.c(slot_off, F if slot_off is not None else None)
    call("gnn_halo_quant_pack_slots", ctypes.byref(cb), _ptr(G), G.stride(0), F, int(s0), int(s1),
         seed & 0xFFFFFFFF, _ptr(packed), _ptr(meta), _stream(stream))


def gnn_spmm_bwd_local(csr: Csr, bnd: Boundary, G, F: int, packed, meta, dH, slot_off=None,
                       ws=None, stream=None) -> None:
    """Owner-side backward aggregation: local transpose entries plus the
    dequantised backward messages in packed/meta."""
    c = csr.c()
    cb = bnd.c(slot_off, F if slot_off is not None else None)
    wp, wn = _ws_args(csr, F, ws, G.device)
    call("gnn_spmm_bwd_local", ctypes.byref(c), ctypes.byref(cb), _ptr(G), G.stride(0), F,
         _ptr(packed), _ptr(meta), _ptr(dH), dH.stride(0), wp, wn, _stream(stream))


def gnn_spmm_bwd_masked(csr: Csr, bnd: Optional[Boundary], G, F: int, seed: int, packed_ws, meta_ws,
                        H_mask, dZ, slot_off=None, ws=None, stream=None) -> None:
    """dZ (bf16, row stride >= ldz_for(F)) = bf16((A^T G) * 1[H_mask > 0])."""
    c = csr.c()
    cb = bnd.c(slot_off, F if slot_off is not None else None) if bnd is not None else None
    wp, wn = _ws_args(csr, F, ws, G.device)
    call("gnn_spmm_bwd_masked", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None,
         _ptr(G), G.stride(0), F, seed & 0xFFFFFFFF, _ptr(packed_ws), _ptr(meta_ws), _ptr(H_mask),
         H_mask.stride(0) if H_mask is not None else 0, _ptr(dZ), dZ.stride(0), wp, wn,
         _stream(stream))


def gnn_spmm_bwd_local_masked(csr: Csr, bnd: Boundary, G, F: int, packed, meta, H_mask, dZ,
                              slot_off=None, ws=None, stream=None) -> None:
    """The owner-side half of gnn_spmm_bwd_masked: dZ = bf16((local A^T G +
    the dequantised messages in packed/meta) * 1[H_mask > 0])."""
    c = csr.c()
    cb = bnd.c(slot_off, F if slot_off is not None else None)
    wp, wn = _ws_args(csr, F, ws, G.device)
    call("gnn_spmm_bwd_local_masked", ctypes.byref(c), ctypes.byref(cb), _ptr(G), G.stride(0), F,
         _ptr(packed), _ptr(meta), _ptr(H_mask), H_mask.stride(0) if H_mask is not None else 0,
         _ptr(dZ), dZ.stride(0), wp, wn, _stream(stream))


def gnn_kernel_launches() -> int:
    """Kernels launched through the library by this process so far."""
    return int(load().gnn_kernel_launches())


def gnn_sync_check(stream=None) -> None:
    call("gnn_sync_check", _stream(stream))


# ---------------------------------------------------------------- dense transform and layers
def gnn_dense_workspace(n: int, F_in: int, F_out: int) -> int:
    nb = ctypes.c_size_t()
    call("gnn_dense_workspace", n, F_in, F_out, ctypes.byref(nb))
    return nb.value


def gnn_dense_fwd(Mb, n: int, F_in: int, W, F_out: int, relu: bool, H_out, ws=None,
                  stream=None) -> None:
    """H_out = act(Mb W) on tcgen05 (Mb, W bf16 tensors; H_out fp32)."""
    if ws is None:
        ws = _workspace(gnn_dense_workspace(n, F_in, F_out), Mb.device)
    call("gnn_dense_fwd", _ptr(Mb), Mb.stride(0), n, F_in, _ptr(W), F_out, int(relu), _ptr(H_out),
         H_out.stride(0), _ptr(ws), ws.numel(), _stream(stream))


def gnn_dense_bwd(Mb, n: int, F_in: int, W, F_out: int, dH_out, H_out, relu: bool, dM, dW,
                  ws=None, stream=None) -> None:
    if ws is None:
        ws = _workspace(gnn_dense_workspace(n, F_in, F_out), Mb.device)
    call("gnn_dense_bwd", _ptr(Mb), Mb.stride(0), n, F_in, _ptr(W), F_out, _ptr(dH_out),
         dH_out.stride(0), _ptr(H_out), H_out.stride(0) if H_out is not None else 0, int(relu),
         _ptr(dM), dM.stride(0) if dM is not None else 0, _ptr(dW), _ptr(ws), ws.numel(),
         _stream(stream))


def gnn_dense_bwd_z(Mb, n: int, F_in: int, W, F_out: int, dZ, dM, dW, ws=None, stream=None) -> None:
    if ws is None:
        ws = _workspace(gnn_dense_workspace(n, F_in, F_out), Mb.device)
    call("gnn_dense_bwd_z", _ptr(Mb), Mb.stride(0), n, F_in, _ptr(W), F_out, _ptr(dZ), dZ.stride(0),
         _ptr(dM), dM.stride(0) if dM is not None else 0, _ptr(dW), _ptr(ws), ws.numel(),
         _stream(stream))


def gnn_layer_workspace(csr: Csr, F_in: int, F_out: int) -> int:
    nb = ctypes.c_size_t()
    c = csr.c()
    call("gnn_layer_workspace", ctypes.byref(c), F_in, F_out, ctypes.byref(nb))
    return nb.value


def gnn_layer_fwd(csr: Csr, bnd: Optional[Boundary], H_in, F_in: int, W, F_out: int, relu: bool,
                  seed: int, packed_ws, meta_ws, Mb, H_out, slot_off=None, ws=None,
                  stream=None) -> None:
    c = csr.c()
    cb = bnd.c(slot_off, F_in if slot_off is not None else None) if bnd is not None else None
    if ws is None:
        ws = _workspace(gnn_layer_workspace(csr, F_in, F_out), H_in.device)
    call("gnn_layer_fwd", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None, _ptr(H_in),
         H_in.stride(0), F_in, _ptr(W), F_out, int(relu), seed & 0xFFFFFFFF, _ptr(packed_ws),
         _ptr(meta_ws), _ptr(Mb), Mb.stride(0), _ptr(H_out), H_out.stride(0), _ptr(ws), ws.numel(),
         _stream(stream))


def gnn_layer_bwd(csr: Csr, bnd: Optional[Boundary], dH_out, H_out, relu: bool, Mb, W, F_in: int,
                  F_out: int, seed: int, packed_ws, meta_ws, dW, dH_in=None, slot_off=None,
                  ws=None, stream=None) -> None:
    c = csr.c()
    cb = bnd.c(slot_off, F_in if slot_off is not None else None) if bnd is not None else None
    if ws is None:
        ws = _workspace(gnn_layer_workspace(csr, F_in, F_out), dH_out.device)
    call("gnn_layer_bwd", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None,
         _ptr(dH_out), dH_out.stride(0), _ptr(H_out), H_out.stride(0) if H_out is not None else 0,
         int(relu), _ptr(Mb), Mb.stride(0), _ptr(W), F_in, F_out, seed & 0xFFFFFFFF, _ptr(packed_ws),
         _ptr(meta_ws), _ptr(dW), _ptr(dH_in), dH_in.stride(0) if dH_in is not None else 0,
         _ptr(ws), ws.numel(), _stream(stream))


def gnn_layer_fwd_async(csr: Csr, bnd: Boundary, H_in, F_in: int, W, F_out: int, relu: bool,
                        seed: int, packed_prev, meta_prev, packed_next, meta_next, Mb, H_out,
                        aux, slot_off=None, ws=None, stream=None) -> None:
    """Forward layer of an asynchronous epoch: remote sources read the
    previous epoch's messages; this epoch's are packed on ``aux`` meanwhile."""
    c = csr.c()
    cb = bnd.c(slot_off, F_in if slot_off is not None else None)
    if ws is None:
        ws = _workspace(gnn_layer_workspace(csr, F_in, F_out), H_in.device)
    call("gnn_layer_fwd_async", ctypes.byref(c), ctypes.byref(cb), _ptr(H_in), H_in.stride(0), F_in,
         _ptr(W), F_out, int(relu), seed & 0xFFFFFFFF, _ptr(packed_prev), _ptr(meta_prev),
         _ptr(packed_next), _ptr(meta_next), _ptr(Mb), Mb.stride(0), _ptr(H_out), H_out.stride(0),
         _ptr(ws), ws.numel(), _stream(stream), aux.cuda_stream)


def gnn_layer_bwd_async(csr: Csr, bnd: Boundary, dH_out, H_out, relu: bool, Mb, W, F_in: int,
                        F_out: int, seed: int, packed_prev, meta_prev, packed_next, meta_next, dW,
                        dH_in, aux, slot_off=None, ws=None, stream=None) -> None:
    c = csr.c()
    cb = bnd.c(slot_off, F_in if slot_off is not None else None)
    if ws is None:
        ws = _workspace(gnn_layer_workspace(csr, F_in, F_out), dH_out.device)
    call("gnn_layer_bwd_async", ctypes.byref(c), ctypes.byref(cb), _ptr(dH_out), dH_out.stride(0),
         _ptr(H_out), H_out.stride(0) if H_out is not None else 0, int(relu), _ptr(Mb), Mb.stride(0),
         _ptr(W), F_in, F_out, seed & 0xFFFFFFFF, _ptr(packed_prev), _ptr(meta_prev),
         _ptr(packed_next), _ptr(meta_next), _ptr(dW), _ptr(dH_in),
         dH_in.stride(0) if dH_in is not None else 0, _ptr(ws), ws.numel(), _stream(stream),
         aux.cuda_stream)


# ---------------------------------------------------------------- transform-first layers
def gnn_layer_tf_workspace(csr: Csr, F_in: int, F_out: int) -> int:
    nb = ctypes.c_size_t()
    c = csr.c()
    call("gnn_layer_tf_workspace", ctypes.byref(c), F_in, F_out, ctypes.byref(nb))
    return nb.value


def gnn_layer_fwd_tf(csr: Csr, bnd: Optional[Boundary], H_in, F_in: int, W, F_out: int,
                     relu: bool, seed: int, packed_ws, meta_ws, Hb, Y, H_out, slot_off=None,
                     ws=None, stream=None) -> None:
    """Y = bf16(H_in) W, messages from Y, H_out = act(A Y) (aggregation at
    width F_out; bnd offsets for F_out)."""
    c = csr.c()
    cb = bnd.c(slot_off, F_out if slot_off is not None else None) if bnd is not None else None
    if ws is None:
        ws = _workspace(gnn_layer_tf_workspace(csr, F_in, F_out), H_in.device)
    call("gnn_layer_fwd_tf", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None,
         _ptr(H_in), H_in.stride(0), F_in, _ptr(W), F_out, int(relu), seed & 0xFFFFFFFF,
         _ptr(packed_ws), _ptr(meta_ws), _ptr(Hb), Hb.stride(0), _ptr(Y), Y.stride(0), _ptr(H_out),
         H_out.stride(0), _ptr(ws), ws.numel(), _stream(stream))


def gnn_layer_bwd_tf(csr: Csr, bnd: Optional[Boundary], dH_out, H_out, relu: bool, Hb, W,
                     F_in: int, F_out: int, seed: int, packed_ws, meta_ws, dW, dH_in=None,
                     slot_off=None, ws=None, stream=None) -> None:
    c = csr.c()
    cb = bnd.c(slot_off, F_out if slot_off is not None else None) if bnd is not None else None
    if ws is None:
        ws = _workspace(gnn_layer_tf_workspace(csr, F_in, F_out), dH_out.device)
    call("gnn_layer_bwd_tf", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None,
         _ptr(dH_out), dH_out.stride(0), _ptr(H_out), H_out.stride(0) if H_out is not None else 0,
         int(relu), _ptr(Hb), Hb.stride(0), _ptr(W), F_in, F_out, seed & 0xFFFFFFFF,
         _ptr(packed_ws), _ptr(meta_ws), _ptr(dW), _ptr(dH_in),
         dH_in.stride(0) if dH_in is not None else 0, _ptr(ws), ws.numel(), _stream(stream))


# ---------------------------------------------------------------- cluster-blocked aggregation
@dataclass
class Blocked:
    T: int
    n_rb: int
    n_tiles: int
    n_entries: int
    arrays: dict
    residual: Csr

    def c(self) -> GnnBlocked:
        a = self.arrays
        b = GnnBlocked()
        b.T, b.n_rb, b.n_tiles, b.n_entries = self.T, self.n_rb, self.n_tiles, self.n_entries
        for k in ("rb_tile_ptr", "tile_cb", "tile_ptr", "tile_rowptr", "ent_col", "ent_val",
                  "res_local_cnt"):
            setattr(b, k, _ptr(a.get(k)))
        b.residual = self.residual.c()
        return b


def gnn_blocked_build(csr: Csr, bnd: Optional[Boundary], min_entries: int = 1024, T: int = 128,
                      split_len: int = 128, stream=None) -> Blocked:
    """Dense T x T tiles (at least min_entries entries) and the residual CSR,
    with a split plan of split_len entries for the residual (0: none)."""
    torch = _torch()
    dev = csr.rowptr.device
    c = csr.c()
    cb = bnd.c() if bnd is not None else None
    pb = ctypes.byref(cb) if cb is not None else None
    nb = ctypes.c_size_t()
    call("gnn_blocked_workspace", ctypes.byref(c), pb, T, min_entries, ctypes.byref(nb))
    ws = _workspace(nb.value, dev)
    nt, ne, nr = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    st = _stream(stream)
    call("gnn_blocked_count", ctypes.byref(c), pb, T, min_entries, ctypes.byref(nt), ctypes.byref(ne),
         ctypes.byref(nr), _ptr(ws), ws.numel(), st)
    nt, ne, nr, n = nt.value, ne.value, nr.value, csr.n
    n_rb = (n + T - 1) // T

    def e(k, dt):
        return torch.empty(max(k, 1), dtype=dt, device=dev)

    a = dict(rb_tile_ptr=e(n_rb + 1, torch.int64), tile_cb=e(nt, torch.int32),
             tile_ptr=e(nt + 1, torch.int64), tile_rowptr=e(nt * (T + 1), torch.int32),
             ent_col=e(ne + 16, torch.uint8), ent_val=e(ne, torch.float32))
    if bnd is not None:
        a["res_local_cnt"] = e(n, torch.int32)
    res = Csr(n=n, nnz=nr, symmetric=False, rowptr=e(n + 1, torch.int64), col=e(nr, torch.int32),
              val=e(nr, torch.float32))
    bl = Blocked(T=T, n_rb=n_rb, n_tiles=nt, n_entries=ne, arrays=a, residual=res)
    out = bl.c()
    call("gnn_blocked_build", ctypes.byref(c), pb, T, min_entries, ctypes.byref(out), _ptr(ws), ws.numel(), st)
    res.col, res.val = res.col[:nr], res.val[:nr]
    if split_len and nr > 0:
        bl.residual = gnn_csr_split(res, split_len, stream)
    return bl


def _blocked_ws(bl: Blocked, F: int, device, ws):
    if ws is not None:
        return ws
    nb = ctypes.c_size_t()
    b = bl.c()
    call("gnn_blocked_spmm_workspace", ctypes.byref(b), F, ctypes.byref(nb))
    return _workspace(nb.value, device)


def gnn_spmm_fwd_blocked(csr: Csr, bnd: Optional[Boundary], bl: Blocked, H, F: int, packed=None,
                         meta=None, M=None, Mb=None, slot_off=None, ws=None, stream=None) -> None:
    c = csr.c()
    cb = bnd.c(slot_off, F if slot_off is not None else None) if bnd is not None else None
    b = bl.c()
    ws = _blocked_ws(bl, F, H.device, ws)
    call("gnn_spmm_fwd_blocked", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None,
         ctypes.byref(b), _ptr(H), H.stride(0), F, _ptr(packed), _ptr(meta), _ptr(M),
         M.stride(0) if M is not None else 0, _ptr(Mb), Mb.stride(0) if Mb is not None else 0,
         _ptr(ws), ws.numel(), _stream(stream))


def gnn_spmm_bwd_blocked(csr: Csr, bnd: Optional[Boundary], bl: Blocked, G, F: int, seed: int,
                         packed_ws=None, meta_ws=None, H_mask=None, dH=None, dZ=None, slot_off=None,
                         ws=None, stream=None) -> None:
    c = csr.c()
    cb = bnd.c(slot_off, F if slot_off is not None else None) if bnd is not None else None
    b = bl.c()
    ws = _blocked_ws(bl, F, G.device, ws)
    call("gnn_spmm_bwd_blocked", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None,
         ctypes.byref(b), _ptr(G), G.stride(0), F, seed & 0xFFFFFFFF, _ptr(packed_ws), _ptr(meta_ws),
         _ptr(H_mask), H_mask.stride(0) if H_mask is not None else 0, _ptr(dH),
         dH.stride(0) if dH is not None else 0, _ptr(dZ), dZ.stride(0) if dZ is not None else 0,
         _ptr(ws), ws.numel(), _stream(stream))


# ---------------------------------------------------------------- attention aggregator
def gnn_gat_index(csr: Csr, bnd: Optional[Boundary], stream=None):
    """Position maps (tpos [nnz], spos [nnz_cut] or None) for the backward."""
    torch = _torch()
    dev = csr.rowptr.device
    tpos = torch.empty(max(csr.nnz, 1), dtype=torch.int64, device=dev)
    spos = torch.empty(max(bnd.nnz_cut, 1), dtype=torch.int64, device=dev) if bnd is not None else None
    c = csr.c()
    cb = bnd.c() if bnd is not None else None
    call("gnn_gat_index", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None, _ptr(tpos),
         _ptr(spos), _stream(stream))
    return tpos, spos


def gnn_gat_workspace(csr: Csr, bnd: Optional[Boundary], F_in: int, F_out: int) -> int:
    nb = ctypes.c_size_t()
    c = csr.c()
    cb = bnd.c() if bnd is not None else None
    call("gnn_gat_workspace", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None, F_in,
         F_out, ctypes.byref(nb))
    return nb.value


def _gat_bnd(bnd, slot_off, F_out):
    return bnd.c(slot_off, F_out if slot_off is not None else None) if bnd is not None else None


def gnn_gat_layer_fwd(csr: Csr, bnd: Optional[Boundary], H_in, F_in: int, W, F_out: int, a_l, a_r,
                      relu: bool, seed: int, packed, meta, Hb, Y, alpha, H_out, slot_off=None,
                      ws=None, stream=None) -> None:
    c = csr.c()
    cb = _gat_bnd(bnd, slot_off, F_out)
    if ws is None:
        ws = _workspace(gnn_gat_workspace(csr, bnd, F_in, F_out), H_in.device)
    call("gnn_gat_layer_fwd", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None,
         _ptr(H_in), H_in.stride(0), F_in, _ptr(W), F_out, _ptr(a_l), _ptr(a_r), int(relu),
         seed & 0xFFFFFFFF, _ptr(packed), _ptr(meta), _ptr(Hb), Hb.stride(0), _ptr(Y), Y.stride(0),
         _ptr(alpha), _ptr(H_out), H_out.stride(0), _ptr(ws), ws.numel(), _stream(stream))


def gnn_gat_layer_bwd(csr: Csr, bnd: Optional[Boundary], tpos, spos, dH_out, H_out, relu: bool, Hb,
                      Y, alpha, packed_fwd, meta_fwd, W, a_l, a_r, F_in: int, F_out: int, seed: int,
                      packed_ws, meta_ws, dW, da_l, da_r, dH_in=None, g_out=None, slot_off=None,
                      ws=None, stream=None) -> None:
    c = csr.c()
    cb = _gat_bnd(bnd, slot_off, F_out)
    if ws is None:
        ws = _workspace(gnn_gat_workspace(csr, bnd, F_in, F_out), dH_out.device)
    call("gnn_gat_layer_bwd", ctypes.byref(c), ctypes.byref(cb) if cb is not None else None,
         _ptr(tpos), _ptr(spos), _ptr(dH_out), dH_out.stride(0), _ptr(H_out),
         H_out.stride(0) if H_out is not None else 0, int(relu), _ptr(Hb), Hb.stride(0), _ptr(Y),
         Y.stride(0), _ptr(alpha), _ptr(packed_fwd), _ptr(meta_fwd), _ptr(W), _ptr(a_l), _ptr(a_r),
         F_in, F_out, seed & 0xFFFFFFFF, _ptr(packed_ws), _ptr(meta_ws), _ptr(dW), _ptr(da_l),
         _ptr(da_r), _ptr(dH_in), dH_in.stride(0) if dH_in is not None else 0, _ptr(g_out),
         _ptr(ws), ws.numel(), _stream(stream))


# ---------------------------------------------------------------- epoch control (host only)
def gnn_ldr_init(lam: float = 0.9, delta: int = 5, b_min: int = 1, b_max: int = 8) -> LdrState:
    st = LdrState()
    call("gnn_ldr_init", ctypes.byref(st), float(lam), delta, b_min, b_max)
    return st


def gnn_ldr_update(st: LdrState, partition_losses: Sequence[float], epoch_seconds: float):
    """Reports one epoch; returns (base width, asynchronous?) for the next."""
    n = len(partition_losses)
    arr = (ctypes.c_double * max(n, 1))(*[float(x) for x in partition_losses])
    call("gnn_ldr_update", ctypes.byref(st), arr, n, float(epoch_seconds))
    return st.base_bits, bool(st.async_next)
