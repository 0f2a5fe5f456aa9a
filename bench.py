"""Throughput of the boundary-quantised GCN aggregation hot path on GB300.

One step = one full forward + backward pass of a GCN over a synthetic graph
with P virtual partitions (contiguous node blocks): per layer, quantise and
pack the boundary rows, aggregate with dequantised remote rows (bf16 output),
transform on tcgen05 with ReLU; backward, mask and transform, weight gradient,
halo partials quantised and packed, local transpose aggregation plus owner
dequant-add (skipped for the first layer).

Metric: algorithmic bytes of every kernel of the step (the per-call byte
counts documented in the design notes) divided by the step time, in GB/s;
the JSON line also carries per-kernel GB/s, GFLOP/s and TFLOP/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload yelp]
  python bench.py --impl reference ...   (the oracle on host cores)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from synth.graphs import CONFIGS  # noqa: E402

METRIC = "SpMM fwd+bwd GB/s & GFLOP/s, quant-pack GB/s; % of GB300 HBM roofline"
UNIT = "GB/s"

WORKLOAD_TEXT = {
    "tiny": "4,096-node planted partition (4 communities, avg degree 8), F=16, 2-layer GCN hidden 16, P=4, top-10% 8 bits else 2",
    "yelp": "Yelp-shaped DC-SBM: 716,847 nodes, 6.975M undirected edges (14.67M CSR entries), power-law degrees over 64 communities, F=300, 3-layer GCN hidden 256, P=8, top-20% 8 bits else 4",
    "reddit": "Reddit-shaped DC-SBM: 232,965 nodes, 57.3M undirected edges, heavy tail capped at 20k, 50 communities, F=602, 2-layer GCN hidden 128, P=8, top-10% 8 bits else 2",
    "products": "ogbn-products-shaped DC-SBM: 2,449,029 nodes, 30,929,570 undirected edges, 128 communities, F=100, 4-layer GCN hidden 256, P=8, width quartiles {1,2,4,8}",
    "scale": "R-MAT scale 24 (16.8M nodes, 128M edge draws), BFS-ordered into 16 blocks, F=256, 3-layer GCN hidden 256, P=16, top-5% 8 bits else base 1",
    "rmat20": "R-MAT scale 20 (1.05M nodes, 8M edge draws), BFS-ordered into 16 blocks, F=256, 3-layer GCN hidden 256, P=16, top-5% 8 bits else base 1 (the scale workload's generator at 1/16 size, for counter captures)",
}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def rowbytes(b, F):
    b = np.asarray(b, np.int64)
    return np.where(b == 32, 16 * ((4 * F + 15) // 16), 16 * ((F * b + 127) // 128))


# --------------------------------------------------------------- byte models
def kernel_bytes(n, nnz, nnz_cut, S, F, slot_bits, slot_cut, out_bytes_per_row):
    """Gather-model bytes of the aggregation calls and the quantiser at width
    F: every gathered row counted at every use.  slot_cut[s] = cut entries of
    slot s (forward remote reads per slot).  bwd = halo + local."""
    rb = rowbytes(slot_bits, F)
    Q = int(rb.sum())
    remote = int((slot_cut * (rb + 8)).sum())
    fwd = 8 * (n + 1) + 8 * nnz + (nnz - nnz_cut) * 4 * F + remote + out_bytes_per_row * n
    qp = 4 * S + 4 * F * S + Q + 8 * S + 1 * S + 8 * S
    halo = 8 * (S + 1) + 8 * nnz_cut + nnz_cut * 4 * F + Q + 8 * S          # halo partials + pack
    local = 8 * (n + 1) + 8 * nnz + (nnz - nnz_cut) * 4 * F + Q + 8 * S + 4 * F * n  # local + owned
    return dict(fwd=fwd, quant=qp, bwd=halo + local, halo=halo, local=local, Q=Q)


def compulsory_bytes(n, nnz, nnz_cut, S, F, Q, n_pool, n_halo_src, out_fwd, out_bwd):
    """Each array a kernel touches counted once (the least any schedule of the
    same algorithm moves between HBM and the chip): CSR metadata, every
    distinct source row, the messages and their per-slot tables, the outputs.
    n_pool = distinct message nodes (rows the quantiser reads); n_halo_src =
    distinct rows the halo partials read; out_* = output bytes per row."""
    tables = 17 * S  # slot width (1), offset (8), meta (8)
    return dict(
        quant=4 * S + 4 * F * n_pool + Q + tables,
        fwd=8 * (n + 1) + 8 * nnz + 4 * n + 4 * F * n + Q + tables + out_fwd * n,
        halo=8 * (S + 1) + 8 * nnz_cut + 4 * F * n_halo_src + Q + tables,
        local=8 * (n + 1) + 8 * nnz + 4 * n + 4 * F * n + 8 * (n + 1) + 4 * S + Q + tables
        + out_bwd * n,
    )


def gemm_bytes(n, F_in, F_out):
    ldb = (F_in + 15) // 16 * 16
    ldz = (F_out + 63) // 64 * 64
    fwd = 2 * n * ldb + 2 * F_in * F_out + 4 * n * F_out
    mask = 4 * n * F_out * 2 + 2 * n * ldz
    dM = 2 * n * ldz + 2 * F_in * F_out + 4 * n * ((F_in + 3) // 4 * 4)
    dW = 2 * n * ldb + 2 * n * ldz + 4 * F_in * F_out
    return dict(fwd=fwd, mask=mask, dM=dM, dW=dW)


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.md")
# the sources each kernel kind is built from
TRAFFIC_SOURCES = {"quant": ("quant.cu", "device.cuh"), "spmm_fwd": ("spmm.cu", "device.cuh"),
                   "halo": ("spmm.cu", "device.cuh"), "spmm_bwd": ("spmm.cu", "device.cuh")}


def traffic_source_hash(kind, read=None):
    """Hash of the sources a kernel kind is built from: committed DRAM
    counters count only while the kernels they were taken on are unchanged.
    ``read(name) -> bytes`` reads a source (default: today's files)."""
    import hashlib

    csrc = os.path.join(ROOT, "sparse_aggregation_message_gb300", "csrc")
    if read is None:
        def read(f):
            with open(os.path.join(csrc, f), "rb") as fh:
                return fh.read()
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES[kind]:
        h.update(read(f))
    return h.hexdigest()[:16]


def committed_traffic(workload, base_bits=None, path=TRAFFIC_FILE):
    """DRAM bytes (read + write) per launch of each aggregation-path kernel on
    this workload, from the committed ncu summary: lines of the form
    ``traffic workload=W base=B kind=K bytes_per_launch=N source=H``.  Kernels
    whose source hash differs from today's sources are left out."""
    import re

    if not os.path.exists(path):
        return {}
    out = {}
    with open(path) as f:
        for ln in f:
            m = re.match(r"^traffic workload=(\S+) base=(\d+) kind=(\S+) bytes_per_launch=(\d+) "
                         r"source=([0-9a-f]+)\s*$", ln.strip())
            if not m or m.group(1) != workload or m.group(3) not in TRAFFIC_SOURCES:
                continue
            if m.group(5) != traffic_source_hash(m.group(3)):
                continue
            if base_bits is not None and int(m.group(2)) != int(base_bits):
                continue
            out[m.group(3)] = int(m.group(4))
    return out


def default_variant(args):
    """The aggregate-first GCN path with the row kernels (the counters in the
    committed summary were taken on it)."""
    return args.order == "af" and args.aggregator == "gcn" and not args.blocked


def max_over_ranks(value, world, device="cpu"):
    """The slowest rank's value (every rank gets it); identity for one rank."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(bytes_per_rank, world, ms):
    """GB/s of the whole job: every replica moves bytes_per_rank in ms."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


# --------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- GPU arm
def layer_orders(order, dims):
    """Per layer: True to transform first (aggregate Y = H W at width F_out).
    "auto" does so where it gathers fewer bytes: the first layer runs one
    aggregation aggregate-first (its input gradient is never formed) but two
    transform-first (dY is needed for dW); later layers run two either way."""
    L = len(dims) - 1
    if order == "af":
        return [False] * L
    if order == "tf":
        return [dims[l + 1] < dims[l] for l in range(L)]
    return [2 * dims[l + 1] < dims[l] * (1 if l == 0 else 2) for l in range(L)]


def run_gpu(args, rank, world, local_rank):
    import torch

    import sparse_aggregation_message_gb300 as G
    from synth import make_workload
    from synth.graphs import make_weight_bf16

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    G.load()
    wl = make_workload(args.workload)
    n, P, dims, L = wl.n, wl.P, wl.dims, wl.layers
    base = args.base_bits if args.base_bits else wl.base_bits[0]
    flags = G.CSR_GCN | (G.CSR_MEAN if args.aggregator == "mean" else 0)  # gat: GCN pattern
    csr = G.gnn_csr_build(n, torch.from_numpy(wl.src).to(dev), torch.from_numpy(wl.dst).to(dev),
                          flags)
    csr = G.gnn_csr_split(csr, args.split_len)
    rule = G.BitRule(wl.rule_pct, wl.rule_bits)
    F0 = dims[0]
    bnd = G.gnn_boundary_index(csr, P, rule, base, F0)
    G.gnn_boundary_long_slots(csr, bnd, args.long_slot_len)
    S = bnd.n_slots
    gat = args.aggregator == "gat"
    # attention layers aggregate the transformed rows
    tf = [True] * L if gat else layer_orders(args.order, dims)
    # message (and aggregation) width of each layer
    mwid = [dims[l + 1] if tf[l] else dims[l] for l in range(L)]
    widths = sorted(set(mwid))
    offs = {F: (bnd.slot_off if F == F0 else G.gnn_slot_offsets(bnd.slot_bits, S, F)) for F in widths}
    Qmax = max(int(offs[F][-1].item()) for F in widths)
    packed = torch.zeros(max(Qmax, 16), dtype=torch.uint8, device=dev)
    meta = torch.zeros((max(S, 1), 2), device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(wl.seed + 1 + rank)
    ld = [G.ld_for(F) for F in dims]
    ldb = [G.ldb_for(F) for F in dims]
    H = [torch.zeros((n, ld[0]), device=dev)]
    H[0][:, :F0] = torch.randn((n, F0), generator=g, device=dev)
    for l in range(1, L + 1):
        H.append(torch.empty((n, ld[l]), device=dev))
    Mb = [torch.empty((n, ldb[l]), dtype=torch.bfloat16, device=dev) for l in range(L)]
    W = [torch.from_numpy(make_weight_bf16(dims[l], dims[l + 1], wl.seed, l).view(np.int16)).to(dev)
         for l in range(L)]
    dW = [torch.empty((dims[l], dims[l + 1]), device=dev) for l in range(L)]
    # transform-first layers keep Y = bf16(H) W (their Mb holds bf16(H))
    Y = [torch.empty((n, ld[l + 1]), device=dev) if tf[l] else None for l in range(L)]
    # gradients w.r.t. each layer's input; the first layer's is never formed
    dH = [None] + [torch.empty((n, ld[l]), device=dev) for l in range(1, L + 1)]
    dH[L].copy_(torch.randn((n, ld[L]), generator=g, device=dev))
    # workspaces sized for the largest layer
    ws_layer = max(G.gnn_layer_tf_workspace(csr, dims[l], dims[l + 1]) if tf[l] else
                   G.gnn_layer_workspace(csr, dims[l], dims[l + 1]) for l in range(L))
    ws = torch.empty(ws_layer, dtype=torch.uint8, device=dev)
    dense_ws = max(G.gnn_dense_workspace(n, dims[l], dims[l + 1]) for l in range(L))
    wsd = torch.empty(dense_ws, dtype=torch.uint8, device=dev)
    spmm_ws = max(G.gnn_spmm_workspace(csr, F) for F in widths)
    wss = torch.empty(max(spmm_ws, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # per-slot cut counts for the byte model
    slot_cut = (bnd.slot_rowptr[1:] - bnd.slot_rowptr[:-1]).cpu().numpy()
    slot_bits = bnd.slot_bits.cpu().numpy()

    kinds = ["quant", "spmm_fwd", "gemm_fwd", "mask_dM_dW", "halo", "spmm_bwd", "tf_fwd", "tf_bwd"]
    ev = {}

    def rec(key):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        ev.setdefault(key, []).append(e)

    # backward aggregation inputs: one dM per row stride
    dM_by_ld = {}
    for l in range(1, L):
        if ld[l] not in dM_by_ld:
            dM_by_ld[ld[l]] = torch.empty((n, ld[l]), device=dev)

    if gat:
        tpos, spos = G.gnn_gat_index(csr, bnd)
        ga = torch.Generator(device=dev)
        ga.manual_seed(wl.seed + 7)
        a_l = [0.1 * torch.randn(dims[l + 1], generator=ga, device=dev) for l in range(L)]
        a_r = [0.1 * torch.randn(dims[l + 1], generator=ga, device=dev) for l in range(L)]
        alpha = [torch.empty(max(csr.nnz, 1), device=dev) for _ in range(L)]
        da_l = [torch.empty(dims[l + 1], device=dev) for l in range(L)]
        da_r = [torch.empty(dims[l + 1], device=dev) for l in range(L)]
        # each layer's forward messages stay for its backward
        fmsg = [(torch.zeros(max(int(offs[dims[l + 1]][-1].item()), 16), dtype=torch.uint8, device=dev),
                 torch.zeros((max(S, 1), 2), device=dev)) for l in range(L)]
        ws_gat = max(G.gnn_gat_workspace(csr, bnd, dims[l], dims[l + 1]) for l in range(L))
        if ws_gat > ws.numel():
            ws = torch.empty(ws_gat, dtype=torch.uint8, device=dev)

    def tf_fwd(l, Hs):
        F, Fo = dims[l], dims[l + 1]
        if gat:
            G.gnn_gat_layer_fwd(csr, bnd, Hs[l], F, W[l], Fo, a_l[l], a_r[l], l < L - 1, 2 * l,
                                fmsg[l][0], fmsg[l][1], Mb[l], Y[l], alpha[l], Hs[l + 1],
                                slot_off=offs[Fo], ws=ws)
            return
        G.gnn_layer_fwd_tf(csr, bnd, Hs[l], F, W[l], Fo, l < L - 1, 2 * l, packed, meta, Mb[l], Y[l],
                           Hs[l + 1], slot_off=offs[Fo], ws=ws)

    def tf_bwd(l, Hs, dHs):
        F, Fo = dims[l], dims[l + 1]
        if gat:
            G.gnn_gat_layer_bwd(csr, bnd, tpos, spos, dHs[l + 1], Hs[l + 1], l < L - 1, Mb[l], Y[l],
                                alpha[l], fmsg[l][0], fmsg[l][1], W[l], a_l[l], a_r[l], F, Fo,
                                2 * l + 1, packed, meta, dW[l], da_l[l], da_r[l],
                                dHs[l] if l > 0 else None, slot_off=offs[Fo], ws=ws)
            return
        G.gnn_layer_bwd_tf(csr, bnd, dHs[l + 1], Hs[l + 1], l < L - 1, Mb[l], W[l], F, Fo, 2 * l + 1,
                           packed, meta, dW[l], dHs[l] if l > 0 else None, slot_off=offs[Fo], ws=ws)

    # the cluster-blocked layout (dense tiles staged in shared memory), one plan
    # for every width
    bl = G.gnn_blocked_build(csr, bnd, args.blocked, split_len=args.split_len) if args.blocked else None
    blk_ws = None
    if bl is not None:
        blk_ws = torch.empty(max(G._blocked_ws(bl, F, dev, None).numel() for F in widths),
                             dtype=torch.uint8, device=dev)

    # with every layer aggregate-first, each backward aggregation stores the
    # layer below's ReLU-gated bf16 gradient directly (one buffer per width)
    fused = not any(tf)
    dZbuf = {}
    if fused:
        for l in range(1, L):
            if dims[l] not in dZbuf:
                dZbuf[dims[l]] = torch.empty((n, G.ldz_for(dims[l])), dtype=torch.bfloat16, device=dev)

    def run_step(timed, Hs=None, dHs=None):
        Hs = H if Hs is None else Hs
        dHs = dH if dHs is None else dHs
        for l in range(L):
            F, Fo = dims[l], dims[l + 1]
            so = offs[mwid[l]]
            if tf[l]:
                if timed:
                    rec(("tf_fwd", l, 0))
                tf_fwd(l, Hs)
                if timed:
                    rec(("tf_fwd", l, 1))
                continue
            if timed:
                rec(("quant", l, 0))
            G.gnn_quant_pack_owned(bnd, Hs[l], F, 2 * l, packed, meta, slot_off=so)
            if timed:
                rec(("quant", l, 1))
            if bl is not None:
                G.gnn_spmm_fwd_blocked(csr, bnd, bl, Hs[l], F, packed, meta, Mb=Mb[l], slot_off=so,
                                       ws=blk_ws)
            else:
                G.gnn_spmm_fwd(csr, bnd, Hs[l], F, packed, meta, Mb=Mb[l], slot_off=so, ws=wss)
            if timed:
                rec(("spmm_fwd", l, 1))
            G.gnn_dense_fwd(Mb[l], n, F, W[l], Fo, l < L - 1, Hs[l + 1], ws=wsd)
            if timed:
                rec(("gemm_fwd", l, 1))
        dZ_in = None  # the gated bf16 gradient the layer above stored for this layer
        for l in reversed(range(L)):
            F, Fo = dims[l], dims[l + 1]
            so = offs[mwid[l]]
            dMl = dM_by_ld.get(ld[l])
            if tf[l]:
                if timed:
                    rec(("tf_bwd", l, 0))
                tf_bwd(l, Hs, dHs)
                if timed:
                    rec(("tf_bwd", l, 1))
                continue
            if timed:
                rec(("mask_dM_dW", l, 0))
            if dZ_in is not None:
                G.gnn_dense_bwd_z(Mb[l], n, F, W[l], Fo, dZ_in, dMl if l > 0 else None, dW[l], ws=wsd)
            else:
                G.gnn_dense_bwd(Mb[l], n, F, W[l], Fo, dHs[l + 1], Hs[l + 1], l < L - 1,
                                dMl if l > 0 else None, dW[l], ws=wsd)
            if timed:
                rec(("mask_dM_dW", l, 1))
            if l > 0:
                # the backward messages (halo partials, quantised and packed)
                # and the owner-side aggregation are timed apart
                if bl is None:
                    G.gnn_halo_quant_pack(bnd, dMl, F, 2 * l + 1, packed, meta, slot_off=so)
                if timed:
                    rec(("halo", l, 1))
                if fused and bl is not None:
                    dZ_in = dZbuf[F]
                    G.gnn_spmm_bwd_blocked(csr, bnd, bl, dMl, F, 2 * l + 1, packed, meta, H_mask=Hs[l],
                                           dZ=dZ_in, slot_off=so, ws=blk_ws)
                elif fused:
                    dZ_in = dZbuf[F]
                    G.gnn_spmm_bwd_local_masked(csr, bnd, dMl, F, packed, meta, Hs[l], dZ_in,
                                                slot_off=so, ws=wss)
                else:
                    G.gnn_spmm_bwd_local(csr, bnd, dMl, F, packed, meta, dHs[l], slot_off=so, ws=wss)
                if timed:
                    rec(("spmm_bwd", l, 1))


    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(args.warmup):
        run_step(False)
    G.gnn_sync_check()
    torch.cuda.synchronize(dev)

    launches0 = G.gnn_kernel_launches()
    barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        time.sleep(1.5)  # nvidia-smi needs about a second before its first sample
        for _ in range(2):
            run_step(False)
        torch.cuda.synchronize(dev)
        t_start.record(stream)
        for _ in range(args.steps):
            run_step(True)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    launches = G.gnn_kernel_launches() - launches0
    G.gnn_sync_check()
    ms = t_start.elapsed_time(t_end) / args.steps

    # per-kernel times (ms per step)
    per = {k: 0.0 for k in kinds}
    per_layer = {}
    for key, lst in ev.items():
        kind, l, which = key
        if which != 1:
            continue
        start_key = {"quant": ("quant", l, 0), "spmm_fwd": ("quant", l, 1), "gemm_fwd": ("spmm_fwd", l, 1),
                     "mask_dM_dW": ("mask_dM_dW", l, 0), "halo": ("mask_dM_dW", l, 1),
                     "spmm_bwd": ("halo", l, 1),
                     "tf_fwd": ("tf_fwd", l, 0), "tf_bwd": ("tf_bwd", l, 0)}[kind]
        starts = ev[start_key]
        tot = sum(a.elapsed_time(b) for a, b in zip(starts, lst)) / args.steps
        per[kind] += tot
        per_layer[f"{kind}_l{l + 1}"] = tot

    # algorithmic bytes per step: the gather model (every gathered row at
    # every use) and the compulsory bytes (every array once)
    nnz, nc = csr.nnz, bnd.nnz_cut
    byt = {k: 0 for k in kinds}
    comp = {k: 0 for k in kinds}
    launches_k = {k: 0 for k in kinds}
    n_pool = int(torch.unique(bnd.slot_node).numel()) if S else 0
    n_halo_src = int(torch.unique(bnd.slot_col).numel()) if nc else 0
    flops = {"spmm": 0.0, "gemm": 0.0}
    for l in range(L):
        F, Fo = dims[l], dims[l + 1]
        gb = gemm_bytes(n, F, Fo)
        if tf[l]:
            # cast, transform, messages and aggregation at F_out (fp32 out);
            # backward: mask, aggregation at F_out, dense backward
            kb = kernel_bytes(n, nnz, nc, S, Fo, slot_bits, slot_cut, 4 * Fo)
            byt["tf_fwd"] += 6 * n * F + gb["fwd"] + kb["quant"] + kb["fwd"]
            byt["tf_bwd"] += (12 * n * Fo if l < L - 1 else 0) + kb["bwd"] + gb["mask"] + gb["dW"] + \
                (gb["dM"] if l > 0 else 0)
            if gat:
                # scores (read Y), softmax (entry ids, source scores, attention),
                # and in the backward the SDDMM's second gather of the rows plus
                # the per-entry gradients, transposes and score sums
                byt["tf_fwd"] += 4 * n * Fo + 12 * nnz
                byt["tf_bwd"] += 4 * n * Fo + kb["fwd"] + 40 * nnz
            flops["spmm"] += 4.0 * nnz * Fo
            flops["gemm"] += 2.0 * n * F * Fo * (3 if l > 0 else 2)
            continue
        kb = kernel_bytes(n, nnz, nc, S, F, slot_bits, slot_cut, 2 * ldb[l])
        byt["quant"] += kb["quant"]
        byt["spmm_fwd"] += kb["fwd"]
        byt["gemm_fwd"] += gb["fwd"]
        byt["mask_dM_dW"] += gb["mask"] + gb["dW"] + (gb["dM"] if l > 0 else 0)
        flops["spmm"] += 2.0 * nnz * F
        flops["gemm"] += 2.0 * n * F * Fo * (3 if l > 0 else 2)
        cb = compulsory_bytes(n, nnz, nc, S, F, kb["Q"], n_pool, n_halo_src, 2 * ldb[l],
                              4 * F + 2 * G.ldz_for(F) if fused else 4 * F)
        comp["quant"] += cb["quant"]
        comp["spmm_fwd"] += cb["fwd"]
        launches_k["quant"] += 1
        launches_k["spmm_fwd"] += 1
        if l > 0:
            kb4 = kernel_bytes(n, nnz, nc, S, F, slot_bits, slot_cut, 4 * F)
            # fused: the store reads the gate row (4F) in place of writing fp32
            # dH (4F) and writes the bf16 gradient; the layer below skips its mask
            extra = 2 * G.ldz_for(F) * n if fused else 0
            if bl is None:
                byt["halo"] += kb4["halo"]
                byt["spmm_bwd"] += kb4["local"] + extra
                comp["halo"] += cb["halo"]
                comp["spmm_bwd"] += cb["local"]
                launches_k["halo"] += 1
            else:
                byt["spmm_bwd"] += kb4["bwd"] + extra
                comp["spmm_bwd"] += cb["halo"] + cb["local"]
            launches_k["spmm_bwd"] += 1
            flops["spmm"] += 2.0 * nnz * F
        if fused and l < L - 1:
            byt["mask_dM_dW"] -= gb["mask"]
    total_bytes = sum(byt.values())

    # an asynchronous epoch (SYLVIE guide section 10) through the layer API:
    # each layer aggregates with the previous step's messages while this
    # step's are quantised and packed on a second stream.  Same work and byte
    # model as the synchronous step; per layer and direction two message
    # buffers alternate between steps.
    asy = None
    if args.async_steps > 0 and not any(tf):
        aux = torch.cuda.Stream(dev)

        def msgbufs(F):
            Qf = max(int(offs[F][-1].item()), 16)
            return [(torch.zeros(Qf, dtype=torch.uint8, device=dev),
                     torch.zeros((max(S, 1), 2), device=dev)) for _ in range(2)]

        fwd_msgs = [msgbufs(dims[l]) for l in range(L)]
        bwd_msgs = [msgbufs(dims[l]) if l > 0 else None for l in range(L)]

        def async_step(i):
            cur, prev = i % 2, (i + 1) % 2
            for l in range(L):
                F, Fo = dims[l], dims[l + 1]
                (pp, mp), (pn, mn) = fwd_msgs[l][prev], fwd_msgs[l][cur]
                G.gnn_layer_fwd_async(csr, bnd, H[l], F, W[l], Fo, l < L - 1, 2 * l, pp, mp, pn, mn,
                                      Mb[l], H[l + 1], aux, slot_off=offs[F], ws=ws)
            for l in reversed(range(L)):
                F, Fo = dims[l], dims[l + 1]
                if l > 0:
                    (pp, mp), (pn, mn) = bwd_msgs[l][prev], bwd_msgs[l][cur]
                    G.gnn_layer_bwd_async(csr, bnd, dH[l + 1], H[l + 1], l < L - 1, Mb[l], W[l], F, Fo,
                                          2 * l + 1, pp, mp, pn, mn, dW[l], dH[l], aux,
                                          slot_off=offs[F], ws=ws)
                else:
                    G.gnn_dense_bwd(Mb[0], n, F, W[0], Fo, dH[1], H[1], L > 1, None, dW[0], ws=wsd)

        for i in range(args.warmup):
            async_step(i)
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(args.async_steps):
            async_step(i)
        b.record(stream)
        torch.cuda.synchronize(dev)
        G.gnn_sync_check()
        asy = dict(ms=a.elapsed_time(b) / args.async_steps)
        del fwd_msgs, bwd_msgs
        torch.cuda.empty_cache()

    # e2e through the public API with host buffers: every step copies its inputs
    # (layer-1 features, upstream gradient) from pinned host memory and reads
    # the weight gradients back.  The copy of step i+1's inputs runs on a copy
    # stream into the other of two device buffers while step i computes; each
    # step waits for its own inputs (events), so all copies stay inside the
    # timed region.
    e2e = None
    if args.e2e_steps > 0:
        h_in = torch.empty((n, ld[0]), dtype=torch.float32, pin_memory=True)
        h_in.copy_(H[0].cpu())
        g_in = torch.empty((n, ld[L]), dtype=torch.float32, pin_memory=True)
        g_in.copy_(dH[L].cpu())
        dW_host = [torch.empty(dW[l].shape, dtype=torch.float32, pin_memory=True) for l in range(L)]
        # two input buffers: the step's own H[0] / dH[L] and one more
        bufs = [(H[0], dH[L]), (torch.empty_like(H[0]), torch.empty_like(dH[L]))]
        copy_stream = torch.cuda.Stream(dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        used = [torch.cuda.Event() for _ in range(2)]
        for e in used:
            e.record(stream)

        def issue_copy(i):
            k = i % 2
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(used[k])
                bufs[k][0].copy_(h_in, non_blocking=True)
                bufs[k][1].copy_(g_in, non_blocking=True)
                copied[k].record(copy_stream)

        def e2e_step(i, last):
            k = i % 2
            stream.wait_event(copied[k])
            if not last:
                issue_copy(i + 1)
            H0d, dHLd = bufs[k]
            # the same public calls as the timed step, on this step's inputs
            run_step(False, [H0d] + H[1:], dH[:L] + [dHLd])
            used[k].record(stream)
            for l in range(L):
                dW_host[l].copy_(dW[l], non_blocking=True)

        def e2e_run(steps):
            copy_stream.wait_stream(stream)  # copies start after the timing event
            issue_copy(0)
            for i in range(steps):
                e2e_step(i, i == steps - 1)

        e2e_run(max(1, args.warmup))
        torch.cuda.synchronize(dev)
        barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        t_issue = time.perf_counter()
        e2e_run(args.e2e_steps)
        t_issue = time.perf_counter() - t_issue
        b.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = a.elapsed_time(b) / args.e2e_steps
        G.gnn_sync_check()
        h2d = h_in.numel() * 4 + g_in.numel() * 4
        d2h = sum(x.numel() * 4 for x in dW_host)
        e2e = dict(ms=e2e_ms, h2d=h2d, d2h=d2h, issue_ms=1e3 * t_issue / args.e2e_steps,
                   pinned=bool(h_in.is_pinned() and g_in.is_pinned()))

    return dict(ms=ms, per=per, per_layer=per_layer, byt=byt, comp=comp, launches_k=launches_k,
                flops=flops, total_bytes=total_bytes,
                launches=launches, clocks=clk.summary(), e2e=e2e, asy=asy, S=S, nnz=nnz, nnz_cut=nc, n=n,
                Q=int(offs[mwid[0]][-1].item()), n_long=csr.n_long,
                n_pieces=csr.n_pieces, dims=dims, P=P, tf=tf, n_pool=n_pool, n_halo_src=n_halo_src,
                base=base)


# --------------------------------------------------------------- oracle (CPU) arm
class OracleBaseline:
    """The oracle, as it stands, on bounded samples of the workload: its C
    routines (one OpenMP loop over rows or slots, timed on every host core
    and on one) run the first layer's forward messages, forward aggregation,
    backward messages and backward aggregation over a block of slots and a
    block of rows of one partition per sample.  The GCN/mean aggregations use
    the same routines; for attention layers the GCN-weighted aggregation is
    timed (the attention oracle is plain numpy and not sampled).  Rates use
    the GPU arm's gather-model bytes per slot and per row."""

    def __init__(self, workload, aggregator="gcn"):
        import oracle as O
        from oracle import coracle as C
        from synth import make_workload

        self.C = C
        self.aggregator = aggregator
        wl = make_workload(workload)
        self.n = n = wl.n
        flags = O.FLAGS_GCN | (O.FLAG_MEAN if aggregator == "mean" else 0)
        self.rp, col, val = O.csr_build(n, wl.src, wl.dst, flags)
        vt = O.transpose_values(n, self.rp, col, val) if aggregator == "mean" else None
        self.b = b = O.boundary_index(n, self.rp, col, val, wl.P, vt)
        del wl
        nb = O.node_bits(n, self.rp, b, wl_rule(workload)[0], wl_rule(workload)[1],
                         CONFIGS[workload]["base_bits"][0])
        self.sb = nb[b["slot_node"]].astype(np.uint8)
        self.F = F = CONFIGS[workload]["F"]
        self.off = O.slot_offsets(self.sb, F)
        self.S = S = b["n_slots"]
        self.P = wl_P = CONFIGS[workload]["P"]
        self.H = normal_f32(n, F, CONFIGS[workload]["index"] + 0x5EED0001)
        self.Gm = normal_f32(n, F, CONFIGS[workload]["index"] + 0x5EED1001)
        # the message buffers the aggregations read (set up once, untimed)
        self.fp, self.fm = C.quant_pack(self.H, F, b["slot_node"], self.sb, self.off, 0)
        self.hp, self.hm = C.halo_quant_pack(b, self.Gm, F, self.sb, self.off, 1)
        # gather-model bytes of each row's two aggregations and each slot's two
        # message rows (the GPU arm's byte model, split by row and by slot)
        rb = rowbytes(self.sb, F).astype(np.int64)
        slot_cut = np.diff(b["slot_rowptr"])
        self.slot_bytes = (4 + 4 * F + rb + 17) + (8 + slot_cut * (8 + 4 * F) + rb + 8)
        cr = b["col_remap"]
        rem = cr < 0
        ent = np.where(rem, 8 + np.concatenate([rb, [0]])[np.where(rem, ~cr, S)] + 8, 8 + 4 * F)
        ent_local = np.where(rem, 8, 8 + 4 * F)
        own = np.zeros(n, np.int64)
        np.add.at(own, b["slot_node"], rb + 8)
        rows_of = np.repeat(np.arange(n), np.diff(self.rp))
        self.row_bytes = (np.bincount(rows_of, weights=ent + ent_local, minlength=n)
                          + 16 + 8 * F + own)
        del rows_of, ent, ent_local, rem
        self.part = O.partition_starts(n, wl_P)
        self.q = 0
        self.rng = np.random.default_rng(CONFIGS[workload]["index"] + 0x5EED2001)

    def _one(self, budget_s, threads):
        """Samples until budget_s has passed: per sample one partition's block
        of slots and block of rows.  Returns (GB/s, seconds, slots, rows)."""
        C, b, F = self.C, self.b, self.F
        C.set_threads(threads)
        done_b, t_used, slots_done, rows_done = 0.0, 0.0, 0, 0
        k_rows, k_slots = 2048, 4096
        t0 = time.perf_counter()
        while t_used < budget_s:
            q = self.q % self.P
            self.q += 1
            # a seeded random block of the partition's rows (all degrees mixed)
            p0, p1 = int(self.part[q]), int(self.part[q + 1])
            rows = np.sort(self.rng.choice(p1 - p0, min(k_rows, p1 - p0), replace=False)) + p0
            # a block of the partition's slots from a seeded random start
            a0, a1 = int(b["send_start"][q]), int(b["send_start"][q + 1])
            s0 = a0 + int(self.rng.integers(0, max(1, a1 - a0 - k_slots + 1)))
            s1 = min(a1, s0 + k_slots)
            if s1 > s0:
                C.quant_pack(self.H, F, b["slot_node"][s0:s1], self.sb[s0:s1],
                             self.off[s0:s1 + 1] - self.off[s0], 0, key0=s0)
                C.halo_quant_pack(b, self.Gm, F, self.sb, self.off, 1, s0, s1)
            C.spmm_fwd_rows(self.rp, b, self.H, F, self.fp, self.fm, self.sb, self.off, rows)
            C.spmm_bwd_rows(self.rp, b, self.Gm, F, self.hp, self.hm, self.sb, self.off, rows)
            slots_done += s1 - s0
            rows_done += rows.size
            done_b += float(self.slot_bytes[s0:s1].sum()) + float(self.row_bytes[rows].sum())
            t_used = time.perf_counter() - t0
            k_rows, k_slots = min(k_rows * 2, 1 << 16), min(k_slots * 2, 1 << 17)
        return done_b / t_used / 1e9, t_used, slots_done, rows_done

    def sample(self, budget_s, single_thread_share=0.3):
        """All host cores for (1 - share) of the budget, one core for the rest."""
        C = self.C
        cores = C.max_threads()
        gbs, secs, ns, nr = self._one(budget_s * (1 - single_thread_share), cores)
        gbs1, secs1, ns1, nr1 = self._one(budget_s * single_thread_share, 1)
        C.set_threads(cores)
        what = ("GCN-weighted aggregation; the attention oracle is not sampled"
                if self.aggregator == "gat" else "forward and backward messages and aggregations")
        return dict(value=gbs, unit=UNIT, cores=cores, kind="oracle",
                    sample=f"{ns} of {self.S} slots and {nr} of {self.n} rows ({what}, F={self.F}), "
                           f"{secs:.1f} s on {cores} threads (the oracle's C routines, OpenMP)",
                    single_thread={"value": gbs1, "unit": UNIT, "cores": 1, "seconds": secs1,
                                   "sample": f"{ns1} slots and {nr1} rows"},
                    seconds=secs)


def normal_f32(n, F, seed, chunk=1 << 18):
    """fp32 N(0,1) [n, F], drawn in row chunks by independent seeded streams
    on several threads (numpy releases the GIL while it fills)."""
    import concurrent.futures as cf

    out = np.empty((n, F), np.float32)
    starts = list(range(0, n, chunk))
    seqs = np.random.SeedSequence(seed).spawn(len(starts))

    def fill(i):
        r0 = starts[i]
        np.random.default_rng(seqs[i]).standard_normal(out=out[r0:r0 + chunk], dtype=np.float32)

    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        list(ex.map(fill, range(len(starts))))
    return out


def wl_rule(workload):
    r = CONFIGS[workload]["rule"]
    return r["pct"], r["bits"]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="scale", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--order", default="af", choices=["af", "tf", "auto"],
                    help="aggregate first (the message is H), transform first where F_out < F_in "
                         "(the message is H W), or per layer where it gathers fewer bytes")
    ap.add_argument("--blocked", type=int, default=0,
                    help="aggregate through the cluster-blocked layout, tiles with at least this "
                         "many entries staged in shared memory (0: off; GCN weights only)")
    ap.add_argument("--aggregator", default="gcn", choices=["gcn", "mean", "gat"],
                    help="GCN weights 1/sqrt(d_v d_u), GraphSAGE mean weights 1/d_v, or one-head "
                         "graph attention on the transformed rows")
    ap.add_argument("--split-len", type=int, default=128)
    ap.add_argument("--base-bits", type=int, default=0,
                    help="epoch base width (1, 2, 4, 8); default: the workload's first")
    ap.add_argument("--long-slot-len", type=int, default=128)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--async-steps", type=int, default=10,
                    help="also time asynchronous-epoch steps (0: skip)")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "gpu" else "gloo")
        if args.impl == "gpu":
            import torch
            torch.cuda.set_device(local_rank)

    config = {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload,
              "aggregator": args.aggregator, "order": args.order, "blocked": args.blocked or None,
              "base_bits": args.base_bits or CONFIGS[args.workload]["base_bits"][0],
              "timing": "inputs larger than L2 (no flush); CUDA events on the launching stream",
              "parallelism": f"replicas x{world}"}

    if args.impl == "reference":
        if rank == 0:
            ob = OracleBaseline(args.workload, args.aggregator)
            per_step = max(1.0, args.cpu_budget / max(1, args.steps))
            for _ in range(args.warmup):
                ob.sample(0.2)
            steps = []
            cb = None
            for _ in range(args.steps):
                cb = ob.sample(per_step)
                steps.append(cb["value"])
            val = float(statistics.median(steps))
            line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world,
                    "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                    "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                    "config": config,
                    "cpu_baseline": {"value": val, "unit": UNIT, "cores": cb["cores"], "kind": "oracle",
                                     "sample": cb["sample"], "single_thread": cb["single_thread"]},
                    "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
            print(json.dumps(line), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    r = run_gpu(args, rank, world, local_rank)
    ms = max_over_ranks(r["ms"], world, "cuda")
    hbm, bf16, bf16_sus, peak_src = load_peaks()
    gbs = whole_job_rate(r["total_bytes"], world, ms)
    per = r["per"]

    def rate(k):
        return r["byt"][k] / (per[k] * 1e-3) / 1e9 if per[k] > 0 else None

    spmm_ms = per["spmm_fwd"] + per["halo"] + per["spmm_bwd"]
    gemm_ms = per["gemm_fwd"] + per["mask_dM_dW"]
    names = {"quant": "quant_pack_owned_kernel / quant_pack_kernel (gnn_quant_pack_owned: forward messages)",
             "spmm_fwd": "spmm_rows_kernel (gnn_spmm_fwd: aggregation with in-gather dequantisation)",
             "halo": "halo_quant_pack_kernel (gnn_halo_quant_pack: backward halo partials, "
                     "quantised and packed)",
             "spmm_bwd": "spmm_rows_kernel (gnn_spmm_bwd_local_masked: local transpose aggregation, "
                         "owned messages, ReLU gate)"}
    agg = [k for k in names if r["launches_k"][k] > 0 and per[k] > 0]
    traffic_tab = (committed_traffic(args.workload, r["base"]) if default_variant(args) else {})

    def kstats(k):
        t = per[k] * 1e-3  # s per step
        nl = r["launches_k"][k]
        d = {"ms_per_step": per[k], "launches_per_step": nl,
             "gather_model_GBs": r["byt"][k] / t / 1e9,
             "compulsory_GBs": r["comp"][k] / t / 1e9,
             "compulsory_frac_of_hbm": r["comp"][k] / t / 1e9 / hbm}
        tr = traffic_tab.get(k)
        if tr is not None:
            d["dram_GBs"] = tr * nl / t / 1e9
            d["dram_frac_of_hbm"] = d["dram_GBs"] / hbm
        return d

    kstat = {k: kstats(k) for k in agg}
    # dominant kernel: the aggregation-path kernel with the most time per step
    dom = max(agg, key=lambda k: per[k]) if agg else None
    roof = None
    if dom is not None:
        st = kstat[dom]
        nl = r["launches_k"][dom]
        t_launch = per[dom] / nl * 1e-3
        traffic = traffic_tab.get(dom)
        comp_launch = r["comp"][dom] / nl
        if traffic is not None:
            achieved, basis = traffic / t_launch / 1e9, "dram bytes (ncu, same kernel source and workload)"
        else:
            achieved, basis = comp_launch / t_launch / 1e9, "compulsory bytes (every array once)"
        roof = {"kernel": names[dom], "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic, "basis": basis,
                "launch_ms": t_launch * 1e3, "launches_per_step": nl,
                "compulsory": {"bytes_per_launch": comp_launch, "GBs": comp_launch / t_launch / 1e9,
                               "frac": comp_launch / t_launch / 1e9 / hbm},
                "gather_model": {"bytes_per_launch": r["byt"][dom] / nl, "GBs": st["gather_model_GBs"],
                                 "note": "every gathered row counted at every use; L2 serves the "
                                         "repeats, so this is not an HBM figure"},
                "peak_source": peak_src + " (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                else peak_src}
    line = {
        "metric": METRIC, "value": gbs, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp32 aggregation, bf16 transform, 1-8 bit messages",
        "data": "synthetic (seeded generator; no dataset)",
        "config": config,
        "value_basis": "gather-model bytes of every kernel of the step / step time",
        "kernels": {
            "spmm_GFLOPs": r["flops"]["spmm"] / (spmm_ms * 1e-3) / 1e9 if spmm_ms else None,
            "gemm_TFLOPs": r["flops"]["gemm"] / (gemm_ms * 1e-3) / 1e12 if gemm_ms else None,
            "ms": per, "ms_per_layer": r["per_layer"], "transform_first_layers": r["tf"],
            **kstat,
        },
        "graph": {"n": r["n"], "nnz": r["nnz"], "nnz_cut": r["nnz_cut"], "slots": r["S"],
                  "packed_bytes_layer1": r["Q"], "meta_bytes_layer1": 8 * r["S"],
                  "message_nodes": r["n_pool"], "halo_source_rows": r["n_halo_src"],
                  "long_rows": r["n_long"], "pieces": r["n_pieces"],
                  "dims": r["dims"], "P": r["P"]},
        "roofline": roof,
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if r["e2e"]:
        e = r["e2e"]
        e_ms = max_over_ranks(e["ms"], world, "cuda")
        line["e2e"] = {"value": whole_job_rate(r["total_bytes"], world, e_ms), "unit": UNIT,
                       "ms_per_step": e_ms, "h2d_bytes_per_step": e["h2d"],
                       "d2h_bytes_per_step": e["d2h"],
                       "host_issue_ms_per_step": e["issue_ms"], "pinned_inputs": e["pinned"]}
    if r["asy"]:
        a_ms = max_over_ranks(r["asy"]["ms"], world, "cuda")
        line["async_epoch"] = {"value": whole_job_rate(r["total_bytes"], world, a_ms), "unit": UNIT,
                               "ms_per_step": a_ms,
                               "what": "remote sources read the previous step's messages; this "
                                       "step's are packed on a second stream meanwhile"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = OracleBaseline(args.workload, args.aggregator).sample(args.cpu_budget)
        line["cpu_baseline"] = {k: cb[k] for k in ["value", "unit", "cores", "kind", "sample",
                                                    "single_thread"]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
