"""Benchmark of the sparse-convolution hot path on one or more GPUs.

Default workload (one JSON line): the training step of a 64 -> 64 bf16
submanifold layer on four 192^3 surface shells (498,145 voxels, batch index in
coordinate column 0).  One step = one pass of its hot path:
spc_build_indice_map (validate + key + hash build + probe of all 27 offsets),
spc_conv_fwd, spc_conv_dgrad (dinput through the mirrored map) and
spc_conv_wgrad (dfilter, fp32).  The headline value is conv TFLOP/s over
active pairs (2 * P * Cin * Cout per conv pass, three passes) over the whole
step time; the indice-map rate (Mvoxel/s) and per-phase times are reported
beside it.  Other workloads (--workload) cover the remaining rows of the
path: the LiDAR-like scene (batch 2, 41 x 1600 x 1408, fp16 16 -> 16), the
strided k3 s2 p1 conv (output coordinates + maps + forward), the 256^3 shell
at 128 -> 128 (k3 and k1), and the inverse conv, fused residual block and max
pool built on the same maps.

Timing: every phase is captured once as a CUDA graph (the C ABI allocates
nothing and only enqueues on the current stream) and replayed; CUDA events on
the launching stream bracket each phase.  Inputs are resident in HBM when the
timed region starts and L2 is flushed (256 MiB write) between timed steps,
outside the events.  `e2e` times the calls a user makes through the C ABI from
pinned host buffers, with the host->device copies of the inputs and the
device->host copies of the outputs inside the timed region.

--impl reference times the CPU oracle (the slow fp64 restatement of the
method the tests check against) on the host cores, on a bounded sample.

Multi-GPU: one process per GPU (torchrun); every rank runs its own replica of
the workload (voxels of different scenes never interact, so the path shards by
scene with no data exchange); value = work of all ranks / max time over ranks.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import scenes  # noqa: E402

METRIC = "SubM3d conv TFLOP/s over active pairs (and % roofline); indice-map Mvoxel/s"
DEFAULT_WORKLOAD = "shell192x4_train_bf16"
L2_FLUSH_BYTES = 256 << 20
SHAPES = {"uniform32": (32, 32, 32), "lidar": (41, 1600, 1408), "shell256": (256, 256, 256),
          "shell192x4": (192, 192, 192)}
DESCRIPTIONS = {
    "lidar_subm_f16": "SubMConv3d k3 indice build + forward, batch 2, 41x1600x1408 grid, "
                      "120000 voxels, fp16 16->16, no bias",
    "uniform32_subm_f32": "SubMConv3d k3 indice build + forward, 2000 voxels of 32^3, fp32 16->16, bias",
    "uniform32_strided_bf16": "SparseConv3d k3 s2 p1 output coords + maps + forward, 2000 voxels "
                              "of 32^3, bf16 64->128",
    "shell256_subm_bf16": "SubMConv3d k3 indice build + forward, 256^3 shell, bf16 128->128",
    "shell256_k1_bf16": "SubMConv3d k1 forward (per-voxel GEMM), 256^3 shell, bf16 128->128",
    "shell192x4_train_bf16": "SubMConv3d k3 indice build + forward + dinput + dfilter, "
                             "4 x 192^3 shells, bf16 64->64",
    "shell192x4_resblock_bf16": "SubMConv3d k3 indice build + forward with fused residual add + "
                                "ReLU (relu(conv(x) + x)), 4 x 192^3 shells, bf16 64->64",
    "shell256_maxpool_bf16": "SparseMaxPool3d k2 s2 forward (with argmax) + input gradient "
                             "(maps built once), 256^3 shell, bf16 128 channels",
    "shell256_inverse_bf16": "SparseInverseConv3d of a k3 s2 p1 conv (maps and row order "
                             "built once), 256^3 shell, bf16 128->128",
    "shell256_int8": "quantized SubMConv3d k3 indice build + int8 forward (per-channel scale and "
                     "bias, ReLU, int8 out), 256^3 shell, int8 128->128",
}
ELEM = {"f32": 4, "f16": 2, "bf16": 2, "i8": 1}
ROW_ORDER = [False]  # --row-order on: wide-channel submanifold tiles in mask-grouped row order
COORD_ORDER = ["scene"]  # --coord-order: the order the voxel rows are stored in


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # raw samples; the JSON line carries their summary
        self.path = os.path.join(os.environ.get("SPC_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"spc_clocks_gpu{gpu_index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return None
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = max(smax, float(parts[2]))
                except ValueError:
                    continue
                for name, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(name)
        except OSError:
            return None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return rank, world, local, dist
    return 0, 1, 0, None


def reduce_max(v: float, dist, device) -> float:
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


class Phase:
    def __init__(self, name, fn, kind, bytes_alg, flops=0.0, kernels="", launches=1):
        self.name, self.fn, self.kind = name, fn, kind
        self.bytes_alg, self.flops, self.kernels = float(bytes_alg), float(flops), kernels
        self.launches = launches  # kernels of libspc launched by one call of the phase
        self.graph = None
        self.ms = []


class Case:
    """Device inputs, preallocated outputs and the timed phases of one workload."""

    def __init__(self, name: str, dev):
        import sparse_convolution_hash_gb300 as spc
        from sparse_convolution_hash_gb300 import binding as B

        self.spc, self.B, self.dev = spc, B, dev
        w = scenes.workload(name)
        self.shape = SHAPES[name.split("_")[0]]
        if COORD_ORDER[0] != "scene" and w["subm"] and w["k"] > 1:
            w = self.reorder_rows(w, COORD_ORDER[0])
        self.w, self.name = w, name
        c = w["coords"]
        self.batch = int(c[:, 0].max()) + 1 if c.shape[0] else 1
        self.n = n = c.shape[0]
        self.cin, self.cout, self.ks = w["cin"], w["cout"], w["k"]
        self.K = K = self.ks ** 3
        self.s = s = ELEM[w["dtype"]]
        self.dtype = w["dtype"]
        self.coords_h = torch.from_numpy(c)
        self.coords = self.coords_h.to(dev)
        self.x = w["x"].to(dev)
        self.wt = w["w"].to(dev)
        self.bias = w["bias"].to(dev) if w["bias"] is not None else None
        self.status = B.new_status(dev)
        self.prec = B.SPC_PREC_EXACT
        self.phases = []
        self.host_out = []
        cin, cout = self.cin, self.cout

        if w["subm"]:
            self.n_out = n
            if self.ks > 1:
                self.m = spc.spc_build_indice_map(self.coords, self.batch, self.shape, ksize=self.ks,
                                                  subm=True, status=self.status)
                imap, mask = self.m["imap"], self.m["mask"]
                torch.cuda.synchronize()
                B.check_status(self.status, "setup build")
                self.pairs = int(self.m["pair_count"].sum().item())
                # wide channels: the build also groups the rows by offset mask (one
                # row order serves the forward, the dinput and the int8 forward)
                self.grouped = ROW_ORDER[0] and cin >= 64 and cout >= 64
                if self.grouped:
                    nro = int(B.lib().spc_map_row_order_workspace_size(n))
                    self.ro_ws = torch.empty(max(nro, 256), dtype=torch.uint8, device=dev)
                    self.perm = torch.empty(n, dtype=torch.int32, device=dev)

                def build():
                    spc.spc_build_indice_map(self.coords, self.batch, self.shape, ksize=self.ks,
                                             subm=True, out=self.m)
                    if self.grouped:
                        spc.spc_map_row_order(None, ws=self.ro_ws, mask=self.m["mask"], K=K,
                                              perm=self.perm)

                build()
                torch.cuda.synchronize()
                passes = (K + 7) // 8
                self.phases.append(Phase(
                    "build", build, "build", 16 * n + 4 * K * n + 4 * n + 4 * K + (4 * n if self.grouped else 0),
                    kernels="k_build_init, k_hash_insert, k_map_probe" + (
                        ", row order: k_row_keys_from_mask, k_radix_hist/k_scan_exclusive/k_radix_scatter "
                        f"x{passes}, k_perm_from_keys" if self.grouped else ""),
                    launches=3 + (2 + 3 * passes if self.grouped else 0)))
            else:
                self.m = None
                imap = mask = None
                self.pairs = n
                self.grouped = False
        else:
            self.grouped = False
            st, pd = w["stride"], w["pad"]
            g = B.make_geom(self.ks, st, pd, 1)
            cap = n * K
            self.oc_buf = torch.empty((cap, 4), dtype=torch.int32, device=dev)
            self.n_out_dev = torch.zeros(1, dtype=torch.int64, device=dev)
            nb = int(B.lib().spc_strided_out_coords_workspace_size(n, ctypes.byref(g)))
            self.oc_ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
            self.out_shape = (ctypes.c_int32 * 3)()
            self.geom = g

            def outcoords():
                code = B.lib().spc_strided_out_coords(
                    self.coords.data_ptr(), n, self.batch, (ctypes.c_int32 * 3)(*self.shape),
                    ctypes.byref(self.geom), self.out_shape, self.oc_buf.data_ptr(), cap,
                    self.n_out_dev.data_ptr(), self.status.data_ptr(), self.oc_ws.data_ptr(),
                    self.oc_ws.numel(), torch.cuda.current_stream(dev).cuda_stream)
                assert code == 0, code

            outcoords()
            torch.cuda.synchronize()
            B.check_status(self.status, "setup out coords")
            self.n_out = n_out = int(self.n_out_dev.item())
            self.oc = self.oc_buf[:n_out]
            self.m = spc.spc_build_indice_map(self.coords, self.batch, self.shape, ksize=self.ks,
                                              stride=st, pad=pd, subm=False, out_coords=self.oc,
                                              with_transpose=True, status=self.status)
            torch.cuda.synchronize()
            B.check_status(self.status, "setup strided build")
            self.pairs = int(self.m["pair_count"].sum().item())
            imap, mask = self.m["imap"], self.m["mask"]
            cells = self.batch * int(np.prod(list(self.out_shape)))
            passes = (max(1, int(np.ceil(np.log2(max(cells, 2))))) + 7) // 8
            # the library takes the bitmap path when the output grid's bitmap fits
            # the candidates' key space (one bit per cell vs 16 bytes per candidate)
            bitmap = (cells + 31) // 32 <= 2 * n * K
            if not w.get("inverse"):
                self.phases.append(Phase(
                    "outcoords", outcoords, "build", 16 * n + 16 * n_out + 8,
                    kernels=("k_bm_mark, k_bm_count, k_scan_exclusive, k_bm_write (bitmap)" if bitmap
                             else "k_candidates, k_radix_*, k_unique_*"),
                    launches=4 if bitmap else 1 + 3 * passes + 3))
                self.phases.append(Phase(
                    "build", lambda: spc.spc_build_indice_map(
                        self.coords, self.batch, self.shape, ksize=self.ks, stride=st, pad=pd,
                        subm=False, out_coords=self.oc, with_transpose=True, out=self.m),
                    "build", 16 * n + 16 * n_out + 4 * K * n_out + 4 * K * n + 4 * n_out + 4 * K,
                    kernels="k_build_init, k_hash_insert, k_map_probe<imap_t>", launches=3))
        n_out, P = self.n_out, self.pairs
        self.imap, self.mask = imap, mask
        if w.get("int8"):
            # quantized layer: int8 codes in and out, exact integer sums on the
            # fp16 tensor cores (weights widened, or split into 4-bit halves, per call)
            self.inverse = self.maxpool = self.train = False
            self.int8 = True
            self.scale, self.qbias = w["scale"].to(dev), w["bias"].to(dev)
            self.bias = None
            self.y = torch.empty((n_out, cout), dtype=torch.int8, device=dev)
            nbw = int(B.lib().spc_conv_int8_workspace_size(K, cin, cout))
            self.conv_ws = torch.empty(max(nbw, 256), dtype=torch.uint8, device=dev)
            self.phases.append(Phase(
                "fwd", lambda: spc.spc_conv_fwd_int8(self.x, self.wt, self.scale, self.qbias,
                                                     self.imap, self.mask, perm=self.perm_or_none(),
                                                     act=B.SPC_ACT_RELU, out=self.y,
                                                     status=self.status, ws=self.conv_ws),
                "conv", n * cin + n_out * cout + K * cin * cout + 4 * P + 8 * cout,
                2.0 * P * cin * cout, kernels="k_i8_prep_w + k_conv_i8 (tcgen05 on exact fp16 values)",
                launches=2))
            self.phases[-1].fp16_per_int8 = int8_fp16_products(K, cin, cout)
            return
        self.int8 = False
        if w.get("maxpool"):
            # pooling on the strided map of its window: forward with argmax, then
            # the input gradient through the transposed map
            self.inverse = False
            self.maxpool = True
            self.train = False
            self.y = torch.empty((n_out, cin), dtype=self.x.dtype, device=dev)
            self.arg = torch.empty((n_out, cin), dtype=torch.uint8, device=dev)
            self.dyp = scenes.normal((n_out, cin), 1.0, self.dtype, w["seed"], 6).to(dev)
            self.dxp = torch.empty((n, cin), dtype=self.x.dtype, device=dev)
            self.phases.append(Phase(
                "pool", lambda: spc.spc_maxpool_fwd(self.x, self.imap, self.mask, out=self.y,
                                                    arg=self.arg),
                "conv", s * n * cin + s * n_out * cin + n_out * cin + 4 * P + 4 * n_out,
                float(P * cin), kernels="k_maxpool_fwd"))
            self.phases.append(Phase(
                "pool_dgrad", lambda: spc.spc_maxpool_dgrad(self.dyp, self.m["imap_t"], self.arg,
                                                            out=self.dxp),
                "conv", s * n_out * cin + n_out * cin + 4 * K * n + s * n * cin, float(P * cin),
                kernels="k_maxpool_dgrad"))
            return
        self.maxpool = False
        if w.get("inverse"):
            # the inverse conv runs on the strided conv's maps: its inputs are
            # features on the output set, its outputs rows of the input set
            self.inverse = True
            self.yin = w["y_for"](n_out).to(dev)
            self.y = torch.empty((n, cout), dtype=self.x.dtype, device=dev)
            nbw = int(B.lib().spc_conv_workspace_size(K, n_out, n, cin, cout, B._DTYPES[self.x.dtype]))
            self.conv_ws = torch.empty(max(nbw, 256), dtype=torch.uint8, device=dev)
            self.train = False
            # rows grouped by offset mask, saved with the maps (spc_map_row_order)
            self.mask_t, self.perm = spc.spc_map_row_order(self.m["imap_t"])
            self.phases.append(Phase(
                "inverse", lambda: spc.spc_conv_inverse(self.yin, self.wt, self.bias, self.m["imap_t"],
                                                        precision=self.prec, out=self.y,
                                                        status=self.status, ws=self.conv_ws,
                                                        mask_t=self.mask_t, perm=self.perm),
                "conv", s * n_out * cin + s * n * cout + s * K * cin * cout + 4 * P,
                2.0 * P * cin * cout, kernels=self.fwd_kernel(),
                launches=2 if "k_transpose_w" in self.fwd_kernel() else 1))
            return
        self.inverse = False
        self.y = torch.empty((n_out, cout), dtype=self.x.dtype, device=dev)
        nbw = int(B.lib().spc_conv_workspace_size(K, n, n_out, cin, cout, B._DTYPES[self.x.dtype]))
        self.conv_ws = torch.empty(max(nbw, 256), dtype=torch.uint8, device=dev)
        flops = 2.0 * P * cin * cout
        bias_b = s * cout if self.bias is not None else 0
        if w.get("resblock"):
            # residual block tail: the identity is the block input itself
            self.phases.append(Phase(
                "fwd", lambda: spc.spc_conv_fwd_fused(
                    self.x, self.wt, self.bias, self.imap, self.mask, residual=self.x,
                    add_scale=1.0, act=B.SPC_ACT_RELU, n_out=n_out, precision=self.prec,
                    out=self.y, status=self.status, ws=self.conv_ws, perm=self.perm_or_none()),
                "conv", s * n * cin + 2 * s * n_out * cout + s * K * cin * cout + 4 * P + bias_b,
                flops, kernels=self.fwd_kernel() + ", fused residual + ReLU epilogue",
                launches=2 if "k_transpose_w" in self.fwd_kernel() else 1))
        else:
            self.phases.append(Phase(
                "fwd", lambda: spc.spc_conv_fwd(self.x, self.wt, self.bias, self.imap, self.mask,
                                                n_out=n_out, precision=self.prec, out=self.y,
                                                status=self.status, ws=self.conv_ws,
                                                perm=self.perm_or_none()),
                "conv", s * n * cin + s * n_out * cout + s * K * cin * cout + 4 * P + bias_b, flops,
                kernels=self.fwd_kernel(), launches=2 if "k_transpose_w" in self.fwd_kernel() else 1))
        self.train = bool(w.get("train"))
        if self.train:
            self.dy = w["dy"].to(dev)
            self.dx = torch.empty((n, cin), dtype=self.x.dtype, device=dev)
            self.dw = torch.empty((K, cin, cout), dtype=torch.float32, device=dev)
            nbg = int(B.lib().spc_conv_wgrad_workspace_size(K, n, n_out, cin, cout,
                                                            B._DTYPES[self.x.dtype]))
            self.wg_ws = torch.empty(max(nbg, 256), dtype=torch.uint8, device=dev)
            self.phases.append(Phase(
                "dgrad", lambda: spc.spc_conv_dgrad(self.dy, self.wt, self.imap,
                                                    B.SPC_MAP_SUBM_MIRROR, n, mask=self.mask,
                                                    out=self.dx, status=self.status,
                                                    perm=self.perm_or_none()),
                "conv", s * n_out * cout + s * n * cin + s * K * cin * cout + 4 * P, flops,
                kernels=self.fwd_kernel(dgrad=True)))
            self.phases.append(Phase(
                "wgrad", lambda: spc.spc_conv_wgrad(self.x, self.dy, self.imap, K, out=self.dw,
                                                    ws=self.wg_ws),
                "conv", s * n * cin + s * n_out * cout + 4 * P + 4 * K * cin * cout, flops,
                kernels=("k_wgrad_tc (tcgen05), k_wgrad_reduce"
                         if self.dtype in ("f16", "bf16") and cin % 64 == 0 and cout % 64 == 0
                         else "k_wgrad_partial, k_wgrad_reduce"), launches=2))

    def reorder_rows(self, w, order):
        """The workload with its voxel rows (coordinates and per-row tensors)
        stored in another order: 'mask' groups rows by their submanifold offset
        mask (from the library's own map of the scene), 'shuffled' is a seeded
        random order.  A data layout; every phase still does all its work."""
        c = w["coords"]
        n = c.shape[0]
        batch = int(c[:, 0].max()) + 1
        if order == "mask":
            m = self.spc.spc_build_indice_map(torch.from_numpy(c).to(self.dev), batch, self.shape,
                                              ksize=w["k"])
            self.B.check_status(m["status"], "layout map")
            K = w["k"] ** 3
            mask = m["mask"].cpu().numpy().astype(np.int64) & ((1 << K) - 1)
            perm = np.argsort(mask, kind="stable")
        else:
            perm = scenes.rng(w["seed"], 99).permutation(n)
        w = dict(w)
        w["coords"] = np.ascontiguousarray(c[perm])
        tp = torch.from_numpy(perm)
        for key in ("x", "dy"):
            if key in w:
                w[key] = w[key][tp].contiguous()
        return w

    def perm_or_none(self):
        return self.perm if getattr(self, "grouped", False) else None

    def fwd_kernel(self, dgrad=False):
        """Kernels one forward (or dinput) call launches, following the library's
        dispatch: the CUDA-core narrow kernel when both widths are 8, 16 or 32,
        tcgen05 for 16-bit rows of 16, 32 or a multiple of 64 channels (and
        tf32), else the general CUDA-core gather kernel."""
        cred, co = (self.cout, self.cin) if dgrad else (self.cin, self.cout)
        if cred in (8, 16, 32) and co in (8, 16, 32) and (cred, co) not in ((8, 32), (32, 8)):
            return "k_conv_narrow"
        half = self.dtype in ("f16", "bf16")
        tc = self.K <= 32 and (
            (half and cred % 64 == 0 and co % 64 == 0) or
            (half and cred in (16, 32) and (co in (16, 32) or co % 64 == 0)) or
            (self.dtype == "f32" and self.prec == self.B.SPC_PREC_TF32 and cred % 32 == 0 and co % 64 == 0))
        if tc:
            as_stored = half and cred % 64 == 0 and co % 64 == 0  # W read as stored
            dense = self.K == 1 and half and cred % 64 == 0 and co % 64 == 0
            return ("k_conv_tc (tcgen05" + (", dense TMA rows" if dense else "") + ")" +
                    ("" if dgrad or as_stored else " + k_transpose_w"))
        return "k_gather_gemm_simt"

    def conv_flops(self):
        return sum(p.flops for p in self.phases)

    def capture(self):
        for p in self.phases:
            p.fn()
        torch.cuda.synchronize()
        self.B.check_status(self.status, "pre-capture")
        for p in self.phases:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                p.fn()
            p.graph = g

    def replay_all(self):
        for p in self.phases:
            p.graph.replay()

    # -- end to end through the C ABI from pinned host memory
    def setup_e2e(self):
        """End-to-end step: a step's inputs sit in one pinned host buffer and are
        copied to the device in one transfer, its results come back in one; the
        device tensors the phases use become views into those buffers."""
        if self.maxpool:
            ins = [("x", self.w["x"]), ("dyp", self.dyp.cpu())]
            outs = ["y", "dxp"]
        elif self.inverse:
            # the maps are saved from the strided conv: a step moves features and weights
            ins = [("yin", self.yin.cpu()), ("wt", self.w["w"])]
            outs = ["y"]
        elif self.int8:
            ins = [("coords", self.coords_h), ("x", self.w["x"]), ("wt", self.w["w"]),
                   ("scale", self.w["scale"]), ("qbias", self.w["bias"])]
            outs = ["y"]
        else:
            ins = [("coords", self.coords_h), ("x", self.w["x"]), ("wt", self.w["w"])]
            if self.bias is not None:
                ins.append(("bias", self.w["bias"]))
            if self.train:
                ins.append(("dy", self.w["dy"]))
            outs = ["y"] + (["dx", "dw"] if self.train else [])

        def layout(tensors):
            offs, off = [], 0
            for t in tensors:
                offs.append(off)
                off = (off + t.numel() * t.element_size() + 255) // 256 * 256
            return offs, off

        hs = [h.contiguous() for _, h in ins]
        ds = [getattr(self, name) for name in outs]
        in_offs, in_total = layout(hs)
        out_offs, out_total = layout(ds)
        self.in_host = torch.empty(in_total, dtype=torch.uint8).pin_memory()
        for h, o in zip(hs, in_offs):
            self.in_host[o:o + h.numel() * h.element_size()].copy_(h.view(-1).view(torch.uint8))
        # two device copies of the inputs and outputs, so that one step's copies
        # overlap the neighbouring step's kernels
        self.in_dev = [torch.empty(in_total, dtype=torch.uint8, device=self.dev) for _ in range(2)]
        self.out_dev = [torch.empty(out_total, dtype=torch.uint8, device=self.dev) for _ in range(2)]
        self.out_host = [torch.empty(out_total, dtype=torch.uint8).pin_memory() for _ in range(2)]
        self.views = []
        for b in range(2):
            v = {}
            for (name, _), h, o in zip(ins, hs, in_offs):
                nb = h.numel() * h.element_size()
                v[name] = self.in_dev[b][o:o + nb].view(h.dtype).view(h.shape)
            for name, d, o in zip(outs, ds, out_offs):
                nb = d.numel() * d.element_size()
                v[name] = self.out_dev[b][o:o + nb].view(d.dtype).view(d.shape)
            self.views.append(v)
        # one stream per copy direction (the two directions use separate copy engines)
        self.up_stream = torch.cuda.Stream(self.dev)
        self.down_stream = torch.cuda.Stream(self.dev)
        self.h2d = in_total
        self.d2h = out_total

    def e2e_run(self, steps: int, stream):
        """`steps` end-to-end steps ordered after `stream`'s current point and
        before its next: per step one host->device copy of the inputs, the
        phases, one device->host copy of the results.  The copies run on two copy
        streams, double-buffered: step i + 1's inputs and step i - 1's results
        move while step i's kernels run.  Two events of each kind are reused
        (an event is recorded again only after its last wait was enqueued)."""
        cs, ds = self.up_stream, self.down_stream
        if not hasattr(self, "_ev"):
            self._ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("start", "h2d", "comp", "d2h")}
        h2d, comp, d2h = self._ev["h2d"], self._ev["comp"], self._ev["d2h"]
        self._ev["start"][0].record(stream)
        cs.wait_event(self._ev["start"][0])
        ds.wait_event(self._ev["start"][0])

        def upload(i):
            with torch.cuda.stream(cs):
                if i >= 2:
                    cs.wait_event(comp[i % 2])  # step i - 2, its buffer's last reader
                self.in_dev[i % 2].copy_(self.in_host, non_blocking=True)
                h2d[i % 2].record(cs)

        upload(0)
        for i in range(steps):
            b = i % 2
            if i + 1 < steps:
                upload(i + 1)
            stream.wait_event(h2d[b])
            if i >= 2:
                stream.wait_event(d2h[b])  # step i - 2's results have been read back
            for name, t in self.views[b].items():
                setattr(self, name, t)
            for p in self.phases:
                p.fn()
            comp[b].record(stream)
            ds.wait_event(comp[b])
            with torch.cuda.stream(ds):
                self.out_host[b].copy_(self.out_dev[b], non_blocking=True)
            d2h[b].record(ds)
        stream.wait_event(d2h[(steps - 1) % 2])


def kernel_source_hash() -> str:
    """Hash of the CUDA sources' code (comments and blank space removed):
    traffic figures taken from other code are void, a comment edit is not."""
    import glob
    import hashlib
    import re

    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "sparse_convolution_hash_gb300", "csrc", "*"))):
        with open(f, encoding="utf-8") as fh:
            code = fh.read()
        code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)  # block comments
        code = re.sub(r"//[^\n]*", " ", code)                # line comments (no string here holds //)
        code = " ".join(code.split())
        h.update(os.path.basename(f).encode() + b"\0" + code.encode() + b"\0")
    return h.hexdigest()[:16]


def measured_traffic(workload: str, phase: str):
    """DRAM bytes per launch of a phase from the committed ncu capture, or None
    when the capture was taken on other kernel sources (or is missing)."""
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("src_hash") != kernel_source_hash():
        return None
    v = t.get("workloads", {}).get(workload, {}).get(phase)
    return float(v) if v is not None else None


_UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}


def record_traffic(csv_path: str, workload: str, phases):
    """Store the DRAM bytes (read + write) of one call of each phase -- the sum
    over the libspc kernels the phase launches -- from an ncu --csv metrics log
    into profiles/dram_traffic.json, keyed by the current kernel-source hash.

    Kernels are grouped by phase: out-coords (candidates, radix sort, unique),
    build (table and count init, insert, map probe), conv (weight transpose + gather
    kernels; with a backward pass the conv launches alternate forward, dinput)
    and dfilter.  A phase's bytes are its kernels' bytes divided by the number
    of its calls (counted by one anchor kernel per phase)."""
    import csv
    import re

    per_id = {}
    with open(csv_path) as f:
        rows = [r for r in csv.reader(l for l in f if l.startswith('"'))]
    head, body = rows[0], rows[1:]
    ci = {k: head.index(k) for k in ("ID", "Kernel Name", "Metric Name", "Metric Unit", "Metric Value")}
    for r in body:
        name = r[ci["Metric Name"]]
        if name not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        d = per_id.setdefault(int(r[ci["ID"]]), {"kernel": r[ci["Kernel Name"]], "bytes": 0.0})
        d["bytes"] += float(r[ci["Metric Value"]].replace(",", "")) * _UNITS.get(r[ci["Metric Unit"]], 1)
    launches = [per_id[i] for i in sorted(per_id)]

    def k(pattern):
        return [d for d in launches if re.search(r"::" + pattern, d["kernel"])]

    def per_call(group, anchor):
        n = len(k(anchor))
        return sum(d["bytes"] for d in group) / n if n else None

    got = {}
    if "outcoords" in phases:
        got["outcoords"] = per_call(k(r"k_(candidates|radix|scan|unique|bm_)"),
                                    r"k_(candidates|bm_mark)")
    if "build" in phases:
        # a submanifold build with its row order also runs the mask-key sort
        ro = r"|row_keys_from_mask|radix|scan_exclusive|perm_from_keys" if k(r"k_row_keys_from_mask") else ""
        got["build"] = per_call(k(r"k_(build_init|hash_insert|map_probe" + ro + ")"), r"k_map_probe")
    conv = k(r"k_(conv_|gather_gemm)")
    fwd, dgr = (conv[0::2], conv[1::2]) if "dgrad" in phases else (conv, [])
    tr = k(r"k_(transpose_w|i8_prep_w)")
    if fwd:
        got["inverse" if "inverse" in phases else "fwd"] = sum(d["bytes"] for d in fwd) / len(fwd) + (
            sum(d["bytes"] for d in tr) / len(tr) if tr else 0.0)
    if dgr:
        got["dgrad"] = sum(d["bytes"] for d in dgr) / len(dgr)
    if "wgrad" in phases:
        got["wgrad"] = per_call(k(r"k_wgrad"), r"k_wgrad_(tc|partial)")
    if "pool" in phases:
        got["pool"] = per_call(k(r"k_maxpool_fwd"), r"k_maxpool_fwd")
        got["pool_dgrad"] = per_call(k(r"k_maxpool_dgrad"), r"k_maxpool_dgrad")
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        t = {}
    if t.get("src_hash") != kernel_source_hash():
        t = {"src_hash": kernel_source_hash(), "workloads": {}}
    t["note"] = ("DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one call of each "
                 "phase, summed over the kernels it launches; ncu, cold caches")
    t["workloads"][workload] = {ph: round(v) for ph, v in got.items() if v is not None}
    with open(path, "w") as f:
        json.dump(t, f, indent=1, sort_keys=True)
    print(json.dumps({workload: t["workloads"][workload]}))


def int8_fp16_products(K: int, cin: int, cout: int) -> int:
    """fp16 tensor-core products per int8 product in the library's int8 forward
    (sm_103a has no integer MMA; conv_i8.cu picks the path the same way): 1 on
    the several-accumulator path (no accumulator sums more than 15 stages of 64
    channels, at most 4 accumulators of 128 or 8 of 64 output channels), 2 on
    the 4-bit weight split beyond it."""
    stages = K * (cin // 64)
    nacc = -(-stages // 15)
    return 1 if (cout % 128 == 0 and nacc <= 4) or nacc <= 8 else 2


def i8_src(p: Phase) -> str:
    if getattr(p, "fp16_per_int8", 2) == 1:
        return "bf16_tflops burst: each int8 product runs as one exact fp16 product (accumulator path)"
    return "bf16_tflops burst / 2: each int8 product runs as two fp16 products (weight split)"


def roofline(p: Phase, ms: float, hbm: float, tc_peak: float, alu_peak: float, dtype: str,
             prec_tf32: bool):
    t_hbm = p.bytes_alg / (hbm * 1e9)
    if p.kind != "conv":
        bound, peak, ach, unit = "hbm", hbm, p.bytes_alg / (ms * 1e-3) / 1e9, "GB/s"
        t_bound = t_hbm
    else:
        if dtype == "f32" and not prec_tf32:
            cpeak, cbound = alu_peak, "alu"
        elif dtype == "i8":
            # no integer MMA on sm_103a: int8 products run as exact fp16 ones, one
            # each on the several-accumulator path, two (the weight's 4-bit halves)
            # on the weight split
            cpeak, cbound = tc_peak / getattr(p, "fp16_per_int8", 2), "tensor"
        else:
            cpeak, cbound = (tc_peak * (1.1 / 2.25) if dtype == "f32" else tc_peak), "tensor"
        t_c = p.flops / (cpeak * 1e12)
        if t_c >= t_hbm:
            bound, peak, ach, unit, t_bound = cbound, cpeak, p.flops / (ms * 1e-3) / 1e12, "TFLOP/s", t_c
        else:
            bound, peak, ach, unit, t_bound = "hbm", hbm, p.bytes_alg / (ms * 1e-3) / 1e9, "GB/s", t_hbm
    return {"bound": bound, "achieved": round(ach, 3), "peak": round(peak, 1), "unit": unit,
            "frac": round(ach / peak, 4), "roofline_ms": round(t_bound * 1e3, 5)}


def run_ours(args, rank, world, local, dist):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    case = Case(args.workload, dev)
    case.capture()
    for _ in range(args.warmup):
        case.replay_all()
    torch.cuda.synchronize()
    case.B.check_status(case.status, "bench warmup")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    nph = len(case.phases)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nph + 1)] for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        # keep the device busy while the host enqueues all steps, so that no
        # host gap falls inside a timed step
        torch.cuda._sleep(int(3e5) * args.steps * nph + int(2e6))
        for i in range(args.steps):
            flush.zero_()
            for j, p in enumerate(case.phases):
                ev[i][j].record(stream)
                p.graph.replay()
            ev[i][nph].record(stream)
        torch.cuda.synchronize()
    barrier(dist)
    case.B.check_status(case.status, "bench timed")
    for j, p in enumerate(case.phases):
        p.ms = [ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps)]
    total_ms = reduce_max(sum(sum(p.ms) for p in case.phases), dist, dev)
    ms_step = total_ms / args.steps
    flops = case.conv_flops()
    value = world * flops * args.steps / (total_ms * 1e-3) / 1e12

    case.setup_e2e()
    case.e2e_run(2, stream)
    torch.cuda.synchronize()
    # three timed regions of e2e_steps steps each; the median region counts
    # (host-side copies share the machine's memory system with other work)
    e2e_steps = max(1, min(args.steps, 20))
    regions = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist)
        e0.record(stream)
        case.e2e_run(e2e_steps, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        regions.append(e0.elapsed_time(e1))
    case.B.check_status(case.status, "bench e2e")
    e2e_ms = reduce_max(statistics.median(regions), dist, dev) / e2e_steps

    hbm, bf16_tf, peak_src = peaks()
    props = torch.cuda.get_device_properties(dev)
    alu_peak = props.multi_processor_count * 128 * 2 * 2.07e9 / 1e12  # FP32 FMA lanes x 2 x max clock
    phases = {}
    for p in case.phases:
        avg = sum(p.ms) / len(p.ms)
        r = roofline(p, avg, hbm, bf16_tf, alu_peak, case.dtype, case.prec == case.B.SPC_PREC_TF32)
        phases[p.name] = {"ms": round(avg, 5), "kernels": p.kernels, **r}
        if p.kind == "conv":
            phases[p.name]["tflops"] = round(p.flops / (avg * 1e-3) / 1e12, 3)
    dom = max(case.phases, key=lambda p: sum(p.ms))
    dom_r = phases[dom.name]
    clocks = clk.summary()
    build_ms = sum(phases[k]["ms"] for k in ("outcoords", "build") if k in phases)
    line = {
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": case.dtype,
        "data": "synthetic (seeded scene, random-init weights)",
        "config": {
            "workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}",
            "n_voxels": case.n, "n_out": case.n_out, "pairs": case.pairs, "cin": case.cin,
            "cout": case.cout, "K": case.K,
            "l2": "flushed between timed steps (256 MiB write, outside the events)",
            "timing": "CUDA-graph replay per phase, CUDA events on the launching stream",
            "parallelism": f"replicas x{world}",
            "row_storage": COORD_ORDER[0],
            "tile_order": "mask-grouped (perm)" if ROW_ORDER[0] else "map order",
        },
        "indice_map_mvoxel_s": round(world * case.n / (build_ms * 1e-3) / 1e6, 2) if build_ms else None,
        "phases": phases,
        "roofline": {"kernel": f"{dom.name}: {dom.kernels}", "bound": dom_r["bound"],
                     "achieved": dom_r["achieved"], "peak": dom_r["peak"], "unit": dom_r["unit"],
                     "frac": dom_r["frac"], "traffic": measured_traffic(args.workload, dom.name),
                     "peak_source": f"{peak_src} ({'hbm_gbs burst copy' if dom_r['unit'] == 'GB/s' else (i8_src(dom) if case.dtype == 'i8' else 'bf16_tflops burst') if dom_r['bound'] == 'tensor' else 'FP32 lanes x clock'})",
                     "alg_bytes_per_launch": dom.bytes_alg, "alg_flops_per_launch": dom.flops},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 4), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": int(case.h2d),
                "d2h_bytes_per_step": int(case.d2h),
                "timing": f"median of 3 regions of {e2e_steps} steps"},
        "gpu_launches": args.steps * sum(p.launches for p in case.phases),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, budget_s=args.cpu_seconds)
    return line


_THREADS = [1]  # oracle threads of the current sample (for its description)


def oracle_threads(n: int) -> int:
    """Sets the oracle's row-loop threads; returns the count in effect."""
    import oracle

    oracle.build()
    _THREADS[0] = oracle.set_threads(n)
    return _THREADS[0]


def cpu_sample(case_w, batch, shape, ks, subm, pairs_total, budget_s, stride=1, pad=0):
    """Times the oracle on a bounded sample; returns (TFLOP/s, description)."""
    import oracle

    oracle.build()
    c = case_w["coords"]
    n = c.shape[0]
    if not case_w.get("int8"):
        x64, w64 = oracle.f64(case_w["x"]), oracle.f64(case_w["w"])
        b64 = oracle.f64(case_w["bias"]) if case_w["bias"] is not None else None
    cin, cout = case_w["cin"], case_w["cout"]
    t0 = time.perf_counter()
    if subm:
        imap, cnt = oracle.subm_map(c, batch, shape, ks)
    else:
        oc = oracle.strided_out_coords(c, batch, shape, ks, stride, pad, 1)
        imap, _, cnt = oracle.strided_map(c, oc, batch, shape, ks, stride, pad, 1, False)
    t_map = time.perf_counter() - t0
    if case_w.get("maxpool"):
        # max pool forward on the saved map (not charged), all rows
        t1 = time.perf_counter()
        oracle.maxpool_fwd(x64, imap)
        t = time.perf_counter() - t1
        return float(cnt.sum()) * cin / t / 1e12, (f"fp64 max pool of all {imap.shape[1]} output "
                                                   f"rows (map built once, not charged), {t:.1f} s, "
                                                   f"{_THREADS[0]} thread(s)")
    if case_w.get("int8"):
        # the oracle's int8 rule on a sample of output rows (the map charged pro rata)
        per_row = 2.0 * float(cnt.sum()) / max(n, 1) * cin * cout
        rows = int(min(n, max(64, budget_s * 0.5e9 * _THREADS[0] / max(per_row, 1.0))))
        sel = np.linspace(0, n - 1, rows).astype(np.int64)
        t1 = time.perf_counter()
        oracle.conv_fwd_int8(case_w["x"], case_w["w"], case_w["scale"], case_w["bias"],
                             imap[:, sel], relu=True)
        t = time.perf_counter() - t1 + t_map * rows / max(n, 1)
        flops = 2.0 * float((imap[:, sel] >= 0).sum()) * cin * cout
        return flops / t / 1e12, (f"map over all {n} voxels ({t_map:.2f} s, charged pro rata) + "
                                  f"int8 forward of {rows} of {n} rows, {t:.1f} s, {_THREADS[0]} thread(s)")
    if case_w.get("inverse"):
        # the inverse conv on the saved maps (not charged): the oracle's forward
        # gathered through the transposed map (the same sums; the oracle pins
        # check that identity) on a sample of the output rows
        oc = oracle.strided_out_coords(c, batch, shape, ks, stride, pad, 1)
        _, imap_t, cnt = oracle.strided_map(c, oc, batch, shape, ks, stride, pad, 1, True)
        y64 = oracle.f64(case_w["y_for"](oc.shape[0]))
        per_row = 2.0 * float(cnt.sum()) / max(n, 1) * cin * cout
        rows = int(min(n, max(64, budget_s * 1.0e9 * _THREADS[0] / max(per_row, 1.0))))
        sel = np.linspace(0, n - 1, rows).astype(np.int64)
        t1 = time.perf_counter()
        oracle.conv_fwd(y64, w64, b64, imap_t, rows=sel)
        t = time.perf_counter() - t1
        flops = 2.0 * float((imap_t[:, sel] >= 0).sum()) * cin * cout
        return flops / t / 1e12, (f"fp64 inverse conv (gather through the transposed map) of {rows} "
                                  f"of {n} output rows (maps built once, not charged), {t:.1f} s, "
                                  f"{_THREADS[0]} thread(s)")
    n_out = imap.shape[1]
    per_row = 2.0 * float(cnt.sum()) / max(n_out, 1) * cin * cout  # flops per output row
    # rows so that the forward sample takes about the budget at ~1 GFLOP/s
    rows = int(min(n_out, max(64, budget_s * 1.0e9 * _THREADS[0] / max(per_row, 1.0))))
    sel = np.linspace(0, n_out - 1, rows).astype(np.int64) if rows < n_out else None
    reps, flops, t_fwd = 0, 0.0, 0.0
    t1 = time.perf_counter()
    while True:
        if sel is None:
            oracle.conv_fwd(x64, w64, b64, imap)
            flops += 2.0 * float(cnt.sum()) * cin * cout
        else:
            oracle.conv_fwd(x64, w64, b64, imap, rows=sel)
            flops += 2.0 * float((imap[:, sel] >= 0).sum()) * cin * cout
        reps += 1
        t_fwd = time.perf_counter() - t1
        if t_fwd >= budget_s or sel is not None:
            break
    frac = (len(sel) if sel is not None else n_out) / max(n_out, 1)
    t = t_map * frac * (reps if sel is None else 1) + t_fwd
    what = (f"{reps} whole steps (map + fp64 forward of all {n_out} rows)" if sel is None else
            f"map over all {n} voxels ({t_map:.2f} s, charged pro rata) + fp64 forward of "
            f"{len(sel)} of {n_out} rows")
    return flops / t / 1e12, f"{what}, {t:.1f} s, {_THREADS[0]} thread(s)"


def cpu_baseline(case, budget_s=10.0):
    """The oracle on the host cores: one thread, then one thread per core (its
    row loops run in parallel; the results do not depend on the count)."""
    w = case.w
    args = (w, case.batch, case.shape, case.ks, w["subm"], case.pairs, budget_s / 2,
            w.get("stride", 1), w.get("pad", 0))
    oracle_threads(1)
    v1, what1 = cpu_sample(*args)
    cores = oracle_threads(os.cpu_count() or 1)
    vn, whatn = cpu_sample(*args)
    oracle_threads(1)
    return {"value": round(vn, 8), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": whatn,
            "single_thread": {"value": round(v1, 8), "cores": 1, "sample": what1}}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = scenes.workload(args.workload)
    kind = args.workload.split("_")[0]
    shape = SHAPES[kind]
    c = w["coords"]
    batch = int(c[:, 0].max()) + 1
    vals = []
    cores = oracle_threads(os.cpu_count() or 1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, what = cpu_sample(w, batch, shape, w["k"], w["subm"], None,
                             args.cpu_seconds / max(args.steps, 1), w.get("stride", 1),
                             w.get("pad", 0))
        vals.append(v)
    tot = time.perf_counter() - t0
    value = statistics.mean(vals)
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 8), "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "i8" if w.get("int8") else "f64",
        "data": "synthetic (seeded scene, random-init weights)",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}",
                   "n_voxels": int(c.shape[0])},
        "cpu_baseline": {"value": round(value, 8), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {what}"},
        "e2e": {"value": round(value, 8), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(DESCRIPTIONS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--row-order", choices=["on", "off"], default="off",
                    help="compute the wide-channel submanifold convs' tiles in mask-grouped "
                         "row order (built with the map) or in map order")
    ap.add_argument("--coord-order", choices=["scene", "mask", "shuffled"], default="scene",
                    help="store the submanifold workloads' voxel rows in the scene's order, "
                         "grouped by offset mask, or shuffled")
    ap.add_argument("--record-traffic", metavar="NCU_CSV",
                    help="store the DRAM bytes of an ncu metrics log of this workload and exit")
    args = ap.parse_args()
    ROW_ORDER[0] = args.row_order == "on"
    COORD_ORDER[0] = args.coord_order
    if args.record_traffic:
        w = scenes.workload(args.workload)
        phases = (["build"] if w["subm"] and w["k"] > 1 else []) + \
                 ([] if w["subm"] else ["outcoords", "build"]) + ["fwd"] + \
                 (["dgrad", "wgrad"] if w.get("train") else [])
        if w.get("inverse"):
            phases = ["inverse"]
        if w.get("maxpool"):
            phases = ["outcoords", "build", "pool", "pool_dgrad"]
        record_traffic(args.record_traffic, args.workload, phases)
        return
    args.warmup = max(args.warmup, 3)
    rank, world, local, dist = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        import __graft_entry__

        if rank == 0:
            __graft_entry__.build()
        barrier(dist)
        __graft_entry__.build()
        line = run_ours(args, rank, world, local, dist)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
