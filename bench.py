#!/usr/bin/env python3
"""Benchmark of the BitDelta hot path on one GB300 (or N replicas).

A step is one pass of the whole hot path over one batch of synthetic input:
compression of every matrix of the workload (delta, sign packing, alpha) and
the fused linear of every matrix at every token count of the workload; the
multi-tenant workload adds the per-token-variant linear.  Inputs are resident
in HBM when the timed region starts; each phase is captured once as a CUDA
graph and replayed, so host launch overhead is not timed, and CUDA events on
the replay stream bracket every phase (they give the per-kernel roofline).

The default workload is the 32-layer Llama-3-8B-shape stack (q 4096x4096, k/v
1024x4096, o 4096x4096, gate/up 14336x4096, down 4096x14336 per layer): the
compression of its 224 matrices, the fused linear of each at m = 1 (decode)
and m = 2048 (prefill), the stack's multi-tenant decode (64 tokens over 14
resident variants of the same base) and the 14-variant batch over one
8192x8192 base (its compressions, 64 decode tokens, 2048 Zipf prefill tokens).
`value` is the decode phase's fused-linear GB/s (algorithmic bytes over that
phase's CUDA-event time); `prefill` gives the m = 2048 phase in TFLOP/s with its
own roofline and CPU baseline.  Every input is far larger than L2 (14 GB of
base weights per pass over the stack), so kernels read from HBM.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
Prints one JSON line (rank 0).  --impl reference times the fp64 CPU oracle on
the host cores (a bounded sample of the same workload per step).
"""
from __future__ import annotations

import argparse
import json
import math
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
import torch  # noqa: E402

from bit_delta_tenant_gb300 import synth, workloads  # noqa: E402

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# --------------------------------------------------------------------------- helpers

def load_peaks():
    try:
        with open(PEAKS_PATH) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), source="measured")
    except Exception:
        return dict(hbm=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS, bf16_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm), "reasons": sorted(reasons)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, value: float) -> float:
    if ws == 1:
        return value
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(ws: int, steps: int, step_work: float, t_max_ms: float) -> float:
    """Whole-job throughput of N replicas (weak scaling): every rank processes
    `steps` steps of `step_work` units; the slowest rank's time counts."""
    return ws * steps * step_work / (t_max_ms * 1e-3) / 1e9


# --------------------------------------------------------------------------- workloads

class Phase:
    """A list of C-ABI calls replayed as one CUDA graph; algorithmic work per replay."""

    def __init__(self, name, calls, bytes_=0.0, flops=0.0, launches=0, bound="hbm", weight_prefetch=False):
        self.name, self.calls, self.bytes, self.flops, self.launches, self.bound = \
            name, calls, bytes_, flops, launches, bound
        self.weight_prefetch = weight_prefetch
        self.graph = None

    @property
    def unit(self):
        return "GB/s" if self.bound == "hbm" else "TFLOP/s"

    def run(self):
        for c in self.calls:
            c()

    def capture(self, stream, bd=None):
        """Graph of the calls.  With `weight_prefetch`, the launches are recorded with
        bd_set_weight_prefetch(1): inside the graph every fused linear follows another
        fused linear, which never writes weights, so the knob's condition holds."""
        prev = bd.bd_set_weight_prefetch(1 if self.weight_prefetch else 0) if bd is not None else None
        try:
            self.run()                     # eager warm-up: sets kernel attributes, caches device info
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                self.run()
            self.graph = g
        finally:
            if bd is not None:
                bd.bd_set_weight_prefetch(prev)

    def replay(self):
        self.graph.replay()


def compress_phase(bd, mats, mode, dev):
    """Every (W_base, W_ft) of `mats` compressed -- in bd_compress_batch calls of up to 8
    matrices (COMPRESS_BATCH), else one bd_compress per matrix; outputs kept for the
    linear phases."""
    calls, nbytes, launches = [], 0.0, 0
    outs = []
    for (wb, wf) in mats:
        n_out, n_in = wb.shape
        bits = torch.empty((n_out, n_in // 8), dtype=torch.uint8, device=dev)
        alpha = torch.empty((n_out if mode == 1 else 1,), dtype=torch.float32, device=dev)
        nbytes += 4.0 * n_out * n_in + n_out * n_in / 8 + 4.0 * (n_out if mode == 1 else 1)
        outs.append((bits, alpha))
        if not COMPRESS_BATCH:
            ws = torch.empty((max(16, bd.bd_compress_workspace_size(n_out, n_in, mode)),), dtype=torch.uint8,
                             device=dev)
            calls.append(lambda wb=wb, wf=wf, bits=bits, alpha=alpha, ws=ws:
                         bd.bd_compress(wb, wf, mode, bits, alpha, ws))
            launches += 2
    if COMPRESS_BATCH:
        for i in range(0, len(mats), 8):
            descs = bd.compress_descs([(wb, wf, mode, bits, alpha) for (wb, wf), (bits, alpha)
                                       in zip(mats[i:i + 8], outs[i:i + 8])])
            ws = torch.empty((max(256, bd.bd_compress_batch_workspace_size(descs)),), dtype=torch.uint8, device=dev)
            calls.append(lambda descs=descs, ws=ws: bd.bd_compress_batch(descs, ws))
            launches += 2
    return Phase("compress", calls, bytes_=nbytes, launches=launches), outs


# Fused linears of the device-resident decode/prefill phases are captured with
# bd_set_weight_prefetch(1) (static weights, as when serving); --weight-prefetch 0
# turns it off.  The end-to-end leg replays the same graphs: a graph launch starts
# only after the previous one (the compression that writes the bits) has completed,
# and inside the linear graph no kernel writes weights.
WEIGHT_PREFETCH = True

# How a layer's fused linears are issued: "layer" passes the projections that share their
# input in a real layer -- q, k, v and gate, up -- to one bd_linear_batch call each; "qkv"
# batches q, k, v only; "none" calls bd_linear per matrix (a call of one problem runs as
# bd_linear either way).  "auto" takes the workload's own choice, measured on GB300: the
# Llama-7B layer batches q/k/v only (its 11008-row gate and up run faster alone, on the
# cluster-split kernel's balanced plan), the Llama-3-8B stack batches both groups.
LINEAR_BATCH = "auto"
FUSED_GROUPS = ({"q", "k", "v"}, {"gate", "up"})
# Compressions issued through bd_compress_batch (up to 8 matrices per call); --compress-batch 0
# issues one bd_compress per matrix.
COMPRESS_BATCH = True


def layer_groups(names, fused=FUSED_GROUPS):
    """Consecutive indices of `names` ("L<l>.<matrix>") that one batched call takes."""
    groups, i = [], 0
    while i < len(names):
        layer, base = names[i].split(".", 1)
        grp = next((g for g in fused if base in g), None)
        j = i + 1
        while grp is not None and j < len(names) and names[j].split(".", 1)[0] == layer \
                and names[j].split(".", 1)[1] in grp:
            j += 1
        groups.append(list(range(i, j)))
        i = j
    return groups


def decode_bytes(m, n_out, n_in, mode):
    return 2.0 * n_out * n_in + n_out * n_in / 8 + 4.0 * (n_out if mode == 1 else 1) + 2.0 * m * n_in + 2.0 * m * n_out


class Workload:
    """Matrices, phases (each a list of C-ABI calls), e2e buffers and an oracle sample.

    `value` of the JSON line = the step's work in `metric_unit` (algorithmic bytes
    for GB/s, 2*m*N*K flops for TFLOP/s) / step time; phases measured in the
    other unit still count in the time.
    """
    metric_unit = "GB/s"

    def step_work(self):
        if self.metric_unit == "GB/s":
            return sum(p.bytes for p in self.phases if p.bound == "hbm")
        return sum(p.flops for p in self.phases if p.bound == "tensor") / 1e3  # TFLOP/s with the GB/s scaling

    def e2e_buffers(self):
        """Per-step host->device inputs (fine-tuned weights, activations) and device->host results."""
        h2d = [(torch.empty_like(t, device="cpu").pin_memory(), t) for t in self.h2d_tensors]
        for host, devt in h2d:
            host.copy_(devt)
        d2h = [(torch.empty_like(t, device="cpu").pin_memory(), t) for t in self.d2h_tensors]
        return h2d, d2h


class LayerWorkload(Workload):
    """Every matrix of `cfg` compressed, then its fused linear at every m of `ms`.

    Used for the Llama-7B layer at decode sizes (the default), the 70B-shape
    prefill linears and the Llama-3-8B-shape stack (decode or prefill)."""

    def __init__(self, bd, dev, cfg, ms, unit, name, layers=1, private_io=True, batch="layer", phase_per_m=False):
        self.cfg, self.metric_unit = cfg, unit
        mode = cfg["mode"]
        shapes = [(f"L{l}.{n}", a, b) for l in range(layers) for (n, a, b) in cfg["matrices"]]
        self.shapes = shapes
        self.mats = [synth.matrix_pair(n_out, n_in, cfg["sigma"], cfg["b"], workloads.matrix_seed(cfg["seed"], i), dev)
                     for i, (_, n_out, n_in) in enumerate(shapes)]
        self.comp, self.packed = compress_phase(bd, self.mats, mode, dev)
        self.xs, self.ys = {}, {}
        calls, nbytes, flops, launches = [], 0.0, 0.0, 0
        names = [n for n, _, _ in shapes]
        self.batch = batch if LINEAR_BATCH == "auto" else LINEAR_BATCH
        groups = layer_groups(names) if self.batch == "layer" else \
            layer_groups(names, FUSED_GROUPS[:1]) if self.batch == "qkv" else [[i] for i in range(len(shapes))]
        self.batch_ws = None
        self.linear_plan = []  # (matrices the call needs, call) for the pipelined end-to-end step
        self.lins = []  # one linear phase per token count (phase_per_m), else one for all of ms
        bound = "hbm" if unit == "GB/s" else "tensor"
        for mi, m in enumerate(ms):
            if phase_per_m and mi > 0:
                self.lins.append(Phase(f"fused_linear_m{ms[mi - 1]}", calls, bytes_=nbytes, flops=flops,
                                       launches=launches, bound="hbm" if ms[mi - 1] <= 16 else "tensor",
                                       weight_prefetch=WEIGHT_PREFETCH))
                calls, nbytes, flops, launches = [], 0.0, 0.0, 0
            for grp in groups:
                probs = []
                for j, i in enumerate(grp):
                    _, n_out, n_in = shapes[i]
                    xk = (m, i) if private_io else (m, n_in)
                    # shared outputs are reused across calls, never within one (bd_linear_batch's
                    # problems may not share a y)
                    yk = (m, i) if private_io else (m, n_out, j)
                    if xk not in self.xs:
                        self.xs[xk] = synth.activations(m, n_in, 10_000 + 97 * len(self.xs) + m, dev)
                    if yk not in self.ys:
                        self.ys[yk] = torch.empty((m, n_out), dtype=torch.bfloat16, device=dev)
                    bits, alpha = self.packed[i]
                    probs.append((self.xs[xk], self.mats[i][0], bits, alpha, mode, self.ys[yk]))
                    nbytes += decode_bytes(m, n_out, n_in, mode)
                    flops += 2.0 * m * n_out * n_in
                if self.batch in ("layer", "qkv"):
                    descs = bd.linear_descs(probs)
                    need = bd.bd_linear_batch_workspace_size(descs)
                    if need > 0 and (self.batch_ws is None or self.batch_ws.numel() < need):
                        self.batch_ws = torch.zeros(need, dtype=torch.uint8, device=dev)
                    calls.append(lambda descs=descs: bd.bd_linear_batch(descs, self.batch_ws))
                    # one launch: the batched streaming kernel (m <= 16), or the pair kernel over the
                    # group (m > 64) when its 256 x 256 tiles fill the SMs (152 on GB300)
                    pair_tiles = sum(-(-p[5].shape[1] // 256) * -(-m // 256) for p in probs)
                    batched = len(probs) > 1 and ((m <= 16 and all(p[1].shape[1] % 128 == 0 for p in probs))
                                                  or (m > 64 and 2 * pair_tiles >= 152))
                    launches += 1 if batched else len(probs)
                else:
                    x, wb, bits, alpha, _, y = probs[0]
                    calls.append(lambda x=x, wb=wb, bits=bits, alpha=alpha, y=y:
                                 bd.bd_linear(x, wb, bits, alpha, mode, y))
                    launches += 1
                self.linear_plan.append((set(grp), calls[-1]))
        if phase_per_m:
            self.lins.append(Phase(f"fused_linear_m{ms[-1]}", calls, bytes_=nbytes, flops=flops, launches=launches,
                                   bound="hbm" if ms[-1] <= 16 else "tensor", weight_prefetch=WEIGHT_PREFETCH))
        else:
            self.lins.append(Phase("fused_linear", calls, bytes_=nbytes, flops=flops, launches=launches, bound=bound,
                                   weight_prefetch=WEIGHT_PREFETCH))
        self.lin = self.lins[0]
        self.phases = [self.comp] + self.lins
        self.dominant = self.lin
        # one compression call per matrix, for the pipelined end-to-end step
        self.compress_one = []
        for (wb, wf), (bits, alpha) in zip(self.mats, self.packed):
            descs = bd.compress_descs([(wb, wf, mode, bits, alpha)])
            ws = torch.empty((max(256, bd.bd_compress_batch_workspace_size(descs)),), dtype=torch.uint8, device=dev)
            self.compress_one.append(lambda descs=descs, ws=ws: bd.bd_compress_batch(descs, ws))
        self.h2d_tensors = [wf for (_, wf) in self.mats] + list(self.xs.values())
        self.d2h_tensors = list(self.ys.values()) + [a for (_, a) in self.packed]
        self.config = {"workload": name, "matrices": sorted({f"{a}x{b}" for _, a, b in shapes}),
                       "matrix_count": len(shapes), "tokens": list(ms),
                       "alpha": "per-row" if mode == 1 else "scalar", "dtype_in": "bf16 weights/activations",
                       "weight_prefetch": WEIGHT_PREFETCH, "linear_batch": self.batch,
                       "compress_batch": COMPRESS_BATCH,
                       "l2": "inputs larger than L2 (consecutive uses of a matrix separated by >250 MB of traffic)"}

    def oracle_sample(self, oracle, frac_rows: float, ms=None, compress=True):
        """Bounded CPU sample of one step: the first `frac_rows` of the first layer's rows
        (compression unless `compress` is false, then the fused linear at each m of `ms`,
        default every m of the step, in the unit of that m's phase)."""
        cfg = self.cfg
        mode = cfg["mode"]
        first_layer = len(cfg["matrices"])
        host = []
        for i, (wb, wf) in enumerate(self.mats[:first_layer]):
            n = max(8, int(wb.shape[0] * frac_rows))
            host.append((synth.as_u16(wb[:n]), synth.as_u16(wf[:n])))
        ms = sorted({k[0] for k in self.xs}) if ms is None else sorted(ms)
        unit = self.metric_unit if len(ms) > 1 else ("GB/s" if ms[0] <= 16 else "TFLOP/s")
        tok_cap = 64  # at most the first 64 tokens of each batch (prefill batches are thousands)
        xs = {}
        for m in ms:
            for i, (_, _, n_in) in enumerate(self.shapes[:first_layer]):
                key = (m, i) if (m, i) in self.xs else (m, n_in)
                xs[(m, i)] = synth.as_u16(self.xs[key][:tok_cap])

        # without the compression in the sample, its bits and alpha are made once outside it
        pre = None if compress else [oracle.compress(wb, wf, mode)[:2] for (wb, wf) in host]

        def run():
            nbytes, flops = 0.0, 0.0
            packed = []
            for (wb, wf) in host:
                if pre is None:
                    bits, a32, _ = oracle.compress(wb, wf, mode)
                    packed.append((bits, a32))
                    nbytes += 4.0 * wb.size + wb.size / 8 + 4.0
            if pre is not None:
                packed = pre
            for (m, i), x in xs.items():
                wb = host[i][0]
                bits, a32 = packed[i]
                oracle.linear(x, wb, bits, a32, mode)
                nbytes += decode_bytes(x.shape[0], wb.shape[0], wb.shape[1], mode)
                flops += 2.0 * x.shape[0] * wb.shape[0] * wb.shape[1]
            return nbytes if unit == "GB/s" else flops / 1e3
        desc = (f"first layer, each matrix's first {frac_rows:.4g} of rows: "
                + ("compression + " if compress else "") + "fused linear "
                f"at m={','.join(str(min(m, tok_cap)) for m in ms)}"
                + (" (first tokens of each batch)" if max(ms) > tok_cap else ""))
        return run, desc


class GroupedWorkload(Workload):
    """14 variants over one 8192x8192 base: compress every variant, then one
    multi-tenant linear per kind -- 64 decode tokens with uniform ids, and/or
    2048 prefill tokens in Zipf(1.1) segments."""

    def __init__(self, bd, dev, kinds=("decode",)):
        c = workloads.GROUPED_14
        self.cfg, self.kinds = c, tuple(kinds)
        self.metric_unit = "GB/s" if self.kinds[0] == "decode" else "TFLOP/s"
        n_out, n_in, nv = c["n_out"], c["n_in"], c["n_variants"]
        g = synth.generator(c["seed"], dev)
        self.w_base = synth.bf16_normal((n_out, n_in), c["sigma"], g, dev)
        self.fts = []
        for v, b in enumerate(workloads.variant_scales(c)):
            d = synth.laplace_f32((n_out, n_in), b, g, dev)
            self.fts.append((self.w_base.float() + d).to(torch.bfloat16))
            del d
        self.mats = [(self.w_base, wf) for wf in self.fts]
        self.comp, self.packed = compress_phase(bd, self.mats, c["mode"], dev)
        bits_v = [b for b, _ in self.packed]
        alpha_v = [a for _, a in self.packed]
        modes = [c["mode"]] * nv
        self.lins, self.io, self.ids_h = [], [], {}
        for kind in self.kinds:
            m = c["decode_m"] if kind == "decode" else c["prefill_m"]
            ids = synth.uniform_ids(m, nv, c["seed"]) if kind == "decode" else \
                synth.zipf_ids(m, nv, c["zipf_s"], c["seed"])
            self.ids_h[kind] = ids
            ids_d = torch.from_numpy(ids).to(dev)
            x = synth.activations(m, n_in, c["seed"] + 1, dev)
            y = torch.empty((m, n_out), dtype=torch.bfloat16, device=dev)
            ws = torch.empty((bd.bd_linear_grouped_workspace_size(m, nv, n_out, n_in),), dtype=torch.uint8,
                             device=dev)
            call = lambda x=x, ids_d=ids_d, y=y, ws=ws: bd.bd_linear_grouped(x, ids_d, self.w_base, bits_v, alpha_v,
                                                                             modes, y, ws)
            active = len(set(ids.tolist()))
            nbytes = 2.0 * n_out * n_in + active * n_out * n_in / 8 + 4.0 * nv + 2.0 * m * n_in + 2.0 * m * n_out
            flops = 2.0 * m * n_out * n_in
            # the sort and gather kernels are tiny; the launch count is the library's whole call
            self.lins.append(Phase(f"grouped_linear_{kind}", [call], bytes_=nbytes, flops=flops, launches=3,
                                   bound="hbm" if kind == "decode" else "tensor"))
            self.io.append(([x, ids_d], [y]))
        self.lin = self.lins[0]
        self.phases = [self.comp] + self.lins
        self.dominant = self.lin
        self.h2d_tensors = list(self.fts) + [t for ins, _ in self.io for t in ins]
        self.d2h_tensors = [t for _, outs in self.io for t in outs] + [a for (_, a) in self.packed]
        k = self.kinds[0]
        self.config = {"workload": f"grouped_14_variants_8192_{k}", "variants": nv,
                       "tokens": c["decode_m"] if k == "decode" else c["prefill_m"],
                       "ids": "uniform" if k == "decode" else "zipf(1.1) segments, shuffled",
                       "active_variants": len(set(self.ids_h[k].tolist())), "alpha": "scalar per variant",
                       "l2": "inputs larger than L2 (14 W_ft of 128 MB each are compressed every step)"}

    def oracle_sample(self, oracle, frac_rows: float, kind=None):
        c = self.cfg
        kind = kind or self.kinds[0]
        n = max(8, int(c["n_out"] * frac_rows))
        wb = synth.as_u16(self.w_base[:n])
        fts = [synth.as_u16(wf[:n]) for wf in self.fts]
        x = synth.as_u16(self.io[self.kinds.index(kind)][0][0])
        ids = self.ids_h[kind]
        modes = np.zeros(len(fts), np.int32)
        unit = "GB/s" if kind == "decode" else "TFLOP/s"

        def run():
            bits, alphas = [], []
            nbytes = 0.0
            for wf in fts:
                b, a, _ = oracle.compress(wb, wf, 0)
                bits.append(b), alphas.append(a)
                nbytes += 4.0 * wb.size + wb.size / 8
            oracle.linear_grouped(x, ids, wb, bits, alphas, modes)
            m = x.shape[0]
            if unit == "GB/s":
                return nbytes + 2.0 * wb.size + len(fts) * wb.size / 8 + 2.0 * m * wb.shape[1] + 2.0 * m * n
            return 2.0 * m * wb.size / 1e3
        return run, f"first {frac_rows:.4g} of the rows: 14 compressions + the multi-tenant linear ({kind})"


def compress_variants(bd, dev, w_base, scales, seed, mode=0):
    """Bits and alpha of one fine-tuned variant per scale of `scales` over `w_base`: W_ft =
    bf16(fp32(W_base) + Laplace(0, b)) drawn on the device and compressed by the library, in
    bd_compress_batch calls of up to 8 variants; the W_ft are freed afterwards."""
    n_out, n_in = w_base.shape
    out = []
    for v0 in range(0, len(scales), 8):
        fts, descs_in = [], []
        for v in range(v0, min(len(scales), v0 + 8)):
            g = synth.generator(seed * 131 + v, dev)
            d = synth.laplace_f32((n_out, n_in), scales[v], g, dev)
            wf = d.add_(w_base.float()).to(torch.bfloat16)
            del d
            bits = torch.empty((n_out, n_in // 8), dtype=torch.uint8, device=dev)
            alpha = torch.empty((n_out if mode == 1 else 1,), dtype=torch.float32, device=dev)
            fts.append(wf)
            descs_in.append((w_base, wf, mode, bits, alpha))
            out.append((bits, alpha))
        descs = bd.compress_descs(descs_in)
        ws = torch.empty((max(256, bd.bd_compress_batch_workspace_size(descs)),), dtype=torch.uint8, device=dev)
        bd.bd_compress_batch(descs, ws)
        torch.cuda.synchronize()
        del fts
    return out


class GroupedStackWorkload(Workload):
    """The serving decode step over a whole model: every linear of the 32-layer
    Llama-3-8B-shape stack as one multi-tenant call, 64 tokens whose ids are
    uniform over 14 variants, all 224 calls replayed as one CUDA graph.

    Each variant's delta of each matrix is compressed by the library from a
    fine-tuned W_ft = bf16(W_base + Laplace(0, b_v)) drawn on the device (b_v the
    14 evenly spaced scales of the 14-variant workload) and resident afterwards, as
    behind the delta cache; the W_ft are not kept (14 x 14 GB).  `bases` shares
    the W_base matrices of another workload (one resident base for every tenant)."""

    def __init__(self, bd, dev, bases=None):
        c = workloads.LLAMA3_8B_STACK
        g14 = workloads.GROUPED_14
        self.cfg = c
        self.metric_unit = "GB/s"
        nv, m = g14["n_variants"], g14["decode_m"]
        scales = workloads.variant_scales(g14)
        ids = synth.uniform_ids(m, nv, g14["seed"])
        self.ids_h = ids
        self.ids = torch.from_numpy(ids).to(dev)
        active = len(set(ids.tolist()))
        shapes = [(n, k) for _ in range(c["layers"]) for (_, n, k) in c["matrices"]]
        self.xs, self.ys, self.wss = {}, {}, {}
        calls, nbytes, flops = [], 0.0, 0.0
        self.first = None
        for i, (n_out, n_in) in enumerate(shapes):
            if bases is not None:
                wb = bases[i]
            else:
                gen = synth.generator(workloads.matrix_seed(c["seed"], 1000 + i), dev)
                wb = synth.bf16_normal((n_out, n_in), c["sigma"], gen, dev)
            packed = compress_variants(bd, dev, wb, scales, workloads.matrix_seed(c["seed"], 5000 + i))
            bits_v = [b for b, _ in packed]
            alpha_v = [a for _, a in packed]
            if n_in not in self.xs:
                self.xs[n_in] = synth.activations(m, n_in, 20_000 + n_in, dev)
                self.wss[n_in] = {}
            if n_out not in self.ys:
                self.ys[n_out] = torch.empty((m, n_out), dtype=torch.bfloat16, device=dev)
            key = (n_out, n_in)
            if key not in self.wss[n_in]:
                self.wss[n_in][key] = torch.empty((bd.bd_linear_grouped_workspace_size(m, nv, n_out, n_in),),
                                                  dtype=torch.uint8, device=dev)
            x, y, ws = self.xs[n_in], self.ys[n_out], self.wss[n_in][key]
            calls.append(lambda x=x, wb=wb, bv=bits_v, av=alpha_v, y=y, ws=ws:
                         bd.bd_linear_grouped(x, self.ids, wb, bv, av, [0] * nv, y, ws))
            nbytes += 2.0 * n_out * n_in + active * n_out * n_in / 8 + 4.0 * nv + 2.0 * m * n_in + 2.0 * m * n_out
            flops += 2.0 * m * n_out * n_in
            if self.first is None:
                self.first = (wb, bits_v, alpha_v, x)
        self.lin = Phase("grouped_linear", calls, bytes_=nbytes, flops=flops, launches=3 * len(calls), bound="hbm")
        self.phases = [self.lin]
        self.dominant = self.lin
        self.h2d_tensors = list(self.xs.values()) + [self.ids]
        self.d2h_tensors = list(self.ys.values())
        self.config = {"workload": "llama3_8b_stack_grouped14_decode", "layers": c["layers"],
                       "matrices": sorted({f"{a}x{b}" for _, a, b in c["matrices"]}), "variants": nv, "tokens": m,
                       "ids": "uniform", "active_variants": active,
                       "deltas": "resident; each compressed by bd_compress_batch from W_base + Laplace(0, b_v)",
                       "l2": "inputs larger than L2 (14 GB of base weights and 12 GB of bits per step)"}

    def oracle_sample(self, oracle, frac_rows: float):
        wb, bits_v, alpha_v, x = self.first
        n = max(8, int(wb.shape[0] * frac_rows))
        wbh = synth.as_u16(wb[:n])
        bh = [b[:n].cpu().numpy() for b in bits_v]
        ah = [a.cpu().numpy() for a in alpha_v]
        xh = synth.as_u16(x)
        modes = np.zeros(len(bh), np.int32)

        def run():
            oracle.linear_grouped(xh, self.ids_h, wbh, bh, ah, modes)
            mm = xh.shape[0]
            return 2.0 * wbh.size + len(bh) * wbh.size / 8 + 2.0 * mm * wbh.shape[1] + 2.0 * mm * n
        return run, f"first {frac_rows:.4g} of the rows of the first matrix: the multi-tenant linear"


def renamed(phase, name):
    phase.name = name
    return phase


class ServingWorkload(Workload):
    """The default step: the whole hot path over the 32-layer Llama-3-8B-shape stack.

    Phases, each one CUDA graph: compression of the 224 matrices; the fused linear of
    every matrix at m = 1 (decode) and at m = 2048 (prefill); the stack's serving decode
    with 64 tokens over 14 resident variants on the same base (one multi-tenant call per
    matrix); and the 14-variant batch over one 8192x8192 base -- its 14 compressions, 64
    decode tokens with uniform ids and 2048 prefill tokens in Zipf(1.1) segments.
    `value` is the fused-linear GB/s of the decode phase (its algorithmic bytes over its
    own CUDA-event time); the prefill phase reports TFLOP/s beside it.  With
    `reference`, only the first layer is built (the CPU arm samples it)."""

    metric_unit = "GB/s"

    def __init__(self, bd, dev, reference=False):
        c = workloads.LLAMA3_8B_STACK
        self.cfg, self.bd = c, bd
        self.stack = LayerWorkload(bd, dev, c, (1, 2048), "GB/s", "llama3_8b_stack",
                                   layers=1 if reference else c["layers"], private_io=False, phase_per_m=True)
        self.decode = renamed(self.stack.lins[0], "fused_linear_decode")
        self.prefill = renamed(self.stack.lins[1], "fused_linear_prefill")
        self.phases = [self.stack.comp, self.decode, self.prefill]
        self.tenants = self.g14 = None
        if not reference:
            self.tenants = GroupedStackWorkload(bd, dev, bases=[wb for wb, _ in self.stack.mats])
            self.g14 = GroupedWorkload(bd, dev, kinds=("decode", "prefill"))
            self.phases += [renamed(self.tenants.lin, "multi_tenant_stack_decode"),
                            renamed(self.g14.comp, "compress_14_variants"),
                            renamed(self.g14.lins[0], "multi_tenant_decode"),
                            renamed(self.g14.lins[1], "multi_tenant_prefill")]
        self.headline, self.secondary = self.decode, self.prefill
        self.dominant = self.decode
        g14 = workloads.GROUPED_14
        self.config = {"workload": "llama3_8b_stack", "layers": c["layers"],
                       "matrices": sorted({f"{a}x{b}" for _, a, b in c["matrices"]}),
                       "matrix_count": c["layers"] * len(c["matrices"]), "tokens": {"decode": 1, "prefill": 2048},
                       "alpha": "scalar", "dtype_in": "bf16 weights/activations",
                       "value": "fused-linear GB/s of the m = 1 phase (its algorithmic bytes / its CUDA-event time)",
                       "weight_prefetch": WEIGHT_PREFETCH, "linear_batch": self.stack.batch,
                       "compress_batch": COMPRESS_BATCH,
                       "multi_tenant": {"stack_decode": f"{g14['decode_m']} tokens, uniform ids over "
                                                       f"{g14['n_variants']} variants, every stack matrix",
                                        "batch_8192": f"{g14['n_variants']} variants over one 8192x8192 base: "
                                                      f"{g14['decode_m']} decode tokens (uniform ids), "
                                                      f"{g14['prefill_m']} prefill tokens (Zipf(1.1) segments)"},
                       "l2": "inputs larger than L2 (14 GB of base weights per pass over the stack)"}

    def oracle_sample(self, oracle, frac_rows: float, phase="decode"):
        return self.stack.oracle_sample(oracle, frac_rows, ms=(1,) if phase == "decode" else (2048,), compress=False)


WORKLOADS = {
    "llama7b_layer_decode": lambda bd, dev: LayerWorkload(
        bd, dev, workloads.LLAMA7B_LAYER, workloads.LLAMA7B_LAYER["ms"], "GB/s", "llama7b_layer_decode",
        batch="qkv"),
    "llama70b_linears_prefill": lambda bd, dev: LayerWorkload(
        bd, dev, workloads.LLAMA70B_PREFILL, workloads.LLAMA70B_PREFILL["ms"], "TFLOP/s", "llama70b_linears_prefill",
        private_io=False),
    "grouped14_decode": lambda bd, dev: GroupedWorkload(bd, dev, ("decode",)),
    "grouped14_prefill": lambda bd, dev: GroupedWorkload(bd, dev, ("prefill",)),
    "llama3_8b_stack": lambda bd, dev: ServingWorkload(bd, dev),
    "llama3_8b_stack_decode": lambda bd, dev: LayerWorkload(
        bd, dev, workloads.LLAMA3_8B_STACK, (1,), "GB/s", "llama3_8b_stack_decode",
        layers=workloads.LLAMA3_8B_STACK["layers"], private_io=False),
    "llama3_8b_stack_grouped14_decode": lambda bd, dev: GroupedStackWorkload(bd, dev),
    "llama3_8b_stack_prefill": lambda bd, dev: LayerWorkload(
        bd, dev, workloads.LLAMA3_8B_STACK, (2048,), "TFLOP/s", "llama3_8b_stack_prefill",
        layers=workloads.LLAMA3_8B_STACK["layers"], private_io=False),
}


# --------------------------------------------------------------------------- arms

def run_ours(args, ws, rank, local):
    from bit_delta_tenant_gb300 import build as lib_build
    if rank == 0:
        lib_build.build()
    barrier(ws)
    from bit_delta_tenant_gb300 import bitdelta as bd
    bd.load_library()
    dev = torch.device("cuda", local if ws > 1 else 0)
    peaks = load_peaks()
    wl = WORKLOADS[args.workload](bd, dev)
    stream = torch.cuda.Stream(device=dev)
    for p in wl.phases:
        p.capture(stream, bd)
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for p in wl.phases:
                p.replay()
    torch.cuda.synchronize()
    assert bd.bd_get_device_status() == bd.BD_OK

    n_ev = len(wl.phases)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev + 1)] for _ in range(args.steps)]
    clocks = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for k in range(args.steps):
            ev[k][0].record(stream)
            for j, p in enumerate(wl.phases):
                p.replay()
                ev[k][j + 1].record(stream)
        end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clock_info = clocks.stop() if clocks else None
    total_ms = start.elapsed_time(end)
    phase_ms = [0.0] * n_ev
    for k in range(args.steps):
        for j in range(n_ev):
            phase_ms[j] += ev[k][j].elapsed_time(ev[k][j + 1])
    status = bd.bd_get_device_status()
    if status != bd.BD_OK:
        raise RuntimeError(f"device status after timing: {bd.bd_status_string(status)}")

    t_max = max_over_ranks(ws, total_ms)
    head = getattr(wl, "headline", None)
    if head is not None:
        # value: the headline phase's work over its own time (summed over the timed steps)
        h_ms = max_over_ranks(ws, phase_ms[wl.phases.index(head)])
        value = aggregate_value(ws, args.steps, head.bytes if head.bound == "hbm" else head.flops / 1e3, h_ms)
    else:
        value = aggregate_value(ws, args.steps, wl.step_work(), t_max)

    def roofline(p):
        t = phase_ms[wl.phases.index(p)] * 1e-3 / (args.steps * p.launches)  # average launch
        if p.bound == "hbm":
            achieved, peak, unit = p.bytes / p.launches / t / 1e9, peaks["hbm"], "GB/s"
        else:
            achieved, peak, unit = p.flops / p.launches / t / 1e12, peaks["bf16"], "TFLOP/s"
        r = {"bound": p.bound, "kernel": p.name, "achieved": achieved, "peak": peak, "unit": unit,
             "frac": achieved / peak, "peak_source": peaks["source"], "traffic": lookup_traffic(args.workload, p)}
        if p.bound == "tensor":
            r["frac_of_sustained"] = achieved / peaks["bf16_sustained"]
        return r

    dom = wl.dominant
    breakdown = {}
    for j, p in enumerate(wl.phases):
        t = phase_ms[j] * 1e-3 / args.steps
        if p.bound == "hbm":
            breakdown[p.name] = {"ms_per_step": t * 1e3, "GB/s": p.bytes / t / 1e9,
                                 "frac_of_measured_hbm": p.bytes / t / 1e9 / peaks["hbm"],
                                 "launches": p.launches}
        else:
            breakdown[p.name] = {"ms_per_step": t * 1e3, "TFLOP/s": p.flops / t / 1e12,
                                 "frac_of_measured_bf16": p.flops / t / 1e12 / peaks["bf16"],
                                 "launches": p.launches}

    if args.no_e2e:
        e2e = None
    elif isinstance(wl, ServingWorkload):
        e2e = run_e2e_serving(args, wl, stream, ws)
    else:
        e2e = run_e2e(args, wl, stream, ws)
    cpu = cpu_baseline(wl, args) if (rank == 0 and not args.no_cpu) else None

    line = {
        "metric": "BitDelta fused linear GB/s (decode) & TFLOP/s (prefill), % of roofline",
        "value": value, "unit": head.unit if head is not None else wl.metric_unit, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_max / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded; N(0,sigma) bf16 base, Laplace deltas, N(0,1) activations)",
        "config": dict(wl.config, parallelism=f"replicas{ws}" if ws > 1 else "single"),
        "roofline": roofline(dom),
        "breakdown": breakdown,
        "e2e": e2e,
        "gpu_launches": args.steps * sum(p.launches for p in wl.phases),
        "clocks": clock_info,
        "cpu_baseline": cpu,
    }
    sec = getattr(wl, "secondary", None)
    if sec is not None:
        s_ms = max_over_ranks(ws, phase_ms[wl.phases.index(sec)])
        sv = aggregate_value(ws, args.steps, sec.bytes if sec.bound == "hbm" else sec.flops / 1e3, s_ms)
        line["prefill"] = {"value": sv, "unit": sec.unit, "tokens": 2048, "roofline": roofline(sec),
                           "e2e": (e2e or {}).get("segments", {}).get(sec.name),
                           "cpu_baseline": cpu_baseline(wl, args, phase="prefill")
                           if (rank == 0 and not args.no_cpu) else None}
    if isinstance(wl, ServingWorkload):
        line["multi_tenant"] = {p.name: roofline(p) for p in wl.phases
                                if p.name.startswith("multi_tenant")}
    if rank == 0:
        print(json.dumps(line), flush=True)


# Sources whose change invalidates a stored traffic figure, by phase bound.
KERNEL_SOURCES = {"hbm": ("decode_tma.cu", "decode_batch.cu", "decode_stage.cuh", "grouped_decode.cu", "grouped.cu",
                          "compress.cu", "api.cu"),
                  "tensor": ("prefill.cu", "prefill_pair.cu", "grouped.cu", "api.cu")}


def traffic_path(workload: str) -> str:
    return os.path.join(ROOT, "profiles", f"traffic_{workload}.json")


def sources_sha1(bound: str) -> str:
    import hashlib
    h = hashlib.sha1()
    for name in KERNEL_SOURCES[bound]:
        with open(os.path.join(ROOT, "bit_delta_tenant_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def lookup_traffic(workload: str, phase):
    """DRAM bytes per launch of `phase` from profiles/traffic_<workload>.json (written by
    --ingest-traffic from a one-kernel ncu capture), if the kernel sources are unchanged since."""
    try:
        with open(traffic_path(workload)) as f:
            rec = json.load(f).get(phase.name)
        if rec is None or rec.get("source_sha1") != sources_sha1(phase.bound):
            return None
        return float(rec["traffic_per_launch_bytes"])
    except (OSError, ValueError, KeyError):
        return None


def ingest_traffic(args):
    """--ingest-traffic CSV --phase NAME: the mean dram__bytes_read.sum + dram__bytes_write.sum per
    launch of an ncu --csv capture (one kernel, a few launches) into profiles/traffic_<workload>.json."""
    import csv
    per = {}
    with open(args.ingest_traffic, newline="") as f:
        rows = [r for r in csv.reader(f) if r]
    hdr = next(i for i, r in enumerate(rows) if "Metric Name" in r)
    cols = rows[hdr]
    ci, cm, cv, cu = (cols.index(k) for k in ("ID", "Metric Name", "Metric Value", "Metric Unit"))
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}
    for r in rows[hdr + 1:]:
        if len(r) <= max(ci, cm, cv, cu) or r[cm] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        per[r[ci]] = per.get(r[ci], 0.0) + float(r[cv].replace(",", "")) * scale.get(r[cu], 1.0)
    if not per:
        raise SystemExit("no dram__bytes_(read|write).sum rows in the capture")
    bound = "tensor" if args.phase in ("fused_linear_prefill", "multi_tenant_prefill") else "hbm"
    path = traffic_path(args.workload)
    try:
        with open(path) as f:
            data = json.load(f)
    except OSError:
        data = {}
    data[args.phase] = {"traffic_per_launch_bytes": sum(per.values()) / len(per), "launches_captured": len(per),
                        "source_sha1": sources_sha1(bound), "sources": list(KERNEL_SOURCES[bound]),
                        "command": args.ingest_command or ""}
    with open(path, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps({args.phase: data[args.phase]}))


def pipelined_step(wl, h2d, d2h, stream, copy_stream):
    """One end-to-end step of a layer workload with the host copies overlapped: each matrix's
    W_ft goes up on `copy_stream` and is compressed on `stream` as soon as it has landed; each
    linear call is issued as soon as the matrices it reads are compressed (weight prefetch off:
    a linear may directly follow the compression of its bits); then the outputs come back.
    Across steps the copies run ahead: a matrix's next W_ft waits only for this step's
    compression of that matrix, and the activations go through two staging buffers (copied
    into place on `stream`, in order with the linears that read them), so the host link never
    waits for a step's tail.  Returns (start, one): `start` orders the copies after work
    already on `stream` (the timer's start event), `one` issues a step."""
    n = len(wl.mats)
    ev = [torch.cuda.Event() for _ in range(n)]      # W_ft i landed (this step)
    cons = [torch.cuda.Event() for _ in range(n)]    # W_ft i read by its compression (previous step)
    xs = h2d[n:]
    staging = [[torch.empty_like(devt) for _, devt in xs] for _ in range(2)]
    x_up = [torch.cuda.Event() for _ in range(2)]    # staging b filled
    x_free = [torch.cuda.Event() for _ in range(2)]  # staging b copied into place
    step = [0]

    def start():
        copy_stream.wait_stream(stream)

    def one():
        b = step[0] % 2
        step[0] += 1
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(x_free[b])
            for (host, _), st in zip(xs, staging[b]):
                st.copy_(host, non_blocking=True)
            x_up[b].record(copy_stream)
            for i in range(n):
                copy_stream.wait_event(cons[i])
                h2d[i][1].copy_(h2d[i][0], non_blocking=True)
                ev[i].record(copy_stream)
        with torch.cuda.stream(stream):
            stream.wait_event(x_up[b])
            for (_, devt), st in zip(xs, staging[b]):
                devt.copy_(st, non_blocking=True)
            x_free[b].record(stream)
            issued = [False] * len(wl.linear_plan)
            done = set()
            for i in range(n):
                stream.wait_event(ev[i])
                wl.compress_one[i]()
                cons[i].record(stream)
                done.add(i)
                for k, (need, call) in enumerate(wl.linear_plan):
                    if not issued[k] and need <= done:
                        call()
                        issued[k] = True
            for host, devt in d2h:
                host.copy_(devt, non_blocking=True)
    return start, one


def run_e2e(args, wl, stream, ws):
    """Same step through the C ABI with host buffers: H2D of the step's inputs, kernels, D2H of
    results.  Layer workloads overlap the copies with the compressions and linears
    (pipelined_step); the others copy, replay the step's graphs and copy back."""
    h2d, d2h = wl.e2e_buffers()
    bi = sum(t.numel() * t.element_size() for t, _ in h2d)
    bo = sum(t.numel() * t.element_size() for t, _ in d2h)
    pipelined = hasattr(wl, "linear_plan")

    if pipelined:
        start, one = pipelined_step(wl, h2d, d2h, stream, torch.cuda.Stream())
    else:
        def start():
            pass

        def one():
            for host, devt in h2d:
                devt.copy_(host, non_blocking=True)
            for p in wl.phases:
                p.replay()
            for host, devt in d2h:
                host.copy_(devt, non_blocking=True)

    with torch.cuda.stream(stream):
        start()
        for _ in range(max(1, args.warmup)):
            one()
    torch.cuda.synchronize()
    barrier(ws)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        s.record(stream)
        start()  # no copy of the timed steps begins before the start event
        for _ in range(args.steps):
            one()
        e.record(stream)
    torch.cuda.synchronize()
    t = max_over_ranks(ws, s.elapsed_time(e))
    if pipelined:
        # the overlapped step must give the graph-replayed step's results, bit for bit
        got = [host.clone() for host, _ in d2h]
        with torch.cuda.stream(stream):
            for p in wl.phases:
                p.replay()
        torch.cuda.synchronize()
        for g, (_, devt) in zip(got, d2h):
            if not torch.equal(g, devt.cpu()):
                raise RuntimeError("end-to-end step and device-resident step disagree")
    return {"value": ws * args.steps * wl.step_work() / (t * 1e-3) / 1e9, "unit": wl.metric_unit,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "ms_per_step": t / args.steps,
            "copies": "overlapped with the compressions and linears, and with the previous step" if pipelined else "before the step"}


def run_e2e_serving(args, wl, stream, ws):
    """The default step end to end through the C ABI with host buffers, in segments whose
    CUDA-event times each include their own copies: (1) every W_ft from pinned host memory,
    each matrix compressed as soon as its copy has landed (copies on a second stream), alpha
    back; (2) the decode activations up, the m = 1 linears, y back; (3) the same at m = 2048;
    (4) the multi-tenant phases, each with its activations and ids up and y back.  W_base and
    the variants' packed deltas stay resident, as on the page.  `value` is the decode
    segment's fused-linear GB/s.  After timing, every output of the last step is checked bit
    for bit against a replay of the device-resident graphs."""
    st = wl.stack
    copy_stream = torch.cuda.Stream()
    pin = lambda t: torch.empty_like(t, device="cpu").pin_memory()

    def host_of(ts):
        out = []
        for t in ts:
            h = pin(t)
            h.copy_(t)
            out.append((h, t))
        return out
    mats = list(st.mats) + (list(wl.g14.mats) if wl.g14 is not None else [])
    comp_one = list(st.compress_one)
    if wl.g14 is not None:
        for (wb, wf), (bits, alpha) in zip(wl.g14.mats, wl.g14.packed):
            descs = wl.bd.compress_descs([(wb, wf, wl.g14.cfg["mode"], bits, alpha)])
            wsb = torch.empty((max(256, wl.bd.bd_compress_batch_workspace_size(descs)),), dtype=torch.uint8,
                              device=wb.device)
            comp_one.append(lambda descs=descs, wsb=wsb: wl.bd.bd_compress_batch(descs, wsb))
    wft_h = host_of([wf for _, wf in mats])
    alphas = [a for _, a in st.packed] + ([a for _, a in wl.g14.packed] if wl.g14 is not None else [])
    alpha_h = [(pin(a), a) for a in alphas]
    segs = []  # (name, phase or None, h2d pairs, d2h pairs)
    xs_of = {m: [t for (mm, _), t in st.xs.items() if mm == m] for m in (1, 2048)}
    ys_of = {m: [t for (mm, _, _), t in st.ys.items() if mm == m] for m in (1, 2048)}
    segs.append(("fused_linear_decode", wl.decode, host_of(xs_of[1]), [(pin(t), t) for t in ys_of[1]]))
    segs.append(("fused_linear_prefill", wl.prefill, host_of(xs_of[2048]), [(pin(t), t) for t in ys_of[2048]]))
    if wl.tenants is not None:
        tn = wl.tenants
        segs.append(("multi_tenant_stack_decode", tn.lin, host_of(list(tn.xs.values()) + [tn.ids]),
                     [(pin(t), t) for t in tn.ys.values()]))
        for ph, (ins, outs) in zip(wl.g14.lins, wl.g14.io):
            segs.append((ph.name, ph, host_of(ins), [(pin(t), t) for t in outs]))
    n = len(mats)
    landed = [torch.cuda.Event() for _ in range(n)]
    ev = []

    def one(record):
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(len(segs) + 2)] if record else None
        with torch.cuda.stream(stream):
            if record:
                marks[0].record(stream)
            copy_stream.wait_stream(stream)  # no copy of this step starts before its first mark
            with torch.cuda.stream(copy_stream):
                for i in range(n):
                    wft_h[i][1].copy_(wft_h[i][0], non_blocking=True)
                    landed[i].record(copy_stream)
            for i in range(n):
                stream.wait_event(landed[i])
                comp_one[i]()
            for h, d in alpha_h:
                h.copy_(d, non_blocking=True)
            if record:
                marks[1].record(stream)
            for k, (_, ph, up, down) in enumerate(segs):
                for h, d in up:
                    d.copy_(h, non_blocking=True)
                ph.replay()
                for h, d in down:
                    h.copy_(d, non_blocking=True)
                if record:
                    marks[k + 2].record(stream)
            stream.wait_stream(copy_stream)
        if record:
            ev.append(marks)

    for _ in range(max(1, args.warmup)):
        one(False)
    torch.cuda.synchronize()
    barrier(ws)
    for _ in range(args.steps):
        one(True)
    torch.cuda.synchronize()
    seg_ms = [0.0] * (len(segs) + 1)
    for marks in ev:
        for k in range(len(segs) + 1):
            seg_ms[k] += marks[k].elapsed_time(marks[k + 1])
    total = sum(ev[i][0].elapsed_time(ev[i][-1]) for i in range(len(ev)))
    # outputs of the last step against the device-resident graphs
    got = [h.clone() for h, _ in alpha_h] + [h.clone() for _, _, _, down in segs for h, _ in down]
    with torch.cuda.stream(stream):
        for p in wl.phases:
            p.replay()
    torch.cuda.synchronize()
    ref = [d for _, d in alpha_h] + [d for _, _, _, down in segs for _, d in down]
    for g, d in zip(got, ref):
        if not torch.equal(g, d.cpu()):
            raise RuntimeError("end-to-end step and device-resident step disagree")
    steps = args.steps
    bi = sum(h.numel() * h.element_size() for h, _ in wft_h) + \
        sum(h.numel() * h.element_size() for _, _, up, _ in segs for h, _ in up)
    bo = sum(h.numel() * h.element_size() for h, _ in alpha_h) + \
        sum(h.numel() * h.element_size() for _, _, _, down in segs for h, _ in down)
    comp_bytes = st.comp.bytes + (wl.g14.comp.bytes if wl.g14 is not None else 0.0)
    segments = {"compress": {"ms_per_step": seg_ms[0] / steps, "unit": "GB/s",
                             "value": ws * steps * comp_bytes / (max_over_ranks(ws, seg_ms[0]) * 1e-3) / 1e9,
                             "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h, _ in wft_h),
                             "d2h_bytes_per_step": sum(h.numel() * h.element_size() for h, _ in alpha_h),
                             "copies": "W_ft per matrix on a second stream, each compressed once landed"}}
    for k, (name, ph, up, down) in enumerate(segs):
        t = max_over_ranks(ws, seg_ms[k + 1])
        work = ph.bytes if ph.bound == "hbm" else ph.flops / 1e3
        segments[name] = {"ms_per_step": seg_ms[k + 1] / steps, "unit": ph.unit,
                          "value": ws * steps * work / (t * 1e-3) / 1e9,
                          "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h, _ in up),
                          "d2h_bytes_per_step": sum(h.numel() * h.element_size() for h, _ in down)}
    dec = segments["fused_linear_decode"]
    return {"value": dec["value"], "unit": "GB/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "ms_per_step": total / steps, "value_segment": "fused_linear_decode (its activations up, y back)",
            "segments": segments}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(wl, args, target_s: float = 12.0, phase=None):
    import oracle
    oracle.build()
    frac = 1.0 / 64
    kw = {"phase": phase} if phase is not None else {}
    unit = wl.metric_unit if phase is None else ("TFLOP/s" if phase == "prefill" else "GB/s")
    run, _ = wl.oracle_sample(oracle, frac, **kw)
    t0 = time.perf_counter()
    run()
    t1 = time.perf_counter() - t0
    frac = min(1.0, frac * max(1.0, target_s / max(t1, 1e-3)))
    run, desc = wl.oracle_sample(oracle, frac, **kw)
    t0 = time.perf_counter()
    nbytes = run()
    dt = time.perf_counter() - t0
    reps = 1
    if frac >= 1.0 and dt < 0.5 * target_s:
        # the whole workload is shorter than the target: repeat it to about target_s
        more = max(1, int(math.ceil(target_s / max(dt, 1e-3))) - 1)
        t0 = time.perf_counter()
        for _ in range(more):
            nbytes += run()
        dt += time.perf_counter() - t0
        reps += more
        desc = desc.replace("each matrix's first 1 of rows", "every row of every matrix") + f", {reps} passes"
    return {"value": nbytes / dt / 1e9, "unit": unit, "cores": cpu_cores(), "kind": "oracle",
            "sample": desc, "seconds": dt}


REFERENCE_BUDGET_S = 90.0


def run_reference(args, ws, rank):
    """The fp64 CPU oracle as it stands, on the host cores; rank 0 only."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    from bit_delta_tenant_gb300 import bitdelta as bd  # noqa: F401  (workload construction only)
    serving = args.workload == "llama3_8b_stack"
    # the default step's CPU arm samples its first layer, so only that layer is built
    wl = ServingWorkload(_NoLib(), dev, reference=True) if serving else WORKLOADS[args.workload](_NoLib(), dev)
    kw = {"phase": "decode"} if serving else {}
    unit = "GB/s" if serving else wl.metric_unit
    # Each step is the largest row sample (up to the whole step) that keeps the run near
    # REFERENCE_BUDGET_S: one 1/64 sample is timed first and scaled.
    frac = 1.0 / 64
    run, desc = wl.oracle_sample(oracle, frac, **kw)
    t0 = time.perf_counter()
    run()
    t_small = time.perf_counter() - t0
    budget_frac = REFERENCE_BUDGET_S / max(1, args.steps + args.warmup) / max(t_small, 1e-4) * frac
    if budget_frac > frac:
        frac = min(1.0, budget_frac)
        run, desc = wl.oracle_sample(oracle, frac, **kw)
        if frac >= 1.0:
            desc = desc.replace("each matrix's first 1 of rows", "every row of every matrix")
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    nbytes = 0.0
    for _ in range(args.steps):
        nbytes = run()
    dt = time.perf_counter() - t0
    v = args.steps * nbytes / dt / 1e9
    line = {"impl": "reference", "metric": "BitDelta fused linear GB/s (decode) & TFLOP/s (prefill), % of roofline",
            "value": v, "unit": unit, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": wl.config,
            "cpu_baseline": {"value": v, "unit": unit, "cores": cpu_cores(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    if serving:
        # the prefill half of the metric: the oracle's fused linear at m = 2048 (first 64 tokens)
        line["prefill"] = {"cpu_baseline": cpu_baseline(wl, args, target_s=8.0, phase="prefill")}
        line["prefill"]["value"] = line["prefill"]["cpu_baseline"]["value"]
        line["prefill"]["unit"] = "TFLOP/s"
    print(json.dumps(line), flush=True)


class _NoLib:
    """Stands in for the library when only the workload's inputs are needed (reference arm)."""

    def bd_compress_workspace_size(self, *a):
        return 16

    def bd_linear_grouped_workspace_size(self, *a):
        return 16

    def bd_compress_batch_workspace_size(self, *a):
        return 256

    def bd_linear_batch_workspace_size(self, *a):
        return 256

    def compress_descs(self, problems):
        return problems

    def linear_descs(self, problems):
        return problems

    def __getattr__(self, name):
        def _never(*a, **k):
            raise RuntimeError("the reference arm does not call the GPU library")
        return _never


def run_kernel_case(args):
    """One kernel on one shape, launched eagerly (no graph): for ncu captures and sweeps.

    --kernel-case linear:N_OUTxN_IN:M[:path], compress:N_OUTxN_IN[:mode],
                  batch:N_OUTxN_IN:M:COUNT (COUNT linears per bd_linear_batch call),
                  grouped:N_OUTxN_IN:M:V[:zipf] (V variants, uniform ids or Zipf(1.1) segments),
                  reconstruct:N_OUTxN_IN
                  (W_eff materialised), reconstruct_mm:N_OUTxN_IN:M (W_eff + a cuBLAS matmul) or
                  cache_load:N_OUTxN_IN (a delta's cold load through the delta cache)
    Rotates over enough copies of the weights that the working set exceeds L2.
    """
    from bit_delta_tenant_gb300 import build as lib_build
    lib_build.build()
    from bit_delta_tenant_gb300 import bitdelta as bd
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    parts = args.kernel_case.split(":")
    kind, shape = parts[0], parts[1]
    n_out, n_in = (int(v) for v in shape.split("x"))
    per = 2.0 * n_out * n_in
    count = int(parts[3]) if kind == "batch" else 1  # linears per batched call
    copies = max(1, int(np.ceil(3 * 129e6 / (per * count)))) * count
    mats = [synth.matrix_pair(n_out, n_in, 0.02, 1e-3, 50 + i, dev) for i in range(copies)] \
        if kind != "cache_load" else []
    if kind == "linear":
        m = int(parts[2])
        path = int(parts[3]) if len(parts) > 3 else 0
        bd.bd_set_linear_path(path)
        packed = []
        for wb, wf in mats:
            bits = torch.empty((n_out, n_in // 8), dtype=torch.uint8, device=dev)
            alpha = torch.empty((1,), dtype=torch.float32, device=dev)
            ws = torch.empty((max(16, bd.bd_compress_workspace_size(n_out, n_in, 0)),), dtype=torch.uint8,
                             device=dev)
            bd.bd_compress(wb, wf, 0, bits, alpha, ws)
            packed.append((bits, alpha))
        x = synth.activations(m, n_in, 7, dev)
        y = torch.empty((m, n_out), dtype=torch.bfloat16, device=dev)

        torch.cuda.synchronize()  # the compressions above are complete before any linear is queued
        bd.bd_set_weight_prefetch(1 if WEIGHT_PREFETCH else 0)  # the rotated copies are never written here

        def call(i):
            bd.bd_linear(x, mats[i][0], packed[i][0], packed[i][1], 0, y)
        work = decode_bytes(m, n_out, n_in, 0)
        flops = 2.0 * m * n_out * n_in
    elif kind == "batch":
        # COUNT linears of one shape per bd_linear_batch call (q/k/v-like); call i takes copies
        # i*COUNT .. i*COUNT+COUNT-1, so the copies rotate as for linear:...
        m = int(parts[2])
        packed = []
        for wb, wf in mats:
            bits = torch.empty((n_out, n_in // 8), dtype=torch.uint8, device=dev)
            alpha = torch.empty((1,), dtype=torch.float32, device=dev)
            ws = torch.empty((max(16, bd.bd_compress_workspace_size(n_out, n_in, 0)),), dtype=torch.uint8,
                             device=dev)
            bd.bd_compress(wb, wf, 0, bits, alpha, ws)
            packed.append((bits, alpha))
        x = synth.activations(m, n_in, 7, dev)
        ys = [torch.empty((m, n_out), dtype=torch.bfloat16, device=dev) for _ in range(count)]
        descs = [bd.linear_descs([(x, mats[c * count + j][0], packed[c * count + j][0], packed[c * count + j][1], 0,
                                   ys[j]) for j in range(count)]) for c in range(copies // count)]
        bws = torch.zeros(max(1, bd.bd_linear_batch_workspace_size(descs[0])), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        bd.bd_set_weight_prefetch(1 if WEIGHT_PREFETCH else 0)
        copies //= count

        def call(i):
            bd.bd_linear_batch(descs[i], bws)
        work = count * decode_bytes(m, n_out, n_in, 0)
        flops = count * 2.0 * m * n_out * n_in
    elif kind in ("reconstruct", "reconstruct_mm"):
        # the page's "standard matmul in decode" reading: rebuild W_eff in HBM (and,
        # for reconstruct_mm, multiply with a cuBLAS GEMM); compare with linear:...
        m = int(parts[2]) if kind == "reconstruct_mm" else 0
        packed = []
        for wb, wf in mats:
            bits = torch.empty((n_out, n_in // 8), dtype=torch.uint8, device=dev)
            alpha = torch.empty((1,), dtype=torch.float32, device=dev)
            ws = torch.empty((max(16, bd.bd_compress_workspace_size(n_out, n_in, 0)),), dtype=torch.uint8,
                             device=dev)
            bd.bd_compress(wb, wf, 0, bits, alpha, ws)
            packed.append((bits, alpha))
        torch.cuda.synchronize()
        w_eff = torch.empty((n_out, n_in), dtype=torch.bfloat16, device=dev)
        x = synth.activations(max(m, 1), n_in, 7, dev)
        y = torch.empty((max(m, 1), n_out), dtype=torch.bfloat16, device=dev)

        def call(i):
            bd.bd_reconstruct(mats[i][0], packed[i][0], packed[i][1], 0, w_eff)
            if m:
                torch.matmul(x, w_eff.t(), out=y)
        # reconstruct alone: its own traffic; with the matmul: the fused linear's algorithmic bytes
        work = decode_bytes(m, n_out, n_in, 0) if m else 4.0 * n_out * n_in + n_out * n_in / 8
        flops = 2.0 * m * n_out * n_in
    elif kind == "cache_load":
        # cold start of a variant through the delta cache: two variants alternate in
        # an arena that holds one, so every request loads its delta from pinned host memory
        bpm = n_out * n_in // 8
        hosts = [(torch.randint(0, 256, (bpm,), dtype=torch.uint8).pin_memory(),
                  torch.full((n_out,), 1e-3, dtype=torch.float32).pin_memory()) for _ in range(2)]
        block = (bpm + 255) // 256 * 256 + (4 * n_out + 255) // 256 * 256
        arena = torch.empty(block + 256, dtype=torch.uint8, device=dev)
        cache = bd.DeltaCache(2, arena, half_life_s=1.0)
        for v, (hb, ha) in enumerate(hosts):
            cache.register(v, hb, ha)
        stream = torch.cuda.Stream()
        for i in range(args.warmup + 1):
            rc, _, _ = cache.acquire(i % 2, stream=stream)
            cache.release(i % 2, stream=stream)
        torch.cuda.synchronize()
        reps = max(args.steps, 4)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(reps):
            rc, _, _ = cache.acquire(i % 2, stream=stream)
            assert rc == bd.BD_OK
            cache.release(i % 2, stream=stream)
        t1.record(stream)
        t1.synchronize()
        sec = t0.elapsed_time(t1) * 1e-3 / reps
        nbytes = bpm + 4 * n_out
        st = cache.stats()
        cache.close()
        print(json.dumps({"kernel_case": args.kernel_case, "load_us": sec * 1e6, "h2d_GB/s": nbytes / sec / 1e9,
                          "loads": st.loads, "evictions": st.evictions,
                          "cold_start_70b_variant_ms": 70e9 / 8 / (nbytes / sec) * 1e3}), flush=True)
        return
    elif kind == "grouped":
        m, nv = int(parts[2]), int(parts[3])
        bd.bd_set_weight_prefetch(0)
        packed = []
        for i, (wb, wf) in enumerate(mats):
            vs = []
            for v in range(nv):
                g = synth.generator(900 + 31 * i + v, dev)
                bits = torch.randint(0, 256, (n_out, n_in // 8), generator=g, device=dev, dtype=torch.uint8)
                vs.append((bits, torch.full((1,), 1e-3, dtype=torch.float32, device=dev)))
            packed.append(vs)
        zipf = len(parts) > 4 and parts[4] == "zipf"  # Zipf(1.1) segments (the 14-variant prefill batch's mix)
        ids = torch.from_numpy(synth.zipf_ids(m, nv, 1.1, 3) if zipf else synth.uniform_ids(m, nv, 3)).to(dev)
        x = synth.activations(m, n_in, 7, dev)
        y = torch.empty((m, n_out), dtype=torch.bfloat16, device=dev)
        gws = torch.empty((bd.bd_linear_grouped_workspace_size(m, nv, n_out, n_in),), dtype=torch.uint8, device=dev)

        def call(i):
            bd.bd_linear_grouped(x, ids, mats[i][0], [b for b, _ in packed[i]], [a for _, a in packed[i]],
                                 [0] * nv, y, gws)
        active = len(set(ids.tolist()))
        work = 2.0 * n_out * n_in + active * n_out * n_in / 8 + 4.0 * nv + 2.0 * m * n_in + 2.0 * m * n_out
        flops = 2.0 * m * n_out * n_in
    else:
        mode = int(parts[2]) if len(parts) > 2 else 0
        bits = torch.empty((n_out, n_in // 8), dtype=torch.uint8, device=dev)
        alpha = torch.empty((n_out if mode else 1,), dtype=torch.float32, device=dev)
        ws = torch.empty((max(16, bd.bd_compress_workspace_size(n_out, n_in, mode)),), dtype=torch.uint8,
                         device=dev)

        def call(i):
            bd.bd_compress(mats[i][0], mats[i][1], mode, bits, alpha, ws)
        work = 4.0 * n_out * n_in + n_out * n_in / 8
        flops = 0.0
    for i in range(args.warmup):
        call(i % copies)
    torch.cuda.synchronize()
    # eager launches (what ncu captures), then the same launches replayed from a graph
    # so that per-launch times exclude host launch overhead
    stream = torch.cuda.Stream()
    reps = max(args.steps, copies)
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            call(k % copies)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for k in range(reps):
            call(k % copies)
    times = []
    with torch.cuda.stream(stream):
        for _ in range(3):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            g.replay()
            s1.record(stream)
            s1.synchronize()
            times.append(s0.elapsed_time(s1) * 1e-3 / reps)
    med = sorted(times)[1]
    assert bd.bd_get_device_status() == bd.BD_OK
    print(json.dumps({"kernel_case": args.kernel_case, "copies": copies, "launches_timed": reps,
                      "us_per_launch": med * 1e6, "GB/s": work / med / 1e9, "TFLOP/s": flops / med / 1e12,
                      "weight_prefetch": WEIGHT_PREFETCH,
                      "env": {k: v for k, v in os.environ.items() if k.startswith("BD_")}}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama3_8b_stack")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--weight-prefetch", type=int, choices=[0, 1], default=1,
                    help="capture the device-resident fused linears with bd_set_weight_prefetch(1)")
    ap.add_argument("--linear-batch", choices=["auto", "none", "qkv", "layer"], default="auto",
                    help="layer: q/k/v and gate/up of a layer in one bd_linear_batch call each; qkv: q/k/v only; "
                         "auto: the workload's own choice")
    ap.add_argument("--compress-batch", type=int, choices=[0, 1], default=1,
                    help="compress through bd_compress_batch (8 matrices per call) or one bd_compress each")
    ap.add_argument("--kernel-case", default=None,
                    help="linear:N_OUTxN_IN:M[:path] or compress:N_OUTxN_IN[:mode] (one kernel, eager)")
    ap.add_argument("--ingest-traffic", default=None,
                    help="ncu --csv capture (dram__bytes_read.sum, dram__bytes_write.sum) to store as the "
                         "traffic of --phase of --workload in profiles/traffic_<workload>.json")
    ap.add_argument("--phase", default="fused_linear_decode")
    ap.add_argument("--ingest-command", default=None, help="the command line of that capture, stored beside it")
    args = ap.parse_args()
    if args.ingest_traffic:
        ingest_traffic(args)
        return
    global WEIGHT_PREFETCH, LINEAR_BATCH, COMPRESS_BATCH
    WEIGHT_PREFETCH = bool(args.weight_prefetch)
    LINEAR_BATCH = args.linear_batch
    COMPRESS_BATCH = bool(args.compress_batch)
    if args.kernel_case:
        run_kernel_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_setup() if args.impl == "ours" else (int(os.environ.get("WORLD_SIZE", "1")),
                                                                 int(os.environ.get("RANK", "0")), 0)
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
