#!/usr/bin/env python3
"""Benchmark of the multi-head scaled dot-product attention hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
for the multi-head workloads that is mha_forward (Q/K/V projections, masked
attention per head, output projection); for the attention-only workloads it
is attn_forward. The metric is attention TFLOP/s counted as
4*B*h*n_q*n_k*d_k (halved for causal) per attention call, over the step time.

Timing: W untimed warm-up steps, then exactly K steps between two CUDA
events on the launching stream, bracketed by a barrier and a device
synchronize; that K-step loop is repeated until at least --min-seconds of
wall time have passed, and the step time is the median over the repeats;
rotating input sets whose total exceeds L2 keep the working set out of
cache; nvidia-smi samples the clocks during the whole timed region. The
dominant kernel's duration is measured in a second event-timed loop where
each kernel is launched through its own entry point, and is compared with
its roofline (MEASURED_PEAKS.json). The CPU baseline is the fp64 oracle on a
bounded sample of the same workload. `--impl reference` times that oracle as
the reference arm.

Multi-GPU: the path has no exchange step; N ranks run N independent replicas
(one GPU each, weak scaling) and only the timing is reduced.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synthetic  # noqa: E402
from synthetic import MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE  # noqa: E402

METRIC = "attention TFLOP/s (bf16) and % of dense BF16 peak / % of HBM BW, 1 GB300"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# --------------------------------------------------------------------------- workloads

WORKLOADS = {
    "base_encoder_mha": dict(
        kind="mha", calls=[dict(B=32, n_q=128, n_k=128, d_model=512, h=8, d=64,
                                mask=MASK_KEY_PADDING, kv_range=(64, 128), add_pe=True,
                                self_attention=True, seed=1001)],
        desc="Transformer-base encoder self-attention MHA: B=32, n=128, d_model=512, h=8, "
             "d_k=d_v=64, key padding kv_len~U[64,128], x~N(0,1)+PE, Xavier-uniform W"),
    "base_decoder_mha": dict(
        kind="mha", calls=[
            dict(B=32, n_q=128, n_k=128, d_model=512, h=8, d=64, mask=MASK_CAUSAL | MASK_KEY_PADDING,
                 kv_range=(64, 128), add_pe=False, self_attention=True, seed=1002),
            dict(B=32, n_q=128, n_k=160, d_model=512, h=8, d=64, mask=MASK_KEY_PADDING,
                 kv_range=(80, 160), add_pe=False, self_attention=False, seed=1012)],
        desc="Transformer-base decoder: masked self-attention MHA (n=128, causal + target "
             "padding U[64,128]) then cross-attention MHA (n_q=128, n_k=160, source padding "
             "U[80,160]); d_model=512, h=8, d_k=64, B=32, N(0,1) activations"),
    "big_self": dict(kind="attn", B=8, h=16, n=1024, d=64, causal=False, seed=1003,
                     desc="Transformer-big self-attention: B=8, h=16, n=1024, d_k=d_v=64"),
    "big_self_causal": dict(kind="attn", B=8, h=16, n=1024, d=64, causal=True, seed=1003,
                            desc="Transformer-big causal self-attention: B=8, h=16, n=1024, d=64"),
    "base_encoder_attn": dict(
        kind="attn", B=32, h=8, n=128, d=64, causal=False, padding=True, kv_range=(64, 128),
        seed=1001,
        desc="Transformer-base encoder self-attention alone (attn_forward, no projections): "
             "B=32, h=8, n=128, d_k=d_v=64, key padding kv_len~U[64,128]; bytes counted with K/V "
             "to kv_len"),
    "base_cross_attn": dict(
        kind="attn", B=32, h=8, n=128, n_k=160, d=64, causal=False, padding=True,
        kv_range=(80, 160), seed=1012,
        desc="Transformer-base decoder cross-attention alone (attn_forward): B=32, h=8, n_q=128, "
             "n_k=160, d_k=d_v=64, source padding kv_len~U[80,160]; bytes counted with K/V to "
             "kv_len"),
    "long": dict(kind="attn", B=4, h=16, n=4096, d=64, causal=False, seed=1004,
                 desc="long-context self-attention with Transformer-big heads: B=4, h=16, "
                      "n=4096, d_k=d_v=64, non-causal, Q/K/V~N(0,1) (the O(n^2 d) row of "
                      "Table 1; --B/--n/--d/--causal select the other sweep points)"),
    "long_causal": dict(kind="attn", B=4, h=16, n=4096, d=64, causal=True, seed=1004,
                        desc="long-context decoder (causal) self-attention with Transformer-big "
                             "heads: B=4, h=16, n=4096, d_k=d_v=64, Q/K/V~N(0,1); TFLOP/s over "
                             "the causal half of 4 B h n^2 d"),
    "base_encoder_layer": dict(
        kind="encoder", B=32, n=128, d_model=512, h=8, d_ff=2048, mask=MASK_KEY_PADDING,
        kv_range=(64, 128), eps=1e-6, seed=1007,
        desc="Transformer-base encoder layer, post-LN: LayerNorm(y + FFN(y)), y = LayerNorm(x "
             "+ MultiHead(x)); B=32, n=128, d_model=512, h=8, d_ff=2048, key padding U[64,128]; "
             "TFLOP/s over all of the layer's matrix FLOPs (projections, attention, FFN)"),
    "decode": dict(kind="decode", B=16, h=16, n_q=1, n_max=8192, d=64, len_range=(4096, 8192),
                   seed=1006,
                   desc="one decoding step against a key/value cache: B=16, h=16, d=64, one new "
                        "token per sequence, cache lengths U[4096, 8192] of 8192 rows; TFLOP/s "
                        "counted over the visible (query, key) pairs, the cache read from HBM"),
    "window": dict(kind="attn", B=4, h=16, n=16384, d=64, causal=False, window=(256, 256),
                   seed=1005,
                   desc="restricted self-attention (Table 1, restricted row): B=4, h=16, n=16384, "
                        "d=64, each query sees the keys within 256 positions of it; TFLOP/s "
                        "counted over the allowed (query, key) pairs"),
}


def attn_flops(B, h, n_q, n_k, d, causal):
    f = 4.0 * B * h * n_q * n_k * d
    return f / 2 if causal else f


def window_pairs(n, left, right, causal):
    """(query, key) pairs of a restricted window over n positions: query i
    sees keys [i - left, i + right] (a negative bound is none), and only j <= i
    when causal."""
    i = np.arange(n, dtype=np.int64)
    lo = np.maximum(0, i - left) if left >= 0 else np.zeros_like(i)
    hi = np.minimum(n - 1, i + right) if right >= 0 else np.full_like(i, n - 1)
    if causal:
        hi = np.minimum(hi, i)
    return int(np.maximum(hi - lo + 1, 0).sum())


# --------------------------------------------------------------------------- helpers

def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha(rels):
    """sha256 of one source file, or of several concatenated in order."""
    h = hashlib.sha256()
    for rel in ((rels,) if isinstance(rels, str) else rels):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


_CSRC = "transformer_scaled_dot_gb300/csrc/"
KERNEL_SOURCES = {
    "attn_fwd_bf16": _CSRC + "attn_bf16.cu",
    "gemm_bf16": _CSRC + "gemm_bf16.cu",
    "mha_fused": _CSRC + "mha_fused.cu",
    "mha_cross": _CSRC + "mha_cross.cu",
    "attn_decode": _CSRC + "attn_decode.cu",
    # the encoder layer's five launches: fused MHA, two LayerNorms, two GEMMs
    "encoder_layer": (_CSRC + "mha_fused.cu", _CSRC + "layernorm.cu", _CSRC + "gemm_bf16.cu"),
}


# the public call the end-to-end leg times, per workload kind
E2E_API = {
    "mha": "mha_forward_host_async + attn_host_join (pinned host x, lengths and result; "
           "weights resident; two staging workspaces in turn; each result copy overlaps the "
           "next call, all joined before the closing event)",
    "attn": "attn_forward_host / attn_forward_window_host (pinned host Q, K, V and O; "
            "two staging workspaces in turn)",
    "encoder": "encoder_layer_forward_host_async + attn_host_join (pinned host x, lengths and "
               "result; parameters resident; two staging workspaces in turn; each result copy "
               "overlaps the next layer, all joined before the closing event)",
    "decode": "attn_decode_host_async + attn_host_join (pinned host queries, cache lengths "
              "and result; caches resident; two staging workspaces in turn; each result copy "
              "overlaps the next step, all joined before the closing event)",
}


def spec_kind(workload):
    return WORKLOADS[workload]["kind"] if workload in WORKLOADS else "attn"


def config_overridden(args):
    """True when --B/--n/--d/--h/--causal change the named workload's shape: its
    committed ncu summary then describes another launch."""
    spec = WORKLOADS.get(args.workload, {})
    for k in ("B", "n", "d", "h"):
        v = getattr(args, k, None)
        if v and v != spec.get(k):
            return True
    return args.causal is not None and bool(args.causal) != bool(spec.get("causal", False))


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, or None when there is
    none for this kernel and workload, or the kernel source changed since."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir) or kernel not in KERNEL_SOURCES:
        return None
    sha = source_sha(KERNEL_SOURCES[kernel])
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".txt", ".md")):
            continue
        fields = {}
        with open(os.path.join(pdir, fn), encoding="utf-8") as f:
            for line in f:
                if ":" in line and line.strip().startswith(("kernel", "workload", "source_sha256",
                                                            "dram_bytes_per_launch")):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if (fields.get("kernel") == kernel and fields.get("workload") == workload
                and fields.get("source_sha256") == sha and "dram_bytes_per_launch" in fields):
            try:
                return float(fields["dram_bytes_per_launch"])
            except ValueError:
                return None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid.lower()
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5:  # wait for the first sample
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t_start, t_end):
        rows = []
        gpus = set()
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            gpus.add(parts[0].lower())
            rows.append((t, parts))
        if self.uuid and any(g.endswith(self.uuid) for g in gpus):
            rows = [r for r in rows if r[1][0].lower().endswith(self.uuid)]
        elif len(gpus) > 1:
            rows = []
        inside = [r for r in rows if t_start <= r[0] <= t_end]
        if not inside and rows:  # region shorter than the sampling period: nearest samples
            inside = sorted(rows, key=lambda r: min(abs(r[0] - t_start), abs(r[0] - t_end)))[:2]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(p[1]) for _, p in inside if p[1].replace(".", "").isdigit()]
        smax = [float(p[2]) for _, p in inside if p[2].replace(".", "").isdigit()]
        reasons = set()
        for _, p in inside:
            for name, val in zip(self.REASONS, p[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        pw = [float(p[3]) for _, p in inside if p[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "power_w_max": max(pw) if pw else None}


# --------------------------------------------------------------------------- distributed

def dist_setup():
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local = _env_int("LOCAL_RANK", 0)
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("TSD_BENCH_BACKEND", "nccl")
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(x: float, world: int) -> float:
    """Maximum of a per-rank scalar over all ranks (host logic; any backend)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_sum(x: float, world: int) -> float:
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------- GPU arm

class MhaCall:
    """Device buffers of one mha_forward call, replicated over rotating sets."""

    def __init__(self, tsd, cfg, nsets, seed_offset):
        import torch
        self.tsd, self.cfg = tsd, cfg
        c = cfg
        self.m = synthetic.mha_inputs(c["seed"] + seed_offset, c["B"], c["n_q"], c["n_k"],
                                      c["d_model"], c["h"], c["d"], c["d"], c["mask"],
                                      c["kv_range"], add_pe=c["add_pe"],
                                      self_attention=c["self_attention"])
        m = self.m
        dev = "cuda"
        bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        host = [m.x_q] + ([] if m.self_attention else [m.x_kv]) + [m.w_q, m.w_k, m.w_v, m.w_o]
        self.wsb = tsd.mha_workspace_bytes(m.B, m.n_q, m.n_k, m.h, m.d_k, m.d_v)
        self.sets = []
        for _ in range(nsets):
            t = [bf(a) for a in host]
            x_q = t[0]
            x_kv = x_q if m.self_attention else t[1]
            w = t[-4:]
            s = dict(x_q=x_q, x_kv=x_kv, w=w,
                     lens=torch.from_numpy(m.kv_lens).to(dev) if m.kv_lens is not None else None,
                     out=torch.empty((m.B, m.n_q, m.d_model), dtype=torch.bfloat16, device=dev),
                     ws=torch.empty(self.wsb, dtype=torch.uint8, device=dev))
            self.sets.append(s)
        hdk, hdv = m.h * m.d_k, m.h * m.d_v
        # workspace regions (the layout mha_workspace_bytes describes)
        al = lambda x: (x + 255) // 256 * 256
        self.q_off = 0
        self.k_off = al(m.B * m.n_q * hdk * 2)
        self.v_off = self.k_off + al(m.B * m.n_k * hdk * 2)
        self.o_off = self.v_off + al(m.B * m.n_k * hdv * 2)
        # host copies for the end-to-end leg (pinned)
        self.h_x_q = torch.from_numpy(np.ascontiguousarray(m.x_q).view(np.int16)).pin_memory()
        self.h_x_kv = None if m.self_attention else \
            torch.from_numpy(np.ascontiguousarray(m.x_kv).view(np.int16)).pin_memory()
        self.h_lens = torch.from_numpy(m.kv_lens).pin_memory() if m.kv_lens is not None else None
        self.h_out = torch.empty((m.B, m.n_q, m.d_model), dtype=torch.bfloat16).pin_memory()
        self.h_ws = None

    def host_workspaces(self):
        """Two staging workspaces of mha_forward_host, taken in turn by the
        end-to-end leg (allocated on first use)."""
        import torch
        if self.h_ws is None:
            m = self.m
            self.h_wsb = self.tsd.mha_host_workspace_bytes(m.B, m.n_q, m.n_k, m.d_model, m.h,
                                                           m.d_k, m.d_v)
            self.h_ws = [torch.empty(self.h_wsb, dtype=torch.uint8, device="cuda")
                         for _ in range(2)]
        return self.h_ws

    def bytes_per_set(self):
        m = self.m
        n = m.x_q.nbytes + (0 if m.self_attention else m.x_kv.nbytes)
        n += m.w_q.nbytes + m.w_k.nbytes + m.w_v.nbytes + m.w_o.nbytes
        return n + self.wsb + m.B * m.n_q * m.d_model * 2

    def run(self, i, stream):
        m, s = self.m, self.sets[i % len(self.sets)]
        self.tsd.mha_forward(s["x_q"], s["x_kv"], *s["w"], s["out"], m.B, m.n_q, m.n_k, m.d_model,
                             m.h, m.d_k, m.d_v, m.mask_kind, s["lens"], 0.0, s["ws"], self.wsb,
                             stream)

    def n_launches(self):
        """Kernels mha_forward launches for this shape, as the library plans
        them: 1 (projections, attention and W_O in one kernel), 2 (that kernel
        up to the merged heads, then the W_O GEMM) or 3 (QKV GEMM, attention,
        W_O GEMM)."""
        if not hasattr(self, "_n_launches"):
            m = self.m
            self._n_launches = self.tsd.mha_forward_launches(m.B, m.n_q, m.n_k, m.d_model, m.h,
                                                             m.d_k, m.d_v, m.self_attention)
            if self._n_launches not in (1, 2, 3):
                raise RuntimeError(f"mha_forward_launches -> {self._n_launches}")
        return self._n_launches

    def fused(self):
        return self.n_launches() < 3

    def run_stage(self, k, i, stream):
        """Launch k of the step's launches through its own entry point, on
        input set i."""
        m, s = self.m, self.sets[i % len(self.sets)]
        base = s["ws"].data_ptr()
        Q, K, V, O = base + self.q_off, base + self.k_off, base + self.v_off, base + self.o_off
        hdk, hdv = m.h * m.d_k, m.h * m.d_v
        if self.n_launches() == 1:
            self.run(i, stream)
            return
        if self.fused():
            if k == 0:
                self.tsd.mha_concat_heads(s["x_q"], s["x_kv"], *s["w"][:3], O, m.B, m.n_q, m.n_k,
                                          m.d_model, m.h, m.d_k, m.d_v, m.mask_kind, s["lens"],
                                          0.0, s["ws"], self.wsb, stream)
            else:
                self.tsd.mha_project_out(O, s["w"][3], s["out"], m.B, m.n_q, m.d_model, m.h,
                                         m.d_v, stream)
            return
        if k == 0:
            self.tsd.mha_project_qkv(s["x_q"], s["x_kv"], *s["w"][:3], Q, K, V, m.B, m.n_q, m.n_k,
                                     m.d_model, m.h, m.d_k, m.d_v, stream)
        elif k == 1:
            self.tsd.attn_forward_strided(Q, m.n_q * hdk, m.d_k, hdk, K, m.n_k * hdk, m.d_k, hdk,
                                          V, m.n_k * hdv, m.d_v, hdv, O, m.n_q * hdv, m.d_v, hdv,
                                          m.B, m.h, m.n_q, m.n_k, m.d_k, m.d_v, m.mask_kind,
                                          s["lens"], 0.0, stream)
        else:
            self.tsd.mha_project_out(O, s["w"][3], s["out"], m.B, m.n_q, m.d_model, m.h, m.d_v,
                                     stream)

    def stage_names(self):
        m = self.m
        # cross-attention over one or two source key tiles has its own kernel
        fused = "mha_cross" if (not m.self_attention and m.n_k > 128) else "mha_fused"
        if self.n_launches() == 1:
            return [fused]
        if self.fused():
            return [fused, "gemm_bf16"]
        return ["gemm_bf16", "attn_fwd_bf16", "gemm_bf16"]

    def stage_work(self):
        """(algorithmic flops, algorithmic bytes) of each stage launch."""
        m = self.m
        dm, hdk, hdv = m.d_model, m.h * m.d_k, m.h * m.d_v
        Mq, Mk = m.B * m.n_q, m.B * m.n_k
        qkv_f = 2.0 * dm * (Mq * hdk + Mk * hdk + Mk * hdv)
        x_b = 2.0 * (Mq * dm + (0 if m.self_attention else Mk * dm))
        w_b = 2.0 * dm * (2 * hdk + hdv)
        qkv_b = x_b + w_b + 2.0 * (Mq * hdk + Mk * (hdk + hdv))
        kv = self.kv_effective()
        causal = bool(m.mask_kind & MASK_CAUSAL)
        att_f = attn_flops(m.B, m.h, m.n_q, m.n_k, m.d_k, causal)
        att_b = 2.0 * m.h * sum(m.n_q * m.d_k + kv[b] * (m.d_k + m.d_v) + m.n_q * m.d_v
                                for b in range(m.B))
        out_f = 2.0 * Mq * hdv * dm
        out_b = 2.0 * (Mq * hdv + hdv * dm + Mq * dm)
        if self.n_launches() == 1:
            # X, the four weights and out cross HBM; Q/K/V and the merged
            # heads stay on chip or in L2
            return [(qkv_f + att_f + out_f, x_b + w_b + 2.0 * (hdv * dm + Mq * dm))]
        if self.fused():
            # X, the weights and the merged heads cross HBM; Q/K/V stay on chip
            return [(qkv_f + att_f, x_b + w_b + 2.0 * Mq * hdv), (out_f, out_b)]
        return [(qkv_f, qkv_b), (att_f, att_b), (out_f, out_b)]

    def kv_effective(self):
        m = self.m
        if m.kv_lens is None:
            return [m.n_k] * m.B
        return [int(min(max(x, 0), m.n_k)) for x in m.kv_lens]

    def metric_flops(self):
        m = self.m
        return attn_flops(m.B, m.h, m.n_q, m.n_k, m.d_k, bool(m.mask_kind & MASK_CAUSAL))

    def useful_flops(self):
        """4 d per (query, key) pair the masks allow (key padding, causal)."""
        m = self.m
        causal = bool(m.mask_kind & MASK_CAUSAL)
        pairs = 0
        for L in self.kv_effective():
            if causal:  # query i sees keys j <= i, j < L
                pairs += sum(min(i + 1, L) for i in range(m.n_q))
            else:
                pairs += m.n_q * L
        return 4.0 * m.h * m.d_k * pairs

    def launches(self):
        return len(self.stage_names())

    def e2e_run(self, i, stream):
        """mha_forward_host_async: pinned host x (and lengths) in, pinned host
        result out (its copy overlapping the next call), the weights resident
        on the device; e2e_finish joins the result copies."""
        m, s = self.m, self.sets[0]
        ws = self.host_workspaces()[i % 2]
        hx = self.h_x_q
        self.tsd.mha_forward_host_async(hx, hx if self.h_x_kv is None else self.h_x_kv, *s["w"],
                                        self.h_out, m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k,
                                        m.d_v, m.mask_kind, self.h_lens, 0.0, ws, self.h_wsb,
                                        stream)

    def e2e_finish(self, stream):
        self.tsd.attn_host_join(stream)

    def e2e_bytes(self):
        m = self.m
        h2d = m.x_q.nbytes + (0 if m.self_attention else m.x_kv.nbytes)
        h2d += 0 if m.kv_lens is None else m.kv_lens.nbytes
        return h2d, m.B * m.n_q * m.d_model * 2


class AttnCall:
    """Device buffers of one attn_forward call over rotating sets."""

    def __init__(self, tsd, cfg, nsets, seed_offset):
        import torch
        self.tsd, self.cfg = tsd, cfg
        c = cfg
        mask = (MASK_CAUSAL if c["causal"] else MASK_NONE) | \
            (MASK_KEY_PADDING if c.get("padding") else MASK_NONE)
        self.a = synthetic.attention_inputs(c["seed"] + seed_offset, c["B"], c["h"], c["n"],
                                            c.get("n_k", c["n"]), c["d"], c["d"], mask,
                                            c.get("kv_range"))
        a = self.a
        bf = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to("cuda").view(torch.bfloat16)
        self.sets = []
        for i in range(nsets):
            q, k, v = (bf(x) for x in (a.q, a.k, a.v))
            lens = torch.from_numpy(a.kv_lens).to("cuda") if a.kv_lens is not None else None
            self.sets.append(dict(q=q, k=k, v=v, lens=lens, out=torch.empty_like(q)))
        self.h_qkv = [torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
                      for x in (a.q, a.k, a.v)]
        self.h_lens = torch.from_numpy(a.kv_lens).pin_memory() if a.kv_lens is not None else None
        self.h_out = torch.empty(a.q.shape, dtype=torch.bfloat16).pin_memory()
        self.window = cfg.get("window")
        self.h_ws = None

    def bytes_per_set(self):
        return 2 * self.a.q.nbytes + self.a.k.nbytes + self.a.v.nbytes

    def kv_effective(self):
        a = self.a
        if a.kv_lens is None:
            return [a.n_k] * a.B
        return [int(min(max(x, 0), a.n_k)) for x in a.kv_lens]

    def run(self, i, stream):
        a, s = self.a, self.sets[i % len(self.sets)]
        if self.window is not None:
            self.tsd.attn_forward_window(s["q"], s["k"], s["v"], s["out"], a.B, a.h, a.n_q, a.n_k,
                                         a.d_k, a.d_v, self.window[0], self.window[1],
                                         a.mask_kind, None, 0.0, stream)
            return
        self.tsd.attn_forward(s["q"], s["k"], s["v"], s["out"], a.B, a.h, a.n_q, a.n_k, a.d_k,
                              a.d_v, a.mask_kind, s["lens"], 0.0, stream)

    def run_stage(self, k, i, stream):
        self.run(i, stream)

    def stage_names(self):
        return ["attn_fwd_bf16"]

    def stage_work(self):
        a = self.a
        causal = bool(a.mask_kind & MASK_CAUSAL)
        if self.window is not None:  # useful FLOPs: the allowed pairs only
            f = 4.0 * a.B * a.h * a.d_k * window_pairs(a.n_q, *self.window, causal)
        else:
            f = attn_flops(a.B, a.h, a.n_q, a.n_k, a.d_k, causal)
        # K/V bytes to each sequence's key length (key tiles past it are never loaded)
        b = 2.0 * a.h * sum(a.n_q * a.d_k + kv * (a.d_k + a.d_v) + a.n_q * a.d_v
                            for kv in self.kv_effective())
        return [(f, b)]

    def metric_flops(self):
        return self.stage_work()[0][0]

    def useful_flops(self):
        a = self.a
        if a.kv_lens is None:
            return self.metric_flops()
        return 4.0 * a.h * a.d_k * a.n_q * sum(self.kv_effective())

    def launches(self):
        return 1

    def e2e_run(self, i, stream):
        """attn_forward_host (attn_forward_window_host): pinned host Q, K, V in,
        pinned host O out, two staging workspaces in turn."""
        import torch
        a = self.a
        if self.h_ws is None:
            self.h_wsb = self.tsd.attn_host_workspace_bytes(a.B, a.h, a.n_q, a.n_k, a.d_k, a.d_v)
            self.h_ws = [torch.empty(self.h_wsb, dtype=torch.uint8, device="cuda")
                         for _ in range(2)]
        ws = self.h_ws[i % 2]
        if self.window is not None:
            self.tsd.attn_forward_window_host(*self.h_qkv, self.h_out, a.B, a.h, a.n_q, a.n_k,
                                              a.d_k, a.d_v, self.window[0], self.window[1],
                                              a.mask_kind, None, 0.0, ws, self.h_wsb, stream)
            return
        self.tsd.attn_forward_host(*self.h_qkv, self.h_out, a.B, a.h, a.n_q, a.n_k, a.d_k, a.d_v,
                                   a.mask_kind, self.h_lens, 0.0, ws, self.h_wsb, stream)

    def e2e_finish(self, stream):
        pass  # results copied on `stream`

    def e2e_bytes(self):
        a = self.a
        lens = 0 if a.kv_lens is None else a.kv_lens.nbytes
        return a.q.nbytes + a.k.nbytes + a.v.nbytes + lens, a.q.nbytes


class EncoderCall:
    """Device buffers of one encoder_layer_forward call over rotating sets."""

    def __init__(self, tsd, cfg, nsets, seed_offset):
        import torch
        self.tsd, self.cfg = tsd, cfg
        c = cfg
        e = synthetic.encoder_inputs(c["seed"] + seed_offset, c["B"], c["n"], c["d_model"], c["h"],
                                     c["d_ff"], c["mask"], c["kv_range"], add_pe=True)
        self.e = e
        m = e.mha
        bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to("cuda").view(torch.bfloat16)
        host = [m.x_q, m.w_q, m.w_k, m.w_v, m.w_o, e.ln1_gamma, e.ln1_beta, e.w_1, e.b_1, e.w_2,
                e.b_2, e.ln2_gamma, e.ln2_beta]
        self.wsb = tsd.encoder_layer_workspace_bytes(m.B, m.n_q, m.d_model, m.h, m.d_k, e.d_ff)
        self.sets = []
        for _ in range(nsets):
            self.sets.append(dict(t=[bf(a) for a in host],
                                  lens=torch.from_numpy(m.kv_lens).to("cuda"),
                                  out=torch.empty((m.B, m.n_q, m.d_model), dtype=torch.bfloat16,
                                                  device="cuda"),
                                  ws=torch.empty(self.wsb, dtype=torch.uint8, device="cuda")))
        self.h_x = torch.from_numpy(np.ascontiguousarray(m.x_q).view(np.int16)).pin_memory()
        self.h_lens = torch.from_numpy(m.kv_lens).pin_memory()
        self.h_out = torch.empty((m.B, m.n_q, m.d_model), dtype=torch.bfloat16).pin_memory()
        self.h_ws = None

    @staticmethod
    def set_bytes(cfg):
        B, n, dm, ff = cfg["B"], cfg["n"], cfg["d_model"], cfg["d_ff"]
        return 2 * (2 * B * n * dm + 4 * dm * dm + 2 * dm * ff) + B * n * (6 * dm + 2 * ff) * 2

    def run(self, i, stream):
        m, e, s = self.e.mha, self.e, self.sets[i % len(self.sets)]
        self.tsd.encoder_layer_forward(*s["t"], s["out"], m.B, m.n_q, m.d_model, m.h, m.d_k,
                                       e.d_ff, m.mask_kind, s["lens"], 0.0, self.cfg["eps"],
                                       s["ws"], self.wsb, stream)

    def run_stage(self, k, i, stream):
        self.run(i, stream)

    def stage_names(self):
        return ["encoder_layer"]

    def stage_work(self):
        m, e = self.e.mha, self.e
        rows = m.B * m.n_q
        f = 2.0 * rows * m.d_model * (4 * m.h * m.d_k) + 4.0 * rows * m.d_model * e.d_ff
        f += attn_flops(m.B, m.h, m.n_q, m.n_k, m.d_k, False)
        b = 2.0 * (2 * rows * m.d_model + 4 * m.d_model * m.h * m.d_k + 2 * m.d_model * e.d_ff)
        return [(f, b)]

    def metric_flops(self):
        return self.stage_work()[0][0]

    def useful_flops(self):
        return self.metric_flops()

    def launches(self):
        m = self.e.mha
        return self.tsd.mha_forward_launches(m.B, m.n_q, m.n_k, m.d_model, m.h, m.d_k, m.d_v,
                                             True) + 4

    def e2e_run(self, i, stream):
        """encoder_layer_forward_host_async: pinned host x and lengths in, pinned
        host output out, the layer's parameters resident on the device;
        e2e_finish joins the result copies."""
        import torch
        m, e, s = self.e.mha, self.e, self.sets[0]
        if self.h_ws is None:
            self.h_wsb = self.tsd.encoder_layer_host_workspace_bytes(m.B, m.n_q, m.d_model, m.h,
                                                                     m.d_k, e.d_ff)
            self.h_ws = [torch.empty(self.h_wsb, dtype=torch.uint8, device="cuda")
                         for _ in range(2)]
        self.tsd.encoder_layer_forward_host_async(self.h_x, *s["t"][1:], self.h_out, m.B, m.n_q,
                                                  m.d_model, m.h, m.d_k, e.d_ff, m.mask_kind,
                                                  self.h_lens, 0.0, self.cfg["eps"],
                                                  self.h_ws[i % 2], self.h_wsb, stream)

    def e2e_finish(self, stream):
        self.tsd.attn_host_join(stream)

    def e2e_bytes(self):
        m = self.e.mha
        return m.x_q.nbytes + m.kv_lens.nbytes, m.B * m.n_q * m.d_model * 2


class DecodeCall:
    """Device buffers of one attn_decode call (queries, the cache, lengths,
    workspace) over rotating sets."""

    def __init__(self, tsd, cfg, nsets, seed_offset):
        import torch
        self.tsd, self.cfg = tsd, cfg
        c = cfg
        B, h, n_q, n_max, d = c["B"], c["h"], c["n_q"], c["n_max"], c["d"]
        self.shape = (B, h, n_q, n_max, d)
        rng = np.random.default_rng(c["seed"] + seed_offset)
        self.lens = synthetic.uniform_lengths(rng, B, *c["len_range"])
        a = synthetic.attention_inputs(c["seed"] + seed_offset, B, h, n_q, n_max, d, d)
        self.a = a
        bf = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to("cuda").view(torch.bfloat16)
        self.wsb = tsd.attn_decode_workspace_bytes(B, h, n_q, n_max, d)
        self.sets = []
        for _ in range(nsets):
            self.sets.append(dict(q=bf(a.q), k=bf(a.k), v=bf(a.v),
                                  lens=torch.from_numpy(self.lens).to("cuda"),
                                  out=torch.empty((B, h, n_q, d), dtype=torch.bfloat16, device="cuda"),
                                  ws=torch.empty(self.wsb, dtype=torch.uint8, device="cuda")))
        self.h_q = torch.from_numpy(np.ascontiguousarray(a.q).view(np.int16)).pin_memory()
        self.h_lens = torch.from_numpy(self.lens).pin_memory()
        self.h_out = torch.empty((B, h, n_q, d), dtype=torch.bfloat16).pin_memory()
        self.h_ws = None

    @staticmethod
    def set_bytes(cfg):
        return 2 * cfg["B"] * cfg["h"] * cfg["n_max"] * cfg["d"] * 2

    def run(self, i, stream):
        B, h, n_q, n_max, d = self.shape
        s = self.sets[i % len(self.sets)]
        self.tsd.attn_decode(s["q"], s["k"], s["v"], s["out"], B, h, n_q, n_max, d, d, s["lens"],
                             0.0, s["ws"], self.wsb, stream)

    def run_stage(self, k, i, stream):
        self.run(i, stream)

    def stage_names(self):
        return ["attn_decode"]

    def visible_pairs(self):
        B, h, n_q, n_max, d = self.shape
        n = 0
        for L in self.lens:
            L = int(min(max(L, 0), n_max))
            n += sum(max(0, min(L, L - n_q + t + 1)) for t in range(n_q))
        return n * h

    def stage_work(self):
        B, h, n_q, n_max, d = self.shape
        f = 4.0 * d * self.visible_pairs()
        rows = sum(int(min(max(L, 0), n_max)) for L in self.lens) * h  # cache rows read
        b = 2.0 * (2 * rows * d + 2 * B * h * n_q * d)
        return [(f, b)]

    def metric_flops(self):
        return self.stage_work()[0][0]

    def useful_flops(self):
        return self.metric_flops()

    def launches(self):
        return 2

    def e2e_run(self, i, stream):
        """attn_decode_host_async: pinned host queries and cache lengths in,
        pinned host output out; the caches (state) resident on the device,
        rotating sets; e2e_finish joins the result copies."""
        import torch
        B, h, n_q, n_max, d = self.shape
        if self.h_ws is None:
            self.h_wsb = self.tsd.attn_decode_host_workspace_bytes(B, h, n_q, n_max, d, d)
            self.h_ws = [torch.empty(self.h_wsb, dtype=torch.uint8, device="cuda")
                         for _ in range(2)]
        s = self.sets[i % len(self.sets)]
        self.tsd.attn_decode_host_async(self.h_q, s["k"], s["v"], self.h_out, B, h, n_q, n_max, d,
                                        d, self.h_lens, 0.0, self.h_ws[i % 2], self.h_wsb, stream)

    def e2e_finish(self, stream):
        self.tsd.attn_host_join(stream)

    def e2e_bytes(self):
        return self.a.q.nbytes + self.lens.nbytes, self.a.q.nbytes


def make_calls(tsd, wl, args, seed_offset):
    spec = WORKLOADS[wl]
    if spec["kind"] in ("decode", "encoder"):
        cls = DecodeCall if spec["kind"] == "decode" else EncoderCall
        per_set = cls.set_bytes(spec)
        nsets = max(2, math.ceil(2.2 * L2_BYTES / per_set))
        return [cls(tsd, spec, nsets, seed_offset)], nsets, per_set
    if spec["kind"] == "mha":
        cfgs = spec["calls"]
        probe = [MhaCall(tsd, c, 1, seed_offset) for c in cfgs]
        per_set = sum(p.bytes_per_set() for p in probe)
        nsets = max(2, math.ceil(2.2 * L2_BYTES / per_set))
        return [MhaCall(tsd, c, nsets, seed_offset) for c in cfgs], nsets, per_set
    cfg = dict(spec)
    for k in ("B", "n", "d", "h"):
        if getattr(args, k, None):
            cfg[k] = getattr(args, k)
    if args.causal is not None:
        cfg["causal"] = bool(args.causal)
    per_set = 2 * cfg["B"] * cfg["h"] * (2 * cfg["n"] + 2 * cfg.get("n_k", cfg["n"])) * cfg["d"]
    nsets = max(2, math.ceil(2.2 * L2_BYTES / per_set))
    return [AttnCall(tsd, cfg, nsets, seed_offset)], nsets, per_set


def workload_config(wl, calls, args, nsets, per_set):
    spec = WORKLOADS[wl]
    cfg = {"workload": wl, "description": spec["desc"]}
    if spec["kind"] == "mha":
        cfg["calls"] = [{k: v for k, v in c.cfg.items() if k not in ("seed",)} for c in calls]
        for c in cfg["calls"]:
            c["mask"] = {0: "none", 1: "causal", 2: "key_padding", 3: "causal+key_padding"}[c["mask"]]
            c["kv_range"] = list(c["kv_range"]) if c["kv_range"] else None
    elif spec["kind"] == "decode":
        cfg.update({k: spec[k] for k in ("B", "h", "n_q", "n_max", "d")})
        cfg["len_range"] = list(spec["len_range"])
    elif spec["kind"] == "encoder":
        cfg.update({k: spec[k] for k in ("B", "n", "d_model", "h", "d_ff", "eps")})
        cfg["kv_range"] = list(spec["kv_range"])
    else:
        a = calls[0].a
        cfg.update(B=a.B, h=a.h, n=a.n_q, d=a.d_k, causal=bool(a.mask_kind & MASK_CAUSAL))
        if a.n_k != a.n_q:
            cfg["n_k"] = a.n_k
        if a.kv_lens is not None:
            cfg["key_padding"] = {"kv_range": list(WORKLOADS[wl]["kv_range"])}
        if calls[0].window is not None:
            cfg["window"] = {"left": calls[0].window[0], "right": calls[0].window[1]}
    cfg["l2"] = f"{nsets} rotating input sets of {per_set / 2**20:.1f} MiB (total > L2)"
    return cfg


def run_gpu_arm(args, world, rank, local):
    import torch
    import transformer_scaled_dot_gb300 as tsd
    from transformer_scaled_dot_gb300 import build as native_build

    if rank == 0 and native_build.is_stale():
        native_build.build()
    dist_barrier(world)
    tsd.library()
    torch.cuda.set_device(local)
    stream = torch.cuda.current_stream()
    calls, nsets, per_set = make_calls(tsd, args.workload, args, seed_offset=rank)
    peaks, peak_src = load_peaks()

    def step(i):
        for c in calls:
            c.run(i, stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if tsd.attn_get_device_status() != tsd.ATTN_OK:
        raise RuntimeError("device error during warm-up")

    # ---------------------------------------------------------------- timed region
    props = torch.cuda.get_device_properties(local)
    sampler = ClockSampler(str(getattr(props, "uuid", "") or ""))
    sampler.start()
    # exactly K steps between two events, bracketed by a barrier and a
    # synchronize on both sides; repeated (the rotating sets run on) until
    # the region has lasted --min-seconds on every rank, so that the clock
    # samples see the GPU under load; the step time is the median repeat
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rep_ms = []
    i_next = 0
    t_start = time.time()
    while True:
        dist_barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(i_next, i_next + args.steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        dist_barrier(world)
        i_next += args.steps
        rep_ms.append(ev0.elapsed_time(ev1))
        if dist_max(time.time() - t_start, world) >= args.min_seconds or len(rep_ms) >= 100000:
            break
    t_end = time.time()
    sampler.stop()
    ms_total_max = dist_max(statistics.median(rep_ms), world)  # one K-step loop
    ms_per_step = ms_total_max / args.steps
    if tsd.attn_get_device_status() != tsd.ATTN_OK:
        raise RuntimeError("device error during the timed region")
    clocks = sampler.summary(t_start, t_end)
    timed = {"repeats": len(rep_ms), "seconds": round(t_end - t_start, 3),
             "ms_per_step_min": round(min(rep_ms) / args.steps, 5),
             "ms_per_step_max": round(max(rep_ms) / args.steps, 5),
             "rule": f"K={args.steps} steps between CUDA events per repeat, repeated for "
                     f">= {args.min_seconds} s; ms_per_step = median repeat / K (max over ranks)"}

    flops_step = sum(c.metric_flops() for c in calls)
    total_flops = dist_sum(flops_step * args.steps, world)
    value = total_flops / (ms_total_max * 1e-3) / 1e12
    useful_value = dist_sum(sum(c.useful_flops() for c in calls) * args.steps, world) / \
        (ms_total_max * 1e-3) / 1e12

    # ---------------------------------------------------------------- per-kernel timing
    # Each kernel on its own: a CUDA graph of back-to-back launches over the
    # rotating input sets, replayed between two events on the launch stream.
    # (Events between the eager launches of a step would time host launch
    # gaps and break the programmatic overlap of consecutive kernels.)
    per_kernel = {}
    g_launches, g_reps = max(2 * nsets, 20), 5
    for c in calls:
        for k, (name, work) in enumerate(zip(c.stage_names(), c.stage_work())):
            graph, cap = torch.cuda.CUDAGraph(), torch.cuda.Stream()
            cap.wait_stream(stream)
            with torch.cuda.graph(graph, stream=cap):
                for i in range(g_launches):
                    c.run_stage(k, i, cap)
            stream.wait_stream(cap)
            graph.replay()
            ka, kb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ka.record(stream)
            for _ in range(g_reps):
                graph.replay()
            kb.record(stream)
            torch.cuda.synchronize()
            d = per_kernel.setdefault(name, {"ms": 0.0, "launches": 0, "flops": 0.0, "bytes": 0.0})
            d["ms"] += ka.elapsed_time(kb) / (g_reps * g_launches)
            d["launches"] += 1
            d["flops"] += work[0]
            d["bytes"] += work[1]
            del graph
    if tsd.attn_get_device_status() != tsd.ATTN_OK:
        raise RuntimeError("device error during the per-kernel timing")
    dominant = max(per_kernel, key=lambda k: per_kernel[k]["ms"])
    d = per_kernel[dominant]
    avg_ms = d["ms"] / d["launches"]
    f_per, b_per = d["flops"] / d["launches"], d["bytes"] / d["launches"]
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if f_per / max(b_per, 1.0) >= ridge:
        achieved = f_per / (avg_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    else:
        achieved = b_per / (avg_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    roof["frac"] = round(achieved / roof["peak"], 4)
    tr = None if config_overridden(args) else profiled_traffic(dominant, args.workload)
    roof["traffic"] = tr
    roof["kernel"] = dominant
    roof["kernel_ms"] = round(avg_ms, 5)
    roof["algorithmic"] = {"flops": f_per, "bytes": b_per}
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured" \
        else "fallback"
    roof["timing"] = (f"each kernel alone: CUDA graph of {g_launches} back-to-back launches over "
                      f"the rotating input sets, CUDA events around {g_reps} replays")
    kernel_table = {k: {"ms_per_launch": round(v["ms"] / v["launches"], 5),
                        "share": round(v["ms"] / sum(x["ms"] for x in per_kernel.values()), 4),
                        "tflops": round(v["flops"] / (v["ms"] * 1e-3) / 1e12, 2),
                        "gbs": round(v["bytes"] / (v["ms"] * 1e-3) / 1e9, 1)}
                    for k, v in per_kernel.items()}

    # ---------------------------------------------------------------- end to end
    e2e_iters = max(args.steps, 10)
    for i in range(2):
        for c in calls:
            c.e2e_run(i, stream)
    for c in calls:
        c.e2e_finish(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist_barrier(world)
    e0.record(stream)
    for i in range(e2e_iters):
        for c in calls:
            c.e2e_run(i, stream)
    for c in calls:  # every result copy inside the timed region
        c.e2e_finish(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = dist_max(e0.elapsed_time(e1), world) / e2e_iters
    h2d = sum(c.e2e_bytes()[0] for c in calls)
    d2h = sum(c.e2e_bytes()[1] for c in calls)
    e2e_value = dist_sum(flops_step * e2e_iters, world) / (e2e_ms * e2e_iters * 1e-3) / 1e12

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "useful_value": round(useful_value, 3),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) / Xavier inputs of the workload's shapes)",
        "config": dict(workload_config(args.workload, calls, args, nsets, per_set),
                       parallelism=f"replicas x{world}" if world > 1 else "single GPU",
                       launch="eager C-ABI calls on the current torch stream"),
        "roofline": roof,
        "kernels": kernel_table,
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 5),
                "api": E2E_API[spec_kind(args.workload)]},
        "clocks": clocks,
        "timed_region": dict(timed, launches_all_repeats=int(
            sum(c.launches() for c in calls) * args.steps * timed["repeats"])),
        "gpu_launches": int(sum(c.launches() for c in calls) * args.steps),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args, calls, budget_s=args.cpu_seconds)
    return line, rank


# --------------------------------------------------------------------------- oracle (CPU)

def oracle_sample_runner(args):
    """A function running the oracle on a bounded sample of the workload, and
    the metric FLOPs that sample represents."""
    import oracle
    spec = WORKLOADS[args.workload]
    if spec["kind"] == "mha":
        ms = []
        for c in spec["calls"]:
            m = synthetic.mha_inputs(c["seed"], c["B"], c["n_q"], c["n_k"], c["d_model"], c["h"],
                                     c["d"], c["d"], c["mask"], c["kv_range"], add_pe=c["add_pe"],
                                     self_attention=c["self_attention"])
            ms.append((m, m.as_f64()))
        flops = sum(attn_flops(m.B, m.h, m.n_q, m.n_k, m.d_k, bool(m.mask_kind & MASK_CAUSAL))
                    for m, _ in ms)

        def run(nthreads=0):
            for m, f64 in ms:
                oracle.mha(*f64, m.h, m.mask_kind, kv_lens=m.kv_lens, nthreads=nthreads)
        return run, flops, "the whole batch through oracle.mha (projections, attention, W_O)"
    if spec["kind"] == "encoder":
        nb = 4  # the first four sequences of the batch
        e = synthetic.encoder_inputs(spec["seed"], nb, spec["n"], spec["d_model"], spec["h"],
                                     spec["d_ff"], spec["mask"], spec["kv_range"], add_pe=True)
        m = e.mha
        x, _, wq, wk, wv, wo = m.as_f64()
        params = e.params_f64()
        rows = nb * m.n_q
        flops = 2.0 * rows * m.d_model * 4 * m.h * m.d_k + 4.0 * rows * m.d_model * e.d_ff
        flops += attn_flops(nb, m.h, m.n_q, m.n_k, m.d_k, False)

        def run(nthreads=0):
            oracle.encoder_layer(x, wq, wk, wv, wo, *params, m.h, m.mask_kind, kv_lens=m.kv_lens,
                                 eps=spec["eps"], nthreads=nthreads)
        return run, flops, f"{nb} sequences of the batch through oracle.encoder_layer"
    if spec["kind"] == "decode":
        B, h, n_q, n_max, d = (spec[k] for k in ("B", "h", "n_q", "n_max", "d"))
        nb = 2  # every head of the first two sequences
        a = synthetic.attention_inputs(spec["seed"], nb, h, n_q, n_max, d, d)
        rng = np.random.default_rng(spec["seed"])
        lens = synthetic.uniform_lengths(rng, B, *spec["len_range"])[:nb]
        q, k, v = (synthetic.bf16_bits_to_f64(x) for x in (a.q, a.k, a.v))
        flops = 4.0 * d * h * sum(max(0, min(int(L), int(L) - n_q + t + 1))
                                  for L in lens for t in range(n_q))

        def run(nthreads=0):
            oracle.decode(q, k, v, cache_lens=lens, nthreads=nthreads)
        return run, flops, (f"all {h} heads of {nb} sequences (cache lengths {list(map(int, lens))}, "
                            f"d={d}) via oracle.decode")
    cfg = dict(spec)
    for k in ("B", "n", "d", "h"):
        if getattr(args, k, None):
            cfg[k] = getattr(args, k)
    if args.causal is not None:
        cfg["causal"] = bool(args.causal)
    n, d, causal = cfg["n"], cfg["d"], cfg["causal"]
    if cfg.get("padding"):  # short padded shapes: every head of the first sequences
        nb = 4
        a = synthetic.attention_inputs(cfg["seed"], nb, cfg["h"], n, cfg.get("n_k", n), d, d,
                                       MASK_KEY_PADDING, cfg["kv_range"])
        q, k, v = a.as_f64()
        flops = attn_flops(nb, a.h, a.n_q, a.n_k, d, False)

        def run(nthreads=0):
            oracle.attention(q, k, v, MASK_KEY_PADDING, kv_lens=a.kv_lens, nthreads=nthreads)
        return run, flops, (f"all {a.h} heads of {nb} sequences (n_q={a.n_q}, n_k={a.n_k}, kv_lens "
                            f"{list(map(int, a.kv_lens))}) via oracle.attention")
    window = cfg.get("window")
    rng = np.random.default_rng(cfg["seed"])
    # one head of the workload, a seeded subset of its query rows
    q = synthetic.bf16_bits_to_f64(synthetic.normal_bf16(rng, (n, d)))
    k = synthetic.bf16_bits_to_f64(synthetic.normal_bf16(rng, (n, d)))
    v = synthetic.bf16_bits_to_f64(synthetic.normal_bf16(rng, (n, d)))
    rows = np.sort(rng.choice(n, size=min(n, 256), replace=False)).astype(np.int32)
    if window is not None:  # keys each sampled row is allowed to see
        lo = np.maximum(0, rows - window[0]) if window[0] >= 0 else np.zeros_like(rows)
        hi = np.minimum(n - 1, rows + window[1]) if window[1] >= 0 else np.full_like(rows, n - 1)
        if causal:
            hi = np.minimum(hi, rows)
        keys_seen = int(np.maximum(hi - lo + 1, 0).sum())
    else:
        keys_seen = (rows + 1).sum() if causal else len(rows) * n
    flops = 4.0 * keys_seen * d

    def run(nthreads=0):
        oracle.attention_rows(q[rows], rows, k, v, causal=causal, window=window, nthreads=nthreads)
    return run, flops, f"{len(rows)} query rows of one head (n={n}, d={d}) via oracle.attention_rows"


def cpu_baseline(args, calls, budget_s=10.0):
    import oracle
    run, flops, what = oracle_sample_runner(args)
    run()  # warm-up (also builds the oracle library)
    reps, t0 = 0, time.perf_counter()
    while True:
        run()
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 100000:
            break
    tflops = flops * reps / el / 1e12
    # the same sample on one thread (the parallel figure's scaling reference)
    reps1, t1 = 0, time.perf_counter()
    while True:
        run(nthreads=1)
        reps1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= budget_s / 3 or reps1 >= 100000:
            break
    return {"value": tflops, "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{what}; {reps} repetitions in {el:.1f} s",
            "single_thread": {"value": flops * reps1 / el1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                              "sample": f"the same sample, {reps1} repetitions in {el1:.1f} s"}}


def run_reference_arm(args, world, rank):
    if rank != 0:
        return None, rank
    import oracle
    run, flops, what = oracle_sample_runner(args)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    value = flops * args.steps / el / 1e12
    cfg = {"workload": args.workload, "description": WORKLOADS[args.workload]["desc"]}
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": what},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return line, rank


# --------------------------------------------------------------------------- main

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="long")
    ap.add_argument("--min-seconds", type=float, default=2.0,
                    help="repeat the timed K-step loop until this much wall time has passed")
    ap.add_argument("--B", type=int, default=None)
    ap.add_argument("--n", type=int, default=None)
    ap.add_argument("--d", type=int, default=None, choices=[16, 32, 64, 128, 256])
    ap.add_argument("--h", type=int, default=None)
    ap.add_argument("--causal", type=int, default=None, choices=[0, 1])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3  # timing rule: at least 3 warm-up steps
    world, rank, local = dist_setup()
    if args.impl == "reference":
        line, rank = run_reference_arm(args, world, rank)
    else:
        line, rank = run_gpu_arm(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
