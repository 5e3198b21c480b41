"""Benchmark of the DFlash hot path on GB300: draft block-positions per second.

One step = one pass of the whole path over one batch of synthetic inputs:
  dflash_plan -> dflash_project_context -> dflash_body_forward -> dflash_verify_greedy
on the Qwen3-8B-shaped training workload (B=4, L=2048, 8 anchors of 16 slots per row,
W_proj 20480->4096, 5 draft layers), plus greedy verification of every drafted block
against synthetic target logits [B*N, 16, 151936].

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Prints one JSON line.  Under torchrun (N > 1) every rank runs its own shard of rows
(weak scaling, no data-path collective); rank 0 prints.  `--impl reference` times the
fp64 CPU oracle on a bounded sample of the same workload.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dflash_inputs as di  # noqa: E402

DEFAULT_WORKLOAD = "train_8b_b4_l2048"
METRIC = "draft block-positions/sec (DFlash body fwd, 1 GB300) and % of bf16/HBM roofline"


# --------------------------------------------------------------------------------------
# algorithmic work (counts only what the method needs; see the design notes)
# --------------------------------------------------------------------------------------

def algorithmic_work(w: di.Workload, plan: dict, mask: np.ndarray) -> dict:
    """FLOPs of the projections and attention, counting context positions c < max anchor
    (mask = 1) per row, block GEMMs for valid slots only, attention 4*dh*Hq per allowed
    (query, key) pair; verification bytes = B_v * S * V * element size."""
    s = w.shape
    D, Kc, NL = s.hidden, s.concat_width, s.num_layers
    kvw = 2 * s.kv_width
    anchors, valid = plan["anchors"], plan["block_valid"].astype(bool)
    ctx_pos = 0
    pairs = 0
    for b in range(w.batch):
        a_valid = [int(a) for a, v in zip(anchors[b], valid[b]) if a >= 0 and v.any()]
        if a_valid:
            ctx_pos += int(mask[b, :min(max(a_valid), w.seq_len)].sum())
        for k in range(anchors.shape[1]):
            a = int(anchors[b, k])
            nv = int(valid[b, k].sum())
            if a < 0 or nv == 0:
                continue
            keys = int(mask[b, :min(a, w.seq_len)].sum()) + nv
            pairs += nv * keys
    tv = int(valid.sum())
    layer_params = NL * D * (s.qkv_width + s.q_width + 3 * s.intermediate)
    ctx_params = Kc * D + NL * D * kvw   # W_proj and the K/V rows of each layer
    f_proj = 2.0 * ctx_pos * Kc * D
    f_ctxkv = 2.0 * ctx_pos * D * kvw * NL
    f_layers = 2.0 * tv * D * (s.qkv_width + s.q_width + 2 * s.intermediate + s.intermediate) * NL
    f_attn = 4.0 * s.head_dim * s.num_heads * pairs * NL
    # context K/V cache read by attention: every readable position of a row (c < its largest
    # anchor, mask = 1) once per layer, K and V, fp16 (bf16 configuration) or fp32
    cache_elem = 2.0 if s.dtype == "bf16" else 4.0
    attn_bytes = ctx_pos * 2.0 * s.kv_width * cache_elem * NL
    return {"layer_weight_bytes": 2.0 * layer_params, "ctx_weight_bytes": 2.0 * ctx_params,
            "attn_cache_bytes": attn_bytes,
            "ctx_positions": ctx_pos, "valid_slots": tv, "gemm_flops": f_proj + f_ctxkv + f_layers,
            "attn_flops": f_attn, "total_flops": f_proj + f_ctxkv + f_layers + f_attn,
            "proj_flops": f_proj, "ctxkv_flops": f_ctxkv, "layer_flops": f_layers}


# --------------------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------------------

class NvmlPoller:
    """Read-only NVML queries (SM clock, its maximum, clock event reasons) polled about every
    millisecond from a thread, so that timed regions of a few milliseconds get samples too."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device_index),
                                                  ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.samples = []
        self.stop_evt = threading.Event()
        self.thread = None

    def query(self):
        ct = self.ct
        mhz, mx, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz)) != 0:
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ct.byref(mx))
        self.reasons_fn(self.h, ct.byref(rs))
        return mhz.value, mx.value, rs.value

    def _run(self):
        while not self.stop_evt.is_set():
            q = self.query()
            if q:
                self.samples.append(q)
            time.sleep(0.001)

    def start(self):
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self):
        self.stop_evt.set()
        if self.thread:
            self.thread.join(timeout=2)
        return self.samples


class ClockSampler:
    """Clocks during the timed region: NVML polled about every millisecond, plus the
    nvidia-smi query loop (200 ms) beside it; the median SM clock and every active slowdown
    reason of both."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None
        try:
            self.nvml = NvmlPoller(device_index)
        except (OSError, AttributeError):
            self.nvml = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        if self.proc is not None:
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        if self.nvml:
            self.nvml.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        nv = self.nvml.stop() if self.nvml else []
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)
        if self.proc is None and not nv:
            return {"sm_mhz": None, "sm_max_mhz": None,
                    "reasons": ["nvidia-smi and NVML unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        n_smi = 0
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            n_smi += 1
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        for mhz, mx, rs in nv:
            sm.append(float(mhz))
            smax.append(float(mx))
            for bit, n in NvmlPoller.REASONS.items():
                if rs & bit:
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm), "samples_nvml": len(nv), "samples_nvidia_smi": n_smi}


# --------------------------------------------------------------------------------------
# the GPU arm
# --------------------------------------------------------------------------------------

def profiled_traffic(workload: str):
    """DRAM bytes per GEMM launch from the committed ncu capture of this workload, or None
    when there is none or the GEMM kernel's sources changed since it was taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"gemm_traffic_{workload}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    h = hashlib.sha256()
    for src in rec["sources"]:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return rec["dram_bytes_per_launch"] if h.hexdigest() == rec["source_sha256"] else None


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class GpuStep:
    """Device-resident inputs and workspaces for one rank; step() runs the whole path."""

    def __init__(self, w: di.Workload, model_w: di.Workload, device):
        import torch
        import block_draft_model_proj_gb300 as dflash
        self.torch, self.dflash = torch, dflash
        self.w = w
        s = w.shape
        self.dev = device
        B, L, N, S = w.batch, w.seq_len, w.num_anchors, s.block_size
        self.B, self.L, self.N, self.S = B, L, N, S

        def dev(t):
            if t.dtype == "bf16":
                return torch.from_numpy(np.ascontiguousarray(t.data).view(np.int16)).to(device).view(
                    torch.bfloat16)
            return torch.from_numpy(np.ascontiguousarray(t.data)).to(device)
        self._dev = dev
        top = di.gen_top_weights(model_w)
        layers = [di.gen_layer_weights(model_w, l) for l in range(s.num_layers)]
        # the model's bf16 weights as given: the training workloads pass them to every call
        # (the weights change with every optimizer step; the library converts what its
        # large-token GEMMs need inside the call).  Inference prepares fp16 copies of the layer
        # matrices once, with the model (DFLASH_FLAG_F16_LAYERS).
        self.wts_bf16 = dflash.Weights({k: dev(v) for k, v in top.items()},
                                       [{k: dev(v) for k, v in lw.items()} for lw in layers])
        self.cfg_bf16 = dflash.make_config(s)
        self.wts_f16, self.cfg_f16 = self.wts_bf16, self.cfg_bf16
        if s.dtype == "bf16":
            self.wts_f16 = dflash.prepare_f16_layers(self.wts_bf16)
            self.cfg_f16 = dflash.make_config(s, f16_layers=True)
        self.use_f16_weights(w.inference)
        # host inputs (pinned for the end-to-end leg) and their device copies
        self.h_mask = torch.from_numpy(di.gen_mask(w)).pin_memory()
        self.h_sids = torch.from_numpy(di.gen_sample_ids(w)).pin_memory()
        H = di.gen_target_hidden(w)
        self.h_hidden = torch.from_numpy(H.data.view(np.int16)).view(torch.bfloat16).pin_memory() \
            if H.dtype == "bf16" else torch.from_numpy(H.data).pin_memory()
        emb = di.gen_block_emb(w)
        self.h_emb = torch.from_numpy(emb.data.view(np.int16)).view(torch.bfloat16).pin_memory() \
            if emb.dtype == "bf16" else torch.from_numpy(emb.data).pin_memory()
        if w.verify_batch == 0:  # verify every drafted block, as on the headline workload
            w = di.scaled(w, verify_batch=B * N, vocab=151936)
        vi = di.gen_verify(w)
        self.Bv = vi.draft.shape[0]
        self.V = w.vocab
        self.h_logits = torch.from_numpy(vi.logits.data.view(np.int16)).view(torch.bfloat16) \
            .pin_memory() if vi.logits.dtype == "bf16" else torch.from_numpy(vi.logits.data).pin_memory()
        self.h_draft = torch.from_numpy(vi.draft).pin_memory()
        self.inference = w.inference
        self.d_mask = self.h_mask.to(device)
        self.d_sids = self.h_sids.to(device)
        self.d_hidden = self.h_hidden.to(device)
        self.d_emb = self.h_emb.to(device)
        self.d_logits = self.h_logits.to(device)
        self.d_draft = self.h_draft.to(device)
        self.kv = torch.empty((s.num_layers, B, 2, s.num_kv_heads, L, s.head_dim),
                              dtype=dflash.kv_cache_dtype(self.cfg), device=device)
        self.anchors = torch.empty((B, N), dtype=torch.int32, device=device)
        self.bv = torch.empty((B, N, S), dtype=torch.uint8, device=device)
        self.lm = torch.empty_like(self.bv)
        self.pid = torch.empty((B, N, S), dtype=torch.int32, device=device)
        if w.inference:
            # one block per request right after the cached context (anchor = L)
            a_np, v_np, p_np = di.inference_block_layout(w)
            self.anchors.copy_(torch.from_numpy(a_np))
            self.bv.copy_(torch.from_numpy(v_np))
            self.pid.copy_(torch.from_numpy(p_np))
        self.ctx_len = torch.empty((B,), dtype=torch.int32, device=device)
        self.out = torch.empty((B, N, S, s.hidden), dtype=torch.float32, device=device)
        self.em = torch.empty((self.Bv, S), dtype=torch.int32, device=device)
        self.ne = torch.empty((self.Bv,), dtype=torch.int32, device=device)
        self.ac = torch.empty_like(self.ne)
        ws = max(dflash.dflash_project_context_workspace_size(self.cfg, B, L),
                 dflash.dflash_body_workspace_size(self.cfg, B, L, N),
                 dflash.dflash_verify_workspace_size(self.Bv, S - 1, self.V))
        self.ws = dflash.workspace(ws, device)
        self.h_out = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        self.h_em = torch.empty(self.em.shape, dtype=torch.int32).pin_memory()
        self.h_ne = torch.empty(self.ne.shape, dtype=torch.int32).pin_memory()
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in
                             (self.h_mask, self.h_sids, self.h_emb, self.h_logits, self.h_draft) +
                             (() if w.inference else (self.h_hidden,)))
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in (self.h_out, self.h_em, self.h_ne))
        self.stream = torch.cuda.current_stream(device)

    def use_f16_weights(self, on: bool):
        self.wts, self.cfg = (self.wts_f16, self.cfg_f16) if on else (self.wts_bf16, self.cfg_bf16)

    def build_cache(self):
        """The projected context of the inference workloads: built once, outside timing."""
        self.dflash.dflash_project_context(self.cfg, self.wts, self.d_hidden, self.B, self.L, 0,
                                           self.L, self.kv, ws=self.ws,
                                           stream=self.stream.cuda_stream)

    def step(self):
        d, w = self.dflash, self.w
        st = self.stream.cuda_stream
        if self.inference:
            d.dflash_body_forward(self.cfg, self.wts, self.d_emb, self.anchors, self.bv, self.pid,
                                  self.d_mask, self.kv, self.B, self.L, self.N, self.out,
                                  ws=self.ws, stream=st)
            d.dflash_verify_greedy(self.d_logits, d.DFLASH_DTYPE_BF16, self.d_draft, self.Bv,
                                   self.S - 1, self.V, -1, self.em, self.ne, self.ac, ws=self.ws,
                                   stream=st)
            return
        d.dflash_plan(self.d_mask, self.d_sids, w.plan_step, w.plan_seed, self.N, self.S,
                      self.anchors, self.bv, self.lm, self.pid, ctx_len=self.ctx_len, stream=st)
        d.dflash_project_context(self.cfg, self.wts, self.d_hidden, self.B, self.L, 0, self.L,
                                 self.kv, ctx_len=self.ctx_len, ws=self.ws, stream=st)
        d.dflash_body_forward(self.cfg, self.wts, self.d_emb, self.anchors, self.bv, self.pid,
                              self.d_mask, self.kv, self.B, self.L, self.N, self.out, ws=self.ws,
                              stream=st)
        d.dflash_verify_greedy(self.d_logits, d.DFLASH_DTYPE_BF16 if self.h_logits.dtype ==
                               self.torch.bfloat16 else d.DFLASH_DTYPE_F32, self.d_draft, self.Bv,
                               self.S - 1, self.V, -1, self.em, self.ne, self.ac, ws=self.ws,
                               stream=st)

    def step_e2e(self):
        """Same step from pinned host buffers: H2D of the step's inputs, D2H of the results."""
        nb = True
        self.d_mask.copy_(self.h_mask, non_blocking=nb)
        self.d_sids.copy_(self.h_sids, non_blocking=nb)
        if not self.inference:  # the inference context is a cache, not a per-step input
            self.d_hidden.copy_(self.h_hidden, non_blocking=nb)
        self.d_emb.copy_(self.h_emb, non_blocking=nb)
        self.d_logits.copy_(self.h_logits, non_blocking=nb)
        self.d_draft.copy_(self.h_draft, non_blocking=nb)
        self.step()
        self.h_out.copy_(self.out, non_blocking=nb)
        self.h_em.copy_(self.em, non_blocking=nb)
        self.h_ne.copy_(self.ne, non_blocking=nb)

    def host_plan(self):
        from_dev = {"anchors": self.anchors.cpu().numpy(), "block_valid": self.bv.cpu().numpy()}
        return from_dev


def timed(fn, steps, torch, stream, barrier):
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        fn()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    return t0.elapsed_time(t1)


def attention_roofline(work: dict, a_ms: float, steps: int, peak_tflops: float,
                       hbm_gbs: float) -> dict:
    """Attention against the roofline that binds it: its FLOPs at the tensor peak or its
    context K/V bytes at the HBM peak, whichever takes longer (decode steps read a long cache
    for few queries and are HBM-bound)."""
    flops, nbytes = work["attn_flops"], work["attn_cache_bytes"]
    t_tensor = flops / (peak_tflops * 1e12)
    t_hbm = nbytes / (hbm_gbs * 1e9)
    sec = a_ms / 1e3 / steps if a_ms else None
    out = {"flop_per_step": flops, "bytes_per_step": nbytes,
           "frac_tensor": t_tensor / sec if sec else None,
           "frac_hbm": t_hbm / sec if sec else None}
    if t_hbm > t_tensor:
        out.update({"bound": "hbm", "achieved": nbytes / sec / 1e9 if sec else None,
                    "peak": hbm_gbs, "unit": "GB/s", "frac": out["frac_hbm"]})
    else:
        out.update({"bound": "tensor", "achieved": flops / sec / 1e12 if sec else None,
                    "peak": peak_tflops, "unit": "TFLOP/s", "frac": out["frac_tensor"]})
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import block_draft_model_proj_gb300 as dflash
    from block_draft_model_proj_gb300 import build as dbuild
    dbuild.build()
    dflash.load()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    base = di.WORKLOADS[args.workload]
    # every rank owns its own rows (a different data stream), all ranks share the model
    w = di.scaled(base, index=base.index + 97 * rank) if rank else base
    g = GpuStep(w, base, device)
    stream = g.stream
    if w.inference:
        g.build_cache()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        g.step()
    torch.cuda.synchronize()
    dflash.dflash_device_status()
    plan = {"anchors": g.anchors.cpu().numpy(), "block_valid": g.bv.cpu().numpy()}
    work = algorithmic_work(w, plan, g.h_mask.numpy())
    if w.inference:  # the cached context is not projected inside the step
        work["gemm_flops"] -= work["proj_flops"] + work["ctxkv_flops"]
        work["total_flops"] -= work["proj_flops"] + work["ctxkv_flops"]

    # headline: the step as a user runs it (no per-kernel events between the launches, which
    # would serialise the programmatically dependent launches)
    sampler = ClockSampler(local_rank)
    launches0 = dflash.dflash_launch_count()
    sampler.start()
    ms = timed(g.step, args.steps, torch, stream, barrier)
    clocks = sampler.stop()
    launches = dflash.dflash_launch_count() - launches0
    dflash.dflash_device_status()
    # per-kernel split: the same steps again with CUDA events around every launch
    dflash.dflash_profile_enable(True)
    prof_ms = timed(g.step, args.steps, torch, stream, barrier)
    prof = dflash.dflash_profile_read()
    dflash.dflash_profile_enable(False)
    dflash.dflash_device_status()

    # end to end: host buffers in, results out, inside the timed region
    for _ in range(2):
        g.step_e2e()
    e2e_ms = timed(g.step_e2e, args.steps, torch, stream, barrier)

    # secondary figure for the training workloads: the same step with the layer weights held
    # as fp16 by the trainer (its optimizer writes the fp16 working copy), i.e. without the
    # per-step bf16 -> fp16 conversion that the headline number includes
    held_ms = 0.0
    if not w.inference and w.shape.dtype == "bf16":
        g.use_f16_weights(True)
        for _ in range(2):
            g.step()
        held_ms = timed(g.step, args.steps, torch, stream, barrier)
        g.use_f16_weights(False)

    t = torch.tensor([ms, e2e_ms, held_ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms, e2e_ms, held_ms = float(t[0]), float(t[1]), float(t[2])
    units = w.tokens * world * args.steps
    value = units / (ms / 1e3)
    e2e_value = units / (e2e_ms / 1e3)

    peaks = measured_peaks()
    gemm_ms, gemm_n = prof["gemm"]
    gemm_s_per_launch = gemm_ms / 1e3 / max(gemm_n, 1)
    flops_per_launch = work["gemm_flops"] * args.steps / max(gemm_n, 1)
    peak = peaks["bf16_tflops_sustained"]
    step_s = ms / 1e3 / args.steps
    # the projection GEMMs' roofline: tensor-bound, or weight-read-bound when the FLOP per
    # weight byte (2 * tokens / 2 bytes) is below the ridge point (a decode step)
    wbytes = work["layer_weight_bytes"] + (0 if w.inference else work["ctx_weight_bytes"])
    gemm_intensity = work["gemm_flops"] / max(wbytes, 1)
    hbm = peaks["hbm_gbs"]
    if gemm_intensity < peak * 1e12 / (hbm * 1e9):
        bytes_per_launch = wbytes * args.steps / max(gemm_n, 1)
        achieved = bytes_per_launch / gemm_s_per_launch / 1e9 if gemm_n else None
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": (achieved / hbm) if achieved else None,
                "algorithmic": "weight bytes read once per projection (bf16 layer matrices)",
                "peak_source": f"{peaks['source']} hbm_gbs"}
    else:
        achieved = flops_per_launch / gemm_s_per_launch / 1e12 if gemm_n else None
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": (achieved / peak) if achieved else None,
                "algorithmic": "2*M*N*K over context rows below each row's largest anchor and "
                               "valid slots",
                "peak_source": f"{peaks['source']} bf16_tflops_sustained (fp16 dense rate = "
                               "bf16 dense rate, nominal ratio 1)"}
    roof.update({"traffic": profiled_traffic(base.name),
                 "traffic_unit": "bytes per launch (ncu dram read + write)",
                 "kernel": "projection GEMMs (gemm_tc_kernel, gemm_ws_kernel)",
                 "launches_per_step": gemm_n / args.steps})
    # verification and attention against their own rooflines
    v_ms, v_n = prof["verify"]
    v_bytes = g.Bv * g.S * g.V * 2
    a_ms, a_n = prof["attention"]
    kernel_rooflines = {
        "verify": {"bound": "hbm", "bytes_per_call": v_bytes,
                   "achieved": v_bytes * args.steps / (v_ms / 1e3) / 1e9 if v_ms else None,
                   "peak": hbm, "unit": "GB/s",
                   "frac": v_bytes * args.steps / (v_ms / 1e3) / 1e9 / hbm if v_ms else None},
        "attention": attention_roofline(work, a_ms, args.steps, peak, hbm),
    }
    result = {
        "metric": METRIC, "value": value, "unit": "block-positions/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16+f16",
        "precision": "bf16 inputs and weights; W_proj bf16 x bf16, draft-layer projections "
                     "f16 x f16 (bf16 weight tiles converted to fp16 on chip for <= 512 tokens, "
                     "fp16 copies converted inside the call above that; fp16 activations), "
                     "fp32 accumulation and residual stream, attention f16 x f16 over an "
                     "fp16 context K/V cache",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, bf16)",
        "config": {"workload": f"{w.name}: B={w.batch} L={w.seq_len} N={w.num_anchors} "
                               f"S={w.shape.block_size} D={w.shape.hidden} "
                               f"W_proj {w.shape.concat_width}->{w.shape.hidden} "
                               f"NL={w.shape.num_layers} Hq/Hkv/dh={w.shape.num_heads}/"
                               f"{w.shape.num_kv_heads}/{w.shape.head_dim} I={w.shape.intermediate}"
                               f"; verify [{g.Bv},{g.S},{g.V}]",
                   "block_positions_per_step": w.tokens, "valid_slots_per_step": work["valid_slots"],
                   "l2": "inputs larger than L2 (weights 2.1 GB + hidden states 0.34 GB + "
                         "logits 0.16 GB read per step)",
                   "parallelism": f"replicas: {world} rank(s), each its own rows, no collective"},
        "roofline": roof,
        "kernel_rooflines": kernel_rooflines,
        "step_roofline": {"algorithmic_tflop_per_step": work["total_flops"] / 1e12,
                          "achieved_tflops": work["total_flops"] / step_s / 1e12,
                          "frac_of_sustained_bf16": work["total_flops"] / step_s / 1e12 / peak},
        "kernel_ms_per_step": {k: v[0] / args.steps for k, v in prof.items()},
        "profiled_ms_per_step": prof_ms / args.steps,
        "clocks": clocks,
        "gpu_launches": launches,
        "e2e": {"value": e2e_value, "unit": "block-positions/s",
                "h2d_bytes_per_step": g.h2d_bytes, "d2h_bytes_per_step": g.d2h_bytes},
    }
    result["kernel_flops_per_step"] = {k: work[k] for k in ("proj_flops", "ctxkv_flops",
                                                          "layer_flops", "attn_flops")}
    if held_ms > 0:
        held_s = held_ms / 1e3 / args.steps
        result["fp16_weights_held"] = {
            "value": units / (held_ms / 1e3), "unit": "block-positions/s",
            "ms_per_step": held_ms / args.steps,
            "frac_of_sustained_bf16": work["total_flops"] / held_s / 1e12 / peak,
            "note": "same step with fp16 copies of the layer weights held by the trainer (its "
                    "optimizer writes the fp16 working copy) instead of the bf16 weights; not "
                    "the headline"}
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(base, g.h_mask.numpy(), g.h_sids.numpy())
    return result


# --------------------------------------------------------------------------------------
# the oracle on the host cores
# --------------------------------------------------------------------------------------

def oracle_row_step(w: di.Workload, b: int, mask, sids, model=None):
    """The oracle on one row of the workload: plan, context for the positions the row's
    blocks read, every block of the row, and verification of its blocks.  Returns the
    number of block positions processed."""
    from oracle import dflash_oracle as orc
    s = w.shape
    if model is None:
        model = OracleModel(w)
    plan = orc.build_plan(mask, sids, w.plan_step, w.plan_seed, w.num_anchors, s.block_size)
    anchors, valid = plan["anchors"][b], plan["block_valid"][b]
    need = max([int(a) for a in anchors if a >= 0] + [1])
    rows = di.gen_target_hidden_rows(w, b, 0, min(need, w.seq_len)).f64()
    kv = orc.project_context_row(s, model.top, model.layer, rows)
    e = model.emb
    emb = di.Tensor(e.data[b], e.dtype).f64()
    for k in range(w.num_anchors):
        orc.block_forward(s, model.top, model.layer, emb[k], int(anchors[k]), valid[k], mask[b],
                          kv, plan["position_ids"][b, k])
    vi = model.verify
    lo, hi = b * w.num_anchors, (b + 1) * w.num_anchors
    orc.verify_greedy(di.Tensor(vi.logits.data[lo:hi], vi.logits.dtype).f64(), vi.draft[lo:hi])
    return w.num_anchors * s.block_size


class OracleModel:
    def __init__(self, w: di.Workload):
        top = di.gen_top_weights(w)
        self.top = {k: v.f64() for k, v in top.items()}
        self._layers = {}
        self.w = w
        self.verify = di.gen_verify(w)
        self.emb = di.gen_block_emb(w)

    def layer(self, l):
        if l not in self._layers:
            self._layers[l] = {k: v.f64() for k, v in di.gen_layer_weights(self.w, l).items()}
        return self._layers[l]


def cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w: di.Workload, mask, sids) -> dict:
    model = OracleModel(w)
    for l in range(w.shape.num_layers):
        model.layer(l)
    t0 = time.perf_counter()
    units = oracle_row_step(w, 0, mask, sids, model)
    dt = time.perf_counter() - t0
    return {"value": units / dt, "unit": "block-positions/s", "cores": cores(), "kind": "oracle",
            "sample": f"row 0 of {w.name} ({w.num_anchors} blocks x {w.shape.block_size} slots): "
                      f"plan, context projection of the row's prefix, body, verification; "
                      f"{dt:.1f} s fp64 NumPy"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = di.WORKLOADS[args.workload]
    mask, sids = di.gen_mask(w), di.gen_sample_ids(w)
    model = OracleModel(w)
    for l in range(w.shape.num_layers):
        model.layer(l)
    valid_rows = [b for b in range(w.batch) if not any(r == b for r, _ in w.padded_rows)]
    for i in range(args.warmup):
        oracle_row_step(w, valid_rows[i % len(valid_rows)], mask, sids, model)
    t0 = time.perf_counter()
    units = 0
    for i in range(args.steps):
        units += oracle_row_step(w, valid_rows[i % len(valid_rows)], mask, sids, model)
    dt = time.perf_counter() - t0
    value = units / dt
    sample = (f"each step = one valid row of {w.name} ({w.num_anchors} blocks x "
              f"{w.shape.block_size} slots: plan, context prefix, body, verification)")
    return {"metric": METRIC, "value": value, "unit": "block-positions/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "block-positions/s", "cores": cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "block-positions/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(di.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
