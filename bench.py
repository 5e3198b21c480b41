"""Benchmark of the DFlash hot path on GB300: draft block-positions per second.

One step = one pass of the whole path over one batch of synthetic inputs:
  dflash_plan -> dflash_project_context -> dflash_body_forward -> dflash_verify_greedy
The headline workload is the largest single-GPU training configuration (B=16, L=4096,
32 anchors of 16 slots per row, W_proj 20480->4096, 5 draft layers of the Qwen3-8B shape,
four row pairs sharing sample ids), with greedy verification of every drafted block against
synthetic target logits [B*N, 16, 151936].  The same JSON line carries the B=4 L=2048
training step, the long-context step (B=1 L=32768, 64 anchors), the decode steps at batch 1
and 64 over a cached 4096-position context, and verification alone on [32|64, 16, 151936].

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--headline-only] [--no-cpu-baseline]

Prints one JSON line.  Under torchrun (N > 1) every rank runs its own rows (weak scaling,
no data-path collective); rank 0 prints.  `--impl reference` times the fp64 CPU oracle on
bounded samples of the same workload.
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

DEFAULT_WORKLOAD = "train_8b_b16_l4096"
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

    def __init__(self, w: di.Workload, model_w: di.Workload, device, pinned: bool = True):
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

        def host(t):
            h = torch.from_numpy(np.ascontiguousarray(t.data).view(np.int16)).view(torch.bfloat16) \
                if t.dtype == "bf16" else torch.from_numpy(np.ascontiguousarray(t.data))
            return h.pin_memory() if pinned else h
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
        self.inference = w.inference
        # host inputs (pinned for the end-to-end leg) and their device copies
        self.h_mask = host(di.Tensor(di.gen_mask(w), "u8"))
        self.h_sids = host(di.Tensor(di.gen_sample_ids(w), "i64"))
        if w.inference:
            # the cached context is not a per-step input: its hidden states go to the device
            # row by row (only to build the cache) and are not kept on the host
            self.h_hidden = None
            self.d_hidden = torch.empty((B, L, s.concat_width), dtype=torch.bfloat16,
                                        device=device)
            for b in range(B):
                self.d_hidden[b].copy_(dev(di.gen_target_hidden_rows(w, b, 0, L)))
        else:
            self.h_hidden = host(di.gen_target_hidden(w))
            self.d_hidden = self.h_hidden.to(device)
        self.h_emb = host(di.gen_block_emb(w))
        if w.verify_batch == 0:  # verify every drafted block, as on the training workloads
            w = di.scaled(w, verify_batch=B * N, vocab=151936)
        vi = di.gen_verify(w)
        self.Bv = vi.draft.shape[0]
        self.V = w.vocab
        self.h_logits = host(vi.logits)
        self.h_draft = host(di.Tensor(vi.draft, "i32"))
        del vi
        self.d_mask = self.h_mask.to(device)
        self.d_sids = self.h_sids.to(device)
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
        self.h_out = torch.empty(self.out.shape, dtype=torch.float32)
        self.h_em = torch.empty(self.em.shape, dtype=torch.int32)
        self.h_ne = torch.empty(self.ne.shape, dtype=torch.int32)
        if pinned:
            self.h_out, self.h_em, self.h_ne = (t.pin_memory() for t in
                                                (self.h_out, self.h_em, self.h_ne))
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in
                             (self.h_mask, self.h_sids, self.h_emb, self.h_logits, self.h_draft) +
                             (() if w.inference else (self.h_hidden,)))
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in (self.h_out, self.h_em, self.h_ne))
        self.stream = torch.cuda.current_stream(device)
        if w.inference:
            self.build_cache()

    def use_f16_weights(self, on: bool):
        self.wts, self.cfg = (self.wts_f16, self.cfg_f16) if on else (self.wts_bf16, self.cfg_bf16)

    def build_cache(self):
        """The projected context of the inference workloads: built once, outside timing."""
        self.dflash.dflash_project_context(self.cfg, self.wts, self.d_hidden, self.B, self.L, 0,
                                           self.L, self.kv, ws=self.ws,
                                           stream=self.stream.cuda_stream)
        self.torch.cuda.synchronize()
        self.d_hidden = None

    def verify(self):
        d = self.dflash
        d.dflash_verify_greedy(self.d_logits, d.DFLASH_DTYPE_BF16 if self.h_logits.dtype ==
                               self.torch.bfloat16 else d.DFLASH_DTYPE_F32, self.d_draft, self.Bv,
                               self.S - 1, self.V, -1, self.em, self.ne, self.ac, ws=self.ws,
                               stream=self.stream.cuda_stream)

    def step(self):
        d, w = self.dflash, self.w
        st = self.stream.cuda_stream
        if not self.inference:
            d.dflash_plan(self.d_mask, self.d_sids, w.plan_step, w.plan_seed, self.N, self.S,
                          self.anchors, self.bv, self.lm, self.pid, ctx_len=self.ctx_len,
                          stream=st)
            d.dflash_project_context(self.cfg, self.wts, self.d_hidden, self.B, self.L, 0,
                                     self.L, self.kv, ctx_len=self.ctx_len, ws=self.ws, stream=st)
        d.dflash_body_forward(self.cfg, self.wts, self.d_emb, self.anchors, self.bv, self.pid,
                              self.d_mask, self.kv, self.B, self.L, self.N, self.out, ws=self.ws,
                              stream=st)
        self.verify()

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


def gemm_roofline(work: dict, inference: bool, gemm_ms: float, gemm_n: int, steps: int,
                  peaks: dict) -> dict:
    """The projection GEMMs (the dominant kernels) per launch: tensor-bound, or weight-read-
    bound when the FLOP per weight byte (2 * tokens / 2 bytes) is below the ridge point (a
    decode step).  Against the burst bf16 peak (the GEMMs are timed a launch at a time)."""
    peak, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    s_per_launch = gemm_ms / 1e3 / max(gemm_n, 1)
    wbytes = work["layer_weight_bytes"] + (0 if inference else work["ctx_weight_bytes"])
    intensity = work["gemm_flops"] / max(wbytes, 1)
    if intensity < peak * 1e12 / (hbm * 1e9):
        per_launch = wbytes * steps / max(gemm_n, 1)
        achieved = per_launch / s_per_launch / 1e9 if gemm_n else None
        return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm if achieved else None,
                "algorithmic_per_launch": per_launch,
                "algorithmic": "weight bytes read once per projection (bf16 layer matrices)",
                "peak_source": f"{peaks['source']} hbm_gbs"}
    per_launch = work["gemm_flops"] * steps / max(gemm_n, 1)
    achieved = per_launch / s_per_launch / 1e12 if gemm_n else None
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak if achieved else None,
            "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"] if achieved else None,
            "algorithmic_per_launch": per_launch,
            "algorithmic": "2*M*N*K over context rows below each row's largest anchor and "
                           "valid slots",
            "peak_source": f"{peaks['source']} bf16_tflops (burst; fp16 dense rate = bf16 dense "
                           "rate, nominal ratio 1)"}


BODY_TARGET = 0.50    # body forward: fraction of the bf16 dense peak on the 8B-shaped configs
VERIFY_TARGET = 0.70  # verification: fraction of HBM bandwidth


def measure(args, w: di.Workload, base: di.Workload, device, barrier, headline: bool) -> dict:
    """Times one workload.  Headline: the plain step (clocks sampled, launches counted), the
    same steps with per-kernel events, the end-to-end step from pinned host buffers and the
    fp16-weights-held variant.  Secondary: the plain and the per-kernel passes only."""
    import torch
    import block_draft_model_proj_gb300 as dflash
    steps = args.steps if headline else max(3, min(args.steps, 10))
    warmup = args.warmup if headline else max(3, min(args.warmup, 3))
    g = GpuStep(w, base, device, pinned=headline)
    stream = g.stream
    for _ in range(warmup):
        g.step()
    torch.cuda.synchronize()
    dflash.dflash_device_status()
    plan = {"anchors": g.anchors.cpu().numpy(), "block_valid": g.bv.cpu().numpy()}
    work = algorithmic_work(w, plan, g.h_mask.numpy())
    if w.inference:  # the cached context is not projected inside the step
        work["gemm_flops"] -= work["proj_flops"] + work["ctxkv_flops"]
        work["total_flops"] -= work["proj_flops"] + work["ctxkv_flops"]
    res = {"workload": w.name, "steps": steps}
    sampler = ClockSampler(device.index or 0) if headline else None
    launches0 = dflash.dflash_launch_count()
    if sampler:
        sampler.start()
    # the step as a user runs it (no per-kernel events between the launches, which would
    # serialise the programmatically dependent launches)
    ms = timed(g.step, steps, torch, stream, barrier)
    if sampler:
        res["clocks"] = sampler.stop()
    res["gpu_launches"] = dflash.dflash_launch_count() - launches0
    dflash.dflash_device_status()
    dflash.dflash_profile_enable(True)
    prof_ms = timed(g.step, steps, torch, stream, barrier)
    prof = dflash.dflash_profile_read()
    dflash.dflash_profile_enable(False)
    dflash.dflash_device_status()
    res.update({"ms": ms, "prof_ms": prof_ms, "prof": prof, "work": work, "g": g})
    if headline:
        for _ in range(2):
            g.step_e2e()
        res["e2e_ms"] = timed(g.step_e2e, steps, torch, stream, barrier)
        res["held_ms"] = 0.0
        if not w.inference and w.shape.dtype == "bf16":
            g.use_f16_weights(True)
            for _ in range(2):
                g.step()
            res["held_ms"] = timed(g.step, steps, torch, stream, barrier)
            g.use_f16_weights(False)
    return res


def summarize(r: dict, peaks: dict) -> dict:
    """Per-workload figures of one measured run (ms per step, throughput, rooflines)."""
    w, g, work, prof, steps = r["g"].w, r["g"], r["work"], r["prof"], r["steps"]
    step_s = r["ms"] / 1e3 / steps
    peak, hbm = peaks["bf16_tflops"], peaks["hbm_gbs"]
    gemm_ms, gemm_n = prof["gemm"]
    v_ms, v_n = prof["verify"]
    v_bytes = g.Bv * g.S * g.V * 2
    a_ms, _ = prof["attention"]
    # the body steps at small batch are bound by reading the weights, not by the tensor
    # cores: their step is measured against the weight-and-cache bytes at the HBM peak
    wbytes = work["layer_weight_bytes"] + work["attn_cache_bytes"] + \
        (0 if w.inference else work["ctx_weight_bytes"])
    t_tensor = work["total_flops"] / (peak * 1e12)
    t_hbm = wbytes / (hbm * 1e9)
    step = {"algorithmic_tflop_per_step": work["total_flops"] / 1e12,
            "achieved_tflops": work["total_flops"] / step_s / 1e12,
            "frac_of_burst_bf16": work["total_flops"] / step_s / 1e12 / peak,
            "frac_of_sustained_bf16": work["total_flops"] / step_s / 1e12 /
            peaks["bf16_tflops_sustained"],
            "bound": "tensor" if t_tensor >= t_hbm else "hbm",
            "frac_of_binding_roofline": max(t_tensor, t_hbm) / step_s}
    if step["bound"] == "tensor":
        step["target"] = f">= {BODY_TARGET} of the bf16 dense peak (burst)"
        step["target_met"] = step["frac_of_burst_bf16"] >= BODY_TARGET
    else:
        step["target"] = "HBM-bound step: fraction of the binding roofline reported"
        step["target_met"] = None
    verify = {"bound": "hbm", "bytes_per_call": v_bytes, "shape": [g.Bv, g.S, g.V],
              "achieved": v_bytes * steps / (v_ms / 1e3) / 1e9 if v_ms else None,
              "peak": hbm, "unit": "GB/s"}
    verify["frac"] = verify["achieved"] / hbm if verify["achieved"] else None
    verify["target_met"] = verify["frac"] >= VERIFY_TARGET if verify["frac"] else None
    return {"workload": w.name, "ms_per_step": r["ms"] / steps,
            "value": w.tokens / step_s, "unit": "block-positions/s",
            "valid_slots_per_step": work["valid_slots"], "step_roofline": step,
            "gemm_roofline": gemm_roofline(work, w.inference, gemm_ms, gemm_n, steps, peaks),
            "kernel_rooflines": {"verify": verify,
                                 "attention": attention_roofline(work, a_ms, steps, peak, hbm)},
            "kernel_ms_per_step": {k: v[0] / steps for k, v in prof.items()},
            "profiled_ms_per_step": r["prof_ms"] / steps,
            "kernel_flops_per_step": {k: work[k] for k in ("proj_flops", "ctxkv_flops",
                                                             "layer_flops", "attn_flops")}}


def verify_alone(args, device, Bv: int) -> dict:
    """Greedy verification alone on [Bv, 16, 151936] bf16 logits (larger than L2 at Bv >= 32):
    device time per call against the HBM peak."""
    import torch
    import block_draft_model_proj_gb300 as dflash
    w = di.scaled(di.WORKLOADS["decode_8b_b64_ctx4096"], verify_batch=Bv)
    vi = di.gen_verify(w)
    S, V = w.shape.block_size, w.vocab
    lg = torch.from_numpy(vi.logits.data.view(np.int16)).to(device).view(torch.bfloat16)
    dr = torch.from_numpy(vi.draft).to(device)
    em = torch.empty((Bv, S), dtype=torch.int32, device=device)
    ne = torch.empty((Bv,), dtype=torch.int32, device=device)
    ac = torch.empty_like(ne)
    ws = dflash.workspace(dflash.dflash_verify_workspace_size(Bv, S - 1, V), device)
    st = torch.cuda.current_stream(device)

    def call():
        dflash.dflash_verify_greedy(lg, dflash.DFLASH_DTYPE_BF16, dr, Bv, S - 1, V, -1, em, ne,
                                    ac, ws=ws, stream=st.cuda_stream)
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    dflash.dflash_device_status()
    assert np.array_equal(ac.cpu().numpy(), vi.planted_prefix)
    n = 50
    ms = timed(call, n, torch, st, lambda: None) / n
    nbytes = Bv * S * V * 2
    peaks = measured_peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"shape": [Bv, S, V], "us_per_call": ms * 1e3, "bytes_per_call": nbytes,
            "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": gbs / peaks["hbm_gbs"], "target_met": gbs / peaks["hbm_gbs"] >= VERIFY_TARGET,
            "l2": "logits larger than L2, read once per call"}


SECONDARY = ("train_8b_b4_l2048", "longctx_8b_l32768", "decode_8b_b1_ctx4096",
             "decode_8b_b64_ctx4096")


def run_ours(args, rank, world, local_rank):
    import torch
    import block_draft_model_proj_gb300 as dflash
    from block_draft_model_proj_gb300 import build as dbuild
    dbuild.build()
    dflash.load()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def shard(name):
        base = di.WORKLOADS[name]
        # every rank owns its own rows (a different data stream), all ranks share the model
        return (di.scaled(base, index=base.index + 97 * rank) if rank else base), base

    w, base = shard(args.workload)
    r = measure(args, w, base, device, barrier, headline=True)
    g = r["g"]
    t = torch.tensor([r["ms"], r["e2e_ms"], r["held_ms"]], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms, e2e_ms, held_ms = float(t[0]), float(t[1]), float(t[2])
    r["ms"] = ms
    steps = args.steps
    units = w.tokens * world * steps
    peaks = measured_peaks()
    head = summarize(r, peaks)
    roof = dict(head["gemm_roofline"])
    roof.update({"traffic": profiled_traffic(base.name),
                 "traffic_unit": "bytes per launch (ncu dram read + write)",
                 "kernel": "projection GEMMs (gemm_tc_kernel, gemm_ws_kernel): the dominant "
                           "kernels of the step",
                 "launches_per_step": r["prof"]["gemm"][1] / steps})
    sw = w.shape
    result = {
        "metric": METRIC, "value": units / (ms / 1e3), "unit": "block-positions/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": ms / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16+f16",
        "precision": "bf16 inputs and weights; W_proj bf16 x bf16, draft-layer projections "
                     "f16 x f16 (bf16 weight tiles converted to fp16 on chip for <= 512 tokens, "
                     "fp16 copies converted inside the call above that; fp16 activations), "
                     "fp32 accumulation and residual stream, attention f16 x f16 over an "
                     "fp16 context K/V cache",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, bf16)",
        "config": {"workload": f"{w.name}: B={w.batch} L={w.seq_len} N={w.num_anchors} "
                               f"S={sw.block_size} D={sw.hidden} "
                               f"W_proj {sw.concat_width}->{sw.hidden} "
                               f"NL={sw.num_layers} Hq/Hkv/dh={sw.num_heads}/"
                               f"{sw.num_kv_heads}/{sw.head_dim} I={sw.intermediate}"
                               f"; verify [{g.Bv},{g.S},{g.V}]",
                   "block_positions_per_step": w.tokens,
                   "valid_slots_per_step": head["valid_slots_per_step"],
                   "l2": "inputs larger than L2 (weights 2.1 GB, target hidden states and "
                         "verification logits read every step)",
                   "parallelism": f"replicas: {world} rank(s), each its own rows, no collective"},
        "roofline": roof,
        "step_roofline": head["step_roofline"],
        "kernel_rooflines": head["kernel_rooflines"],
        "kernel_ms_per_step": head["kernel_ms_per_step"],
        "profiled_ms_per_step": head["profiled_ms_per_step"],
        "kernel_flops_per_step": head["kernel_flops_per_step"],
        "peaks": {k: peaks[k] for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained",
                                        "source")},
        "clocks": r["clocks"],
        "gpu_launches": r["gpu_launches"],
        "e2e": {"value": units / (e2e_ms / 1e3), "unit": "block-positions/s",
                "h2d_bytes_per_step": g.h2d_bytes, "d2h_bytes_per_step": g.d2h_bytes},
    }
    if held_ms > 0:
        held_s = held_ms / 1e3 / steps
        result["fp16_weights_held"] = {
            "value": units / (held_ms / 1e3), "unit": "block-positions/s",
            "ms_per_step": held_ms / steps,
            "frac_of_burst_bf16": head["step_roofline"]["algorithmic_tflop_per_step"] /
            held_s / peaks["bf16_tflops"],
            "note": "same step with fp16 copies of the layer weights held by the trainer (its "
                    "optimizer writes the fp16 working copy) instead of the bf16 weights; not "
                    "the headline"}
    del r, g
    torch.cuda.empty_cache()
    if not args.headline_only:
        extra = {}
        for name in SECONDARY:
            if name == args.workload:
                continue
            ws_, wb = shard(name)
            rr = measure(args, ws_, wb, device, barrier, headline=False)
            extra[name] = summarize(rr, peaks)
            del rr
            torch.cuda.empty_cache()
        result["other_workloads"] = extra
        result["verify_alone"] = {f"b{b}": verify_alone(args, device, b) for b in (32, 64)}
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(base)
    return result


# --------------------------------------------------------------------------------------
# the oracle on the host cores
# --------------------------------------------------------------------------------------

def oracle_sample(w: di.Workload, b: int, prefix: int, mask, sids, model) -> int:
    """The oracle on one bounded sample of the workload: row b's plan, the context
    projection of positions [0, prefix), every block of row b anchored below `prefix`, and
    greedy verification of those blocks.  Anchors are spread uniformly over the row, so the
    context work per block position is that of the whole row.  Returns the block positions
    processed."""
    from oracle import dflash_oracle as orc
    s = w.shape
    plan = orc.build_plan(mask[b:b + 1], sids[b:b + 1], w.plan_step, w.plan_seed,
                          w.num_anchors, s.block_size)
    anchors, valid = plan["anchors"][0], plan["block_valid"][0]
    ks = [k for k in range(w.num_anchors) if 0 <= anchors[k] < prefix]
    if not ks:
        return 0
    need = max(1, max(int(anchors[k]) for k in ks))
    rows = di.gen_target_hidden_rows(w, b, 0, min(need, w.seq_len)).f64()
    kv = orc.project_context_row(s, model.top, model.layer, rows)
    emb = di.Tensor(di.gen_block_emb(di.scaled(w, batch=b + 1)).data[b], s.dtype).f64()
    for k in ks:
        orc.block_forward(s, model.top, model.layer, emb[k], int(anchors[k]), valid[k], mask[b],
                          kv, plan["position_ids"][0, k])
    vi = di.gen_verify(di.scaled(w, verify_batch=len(ks), vocab=w.vocab or 151936,
                                 index=w.index + 31 * b))
    orc.verify_greedy(vi.logits.f64(), vi.draft)
    return len(ks) * s.block_size


class OracleModel:
    """The workload's weights widened to fp64 for the oracle."""

    def __init__(self, w: di.Workload):
        top = di.gen_top_weights(w)
        self.top = {k: v.f64() for k, v in top.items()}
        self._layers = {}
        self.w = w

    def layer(self, l):
        if l not in self._layers:
            self._layers[l] = {k: v.f64() for k, v in di.gen_layer_weights(self.w, l).items()}
        return self._layers[l]


def cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_prefix(w: di.Workload) -> int:
    """Context positions per oracle sample: a quarter of the row for long rows."""
    return max(min(w.seq_len, 1024), w.seq_len // 4) if w.seq_len > 1024 else w.seq_len


def valid_rows(w: di.Workload) -> list:
    return [b for b in range(w.batch) if not any(r == b for r, _ in w.padded_rows)]


def cpu_baseline(w: di.Workload, min_s: float = 10.0, max_s: float = 30.0) -> dict:
    """The oracle as it stands on the host cores, samples of the workload until at least
    min_s seconds of work (at most max_s)."""
    mask, sids = di.gen_mask(w), di.gen_sample_ids(w)
    model = OracleModel(w)
    for l in range(w.shape.num_layers):
        model.layer(l)
    P = oracle_prefix(w)
    rows = valid_rows(w)
    t0 = time.perf_counter()
    units, n = 0, 0
    while True:
        units += oracle_sample(w, rows[n % len(rows)], P, mask, sids, model)
        n += 1
        dt = time.perf_counter() - t0
        if dt >= min_s or dt >= max_s or n >= 8 * len(rows):
            break
    return {"value": units / dt, "unit": "block-positions/s", "cores": cores(), "kind": "oracle",
            "sample": f"{n} sample(s) of {w.name}, each one row: plan, context projection of "
                      f"positions [0, {P}), every block of the row anchored below {P}, their "
                      f"verification; {units} block positions in {dt:.1f} s (fp64 NumPy)"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = di.WORKLOADS[args.workload]
    mask, sids = di.gen_mask(w), di.gen_sample_ids(w)
    model = OracleModel(w)
    for l in range(w.shape.num_layers):
        model.layer(l)
    rows = valid_rows(w)
    P = oracle_prefix(w)
    for i in range(args.warmup):
        oracle_sample(w, rows[i % len(rows)], P, mask, sids, model)
    t0 = time.perf_counter()
    units = 0
    for i in range(args.steps):
        units += oracle_sample(w, rows[i % len(rows)], P, mask, sids, model)
    dt = time.perf_counter() - t0
    value = units / dt
    sample = (f"each step = one row of {w.name}: plan, context projection of positions "
              f"[0, {P}), every block of the row anchored below {P}, their verification")
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
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the secondary workloads and the verification-alone timings")
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
