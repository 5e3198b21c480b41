"""Single-kernel cases on synthetic inputs, for profiling one kernel at a time (ncu).

    python -m block_draft_model_proj_gb300.kernel_cases gemm --m 8192 --n 4096 --k 20480
    python -m block_draft_model_proj_gb300.kernel_cases gemm --m 512 --n 24576 --k 4096 --f16
    python -m block_draft_model_proj_gb300.kernel_cases body --workload train_8b_b4_l2048
    python -m block_draft_model_proj_gb300.kernel_cases verify --workload decode_8b_b64_ctx4096
    python -m block_draft_model_proj_gb300.kernel_cases sampling --workload decode_8b_b64_ctx4096
    python -m block_draft_model_proj_gb300.kernel_cases loss --workload train_8b_b4_l2048

Each case builds its inputs once, runs the kernel `--iters` times and prints the mean
CUDA-event time per launch (a number printed under a profiler is not a benchmark).
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _timed(fn, iters):
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record()
    for _ in range(iters):
        fn()
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / iters


def case_gemm(args):
    import torch
    import block_draft_model_proj_gb300 as dflash
    g = torch.Generator(device="cuda").manual_seed(0)
    tdt = torch.float16 if args.f16 else torch.bfloat16
    A = torch.randn((args.m, args.k), generator=g, device="cuda").to(tdt)
    B = (torch.randn((args.n, args.k), generator=g, device="cuda") * 0.02).to(tdt)
    C = torch.empty((args.splits, args.m, args.n), dtype=torch.float32, device="cuda")
    dt = dflash.DFLASH_DTYPE_F16 if args.f16 else dflash.DFLASH_DTYPE_BF16

    def run():
        dflash.dflash_testing_gemm(dflash.DFLASH_TESTING_ENGINE_TC, dt, A, B, C, args.splits)
    run()
    dflash.dflash_device_status()
    ms = _timed(run, args.iters)
    flops = 2.0 * args.m * args.n * args.k
    print(f"gemm M={args.m} N={args.n} K={args.k} {'f16' if args.f16 else 'bf16'} "
          f"splits={args.splits}: {ms:.4f} ms/launch, {flops / ms / 1e9:.1f} TFLOP/s")


def case_gemm_ws(args):
    import torch
    import block_draft_model_proj_gb300 as dflash
    g = torch.Generator(device="cuda").manual_seed(0)
    X = torch.randn((args.m, args.k), generator=g, device="cuda").to(torch.float16)
    W = (torch.randn((args.n, args.k), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    C = torch.empty((args.splits, args.m, args.n), dtype=torch.float32, device="cuda")
    so = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run():
        dflash.dflash_testing_gemm_ws(X, W, dflash.DFLASH_DTYPE_BF16, C, args.splits, so)
    run()
    dflash.dflash_device_status()
    ms = _timed(run, args.iters)
    flops = 2.0 * args.m * args.n * args.k
    print(f"gemm_ws M={args.m} N={args.n} K={args.k} max_splits={args.splits} "
          f"(chose {int(so.cpu()[0])}): {ms:.4f} ms/launch, {flops / ms / 1e9:.1f} TFLOP/s")


def case_body(args):
    import torch
    import block_draft_model_proj_gb300 as dflash
    import dflash_inputs as di
    w = di.WORKLOADS[args.workload]
    if args.batch:
        w = di.scaled(w, batch=args.batch,
                      shared_sid_groups=tuple(g for g in w.shared_sid_groups
                                              if max(g) < args.batch),
                      padded_rows=tuple(r for r in w.padded_rows if r[0] < args.batch))
    s = w.shape
    B, L, N, S = w.batch, w.seq_len, w.num_anchors, s.block_size

    def dev(t):
        if t.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(t.data).view(np.int16)).cuda().view(
                torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(t.data)).cuda()
    top = {k: dev(v) for k, v in di.gen_top_weights(w).items()}
    layers = [{k: dev(v) for k, v in di.gen_layer_weights(w, l).items()} for l in range(s.num_layers)]
    wts = dflash.Weights(top, layers)
    cfg = dflash.make_config(s)
    mask = torch.from_numpy(di.gen_mask(w)).cuda()
    sids = torch.from_numpy(di.gen_sample_ids(w)).cuda()
    H = dev(di.gen_target_hidden(w))
    emb = dev(di.gen_block_emb(w))
    kv = torch.empty((s.num_layers, B, 2, s.num_kv_heads, L, s.head_dim), dtype=dflash.kv_cache_dtype(cfg),
                     device="cuda")
    if w.inference:
        a_np, v_np, p_np = di.inference_block_layout(w)
        anchors = torch.from_numpy(a_np).cuda()
        bv = torch.from_numpy(v_np).cuda()
        pid = torch.from_numpy(p_np).cuda()
    else:
        anchors = torch.empty((B, N), dtype=torch.int32, device="cuda")
        bv = torch.empty((B, N, S), dtype=torch.uint8, device="cuda")
        lm = torch.empty_like(bv)
        pid = torch.empty((B, N, S), dtype=torch.int32, device="cuda")
        dflash.dflash_plan(mask, sids, w.plan_step, w.plan_seed, N, S, anchors, bv, lm, pid)
    out = torch.empty((B, anchors.shape[1], S, s.hidden), dtype=torch.float32, device="cuda")
    ws = dflash.workspace(max(dflash.dflash_project_context_workspace_size(cfg, B, L),
                              dflash.dflash_body_workspace_size(cfg, B, L, anchors.shape[1])))
    dflash.dflash_project_context(cfg, wts, H, B, L, 0, L, kv, ws=ws)

    def run():
        dflash.dflash_body_forward(cfg, wts, emb, anchors, bv, pid, mask, kv, B, L,
                                   anchors.shape[1], out, ws=ws)
    run()
    dflash.dflash_device_status()
    ms = _timed(run, args.iters)
    print(f"body {w.name}: {ms:.4f} ms/call")


def case_verify(args):
    import torch
    import block_draft_model_proj_gb300 as dflash
    import dflash_inputs as di
    w = di.WORKLOADS[args.workload]
    vi = di.gen_verify(w)
    Bv, S, V = vi.logits.shape
    logits = torch.from_numpy(vi.logits.data.view(np.int16)).cuda().view(torch.bfloat16)
    draft = torch.from_numpy(vi.draft).cuda()
    em = torch.empty((Bv, S), dtype=torch.int32, device="cuda")
    ne = torch.empty((Bv,), dtype=torch.int32, device="cuda")
    ac = torch.empty_like(ne)
    ws = dflash.workspace(dflash.dflash_verify_workspace_size(Bv, S - 1, V))

    def run():
        dflash.dflash_verify_greedy(logits, dflash.DFLASH_DTYPE_BF16, draft, Bv, S - 1, V, -1, em,
                                    ne, ac, ws=ws)
    run()
    dflash.dflash_device_status()
    ms = _timed(run, args.iters)
    # device time of the kernels alone (CUDA events around the launches): back-to-back calls
    # from Python can be bound by the host
    dflash.dflash_profile_enable(True)
    _timed(run, args.iters)
    dev_ms, n = dflash.dflash_profile_read()["verify"]
    dflash.dflash_profile_enable(False)
    dev = dev_ms / max(args.iters, 1)
    nbytes = Bv * S * V * 2
    print(f"verify [{Bv},{S},{V}] bf16: {ms * 1e3:.2f} us/call wall, {dev * 1e3:.2f} us/call on "
          f"the device ({n} launches), {nbytes / dev / 1e6:.1f} GB/s")


def case_sampling(args):
    import torch
    import block_draft_model_proj_gb300 as dflash
    import dflash_inputs as di
    w = di.WORKLOADS[args.workload]
    vi = di.gen_verify(w)
    Bv, S, V = vi.logits.shape
    logits = torch.from_numpy(vi.logits.data.view(np.int16)).cuda().view(torch.bfloat16)
    draft = torch.from_numpy(vi.draft).cuda()
    # proposal distributions: the target's own at a higher temperature (a stand-in for the
    # drafter's), normalised per row
    q = torch.softmax(logits[:, :S - 1].float() / 1.3, dim=-1).contiguous()
    em = torch.empty((Bv, S), dtype=torch.int32, device="cuda")
    ne = torch.empty((Bv,), dtype=torch.int32, device="cuda")
    ac = torch.empty_like(ne)
    ws = dflash.workspace(dflash.load().dflash_verify_sampling_workspace_size(Bv, S - 1, V))

    def run():
        dflash.dflash_verify_sampling(logits, dflash.DFLASH_DTYPE_BF16, 1.0, q, draft, Bv, S - 1, V,
                                      1234, -1, em, ne, ac, ws=ws)
    run()
    dflash.dflash_device_status()
    dflash.dflash_profile_enable(True)
    _timed(run, args.iters)
    dev_ms, n = dflash.dflash_profile_read()["verify"]
    dflash.dflash_profile_enable(False)
    dev = dev_ms / max(args.iters, 1)
    nbytes = Bv * S * V * 2
    print(f"sampling verify [{Bv},{S},{V}] bf16: {dev * 1e3:.2f} us/call on the device "
          f"({n} launches), logits read at {nbytes / dev / 1e6:.1f} GB/s")


def case_loss(args):
    import torch
    import block_draft_model_proj_gb300 as dflash
    import dflash_inputs as di
    w = di.WORKLOADS[args.workload]
    s = w.shape
    T = w.tokens
    V = args.vocab
    g = torch.Generator(device="cuda").manual_seed(0)
    hidden = torch.randn((T, s.hidden), generator=g, device="cuda")
    lm = (torch.randn((V, s.hidden), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    targets = torch.randint(0, V, (T,), generator=g, device="cuda", dtype=torch.int32)
    mask = torch.ones((T,), dtype=torch.uint8, device="cuda")
    mask.view(-1, s.block_size)[:, 0] = 0
    ce = torch.empty((T,), dtype=torch.float32, device="cuda")
    loss = torch.empty((1,), dtype=torch.float32, device="cuda")
    ws = dflash.workspace(dflash.load().dflash_decayed_ce_workspace_size(T, s.hidden, V))

    def run():
        dflash.dflash_decayed_ce_loss(hidden, lm, targets, mask, T, s.block_size, s.hidden, V, 4.0,
                                      ce, loss, ws=ws)
    run()
    dflash.dflash_device_status()
    ms = _timed(run, args.iters)
    flops = 2.0 * int(mask.sum()) * V * s.hidden
    print(f"decayed CE T={T} D={s.hidden} V={V}: {ms:.4f} ms/call, {flops / ms / 1e9:.1f} TFLOP/s")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["gemm", "gemm_ws", "body", "verify", "sampling", "loss"])
    ap.add_argument("--m", type=int, default=8192)
    ap.add_argument("--n", type=int, default=4096)
    ap.add_argument("--k", type=int, default=20480)
    ap.add_argument("--splits", type=int, default=1)
    ap.add_argument("--f16", action="store_true", help="fp16 operands (else bf16)")
    ap.add_argument("--workload", default="train_8b_b4_l2048")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--batch", type=int, default=0, help="body: override the workload's batch")
    ap.add_argument("--vocab", type=int, default=151936, help="loss: vocab size")
    args = ap.parse_args(argv)
    from block_draft_model_proj_gb300 import build as b
    b.build()
    {"gemm": case_gemm, "gemm_ws": case_gemm_ws, "body": case_body,
     "verify": case_verify, "sampling": case_sampling, "loss": case_loss}[args.case](args)


if __name__ == "__main__":
    main()
