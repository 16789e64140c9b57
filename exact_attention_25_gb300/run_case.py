"""Run one forward or backward case a few times (for profilers and quick timing).

    python -m exact_attention_25_gb300.run_case --pass fwd --B 1 --H 32 --N 8192 --d 128 --causal

Inputs are seeded standard-normal bf16 tensors created on the device.  ``--pass bwd`` runs the
forward once untimed, then the backward stages; ``--stage`` restricts the backward to one
stage (0 preprocess, 1 dK/dV, 2 dQ) after one full backward.
"""
from __future__ import annotations

import argparse
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def main():
    import torch

    import exact_attention_25_gb300 as fa

    ap = argparse.ArgumentParser()
    ap.add_argument("--pass", dest="which", choices=["fwd", "bwd"], default="fwd")
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--H", type=int, default=32)
    ap.add_argument("--N", type=int, default=8192)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--stage", type=int, default=-1)
    ap.add_argument("--time", action="store_true", help="report CUDA-event timing")
    a = ap.parse_args()
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    shape = (a.B, a.H, a.N, a.d)
    q, k, v, do = (torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
                   for _ in range(4))
    scale = a.d ** -0.5
    o = torch.empty_like(q)
    lse = torch.empty((a.B, a.H, a.N), device="cuda", dtype=torch.float32)
    if a.time:
        from exact_attention_25_gb300 import perfmodel

        fa.fa_fwd(q, k, v, o, lse, scale, a.causal)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        ws = torch.empty(fa.fa_bwd_workspace_bytes(*shape), dtype=torch.uint8, device="cuda")
        run = {"fwd": lambda: fa.fa_fwd(q, k, v, o, lse, scale, a.causal),
               "bwd": lambda: fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, a.causal, ws)}[a.which]
        if a.which == "bwd" and a.stage >= 0:
            fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, a.causal, ws)
            run = lambda: fa.fa_bwd_stage(q, k, v, o, do, lse, dq, dk, dv, scale, a.causal, ws,  # noqa: E731
                                          a.stage)
        for _ in range(3):
            run()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(a.iters):
            run()
        e1.record()
        torch.cuda.synchronize()
        fa.fa_device_status()
        ms = e0.elapsed_time(e1) / a.iters
        fl = (perfmodel.fwd_flops if a.which == "fwd" else perfmodel.bwd_flops)(*shape, a.causal)
        if a.which == "bwd" and a.stage >= 0:
            print(f"bwd stage {a.stage} B={a.B} H={a.H} N={a.N} d={a.d} causal={a.causal}: "
                  f"{ms:.4f} ms")
            return
        print(f"{a.which} B={a.B} H={a.H} N={a.N} d={a.d} causal={a.causal}: {ms:.4f} ms "
              f"{fl / ms / 1e9:.1f} TFLOP/s")
        return
    if a.which == "fwd":
        for _ in range(a.iters):
            fa.fa_fwd(q, k, v, o, lse, scale, a.causal)
    else:
        fa.fa_fwd(q, k, v, o, lse, scale, a.causal)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        ws = torch.empty(fa.fa_bwd_workspace_bytes(*shape), dtype=torch.uint8, device="cuda")
        if a.stage >= 0:
            fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, a.causal, ws)
        for _ in range(a.iters):
            if a.stage >= 0:
                fa.fa_bwd_stage(q, k, v, o, do, lse, dq, dk, dv, scale, a.causal, ws, a.stage)
            else:
                fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, a.causal, ws)
    fa.fa_device_status()
    torch.cuda.synchronize()
    print("ok", a.which, shape, "causal" if a.causal else "full")


if __name__ == "__main__":
    main()
