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
    ap.add_argument("--dtype", choices=["bf16", "fp32", "fp8"], default="bf16",
                    help="fixed layout: fp32 runs the SIMT kernels, fp8 the e4m3 forward")
    ap.add_argument("--Hkv", type=int, default=0,
                    help="packed layout with this many key/value heads (GQA); 0 = fixed layout")
    ap.add_argument("--Nq", type=int, default=0,
                    help="packed layout: queries per sequence (the last Nq of N; 0 = N)")
    ap.add_argument("--decode", action="store_true",
                    help="packed layout through fa_fwd_decode (split-KV); reports GB/s")
    ap.add_argument("--splits", type=int, default=0, help="decode split count (0 = suggested)")
    a = ap.parse_args()
    if a.Hkv and a.decode:
        return run_decode(a)
    if a.Hkv and a.dtype == "fp8":
        return run_packed_fp8(a)
    if a.Hkv:
        return run_packed(a)
    if a.dtype == "fp8":
        return run_fp8(a)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    shape = (a.B, a.H, a.N, a.d)
    dt = torch.float32 if a.dtype == "fp32" else torch.bfloat16
    q, k, v, do = (torch.randn(shape, generator=g, device="cuda").to(dt) for _ in range(4))
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
        print(f"{a.which} {a.dtype} B={a.B} H={a.H} N={a.N} d={a.d} causal={a.causal}: "
              f"{ms:.4f} ms {fl / ms / 1e9:.1f} TFLOP/s")
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


def run_packed(a):
    """B sequences of N keys each and the last Nq of their positions as queries (a chunked
    prefill step), H query heads over Hkv key/value heads, packed token by token."""
    import torch

    import exact_attention_25_gb300 as fa

    nq = a.Nq or a.N
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    mk = lambda rows, heads: torch.randn((rows, heads, a.d), generator=g, device="cuda").to(  # noqa: E731
        torch.bfloat16)
    q, k, v, do = mk(a.B * nq, a.H), mk(a.B * a.N, a.Hkv), mk(a.B * a.N, a.Hkv), mk(a.B * nq, a.H)
    cu_q = torch.arange(0, a.B * nq + 1, nq, dtype=torch.int32, device="cuda")
    cu_k = torch.arange(0, a.B * a.N + 1, a.N, dtype=torch.int32, device="cuda")
    scale = a.d ** -0.5
    o = torch.empty_like(q)
    lse = torch.empty((a.H, a.B * nq), device="cuda", dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_varlen_workspace_bytes(a.B * nq, a.H, a.d), dtype=torch.uint8,
                     device="cuda")
    fwd = lambda: fa.fa_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, nq, a.N, scale, a.causal)  # noqa: E731
    bwd = lambda: fa.fa_bwd_varlen(q, k, v, o, do, lse, dq, dk, dv, cu_q, cu_k, nq, a.N,  # noqa: E731
                                   scale, a.causal, ws)
    fwd()
    run = fwd if a.which == "fwd" else bwd
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
    # visible (query, key) pairs: every key for each query, or under the bottom-right causal
    # mask the keys j <= i + N - Nq of query i
    pairs = nq * a.N if not a.causal else sum(min(a.N, i + a.N - nq + 1) for i in range(nq))
    fl = 4.0 * a.B * a.H * pairs * a.d * (1.0 if a.which == "fwd" else 2.5)
    print(f"{a.which} packed B={a.B} H={a.H} Hkv={a.Hkv} Nq={nq} Nk={a.N} d={a.d} "
          f"causal={a.causal}: {ms:.4f} ms {fl / ms / 1e9:.1f} TFLOP/s")


def run_fp8(a):
    """The e4m3 forward (transpose of V, then the tensor-core kernel) on standard-normal codes
    with unit descale factors; FLOPs by the same convention as the bf16 forward."""
    import torch

    import exact_attention_25_gb300 as fa
    from exact_attention_25_gb300 import perfmodel

    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    shape = (a.B, a.H, a.N, a.d)
    q, k, v = (torch.randn(shape, generator=g, device="cuda").to(torch.float8_e4m3fn)
               for _ in range(3))
    o = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((a.B, a.H, a.N), device="cuda", dtype=torch.float32)
    ws = torch.empty(fa.fa_fwd_fp8_workspace_bytes(*shape), dtype=torch.uint8, device="cuda")
    run = lambda: fa.fa_fwd_fp8(q, k, v, o, lse, a.d ** -0.5, 1.0, 1.0, 1.0, a.causal, ws)  # noqa: E731
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
    fl = perfmodel.fwd_flops(*shape, a.causal)
    print(f"fwd fp8 B={a.B} H={a.H} N={a.N} d={a.d} causal={a.causal}: {ms:.4f} ms "
          f"{fl / ms / 1e9:.1f} TFLOP/s (transpose + forward)")


def run_packed_fp8(a):
    """The packed e4m3 forward on the batch of run_packed (B sequences of N keys, the last Nq
    positions as queries, H query heads over Hkv key/value heads), unit descale factors."""
    import torch

    import exact_attention_25_gb300 as fa

    nq = a.Nq or a.N
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    mk = lambda rows, heads: torch.randn((rows, heads, a.d), generator=g, device="cuda").to(  # noqa: E731
        torch.float8_e4m3fn)
    q, k, v = mk(a.B * nq, a.H), mk(a.B * a.N, a.Hkv), mk(a.B * a.N, a.Hkv)
    cu_q = torch.arange(0, a.B * nq + 1, nq, dtype=torch.int32, device="cuda")
    cu_k = torch.arange(0, a.B * a.N + 1, a.N, dtype=torch.int32, device="cuda")
    o = torch.empty((a.B * nq, a.H, a.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((a.H, a.B * nq), device="cuda", dtype=torch.float32)
    ws = torch.empty(fa.fa_fwd_fp8_varlen_workspace_bytes(a.B, a.N, a.Hkv, a.d), dtype=torch.uint8,
                     device="cuda")
    run = lambda: fa.fa_fwd_fp8_varlen(q, k, v, o, lse, cu_q, cu_k, nq, a.N, a.d ** -0.5,  # noqa: E731
                                       1.0, 1.0, 1.0, a.causal, ws)
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
    pairs = nq * a.N if not a.causal else sum(min(a.N, i + a.N - nq + 1) for i in range(nq))
    fl = 4.0 * a.B * a.H * pairs * a.d
    print(f"fwd fp8 packed B={a.B} H={a.H} Hkv={a.Hkv} Nq={nq} Nk={a.N} d={a.d} "
          f"causal={a.causal}: {ms:.4f} ms {fl / ms / 1e9:.1f} TFLOP/s (transpose + forward)")


def run_decode(a):
    """A decode step: B sequences of N cached keys, the last Nq positions (default 1) as
    queries, H query heads over Hkv key/value heads.  Bandwidth counts the bytes the step must
    move: K and V once, Q, O and the LSE."""
    import torch

    import exact_attention_25_gb300 as fa

    nq = a.Nq or 1
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    mk = lambda rows, heads: torch.randn((rows, heads, a.d), generator=g, device="cuda").to(  # noqa: E731
        torch.bfloat16)
    q, k, v = mk(a.B * nq, a.H), mk(a.B * a.N, a.Hkv), mk(a.B * a.N, a.Hkv)
    cu_q = torch.arange(0, a.B * nq + 1, nq, dtype=torch.int32, device="cuda")
    cu_k = torch.arange(0, a.B * a.N + 1, a.N, dtype=torch.int32, device="cuda")
    splits = a.splits or fa.fa_decode_num_splits(a.B, a.Hkv, a.N)
    o = torch.empty_like(q)
    lse = torch.empty((a.H, a.B * nq), device="cuda", dtype=torch.float32)
    nbytes = fa.fa_decode_workspace_bytes(a.B * nq, a.H, a.d, splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
    run = lambda: fa.fa_fwd_decode(q, k, v, o, lse, cu_q, cu_k, nq, a.N, a.d ** -0.5,  # noqa: E731
                                   a.causal, splits, ws)
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
    moved = 2 * k.numel() * 2 + 2 * q.numel() * 2 + lse.numel() * 4
    print(f"decode B={a.B} H={a.H} Hkv={a.Hkv} Nq={nq} Nk={a.N} d={a.d} causal={a.causal} "
          f"splits={splits}: {ms:.4f} ms {moved / ms / 1e6:.1f} GB/s")


if __name__ == "__main__":
    main()
