"""Backward parity: dQ, dK, dV from the CUDA library (through the C ABI, with O and LSE from the
library's own forward) against the fp64 oracle backward, which recomputes its own P.  Covers
ragged tails, the fp32 path, the SIMT cross-check, canaries, determinism and the named
workloads at full size (every head at N = 4096; at N = 32000 the oracle's row mode on 64
sampled query rows and 64 key rows; identities at every head)."""
import time

import numpy as np
import pytest
import torch

import exact_attention_25_gb300 as fa
import oracle
from exact_attention_25_gb300.inputs import WORKLOADS, generate, random_qkv
from tests.gpu_util import (TOL_GRAD_REL_L2, check_fwd, check_grads, f64, guarded_empty,
                            oracle_threads, record_stats, rel_l2)

pytestmark = pytest.mark.gpu


def run(x, causal, impl=0, scale=None):
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, scale=scale, causal=causal, impl=impl)
    fa.fa_device_status()
    return {"dq": dq, "dk": dk, "dv": dv, "o": o, "lse": lse}


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 2, 17, 64, 65, 127, 129, 255, 300, 1000, 4097])
def test_bf16_tail_sweep(N, d, causal):
    x = random_qkv(1, 2, N, d, seed=500 + N + d)
    got = run(x, causal)
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], d ** -0.5, causal)
    check_grads(got, ref, torch.bfloat16, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 33, 300])
def test_fp32_sweep(N, d, causal):
    x = random_qkv(1, 2, N, d, dtype=torch.float32, seed=900 + N)
    got = run(x, causal)
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], d ** -0.5, causal)
    check_grads(got, ref, torch.float32, f"fp32 N={N} d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_simt_cross_check_path(causal):
    x = random_qkv(1, 2, 400, 128, seed=21)
    got = run(x, causal, impl=1)
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], 128 ** -0.5, causal)
    check_grads(got, ref, torch.bfloat16, "simt")


@pytest.mark.parametrize("scale", [0.0, -0.3])
def test_unusual_scales(scale):
    x = random_qkv(1, 2, 200, 64, seed=31)
    for causal in (False, True):
        got = run(x, causal, scale=scale)
        ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal)
        # scale = 0: dQ and dK are exactly 0 in the oracle; compare dV only there
        if scale == 0.0:
            assert rel_l2(got["dv"], ref["dv"]) <= TOL_GRAD_REL_L2
            assert got["dq"].abs().max().item() == 0.0 and got["dk"].abs().max().item() == 0.0
        else:
            check_grads(got, ref, torch.bfloat16, f"scale={scale}")


@pytest.mark.parametrize("d", [64, 128])
def test_gradients_stay_inside_their_buffers_and_are_deterministic(d):
    B, H, N = 1, 2, 333
    x = random_qkv(B, H, N, d, seed=41)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    for causal in (False, True):
        o, lse = fa.forward(q, k, v, causal=causal)
        outs = []
        for _ in range(2):
            dq, cq = guarded_empty((B, H, N, d), torch.bfloat16)
            dk, ck = guarded_empty((B, H, N, d), torch.bfloat16)
            dv, cv = guarded_empty((B, H, N, d), torch.bfloat16)
            nbytes = fa.fa_bwd_workspace_bytes(B, H, N, d)
            ws, cw = guarded_empty((nbytes,), torch.uint8)
            fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, d ** -0.5, causal, ws)
            fa.fa_device_status()
            for c in (cq, ck, cv):
                c()
            outs.append([t.clone() for t in (dq, dk, dv)])
        for a, b in zip(*outs):
            assert torch.equal(a, b), "backward is not bit-for-bit deterministic"


def test_workload_bwd_b4h16_n4096_d128_causal():
    """Every head of the backward workload against the oracle backward: dQ, dK and dV by
    relative L2 over the whole tensors (and the forward's O and LSE that fed them)."""
    w = WORKLOADS["bf16_b4h16_n4096_d128_causal_bwd"]
    x = generate(w)
    got = run(x, w.causal)
    g = {n: got[n].cpu() for n in ("dq", "dk", "dv")}
    # each oracle thread holds P and dP of one head
    nthr = oracle_threads(16.0 * w.N * (w.N + 2 * w.d) + 64e6)
    t0 = time.perf_counter()
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], w.scale, w.causal, nthreads=nthr)
    oracle_s = time.perf_counter() - t0
    stats = check_grads(g, ref, torch.bfloat16, w.name)
    stats["oracle_s"], stats["oracle_threads"] = oracle_s, nthr
    for n in ("dq", "dk", "dv"):
        per_head = [rel_l2(g[n][b, h], ref[n][b, h]) for b in range(w.B) for h in range(w.H)]
        stats["worst_head_" + n] = max(per_head)
    stats["heads"] = w.B * w.H
    stats["fwd"] = check_fwd(got["o"].cpu(), got["lse"].cpu(), ref["o"], ref["lse"],
                             torch.bfloat16, w.name + " forward")
    record_stats(w.name, stats)
    check_gradient_identities(x, g, w)


def check_gradient_identities(x, g, w):
    """At every head: rows of dS sum to zero, so sum_j dK_j = 0; rows of P sum to one, so
    sum_j dV_j = sum_i dO_i.  Both hold for the exact gradients at any size."""
    dk_sum = g["dk"].double().sum(2)          # [B, H, d]
    dv_sum = g["dv"].double().sum(2)
    do_sum = x["do"].double().sum(2)
    dk_norm = g["dk"].double().abs().sum(2)   # scale of the terms being summed
    assert (dk_sum.abs() <= 2e-2 * dk_norm + 1e-3).all(), float((dk_sum.abs() / dk_norm).max())
    assert torch.allclose(dv_sum, do_sum, rtol=2e-2, atol=0.25), float((dv_sum - do_sum).abs().max())


def long_sequence_key_rows(x, w, n_heads=4, per_head=16):
    """Key rows whose dK and dV are compared at N = 32000: for the first n_heads sampled heads,
    that head's sampled rows plus seeded extra rows up to per_head, and the last row of the
    sequence (n_heads x per_head rows in all).  One pass of the oracle's row mode over a head
    gives all of its key rows at once."""
    by_head = {}
    for h, i in x["samples"]:
        by_head.setdefault(h, []).append(i)
    rng = np.random.default_rng(20260)
    out = {}
    for h in sorted(by_head)[:n_heads]:
        rows = set(by_head[h]) | {w.N - 1}
        while len(rows) < per_head:
            rows.add(int(rng.integers(0, w.N)))
        out[h] = sorted(rows)[:per_head] if len(rows) > per_head else sorted(rows)
    return by_head, out


def test_workload_long_sequence_sampled_rows():
    w = WORKLOADS["bf16_b1h32_n32000_d128_causal_fwdbwd"]
    x = generate(w)
    got = run(x, w.causal)
    g = {n: got[n].cpu() for n in ("dq", "dk", "dv")}
    by_head, key_rows = long_sequence_key_rows(x, w)
    assert sum(len(r) for r in key_rows.values()) == 64
    gq, rq = [], []
    gk, rk, gv, rv = [], [], [], []
    t0 = time.perf_counter()
    for h in sorted(set(by_head) | set(key_rows)):
        rows = by_head.get(h, [])
        krows = key_rows.get(h, [])
        res = oracle.attention_rows_head(x["q"][0, h], x["k"][0, h], x["v"][0, h], x["do"][0, h],
                                         w.scale, w.causal, rows, krows)
        gq.append(f64(g["dq"][0, h, rows]))
        rq.append(res["dq"])
        if krows:
            gk.append(f64(g["dk"][0, h, krows]))
            rk.append(res["dk"])
            gv.append(f64(g["dv"][0, h, krows]))
            rv.append(res["dv"])
    e_q = rel_l2(np.concatenate(gq), np.concatenate(rq))
    e_k = rel_l2(np.concatenate(gk), np.concatenate(rk))
    e_v = rel_l2(np.concatenate(gv), np.concatenate(rv))
    record_stats(w.name, {"dq_rows": sum(len(r) for r in gq), "dkv_rows": 64, "dq": e_q,
                          "dk": e_k, "dv": e_v, "oracle_s": time.perf_counter() - t0})
    assert e_q <= TOL_GRAD_REL_L2 and e_k <= TOL_GRAD_REL_L2 and e_v <= TOL_GRAD_REL_L2
    check_gradient_identities(x, g, w)
