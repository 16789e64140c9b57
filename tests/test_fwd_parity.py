"""Forward parity: the CUDA library (through the C ABI) against the fp64 oracle, element by
element, on seeded inputs.  Covers the fp32 SIMT path, the bf16 tensor-core path with ragged
tails, canary guard regions, and the named workloads at their full sizes (oracle on sampled
heads and rows)."""
import numpy as np
import pytest
import torch

import exact_attention_25_gb300 as fa
import oracle
from exact_attention_25_gb300.inputs import WORKLOADS, generate, random_qkv
from tests.gpu_util import check_fwd, f64, guarded_empty

pytestmark = pytest.mark.gpu

TAIL_NS = [1, 2, 17, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 1000, 4097]


def run_fwd(x, causal, impl=0, scale=None):
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o, lse = fa.forward(q, k, v, scale=scale, causal=causal, impl=impl)
    fa.fa_device_status()
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", TAIL_NS)
def test_bf16_tail_sweep(N, d, causal):
    x = random_qkv(1, 2, N, d, seed=1000 + N + d, with_do=False)
    o, lse = run_fwd(x, causal)
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], d ** -0.5, causal)
    check_fwd(o, lse, ro, rl, torch.bfloat16, f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 17, 129, 1000])
def test_fp32_sweep(N, d, causal):
    x = random_qkv(2, 1, N, d, dtype=torch.float32, seed=77 + N, with_do=False)
    o, lse = run_fwd(x, causal)
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], d ** -0.5, causal)
    check_fwd(o, lse, ro, rl, torch.float32, f"fp32 N={N} d={d} causal={causal}")


def test_workload_fp32_n512_d64():
    w = WORKLOADS["fp32_b1h1_n512_d64"]
    x = generate(w)
    o, lse = run_fwd(x, w.causal)
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], w.scale, w.causal)
    stats = check_fwd(o, lse, ro, rl, torch.float32, w.name)
    print(w.name, stats)


@pytest.mark.parametrize("causal", [False, True])
def test_simt_cross_check_path(causal):
    """The portable SIMT kernel with bf16 inputs also meets the bf16 bounds."""
    x = random_qkv(1, 3, 700, 128, seed=5, with_do=False)
    o, lse = run_fwd(x, causal, impl=1)
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], 128 ** -0.5, causal)
    check_fwd(o, lse, ro, rl, torch.bfloat16, "simt")


@pytest.mark.parametrize("scale", [0.0, -0.2, 1.0])
def test_unusual_scales(scale):
    """scale = 0 gives uniform attention; a negative scale flips the preference."""
    x = random_qkv(1, 2, 300, 64, seed=9, with_do=False)
    for causal in (False, True):
        o, lse = run_fwd(x, causal, scale=scale)
        ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal)
        check_fwd(o, lse, ro, rl, torch.bfloat16, f"scale={scale} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_outputs_stay_inside_their_buffers(d):
    B, H, N = 1, 3, 333
    x = random_qkv(B, H, N, d, seed=3, with_do=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    for causal in (False, True):
        o, chk_o = guarded_empty((B, H, N, d), torch.bfloat16)
        lse, chk_l = guarded_empty((B, H, N), torch.float32)
        fa.fa_fwd(q, k, v, o, lse, d ** -0.5, causal)
        fa.fa_device_status()
        chk_o()
        chk_l()
        ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], d ** -0.5, causal)
        check_fwd(o, lse, ro, rl, torch.bfloat16, "guarded")


def test_tensor_core_and_simt_agree_on_many_heads():
    """All heads of a medium shape: the two device paths agree within the bf16 bounds."""
    x = random_qkv(2, 8, 2048, 128, seed=11, with_do=False)
    for causal in (False, True):
        o1, l1 = run_fwd(x, causal)
        o2, l2 = run_fwd(x, causal, impl=1)
        assert (o1.float() - o2.float()).abs().max().item() <= 1.6e-2
        assert (l1 - l2).abs().max().item() <= 1e-3


def heads_to_check(w, n):
    """The first n (b, h) pairs in a seeded order (the same on every run)."""
    g = np.random.default_rng(1234)
    allh = [(b, h) for b in range(w.B) for h in range(w.H)]
    idx = g.permutation(len(allh))[:n]
    return [allh[i] for i in sorted(idx)]


@pytest.mark.parametrize("name,n_heads", [("bf16_b4h16_n4096_d64_hotrows", 4),
                                          ("bf16_b2h32_n8192_d128_causal", 2)])
def test_workload_full_size_sampled_heads(name, n_heads):
    w = WORKLOADS[name]
    x = generate(w)
    o, lse = run_fwd(x, w.causal)
    o_cpu, lse_cpu = o.cpu(), lse.cpu()
    assert torch.isfinite(o_cpu.float()).all() and torch.isfinite(lse_cpu).all()
    for b, h in heads_to_check(w, n_heads):
        ro, rl = oracle.attention_fwd_head(x["q"][b, h], x["k"][b, h], x["v"][b, h], w.scale,
                                           w.causal)
        stats = check_fwd(o_cpu[b, h], lse_cpu[b, h], ro, rl, torch.bfloat16, f"{name} b={b} h={h}")
        print(name, b, h, stats)
    if w.hot_rows_frac:
        # every hot row of the whole batch, one row at a time
        got_o, got_l, ref_o, ref_l = [], [], [], []
        for r in x["hot_rows"][:64].tolist():
            bh, i = divmod(r, w.N)
            b, h = divmod(bh, w.H)
            res = oracle.attention_rows_head(x["q"][b, h], x["k"][b, h], x["v"][b, h],
                                             torch.zeros(w.N, w.d), w.scale, w.causal, [i], [])
            got_o.append(f64(o_cpu[b, h, i:i + 1]))
            got_l.append(f64(lse_cpu[b, h, i:i + 1]))
            ref_o.append(res["o"])
            ref_l.append(res["lse"])
        stats = check_fwd(np.concatenate(got_o), np.concatenate(got_l), np.concatenate(ref_o),
                          np.concatenate(ref_l), torch.bfloat16, "hot rows", check_mean=False)
        print("hot rows (x10 queries)", stats)


def test_workload_long_sequence_sampled_rows():
    w = WORKLOADS["bf16_b1h32_n32000_d128_causal_fwdbwd"]
    x = generate(w)
    o, lse = run_fwd(x, w.causal)
    o_cpu, lse_cpu = o.cpu(), lse.cpu()
    by_head = {}
    for h, i in x["samples"]:
        by_head.setdefault(h, []).append(i)
    for h, rows in sorted(by_head.items()):
        res = oracle.attention_rows_head(x["q"][0, h], x["k"][0, h], x["v"][0, h],
                                         torch.zeros(w.N, w.d), w.scale, w.causal, rows, [])
        check_fwd(o_cpu[0, h, rows], lse_cpu[0, h, rows], res["o"], res["lse"], torch.bfloat16,
                  f"N=32000 h={h}", check_mean=False)
