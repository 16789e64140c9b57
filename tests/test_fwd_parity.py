"""Forward parity: the CUDA library (through the C ABI) against the fp64 oracle, element by
element, on seeded inputs.  Covers the fp32 SIMT path, the bf16 tensor-core path with ragged
tails, canary guard regions, and the named workloads at their full sizes (every head of the
N = 4096 and N = 8192 workloads; sampled rows at N = 32000)."""
import time

import numpy as np
import pytest
import torch

import exact_attention_25_gb300 as fa
import oracle
from exact_attention_25_gb300.inputs import WORKLOADS, generate, random_qkv
from tests.gpu_util import check_fwd, f64, guarded_empty, oracle_threads, record_stats

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
    t0 = time.perf_counter()
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], w.scale, w.causal)
    stats = check_fwd(o, lse, ro, rl, torch.float32, w.name)
    stats["oracle_s"] = time.perf_counter() - t0
    record_stats(w.name, stats)


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


@pytest.mark.parametrize("name", ["bf16_b4h16_n4096_d64_hotrows",
                                  "bf16_b2h32_n8192_d128_causal"])
def test_workload_full_size_every_head(name):
    """Every head of the workload against the oracle, element by element, with the mean bound
    evaluated over the whole output tensor; for the workload with x10 query rows, every one of
    those rows is also held to the max bounds on its own."""
    w = WORKLOADS[name]
    x = generate(w)
    o, lse = run_fwd(x, w.causal)
    o_cpu, lse_cpu = o.cpu(), lse.cpu()
    # one batch entry per oracle call; each oracle thread holds S (and K^T) of one head
    nthr = oracle_threads(8.0 * w.N * (w.N + w.d) + 64e6)
    ro = np.empty(tuple(o_cpu.shape))
    rl = np.empty(tuple(lse_cpu.shape))
    t0 = time.perf_counter()
    for b in range(w.B):
        rob, rlb = oracle.attention_fwd(x["q"][b:b + 1], x["k"][b:b + 1], x["v"][b:b + 1],
                                        w.scale, w.causal, nthreads=nthr)
        ro[b], rl[b] = rob[0], rlb[0]
    oracle_s = time.perf_counter() - t0
    stats = check_fwd(o_cpu, lse_cpu, ro, rl, torch.bfloat16, name)
    stats["oracle_s"], stats["oracle_threads"] = oracle_s, nthr
    # the worst head by max |dO|, for the record
    per_head = np.abs(f64(o_cpu) - ro).reshape(w.B * w.H, -1).max(axis=1)
    stats["heads"] = w.B * w.H
    stats["worst_head_max_abs_o"] = float(per_head.max())
    record_stats(name, stats)
    if w.hot_rows_frac:
        hot = x["hot_rows"]
        assert len(hot) == round(w.hot_rows_frac * w.B * w.H * w.N)
        hs = check_fwd(o_cpu.reshape(-1, w.d)[hot], lse_cpu.reshape(-1)[hot],
                       ro.reshape(-1, w.d)[hot.numpy()], rl.reshape(-1)[hot.numpy()],
                       torch.bfloat16, "hot rows", check_mean=False)
        hs["rows"] = int(len(hot))
        record_stats(name + " x10 query rows", hs)


def test_workload_long_sequence_sampled_rows():
    w = WORKLOADS["bf16_b1h32_n32000_d128_causal_fwdbwd"]
    x = generate(w)
    o, lse = run_fwd(x, w.causal)
    o_cpu, lse_cpu = o.cpu(), lse.cpu()
    by_head = {}
    for h, i in x["samples"]:
        by_head.setdefault(h, []).append(i)
    got_o, got_l, ref_o, ref_l = [], [], [], []
    t0 = time.perf_counter()
    for h, rows in sorted(by_head.items()):
        res = oracle.attention_rows_head(x["q"][0, h], x["k"][0, h], x["v"][0, h],
                                         torch.zeros(w.N, w.d), w.scale, w.causal, rows, [])
        got_o.append(f64(o_cpu[0, h, rows]))
        got_l.append(f64(lse_cpu[0, h, rows]))
        ref_o.append(res["o"])
        ref_l.append(res["lse"])
    oracle_s = time.perf_counter() - t0
    stats = check_fwd(np.concatenate(got_o), np.concatenate(got_l), np.concatenate(ref_o),
                      np.concatenate(ref_l), torch.bfloat16, "N=32000 sampled rows",
                      check_mean=False)
    stats["rows"], stats["oracle_s"] = sum(len(r) for r in got_o), oracle_s
    record_stats(w.name + " forward", stats)
