"""Pins for the oracle's rectangular head (Nq != Nk, bottom-right causal mask) and its packed,
grouped-head driver.  Each check is fixed by the mathematics or by an already pinned function,
never by the code under test:

  * closed forms with Q = 0 (uniform weights over exactly the visible keys; rows that see no
    key give O = 0, lse = -inf), which pin the direction and the offset of the mask;
  * chunked prefill: the last c rows of a square causal problem are the rectangular problem of
    those c queries against every key ("PagedAttention·Chunked Prefill과의 위치" in "Flash
    Attention IO-awareness principle" puts the kernel inside each chunk);
  * central finite differences of L = sum(dO o O) for the backward;
  * grouped heads ("서빙에서 Flash Attention 이득이 예상보다 작은 경우", same page, on GQA / MQA)
    equal ordinary heads on key/value tensors repeated per group, with the gradients of each
    shared head summed (chain rule);
  * a packed batch equals its sequences run one by one through the square oracle.
"""
import math

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(2468)


def rnd(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def visible_counts(Nq, Nk, causal):
    """Keys row i sees: all Nk, or (causal, bottom-right) clamp(i + Nk - Nq + 1, 0, Nk)."""
    if not causal:
        return np.full(Nq, Nk)
    return np.clip(np.arange(Nq) + Nk - Nq + 1, 0, Nk)


@pytest.mark.parametrize("Nq,Nk", [(3, 7), (7, 3), (5, 5), (4, 1), (1, 6), (6, 0), (0, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_rect_q_zero_closed_form(Nq, Nk, causal):
    """Q = 0: row i averages V over the keys it sees, lse_i = ln(count); no key: O = 0, -inf."""
    d = 5
    q, k, v = np.zeros((Nq, d)), rnd(Nk, d), rnd(Nk, d)
    r = oracle.attention_rect_head(q, k, v, 0.9, causal)
    for i, c in enumerate(visible_counts(Nq, Nk, causal)):
        if c == 0:
            np.testing.assert_array_equal(r["o"][i], np.zeros(d))
            assert r["lse"][i] == -math.inf
        else:
            np.testing.assert_allclose(r["o"][i], v[:c].mean(0), rtol=0, atol=1e-13)
            assert abs(r["lse"][i] - math.log(c)) < 1e-13


@pytest.mark.parametrize("N,c", [(9, 4), (12, 12), (7, 1)])
def test_rect_is_the_tail_chunk_of_a_square_causal_problem(N, c):
    """Queries N-c..N-1 against all N keys (bottom-right) = the last c rows of the square causal
    problem; with dO = 0 on the other rows, dK and dV agree too."""
    d, scale = 6, 0.45
    q, k, v, do = rnd(N, d), rnd(N, d), rnd(N, d), rnd(N, d)
    do[: N - c] = 0.0
    sq = oracle.attention_bwd_head(q, k, v, do, scale, True)
    r = oracle.attention_rect_head(q[N - c:], k, v, scale, True, do=do[N - c:])
    np.testing.assert_allclose(r["o"], sq["o"][N - c:], rtol=0, atol=1e-13)
    np.testing.assert_allclose(r["lse"], sq["lse"][N - c:], rtol=0, atol=1e-13)
    np.testing.assert_allclose(r["dq"], sq["dq"][N - c:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dk"], sq["dk"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["dv"], sq["dv"], rtol=0, atol=1e-12)


@pytest.mark.parametrize("Nq,Nk,causal", [(3, 5, True), (5, 3, True), (4, 6, False), (2, 2, True)])
def test_rect_backward_matches_central_finite_differences(Nq, Nk, causal):
    """dQ, dK, dV of the rectangular head against central differences (h = 1e-6)."""
    d, scale = 3, 0.8
    q, k, v, do = rnd(Nq, d), rnd(Nk, d), rnd(Nk, d), rnd(Nq, d)
    g = oracle.attention_rect_head(q, k, v, scale, causal, do=do)

    def loss(qq, kk, vv):
        return float((oracle.attention_rect_head(qq, kk, vv, scale, causal)["o"] * do).sum())

    h = 1e-6
    for name, idx, arr in (("dq", 0, q), ("dk", 1, k), ("dv", 2, v)):
        num = np.zeros_like(arr)
        for a in range(arr.shape[0]):
            for b in range(d):
                args_p, args_m = [q.copy(), k.copy(), v.copy()], [q.copy(), k.copy(), v.copy()]
                args_p[idx][a, b] += h
                args_m[idx][a, b] -= h
                num[a, b] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(num - g[name]).max() / max(1e-3, np.abs(num).max())
        assert err < 1e-6, (name, err)
    # Delta_i = dO_i . O_i, also on rows that see no key (both 0 there)
    np.testing.assert_allclose(g["delta"], (do * g["o"]).sum(1), atol=1e-12)


def _packed(lens_q, lens_k, H, Hkv, d, scale=1.0):
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    q, do = rnd(int(cu_q[-1]), H, d, scale=scale), rnd(int(cu_q[-1]), H, d)
    k, v = rnd(int(cu_k[-1]), Hkv, d, scale=scale), rnd(int(cu_k[-1]), Hkv, d)
    return cu_q, cu_k, q, k, v, do


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (6, 1), (4, 4)])
def test_grouped_heads_equal_repeated_heads(causal, H, Hkv):
    """Query head h reads key/value head h // (H/Hkv): the same as ordinary heads on K, V
    repeated per group; the shared head's dK, dV are the sums over its group."""
    G = H // Hkv
    cu_q, cu_k, q, k, v, do = _packed([5, 3, 8], [7, 3, 6], H, Hkv, 4)
    g = oracle.attention_varlen(q, k, v, cu_q, cu_k, 0.6, causal, do=do)
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    r = oracle.attention_varlen(q, kr, vr, cu_q, cu_k, 0.6, causal, do=do)
    for name in ("o", "lse", "dq", "delta"):
        np.testing.assert_allclose(g[name], r[name], rtol=0, atol=1e-13)
    for name in ("dk", "dv"):
        summed = r[name].reshape(r[name].shape[0], Hkv, G, -1).sum(2)
        np.testing.assert_allclose(g[name], summed, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_packed_batch_equals_sequences_one_by_one(causal):
    """Equal query and key lengths per sequence: each sequence is the square problem of the
    pinned [B, H, N, d] oracle, including the [H, total] order of lse and Delta."""
    lens, H, d = [6, 1, 9, 4], 3, 5
    cu_q, cu_k, q, k, v, do = _packed(lens, lens, H, H, d)
    g = oracle.attention_varlen(q, k, v, cu_q, cu_k, 0.5, causal, do=do)
    for b, n in enumerate(lens):
        s = slice(cu_q[b], cu_q[b + 1])
        as_bhnd = lambda x: np.ascontiguousarray(x[s].transpose(1, 0, 2))[None]  # noqa: E731
        ref = oracle.attention_bwd(as_bhnd(q), as_bhnd(k), as_bhnd(v), as_bhnd(do), 0.5, causal)
        for name in ("o", "dq", "dk", "dv"):
            np.testing.assert_allclose(g[name][s], ref[name][0].transpose(1, 0, 2), atol=1e-12)
        np.testing.assert_allclose(g["lse"][:, s], ref["lse"][0], atol=1e-13)
        np.testing.assert_allclose(g["delta"][:, s], ref["delta"][0], atol=1e-12)


def test_empty_sequences_give_zero_outputs_and_gradients():
    """A sequence without keys: O = 0, lse = -inf, dQ = 0.  Without queries: dK = dV = 0."""
    cu_q, cu_k, q, k, v, do = _packed([3, 0, 2], [0, 4, 5], 2, 1, 4)
    g = oracle.attention_varlen(q, k, v, cu_q, cu_k, 0.7, True, do=do)
    np.testing.assert_array_equal(g["o"][0:3], 0.0)
    assert np.all(g["lse"][:, 0:3] == -math.inf)
    np.testing.assert_array_equal(g["dq"][0:3], 0.0)
    np.testing.assert_array_equal(g["dk"][0:4], 0.0)
    np.testing.assert_array_equal(g["dv"][0:4], 0.0)
    assert np.all(np.isfinite(g["o"][3:])) and np.abs(g["dk"][4:]).sum() > 0
