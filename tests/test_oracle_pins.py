"""Pins for the fp64 oracle: checks against facts fixed by the mathematics, not by the oracle.

Each test names what it pins.  Together they are chosen so that a plausible slip in
``oracle/oracle.c`` (a wrong mask direction, a dropped scale, a transposed operand, a sign
error in dS, a missing Delta) fails at least one of them; ``test_oracle_mutations.py``
demonstrates that by compiling mutated copies of the oracle.
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle

RNG = np.random.default_rng(12345)


def rnd(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


# ----- closed forms ---------------------------------------------------------------------

@pytest.mark.parametrize("N,d", [(1, 4), (7, 3), (64, 16), (130, 8)])
def test_q_zero_noncausal_gives_column_mean_and_log_n(N, d):
    """Q = 0 => every logit is 0 => P uniform => O = column mean of V, lse = ln N."""
    q = np.zeros((N, d)); k = rnd(N, d); v = rnd(N, d)
    o, lse = oracle.attention_fwd_head(q, k, v, 0.7, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(0), o.shape), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.full(N, math.log(N)), rtol=0, atol=1e-13)


@pytest.mark.parametrize("N,d", [(1, 4), (9, 5), (100, 16)])
def test_q_zero_causal_gives_prefix_mean(N, d):
    """Causal, Q = 0 => row i is the mean of V_0..V_i and lse_i = ln(i+1)."""
    q = np.zeros((N, d)); k = rnd(N, d); v = rnd(N, d)
    o, lse = oracle.attention_fwd_head(q, k, v, 1.3, True)
    prefix = np.cumsum(v, 0) / np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(o, prefix, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.log(np.arange(1, N + 1)), rtol=0, atol=1e-13)


def test_causal_row_zero_is_v0():
    """Causal row 0 sees only key 0: O_0 = V_0 exactly and lse_0 = scale * q_0 . k_0."""
    N, d, scale = 33, 12, 0.25
    q, k, v = rnd(N, d), rnd(N, d), rnd(N, d)
    o, lse = oracle.attention_fwd_head(q, k, v, scale, True)
    np.testing.assert_array_equal(o[0], v[0])
    assert abs(lse[0] - scale * float(q[0] @ k[0])) < 1e-14


def test_scale_zero_is_uniform():
    """scale = 0 => uniform attention over the visible keys, whatever Q and K are."""
    N, d = 20, 6
    q, k, v = rnd(N, d, scale=5), rnd(N, d, scale=5), rnd(N, d)
    o, lse = oracle.attention_fwd_head(q, k, v, 0.0, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(0), o.shape), atol=1e-13)
    np.testing.assert_allclose(lse, math.log(N), atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_single_dominant_logit_selects_one_value_row(causal):
    """K_j = t * Q_i/|Q_i| with large t makes one logit exceed all others by > 40 nats,
    so O_i equals V_j to within exp(-40) relative weight."""
    N, d, scale = 48, 16, 1.0 / 4.0
    q, k, v = rnd(N, d), rnd(N, d), rnd(N, d)
    i, j = 40, 17
    qi = q[i] / np.linalg.norm(q[i])
    t = 400.0
    k[j] = t * qi
    o, _ = oracle.attention_fwd_head(q, k, v, scale, causal)
    s = scale * (k[: i + 1] if causal else k) @ q[i]
    gap = s[j] - np.max(np.delete(s, j))
    assert gap > 40
    np.testing.assert_allclose(o[i], v[j], atol=N * math.exp(-gap) * np.abs(v).max() + 1e-12)


def test_n_equals_one():
    """N = 1: the single row attends to itself only, O = V_0, lse = scale q.k."""
    q, k, v = rnd(1, 8), rnd(1, 8), rnd(1, 8)
    for causal in (False, True):
        o, lse = oracle.attention_fwd_head(q, k, v, 0.5, causal)
        np.testing.assert_array_equal(o, v)
        assert abs(lse[0] - 0.5 * float(q[0] @ k[0])) < 1e-15


def test_two_by_one_worked_by_hand():
    """N=2, d=1, worked by hand: q=(1,2), k=(0,1), v=(10,20), scale=1.
    Logits: row0 (0,1), row1 (0,2).  Non-causal O0 = (10 + 20e)/(1+e), O1 = (10+20e^2)/(1+e^2);
    causal O0 = 10, O1 as non-causal.  lse0 = ln(1+e), lse1 = ln(1+e^2)."""
    e = math.e
    q = np.array([[1.0], [2.0]]); k = np.array([[0.0], [1.0]]); v = np.array([[10.0], [20.0]])
    o, lse = oracle.attention_fwd_head(q, k, v, 1.0, False)
    assert abs(o[0, 0] - (10 + 20 * e) / (1 + e)) < 1e-13
    assert abs(o[1, 0] - (10 + 20 * e * e) / (1 + e * e)) < 1e-13
    assert abs(lse[0] - math.log(1 + e)) < 1e-14 and abs(lse[1] - math.log(1 + e * e)) < 1e-14
    o, lse = oracle.attention_fwd_head(q, k, v, 1.0, True)
    assert o[0, 0] == 10.0 and abs(lse[0] - 0.0) < 1e-15
    assert abs(o[1, 0] - (10 + 20 * e * e) / (1 + e * e)) < 1e-13


# ----- softmax rows ---------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_probabilities_are_rows_of_a_stochastic_matrix(causal):
    """P >= 0, each row sums to 1 (1e-14), and causal P is 0 strictly above the diagonal."""
    N, d = 70, 9
    _, _, P = oracle.attention_fwd_head(rnd(N, d, scale=3), rnd(N, d, scale=3), rnd(N, d), 0.9,
                                        causal, want_p=True)
    assert (P >= 0).all()
    np.testing.assert_allclose(P.sum(1), 1.0, rtol=0, atol=1e-14)
    if causal:
        assert (np.triu(P, 1) == 0).all()
        assert (np.diag(P) > 0).all()


# ----- invariants -----------------------------------------------------------------------

def test_joint_permutation_of_keys_and_values_leaves_output_unchanged():
    N, d = 40, 8
    q, k, v = rnd(N, d), rnd(N, d), rnd(N, d)
    perm = RNG.permutation(N)
    o1, l1 = oracle.attention_fwd_head(q, k, v, 0.4, False)
    o2, l2 = oracle.attention_fwd_head(q, k[perm], v[perm], 0.4, False)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)
    # a permutation that is not joint must change the result (pins the operand pairing)
    o3, _ = oracle.attention_fwd_head(q, k[perm], v, 0.4, False)
    assert np.abs(o3 - o1).max() > 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_shift_of_all_keys(causal):
    """K_j += u for all j shifts row i's logits by scale*q_i.u: O unchanged, lse += scale q_i.u."""
    N, d, scale = 30, 5, 0.6
    q, k, v = rnd(N, d), rnd(N, d), rnd(N, d)
    u = rnd(d)
    o1, l1 = oracle.attention_fwd_head(q, k, v, scale, causal)
    o2, l2 = oracle.attention_fwd_head(q, k + u, v, scale, causal)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, scale * q @ u, atol=1e-12)


def test_output_is_linear_in_v():
    N, d = 25, 7
    q, k, v1, v2 = rnd(N, d), rnd(N, d), rnd(N, d), rnd(N, d)
    a, b = 1.7, -0.3
    o1, _ = oracle.attention_fwd_head(q, k, v1, 0.5, True)
    o2, _ = oracle.attention_fwd_head(q, k, v2, 0.5, True)
    o3, _ = oracle.attention_fwd_head(q, k, a * v1 + b * v2, 0.5, True)
    np.testing.assert_allclose(o3, a * o1 + b * o2, atol=1e-12)


# ----- special cases that reduce to library routines --------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(5, 3), (64, 32), (129, 16)])
def test_matches_library_softmax_and_logsumexp(causal, N, d):
    """Row-by-row scipy.special.softmax / logsumexp on an explicitly masked S."""
    scale = 0.37
    q, k, v = rnd(N, d), rnd(N, d), rnd(N, d)
    o, lse = oracle.attention_fwd_head(q, k, v, scale, causal)
    S = scale * (q @ k.T)
    if causal:
        S = np.where(np.tril(np.ones((N, N), bool)), S, -np.inf)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(S, axis=1), atol=1e-12)
    np.testing.assert_allclose(o, scipy.special.softmax(S, axis=1) @ v, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_and_autograd_in_fp64(causal):
    """torch's scaled_dot_product_attention (CPU, float64) and its autograd gradients."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F

    B, H, N, d, scale = 2, 3, 45, 16, 0.2
    q, k, v, do = (rnd(B, H, N, d) for _ in range(4))
    t = [torch.tensor(x, requires_grad=True) for x in (q, k, v)]
    ref = F.scaled_dot_product_attention(*t, is_causal=causal, scale=scale)
    ref.backward(torch.tensor(do))
    o, lse = oracle.attention_fwd(q, k, v, scale, causal)
    np.testing.assert_allclose(o, ref.detach().numpy(), atol=1e-13)
    g = oracle.attention_bwd(q, k, v, do, scale, causal)
    for i, name in enumerate(("dq", "dk", "dv")):
        np.testing.assert_allclose(g[name], t[i].grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(g["o"], o, atol=1e-14)
    np.testing.assert_allclose(g["lse"], lse, atol=1e-14)


# ----- exactness of tiling (Algorithm 1 reaches Algorithm 0) ------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Br,Bc", [(1, 1), (4, 4), (16, 16), (7, 5), (64, 32), (200, 3), (3, 200)])
def test_tiled_online_softmax_equals_standard(causal, Br, Bc):
    N, d = 97, 12
    q, k, v = rnd(N, d, scale=2), rnd(N, d, scale=2), rnd(N, d)
    o0, l0 = oracle.attention_fwd_head(q, k, v, 0.8, causal)
    o1, l1 = oracle.attention_fwd_tiled_head(q, k, v, 0.8, causal, Br, Bc)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-12)


def test_tiled_path_with_large_logit_rows():
    """Rows scaled x10 (a large running max) still agree to 1e-12."""
    N, d = 80, 16
    q, k, v = rnd(N, d), rnd(N, d), rnd(N, d)
    q[::7] *= 10
    o0, l0 = oracle.attention_fwd_head(q, k, v, 0.25, False)
    o1, l1 = oracle.attention_fwd_tiled_head(q, k, v, 0.25, False, 16, 8)
    np.testing.assert_allclose(o1, o0, atol=1e-12)
    np.testing.assert_allclose(l1, l0, atol=1e-11)


# ----- backward --------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 1), (2, 3), (5, 4), (8, 2)])
def test_backward_matches_central_finite_differences(causal, N, d):
    """dQ, dK, dV against central differences of L = sum(dO o O) in fp64 (h = 1e-6)."""
    scale = 0.7
    q, k, v, do = rnd(N, d), rnd(N, d), rnd(N, d), rnd(N, d)
    g = oracle.attention_bwd_head(q, k, v, do, scale, causal)

    def loss(qq, kk, vv):
        o, _ = oracle.attention_fwd_head(qq, kk, vv, scale, causal)
        return float((o * do).sum())

    h = 1e-6
    for name, idx in (("dq", 0), ("dk", 1), ("dv", 2)):
        num = np.zeros((N, d))
        for a in range(N):
            for b in range(d):
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[idx][a, b] += h
                args_m[idx][a, b] -= h
                num[a, b] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        err = np.abs(num - g[name]).max() / max(1e-3, np.abs(num).max())
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("causal", [False, True])
def test_delta_identity_and_gradient_sums(causal):
    """Delta_i = dO_i . O_i; sum_j dK_j = 0 (rows of dS sum to 0); sum_j dV_j = sum_i dO_i."""
    N, d = 60, 10
    q, k, v, do = rnd(N, d), rnd(N, d), rnd(N, d), rnd(N, d)
    g = oracle.attention_bwd_head(q, k, v, do, 0.3, causal)
    np.testing.assert_allclose(g["delta"], (do * g["o"]).sum(1), atol=1e-12)
    np.testing.assert_allclose(g["dk"].sum(0), 0.0, atol=1e-12)
    np.testing.assert_allclose(g["dv"].sum(0), do.sum(0), atol=1e-12)
    if causal:  # the last key is seen only by the last query
        s = 0.3 * float(q[-1] @ k[-1])
        p = math.exp(s - g["lse"][-1])
        np.testing.assert_allclose(g["dv"][-1], p * do[-1], atol=1e-13)


# ----- sampled-rows mode -------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_rows_mode_equals_full_materialisation(causal):
    N, d = 150, 8
    q, k, v, do = rnd(N, d), rnd(N, d), rnd(N, d), rnd(N, d)
    full = oracle.attention_bwd_head(q, k, v, do, 0.45, causal)
    qr = [0, 1, 77, 149]
    kr = [0, 33, 148, 149]
    r = oracle.attention_rows_head(q, k, v, do, 0.45, causal, qr, kr, nthreads=3)
    np.testing.assert_allclose(r["o"], full["o"][qr], atol=1e-13)
    np.testing.assert_allclose(r["lse"], full["lse"][qr], atol=1e-13)
    np.testing.assert_allclose(r["delta"], full["delta"][qr], atol=1e-13)
    np.testing.assert_allclose(r["dq"], full["dq"][qr], atol=1e-12)
    np.testing.assert_allclose(r["dk"], full["dk"][kr], atol=1e-12)
    np.testing.assert_allclose(r["dv"], full["dv"][kr], atol=1e-12)


def test_batched_driver_equals_per_head():
    B, H, N, d = 2, 3, 19, 4
    q, k, v, do = (rnd(B, H, N, d) for _ in range(4))
    o, lse = oracle.attention_fwd(q, k, v, 0.5, True, nthreads=4)
    g = oracle.attention_bwd(q, k, v, do, 0.5, True, nthreads=4)
    for b in range(B):
        for h in range(H):
            o1, l1 = oracle.attention_fwd_head(q[b, h], k[b, h], v[b, h], 0.5, True)
            np.testing.assert_array_equal(o[b, h], o1)
            np.testing.assert_array_equal(lse[b, h], l1)
            g1 = oracle.attention_bwd_head(q[b, h], k[b, h], v[b, h], do[b, h], 0.5, True)
            for n in ("dq", "dk", "dv"):
                np.testing.assert_array_equal(g[n][b, h], g1[n])
