"""Plants plausible mistakes in a copy of the oracle (on the CPU) and checks that the pins in
``test_oracle_pins.py`` catch every one of them.  The real oracle is never modified."""
import ctypes
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
from tests import test_oracle_pins as pins
from tests import test_oracle_varlen_pins as vpins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement): each is a slip someone could plausibly make.
MUTATIONS = [
    ("mask_direction", "return !causal || j <= i;", "return !causal || j >= i;"),
    ("dropped_scale", "? scale * Si[j] : -INFINITY", "? Si[j] : -INFINITY"),
    ("lse_without_max", "lse[i] = m + log(l);\n        /* O_i", "lse[i] = log(l);\n        /* O_i"),
    ("ds_sign", "P[i * n + j] * (dP[i * n + j] - delta)", "P[i * n + j] * (dP[i * n + j] + delta)"),
    ("missing_delta", "P[i * n + j] * (dP[i * n + j] - delta)", "P[i * n + j] * dP[i * n + j]"),
    ("dk_unscaled", "dQ[i] *= scale; dK[i] *= scale;", "dQ[i] *= scale;"),
    ("dv_transposed", "double* dVj = dV + j * d;\n            const double* dOi = dO + i * d;",
     "double* dVj = dV + i * d;\n            const double* dOi = dO + j * d;"),
    ("dq_uses_q", "dQi[c] += ds * Kj[c];", "dQi[c] += ds * Qi[c];"),
    ("tiled_exponent", "a_new = exp(mt - mnew);", "a_new = exp(mt);"),
    ("tiled_no_rescale", "(l[i] * a_old * O[i * d + c] + a_new * PV[c]) / lnew",
     "(l[i] * O[i * d + c] + a_new * PV[c]) / lnew"),
    ("rows_delta", "ds = p * (jb->dp[j] - delta_i)", "ds = p * jb->dp[j]"),
    ("rect_offset_sign", "if (causal && j > i + off)", "if (causal && j > i - off)"),
    ("rect_top_left_mask", "if (causal && j > i + off)", "if (causal && j > i)"),
    ("rect_empty_row_lse", "lse[i] = -INFINITY;\n        } else {", "lse[i] = 0.0;\n        } else {"),
    ("rect_dk_unscaled", "for (long x = 0; x < nk * d; ++x) dK[x] *= scale;", ""),
    ("rect_missing_delta", "P[i * nk + j] * (dP[i * nk + j] - dl)", "P[i * nk + j] * dP[i * nk + j]"),
    ("rect_dv_uses_ds", "dV[j * d + c] += p * dO[i * d + c];", "dV[j * d + c] += ds * dO[i * d + c];"),
]

# Pin calls run against each mutant; each is (callable, args).
PIN_CALLS = [
    (pins.test_q_zero_causal_gives_prefix_mean, (9, 5)),
    (pins.test_causal_row_zero_is_v0, ()),
    (pins.test_single_dominant_logit_selects_one_value_row, (False,)),
    (pins.test_two_by_one_worked_by_hand, ()),
    (pins.test_shift_of_all_keys, (True,)),
    (pins.test_matches_library_softmax_and_logsumexp, (True, 5, 3)),
    (pins.test_tiled_online_softmax_equals_standard, (True, 7, 5)),
    (pins.test_backward_matches_central_finite_differences, (True, 5, 4)),
    (pins.test_backward_matches_central_finite_differences, (False, 5, 4)),
    (pins.test_delta_identity_and_gradient_sums, (True,)),
    (pins.test_rows_mode_equals_full_materialisation, (True,)),
    (vpins.test_rect_q_zero_closed_form, (7, 3, True)),
    (vpins.test_rect_q_zero_closed_form, (3, 7, True)),
    (vpins.test_rect_is_the_tail_chunk_of_a_square_causal_problem, (9, 4)),
    (vpins.test_rect_backward_matches_central_finite_differences, (3, 5, True)),
    (vpins.test_rect_backward_matches_central_finite_differences, (4, 6, False)),
    (vpins.test_empty_sequences_give_zero_outputs_and_gradients, ()),
]


def _build_mutant(tmp, text, repl):
    src = open(SRC).read()
    assert src.count(text) == 1, f"mutation anchor not unique or missing: {text!r}"
    path = os.path.join(tmp, "oracle_mut.c")
    with open(path, "w") as f:
        f.write(src.replace(text, repl))
    lib = os.path.join(tmp, "liboracle_mut.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", lib,
                           path, "-lm"])
    return lib


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name,text,repl", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(name, text, repl, monkeypatch):
    with tempfile.TemporaryDirectory() as tmp:
        lib_path = _build_mutant(tmp, text, repl)
        real = oracle._load()
        mutant = ctypes.CDLL(lib_path)
        for fn in ("oracle_attention_fwd_head", "oracle_attention_bwd_head",
                   "oracle_attention_fwd_tiled_head", "oracle_attention_rows_head",
                   "oracle_attention_fwd", "oracle_attention_bwd", "oracle_attention_rect_head"):
            f = getattr(mutant, fn)
            f.argtypes = getattr(real, fn).argtypes
            f.restype = ctypes.c_int
        monkeypatch.setattr(oracle, "_lib", mutant)
        caught = []
        for fn, args in PIN_CALLS:
            try:
                fn(*args)
            except (AssertionError, RuntimeError):
                caught.append(fn.__name__)
        assert caught, f"no pin caught mutation {name}"
