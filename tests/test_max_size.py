"""The largest fixed-length problem the ABI accepts: B*H*N*d = 2^31 - 65536 elements per
tensor (B=1, H=512, N=32767, d=128, causal; 4 GB per tensor), so that every 32-bit index or
offset that could overflow is exercised.  Inputs are drawn on the device (seeded); the fp64
oracle checks sampled rows of the first and the last head, where the byte offsets are
smallest and largest."""
import numpy as np
import pytest
import torch

import exact_attention_25_gb300 as fa
import oracle
from tests.gpu_util import TOL_GRAD_REL_L2, check_fwd, f64, rel_l2

pytestmark = pytest.mark.gpu

B, H, N, D = 1, 512, 32767, 128


def test_largest_accepted_problem_sampled_rows():
    assert B * H * N * D < 2 ** 31 and B * H * (N + 1) * D > 2 ** 31 - 2 ** 17
    free, _ = torch.cuda.mem_get_info()
    if free < 40 * 2 ** 30:
        pytest.skip("needs 40 GB of free device memory")
    g = torch.Generator(device="cuda")
    g.manual_seed(31)
    q, k, v, do = (torch.randn((B, H, N, D), generator=g, device="cuda", dtype=torch.bfloat16)
                   for _ in range(4))
    o, lse = fa.forward(q, k, v, causal=True)
    dq, dk, dv = fa.backward(q, k, v, o, do, lse, causal=True)
    fa.fa_device_status()
    rows = [0, 1, 4095, 20000, N - 129, N - 1]
    for h in (0, H - 1):
        x = {n: t[0, h].cpu() for n, t in (("q", q), ("k", k), ("v", v), ("do", do))}
        krows = [N - 1, 7] if h == H - 1 else []
        ref = oracle.attention_rows_head(x["q"], x["k"], x["v"], x["do"], D ** -0.5, True, rows,
                                         krows)
        check_fwd(o[0, h, rows], lse[0, h, rows], ref["o"], ref["lse"], torch.bfloat16,
                  f"head {h}", check_mean=False)
        assert rel_l2(dq[0, h, rows], ref["dq"]) <= TOL_GRAD_REL_L2
        if krows:
            assert rel_l2(dk[0, h, krows], ref["dk"]) <= TOL_GRAD_REL_L2
            assert rel_l2(dv[0, h, krows], ref["dv"]) <= TOL_GRAD_REL_L2
    # identities at every head (any size): rows of dS sum to 0, rows of P to 1
    dk_sum = dk.sum(2, dtype=torch.float64)
    dk_norm = dk.abs().sum(2, dtype=torch.float64)
    assert bool((dk_sum.abs() <= 2e-2 * dk_norm + 1e-3).all())
    assert torch.allclose(dv.sum(2, dtype=torch.float64), do.sum(2, dtype=torch.float64),
                          rtol=2e-2, atol=0.25)
    assert np.isfinite(f64(lse[0, :, -1])).all()
