"""The decode kernel's softmax exponential (the hardware 2^x approximation)
against exact 2^x, over the arguments the kernel gives it: x <= 0 (every
weight is 2^(logit - running max)), down to where the result leaves the
normal range. The measured relative error bounds its share of the output
error: every weight p_t carries a relative error of at most e, so the output
sum_t p_t v_t / sum_t p_t moves by at most 2e max|v|, far below the stated
max |d| <= 2e-3 for |v| up to 4 (the synthetic values are N(0, 1)).
"""
import ctypes as C

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_ex2_relative_error(ott):
    rng = np.random.default_rng(0)
    x = np.concatenate([
        -np.linspace(0.0, 126.0, 1_000_003),            # dense sweep of the normal range
        -rng.uniform(0.0, 1.0, 200_000),                # the weights that matter most
        -rng.uniform(0.0, 126.0, 300_000),
        [0.0, -1.0, -0.5, -125.999],
    ]).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    yd = torch.empty_like(xd)
    assert ott.load().ott_ex2_probe(C.c_void_p(xd.data_ptr()), C.c_void_p(yd.data_ptr()), x.size,
                                    C.c_void_p(torch.cuda.current_stream().cuda_stream)) == ott.OTT_OK
    torch.cuda.synchronize()
    y = yd.cpu().numpy().astype(np.float64)
    exact = np.exp2(x.astype(np.float64))
    rel = np.abs(y - exact) / exact
    worst = float(rel.max())
    print(f"ex2 max relative error {worst:.3e} ({np.log2(worst):.2f} in log2)")
    assert worst <= 2.0 ** -21
    assert y[-4] == 1.0                                  # 2^0 exactly: the running max's own weight
    # its effect on an output with values up to 4: far inside max |d| <= 2e-3
    assert 2 * worst * 4.0 < 1e-5
    # -inf (an empty or masked slot) gives exactly 0
    zd = torch.tensor([-float("inf")], device="cuda")
    assert ott.load().ott_ex2_probe(C.c_void_p(zd.data_ptr()), C.c_void_p(zd.data_ptr()), 1,
                                    C.c_void_p(torch.cuda.current_stream().cuda_stream)) == ott.OTT_OK
    torch.cuda.synchronize()
    assert float(zd.item()) == 0.0
