"""GPU parity past 2**31 elements per tensor.

Every byte and element offset of the kernels and of the C ABI must be 64-bit:
these shapes put the last heads' rows past element 2**31 (and past byte
2**32).  Inputs are drawn on the device from a seeded generator (too large to
draw on the host quickly); rows at both ends of the tensors, or whole heads,
are copied back and checked against the float64 oracle at the bf16 bar
(max|gpu - ref| <= 2e-2 * max|ref|).
"""

import gc

import numpy as np
import pytest
import torch

from block_sparse_attention_tra_gb300 import bsa, workloads
from oracle import nsa as onsa
from oracle import tra as otra

pytestmark = pytest.mark.gpu
TOL = 2e-2
LSE_TOL = 1e-2  # absolute, on the log-sum-exp (as the other NSA parity tests)

# 1100 heads of 16384 x 128: 2.31e9 elements per tensor (4.6 GB in bf16)
BIG_TRA = (1, 1100, 16384, 128)


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_attention_tra_gb300 import build

    build.build()
    bsa.load_library()
    yield
    assert bsa.device_error() == 0


@pytest.fixture(autouse=True)
def _release():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(got, ref):
    return float(np.abs(got - ref).max()) / max(float(np.abs(ref).max()), 1e-30)


def test_tra_forward_past_2_31_elements():
    B, H, T, D = BIG_TRA
    q, k, v = workloads.tra_inputs(B, H, T, D, "bf16", seed=11, device="cuda")
    assert q.numel() > 2**31
    out = bsa.tra_forward(q, k, v, 1.0, 2.0)
    torch.cuda.synchronize()
    rows = [0, 1, 127, 128, T // 2, T - 2, T - 1]
    for h in (0, H // 2, H - 1):
        sl = (slice(0, 1), slice(h, h + 1))
        ref = otra.tra_rows(f64(q[sl]), f64(k[sl]), f64(v[sl]), 1.0, 2.0, [(0, 0, i) for i in rows])
        err = rel_err(f64(out[0, h, rows]), ref)
        assert err <= TOL, f"head {h}: max err {err:.3e} of max|ref|"


def test_tra_backward_past_2_31_elements():
    B, H, T, D = BIG_TRA
    q, k, v = workloads.tra_inputs(B, H, T, D, "bf16", seed=12, device="cuda")
    do = torch.randn(q.shape, generator=torch.Generator(device="cuda").manual_seed(13), device="cuda").to(
        torch.bfloat16)
    grads = bsa.tra_backward(q, k, v, do, 1.0, 2.0)
    torch.cuda.synchronize()
    for h in (0, H - 1):
        sl = (slice(0, 1), slice(h, h + 1))
        refs = otra.tra_backward(f64(q[sl]), f64(k[sl]), f64(v[sl]), f64(do[sl]), 1.0, 2.0)
        for name, g, ref in zip(("dq", "dk", "dv"), grads, refs):
            err = rel_err(f64(g[sl]), ref)
            assert err <= TOL, f"{name} head {h}: max err {err:.3e} of max|ref|"


def test_tra_diff_past_2_31_elements():
    B, H, T, D = BIG_TRA
    q1, k1, v = workloads.tra_inputs(B, H, T, D, "bf16", seed=14, device="cuda")
    q2, k2, _ = workloads.tra_inputs(B, H, T, D, "bf16", seed=15, device="cuda")
    del _
    out = bsa.tra_diff_forward(q1, q2, k1, k2, v, 0.05, 0.5, 2.0, normalize=True)
    torch.cuda.synchronize()
    h = H - 1
    sl = (slice(0, 1), slice(h, h + 1))
    ref = otra.tra_diff_forward(f64(q1[sl]), f64(q2[sl]), f64(k1[sl]), f64(k2[sl]), f64(v[sl]), 0.05, 0.5, 2.0,
                                normalize=True)
    err = rel_err(f64(out[sl]), ref)
    assert err <= TOL, f"head {h}: max err {err:.3e} of max|ref|"


def test_nsa_select_past_2_31_elements():
    # 528 query heads (33 kv groups of 16) of 32768 x 128: 2.21e9 elements in q and o
    B, Hq, Hkv, T, D, bs, S = 1, 528, 33, 32768, 128, 64, 16
    q, k, v, idx = workloads.nsa_inputs(B, Hq, Hkv, T, D, bs, S, seed=16, device="cuda")
    assert q.numel() > 2**31
    out, lse = bsa.nsa_select_forward(q, k, v, idx.cuda(), bs, return_lse=True)
    torch.cuda.synchronize()
    G = Hq // Hkv
    for g in (0, Hkv // 2, Hkv - 1):
        for i in (0, 63, 64, T // 2, T - 1):
            toks = torch.as_tensor(onsa.selected_tokens(idx[0, g, i].numpy(), i, bs), device="cuda")
            ref_o, ref_l = onsa.softmax_attend(f64(q[0, g * G:(g + 1) * G, i]), f64(k[0, g, toks]),
                                               f64(v[0, g, toks]), D ** -0.5)
            err = rel_err(f64(out[0, g * G:(g + 1) * G, i]), ref_o)
            assert err <= TOL, f"group {g} row {i}: max err {err:.3e} of max|ref|"
            lerr = float(np.abs(f64(lse[0, g * G:(g + 1) * G, i]) - ref_l).max())
            assert lerr <= LSE_TOL, f"group {g} row {i}: lse err {lerr:.3e}"
