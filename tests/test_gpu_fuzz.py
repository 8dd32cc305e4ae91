"""Seeded random shapes for the GPU paths, each against the float64 oracle.

The parity files check chosen shapes; these draw sizes, powers and group
sizes from a fixed seed so that many combinations of tile counts, ragged
tails, work items per CTA and MMA-issuer organisations (one issuer for the
general and half powers, one per query tile for p = 1, 2) are exercised, for
the forwards, the backward and the differential forward.
Bars: bf16 max|gpu - ref| <= 2e-2 * max|ref|, fp32 <= 1e-4 * max|ref|;
NSA lse within 1e-2 on rows with a valid key; the host-buffer path must be
bit-identical to the device path.
"""

import numpy as np
import pytest
import torch

from block_sparse_attention_tra_gb300 import bsa, workloads
from oracle import nsa as onsa
from oracle import tra as otra

pytestmark = pytest.mark.gpu

_rng = np.random.default_rng(20261202)
TRA_CASES = []
for _ in range(14):
    D = int(_rng.choice([64, 128]))
    p = float(_rng.choice([1.0, 2.0, 1.5, 0.7, 2.5, 3.0]))
    TRA_CASES.append((int(_rng.integers(1, 4)), int(_rng.integers(1, 7)), int(_rng.integers(1, 700)), D,
                      round(float(_rng.uniform(-0.5, 2.0)), 3), p, "bf16"))
for _ in range(3):
    TRA_CASES.append((1, int(_rng.integers(1, 4)), int(_rng.integers(1, 300)), int(_rng.choice([64, 128])),
                      round(float(_rng.uniform(0.0, 1.5)), 3), float(_rng.choice([1.0, 2.0, 1.5])), "f32"))
NSA_CASES = []
for G in (1, 2, 4, 8, 16, 8, 16, 3):
    Hkv = int(_rng.integers(1, 3))
    NSA_CASES.append((int(_rng.integers(1, 3)), G * Hkv, Hkv, 64 * int(_rng.integers(1, 11)),
                      int(_rng.choice([64, 128])), int(_rng.integers(1, 13))))
HOST_CASES = [(int(_rng.integers(1, 4)), int(_rng.integers(1, 12)), int(_rng.integers(1, 600)),
               int(_rng.choice([64, 128]))) for _ in range(3)]


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_attention_tra_gb300 import build

    build.build()
    bsa.load_library()
    torch.cuda.set_device(0)
    yield
    assert bsa.device_error() == 0


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(gpu, ref):
    return float(np.abs(gpu - ref).max()) / max(float(np.abs(ref).max()), 1e-30)


@pytest.mark.parametrize("B,H,T,D,beta,p,dtype", TRA_CASES)
def test_tra_random_shapes(B, H, T, D, beta, p, dtype):
    q, k, v = workloads.tra_inputs(B, H, T, D, dtype, seed=B * 1000 + H * 100 + T)
    out = bsa.tra_forward(q.cuda(), k.cuda(), v.cuda(), beta, p)
    torch.cuda.synchronize()
    ref = otra.tra_forward(f64(q), f64(k), f64(v), beta, p)
    tol = 1e-4 if dtype == "f32" else 2e-2
    err = rel_err(f64(out), ref)
    assert err <= tol, f"max err {err:.3e} of max|ref| (tol {tol})"


@pytest.mark.parametrize("B,Hq,Hkv,T,D,S", NSA_CASES)
def test_nsa_random_shapes_both_forms(B, Hq, Hkv, T, D, S):
    q, k, v, idx = workloads.nsa_inputs(B, Hq, Hkv, T, D, 64, S, seed=Hq * 100 + T + S)
    ro, rl = onsa.nsa_select_forward(f64(q), f64(k), f64(v), idx.numpy(), 64)
    outs = [bsa.nsa_select_forward(q.cuda(), k.cuda(), v.cuda(), idx.cuda(), 64, return_lse=True),
            bsa.nsa_select_forward_fsa(q.cuda(), k.cuda(), v.cuda(), idx.cuda(), 64, return_lse=True)]
    torch.cuda.synchronize()
    valid = rl != -1e9
    for name, (o, lse) in zip(("query-outer", "split-K"), outs):
        err = rel_err(f64(o), ro)
        assert err <= 2e-2, f"{name}: max err {err:.3e} of max|ref|"
        gl = f64(lse)
        assert np.all(gl[~valid] == -1e9), name
        if np.any(valid):
            assert float(np.abs(gl[valid] - rl[valid]).max()) <= 1e-2, name


@pytest.mark.parametrize("B,H,T,D", HOST_CASES)
def test_tra_host_random_shapes(B, H, T, D):
    q, k, v = workloads.tra_inputs(B, H, T, D, "bf16", seed=T + 7)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    got = bsa.tra_forward_host(hq, hk, hv, 0.8, 2.0)
    want = bsa.tra_forward(q.cuda(), k.cuda(), v.cuda(), 0.8, 2.0)
    torch.cuda.synchronize()
    assert torch.equal(got, want.cpu())


# Backward and differential forward: a second seeded stream, so the cases
# above stay as they are.  The backward draws p >= 1 only: for p < 1 the
# gradient p x^(p-1) is unbounded as x -> 0+, and an element-wise bar
# relative to max|ref| would then judge the rounding of x itself.
_rng2 = np.random.default_rng(20261203)
BWD_CASES = [(int(_rng2.integers(1, 3)), int(_rng2.integers(1, 4)), int(_rng2.integers(1, 600)),
              int(_rng2.choice([64, 128])), round(float(_rng2.uniform(-0.5, 2.0)), 3),
              float(_rng2.choice([1.0, 2.0, 1.5, 2.5, 3.0]))) for _ in range(8)]
DIFF_CASES = [(int(_rng2.integers(1, 3)), int(_rng2.integers(1, 4)), int(_rng2.integers(1, 600)),
               int(_rng2.choice([64, 128])), round(float(_rng2.uniform(-0.3, 1.0)), 3),
               round(float(_rng2.uniform(-0.5, 1.5)), 3), float(_rng2.choice([1.0, 2.0, 1.5, 0.7])),
               bool(_rng2.integers(0, 2))) for _ in range(8)]


# NSA selection for head dims and block sizes other than (D in {64, 128},
# 64-token blocks): the general query-outer kernel.
NSA_GEN_CASES = []
for _ in range(8):
    bs = int(_rng2.choice([16, 32, 64, 128]))
    D = int(_rng2.choice([16, 32, 64, 128]))
    if bs == 64 and D in (64, 128):
        D = 32  # that pair runs on the TMA kernel, covered above
    G, Hkv = int(_rng2.choice([1, 3, 8, 16])), int(_rng2.integers(1, 3))
    NSA_GEN_CASES.append((int(_rng2.integers(1, 3)), G * Hkv, Hkv, bs * int(_rng2.integers(1, 12)), D, bs,
                          int(_rng2.integers(1, 17))))


@pytest.mark.parametrize("B,Hq,Hkv,T,D,bs,S", NSA_GEN_CASES)
def test_nsa_general_random_shapes(B, Hq, Hkv, T, D, bs, S):
    q, k, v, idx = workloads.nsa_inputs(B, Hq, Hkv, T, D, bs, S, seed=Hq * 10 + T + S + D)
    ro, rl = onsa.nsa_select_forward(f64(q), f64(k), f64(v), idx.numpy(), bs)
    o, lse = bsa.nsa_select_forward(q.cuda(), k.cuda(), v.cuda(), idx.cuda(), bs, return_lse=True)
    torch.cuda.synchronize()
    err = rel_err(f64(o), ro)
    assert err <= 2e-2, f"max err {err:.3e} of max|ref|"
    gl, valid = f64(lse), rl != -1e9
    assert np.all(gl[~valid] == -1e9)
    if np.any(valid):
        assert float(np.abs(gl[valid] - rl[valid]).max()) <= 1e-2


@pytest.mark.parametrize("B,H,T,D,beta,p", BWD_CASES)
def test_tra_backward_random_shapes(B, H, T, D, beta, p):
    q, k, v = workloads.tra_inputs(B, H, T, D, "bf16", seed=T * 7 + D)
    do = torch.randn((B, H, T, D), generator=torch.Generator().manual_seed(T + 1)).to(torch.bfloat16)
    grads = bsa.tra_backward(q.cuda(), k.cuda(), v.cuda(), do.cuda(), beta, p)
    torch.cuda.synchronize()
    refs = otra.tra_backward(f64(q), f64(k), f64(v), f64(do), beta, p)
    for name, g, ref in zip(("dq", "dk", "dv"), grads, refs):
        err = rel_err(f64(g), ref)
        assert err <= 2e-2, f"{name}: max err {err:.3e} of max|ref|"


@pytest.mark.parametrize("B,H,T,D,beta,lam,p,norm", DIFF_CASES)
def test_tra_diff_random_shapes(B, H, T, D, beta, lam, p, norm):
    q1, k1, v = workloads.tra_inputs(B, H, T, D, "bf16", seed=T * 5 + D)
    q2, k2, _ = workloads.tra_inputs(B, H, T, D, "bf16", seed=T * 5 + D + 1)
    out = bsa.tra_diff_forward(q1.cuda(), q2.cuda(), k1.cuda(), k2.cuda(), v.cuda(), beta, lam, p, normalize=norm)
    torch.cuda.synchronize()
    ref = otra.tra_diff_forward(f64(q1), f64(q2), f64(k1), f64(k2), f64(v), beta, lam, p, normalize=norm)
    if float(np.abs(ref).max()) == 0.0:  # every score under its threshold: the output is exactly zero
        assert float(out.abs().max()) == 0.0
        return
    err = rel_err(f64(out), ref)
    assert err <= 2e-2, f"max err {err:.3e} of max|ref|"


# Head dims below the bf16 tile widths (16 .. 48 at width 64, 80 .. 112 at
# width 128, zero-filled columns), and the fp32 kernels built per head dim:
# a third seeded stream, so the cases above stay as they are.
_rng3 = np.random.default_rng(20261204)
_DIMS = [16, 32, 48, 80, 96, 112]
DIM_FWD_CASES = [(int(_rng3.integers(1, 3)), int(_rng3.integers(1, 4)), int(_rng3.integers(1, 500)),
                  int(_rng3.choice(_DIMS)), round(float(_rng3.uniform(-0.5, 2.0)), 3),
                  float(_rng3.choice([1.0, 2.0, 1.5, 0.7, 3.0])), str(_rng3.choice(["bf16", "bf16", "f32"])))
                 for _ in range(10)]
DIM_BWD_CASES = [(1, int(_rng3.integers(1, 3)), int(_rng3.integers(1, 400)), int(_rng3.choice(_DIMS)),
                  round(float(_rng3.uniform(-0.5, 2.0)), 3), float(_rng3.choice([1.0, 2.0, 1.5, 2.5])))
                 for _ in range(6)]
DIM_DIFF_CASES = [(1, int(_rng3.integers(1, 3)), int(_rng3.integers(1, 400)), int(_rng3.choice(_DIMS)),
                   round(float(_rng3.uniform(-0.3, 1.0)), 3), round(float(_rng3.uniform(-0.5, 1.5)), 3),
                   float(_rng3.choice([1.0, 2.0, 1.5])), bool(_rng3.integers(0, 2))) for _ in range(6)]


@pytest.mark.parametrize("B,H,T,D,beta,p,dtype", DIM_FWD_CASES)
def test_tra_forward_random_head_dims(B, H, T, D, beta, p, dtype):
    q, k, v = workloads.tra_inputs(B, H, T, D, dtype, seed=T * 3 + D)
    out = bsa.tra_forward(q.cuda(), k.cuda(), v.cuda(), beta, p)
    torch.cuda.synchronize()
    ref = otra.tra_forward(f64(q), f64(k), f64(v), beta, p)
    if float(np.abs(ref).max()) == 0.0:
        assert float(out.abs().max()) == 0.0
        return
    err = rel_err(f64(out), ref)
    assert err <= (2e-2 if dtype == "bf16" else 1e-4), f"max err {err:.3e} of max|ref|"


@pytest.mark.parametrize("B,H,T,D,beta,p", DIM_BWD_CASES)
def test_tra_backward_random_head_dims(B, H, T, D, beta, p):
    test_tra_backward_random_shapes(B, H, T, D, beta, p)


@pytest.mark.parametrize("B,H,T,D,beta,lam,p,norm", DIM_DIFF_CASES)
def test_tra_diff_random_head_dims(B, H, T, D, beta, lam, p, norm):
    test_tra_diff_random_shapes(B, H, T, D, beta, lam, p, norm)
