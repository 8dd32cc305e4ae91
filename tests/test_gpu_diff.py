"""GPU parity of the fused threshold differential attention (tra_diff_forward
through the C ABI) against the float64 oracle.

Bar: max|gpu - ref| <= 2e-2 * max|ref| over the whole output (bf16 inputs).
"""

import numpy as np
import pytest
import torch

from block_sparse_attention_tra_gb300 import bsa, workloads
from oracle import tra as otra

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_attention_tra_gb300 import build

    build.build()
    bsa.load_library()
    yield
    assert bsa.device_error() == 0


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def inputs(B, H, T, D, seed):
    q1, k1, v = workloads.tra_inputs(B, H, T, D, "bf16", seed=seed)
    q2, k2, _ = workloads.tra_inputs(B, H, T, D, "bf16", seed=seed + 1)
    return q1, q2, k1, k2, v


CASES = [
    # (B, H, T, D, beta, lam, p, normalize)
    (1, 2, 256, 128, 0.0, 0.5, 2.0, True),
    (1, 2, 300, 64, 0.2, 0.8, 1.5, True),   # ragged, general power
    (2, 1, 129, 128, 0.0, 0.3, 1.0, False),
    (1, 1, 1, 64, 1.0, 0.5, 2.0, True),
    (1, 2, 640, 64, 0.0, 1.5, 2.0, True),   # lambda clamps to 1
    (1, 1, 384, 128, 0.5, -1.0, 2.0, False),  # lambda clamps to 0
    (2, 2, 1024, 128, 0.05, 0.5, 2.0, True),
    (2, 3, 500, 64, 0.3, 0.6, 1.0, False),  # D = 64, p = 1: one MMA issuer per stream
    (1, 2, 300, 32, 0.2, 0.5, 2.0, True),   # head dim 32 (width-64 tiles, zero-filled columns)
    (1, 1, 257, 16, 0.0, 0.7, 1.5, True),   # head dim 16, general power
    (1, 2, 130, 32, 0.3, 0.4, 1.0, False),
    (1, 2, 300, 96, 0.2, 0.5, 2.0, True),   # head dims 96, 48, 112 (zero-filled columns)
    (1, 1, 257, 48, 0.0, 0.7, 1.5, True),
    (1, 2, 200, 112, 0.3, 0.4, 1.0, False),
]


@pytest.mark.parametrize("B,H,T,D,beta,lam,p,norm", CASES)
def test_tra_diff_full_output(B, H, T, D, beta, lam, p, norm):
    q1, q2, k1, k2, v = inputs(B, H, T, D, seed=T + D)
    out = bsa.tra_diff_forward(*(t.cuda() for t in (q1, q2, k1, k2, v)), beta, lam, p, normalize=norm)
    torch.cuda.synchronize()
    ref = otra.tra_diff_forward(f64(q1), f64(q2), f64(k1), f64(k2), f64(v), beta, lam, p, normalize=norm)
    err = float(np.abs(f64(out) - ref).max()) / max(float(np.abs(ref).max()), 1e-30)
    assert err <= TOL, f"max err {err:.3e} of max|ref|"


def test_tra_diff_equal_streams_cancel():
    q1, _, k1, _, v = inputs(1, 2, 256, 64, seed=5)
    out = bsa.tra_diff_forward(q1.cuda(), q1.cuda(), k1.cuda(), k1.cuda(), v.cuda(), 0.0, 1.0, 2.0)
    plain = bsa.tra_forward(q1.cuda(), k1.cuda(), v.cuda(), 0.0, 2.0)
    torch.cuda.synchronize()
    # identical streams run identical MMAs into their own fp32 accumulators,
    # so O_0 - 1 * O_1 cancels exactly
    assert float(plain.abs().max()) > 0
    assert float(out.abs().max()) == 0.0


def test_tra_diff_full_workload_sampled_heads():
    # The bench's differential workload (B4 H16 T4096 D128, p=2, lambda=0.5,
    # normalised); three (b, h) heads checked in full against the oracle.
    w = workloads.TRA_WORKLOADS["tra_bf16_B4_H16_T4096_D128"]
    q1, k1, v = workloads.workload_inputs(w)
    gen = torch.Generator().manual_seed(1)
    q2 = torch.randn(q1.shape, generator=gen).to(torch.bfloat16)
    k2 = torch.randn(q1.shape, generator=gen).to(torch.bfloat16)
    out = bsa.tra_diff_forward(q1.cuda(), q2.cuda(), k1.cuda(), k2.cuda(), v.cuda(), w.beta, 0.5, w.p, normalize=True)
    torch.cuda.synchronize()
    for b, h in [(0, 0), (2, 9), (3, 15)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = otra.tra_diff_forward(f64(q1[sl]), f64(q2[sl]), f64(k1[sl]), f64(k2[sl]), f64(v[sl]), w.beta, 0.5, w.p,
                                    normalize=True)
        err = float(np.abs(f64(out[sl]) - ref).max()) / max(float(np.abs(ref).max()), 1e-30)
        assert err <= TOL, f"head ({b},{h}): max err {err:.3e} of max|ref|"


@pytest.mark.parametrize("normalize", [True, False])
def test_tra_diff_head_groups_cover_every_head(normalize):
    # At the bench shape the blocks run in head groups of unequal size (64
    # heads in three groups).  Each output row is computed by one CTA with the
    # same arithmetic whatever the block order (and the row norms per row), so
    # the full call must equal single-head calls bit for bit on every head.
    w = workloads.TRA_WORKLOADS["tra_bf16_B4_H16_T4096_D128"]
    q1, q2, k1, k2, v = (t.cuda() for t in inputs(w.B, w.H, w.T, w.D, seed=5))
    full = bsa.tra_diff_forward(q1, q2, k1, k2, v, w.beta, 0.5, w.p, normalize=normalize)
    for b in range(w.B):
        for h in range(w.H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            one = bsa.tra_diff_forward(q1[sl], q2[sl], k1[sl], k2[sl], v[sl], w.beta, 0.5, w.p, normalize=normalize)
            assert torch.equal(full[sl], one), f"head ({b},{h}) differs from its single-head call"


# fp32 inputs: the CUDA-core FFMA kernel (normalisation folded into the
# scores, no scratch), at the fp32 bar.
F32_TOL = 1e-4
F32_CASES = [
    # (B, H, T, D, beta, lam, p, normalize)
    (1, 2, 256, 64, 0.0, 0.5, 2.0, True),
    (2, 1, 200, 128, 0.2, 0.8, 1.5, True),   # ragged, general power
    (1, 2, 130, 64, 0.5, 0.3, 1.0, False),
    (1, 1, 1, 128, 1.0, 0.5, 2.0, True),
    (1, 1, 320, 64, 0.1, 1.5, 2.0, False),   # lambda clamps to 1
    (1, 2, 150, 32, 0.2, 0.5, 2.0, True),    # head dim 32
    (1, 1, 100, 16, 0.0, 0.6, 1.5, True),    # head dim 16
    (1, 1, 120, 96, 0.2, 0.5, 2.0, True),    # head dim 96
]


@pytest.mark.parametrize("B,H,T,D,beta,lam,p,norm", F32_CASES)
def test_tra_diff_f32(B, H, T, D, beta, lam, p, norm):
    q1, k1, v = workloads.tra_inputs(B, H, T, D, "f32", seed=T + D)
    q2, k2, _ = workloads.tra_inputs(B, H, T, D, "f32", seed=T + D + 1)
    ts = [t.cuda() for t in (q1, q2, k1, k2, v)]
    out = bsa.tra_diff_forward(*ts, beta, lam, p, normalize=norm)
    torch.cuda.synchronize()
    assert out.dtype == torch.float32
    ref = otra.tra_diff_forward(f64(q1), f64(q2), f64(k1), f64(k2), f64(v), beta, lam, p, normalize=norm)
    err = float(np.abs(f64(out) - ref).max()) / max(float(np.abs(ref).max()), 1e-30)
    assert err <= F32_TOL, f"max err {err:.3e} of max|ref|"
    # the allocation-free entry point runs the same fp32 kernel (it needs no scratch)
    out2 = torch.empty_like(out)
    st = bsa.tra_diff_forward_noalloc_raw(*(t.data_ptr() for t in ts), out2.data_ptr(), B, H, T, D, beta, lam, p,
                                          norm, bsa.BSA_F32, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0 and torch.equal(out, out2)


# Gradients of the differential form (tra_diff_backward) against the float64
# oracle: each of dq1, dq2, dk1, dk2, dv within the bar of its own max|ref|,
# and dlambda within the bar of sum|dout * TRA(a2, b2, v)| (the size of the
# terms it sums).  Powers p > 1 only (plus p = 1 without normalisation): the
# gradient's factor p x^(p-1) jumps at x = 0 for p = 1, and normalised scores
# crowd around tau, so bf16 rounding of the inputs flips it for some pairs.
BWD_CASES = [
    # (B, H, T, D, beta, lam, p, normalize, dtype)
    (1, 2, 300, 64, 0.2, 0.5, 2.0, True, "bf16"),
    (1, 2, 257, 128, 0.1, 0.7, 1.5, True, "bf16"),
    (2, 1, 200, 64, 0.5, 0.3, 2.0, False, "bf16"),
    (1, 1, 150, 96, 0.0, 1.3, 2.0, True, "bf16"),   # lambda clamps to 1: dlambda 0
    (1, 2, 130, 48, 0.3, -0.2, 2.0, True, "bf16"),  # lambda clamps to 0: path 2 gives nothing
    (1, 1, 1, 64, 0.1, 0.4, 2.0, True, "bf16"),     # T = 1
    (1, 2, 130, 64, 0.2, 0.5, 2.0, True, "f32"),
    (1, 1, 100, 32, 0.1, 0.6, 1.5, False, "f32"),
]


@pytest.mark.parametrize("B,H,T,D,beta,lam,p,norm,dtype", BWD_CASES)
def test_tra_diff_backward(B, H, T, D, beta, lam, p, norm, dtype):
    g = torch.Generator().manual_seed(T + D)
    scale = D ** -0.25 if not norm else 1.0
    q1, q2, k1, k2, v, do = (torch.randn((B, H, T, D), generator=g) * (scale if i < 4 else 1.0) for i in range(6))
    q1, q2, k1, k2, v, do = (t.to(torch.bfloat16 if dtype == "bf16" else torch.float32) for t in
                             (q1, q2, k1, k2, v, do))
    grads = bsa.tra_diff_backward(*(t.cuda() for t in (q1, q2, k1, k2, v, do)), beta, lam, p, normalize=norm,
                                  want_dlam=True)
    torch.cuda.synchronize()
    h = [f64(t) for t in (q1, q2, k1, k2, v, do)]
    refs = otra.tra_diff_backward(*h, beta, lam, p, normalize=norm)
    tol = 2e-2 if dtype == "bf16" else 1e-4
    for name, got, ref in zip(("dq1", "dq2", "dk1", "dk2", "dv"), grads[:5], refs[:5]):
        scale_ref = float(np.abs(ref).max())
        err = float(np.abs(f64(got) - ref).max())
        assert err <= tol * max(scale_ref, 1e-30) or (scale_ref == 0.0 and err == 0.0), f"{name}: {err:.3e}"
    a2, b2 = (otra.l2_normalize(x) for x in (h[1], h[3])) if norm else (h[1], h[3])
    size = float(np.abs(h[5] * otra.tra_forward(a2, b2, h[4], beta, p)).sum())
    assert abs(float(grads[5].item()) - refs[5]) <= tol * max(size, 1e-30)
    if not 0.0 < lam < 1.0:
        assert float(grads[5].item()) == 0.0


def test_tra_diff_attention_autograd():
    # the autograd form, with lambda a tensor that requires a gradient
    B, H, T, D = 1, 2, 200, 64
    g = torch.Generator().manual_seed(9)
    ts = [torch.randn((B, H, T, D), generator=g).to(torch.bfloat16).cuda().requires_grad_(True) for _ in range(5)]
    lam = torch.tensor(0.4, device="cuda", requires_grad=True)
    w = torch.randn((B, H, T, D), generator=g).cuda()
    out = bsa.tra_diff_attention(*ts, 0.2, lam, 2.0, normalize=True)
    (out.float() * w).sum().backward()
    torch.cuda.synchronize()
    h = [f64(t) for t in ts]
    refs = otra.tra_diff_backward(*h, f64(w.to(torch.bfloat16)), 0.2, 0.4, 2.0, normalize=True)
    for name, t, ref in zip(("dq1", "dq2", "dk1", "dk2", "dv"), ts, refs[:5]):
        err = float(np.abs(f64(t.grad) - ref).max()) / max(float(np.abs(ref).max()), 1e-30)
        assert err <= 2e-2, f"{name}: max err {err:.3e} of max|ref|"
    assert lam.grad is not None
    a2, b2 = otra.l2_normalize(h[1]), otra.l2_normalize(h[3])
    size = float(np.abs(f64(w.to(torch.bfloat16)) * otra.tra_forward(a2, b2, h[4], 0.2, 2.0)).sum())
    assert abs(float(lam.grad) - refs[5]) <= 2e-2 * size
