"""GPU parity of the threshold-attention backward (tcgen05 kernels, through
the C ABI) against the float64 oracle's analytic gradients.

Bar (from the bf16 arithmetic, as for the forward): for each of dq, dk, dv,
max|gpu - ref| <= 2e-2 * max|ref| over the whole tensor.
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


CASES = [
    # (B, H, T, D, beta, p)
    (1, 2, 256, 128, 1.0, 2.0),
    (1, 2, 300, 64, 2.0, 1.5),   # ragged, general power
    (2, 1, 129, 128, 0.0, 1.0),  # p = 1
    (1, 1, 1, 64, 1.0, 2.0),     # T = 1
    (1, 2, 640, 64, 1.0, 2.0),   # 5 tiles each way
    (1, 1, 384, 128, -0.5, 3.7), # beta < 0 reading, large power
    (2, 2, 1024, 128, 1.0, 2.0), # medium size
    (1, 2, 300, 32, 1.0, 2.0),   # head dim 32 (width-64 tiles, zero-filled columns), ragged
    (1, 1, 257, 16, 0.5, 1.5),   # head dim 16, general power
    (1, 2, 300, 96, 1.0, 2.0),   # head dim 96 (tile width 128, zero-filled columns)
    (1, 1, 257, 48, 0.5, 1.5),   # head dim 48 (tile width 64)
    (1, 1, 200, 112, 1.0, 3.0),
    (1, 1, 150, 80, 0.5, 0.75),  # p < 1 at width 128
]


@pytest.mark.parametrize("deterministic", [False, True], ids=["fused", "two_kernel"])
@pytest.mark.parametrize("B,H,T,D,beta,p", CASES)
def test_tra_backward_full_output(B, H, T, D, beta, p, deterministic):
    q, k, v = workloads.tra_inputs(B, H, T, D, "bf16", seed=T + 3 * D)
    g = torch.Generator().manual_seed(T)
    do = torch.randn((B, H, T, D), generator=g).to(torch.bfloat16)
    dq, dk, dv = bsa.tra_backward(q.cuda(), k.cuda(), v.cuda(), do.cuda(), beta, p, deterministic=deterministic)
    torch.cuda.synchronize()
    rq, rk, rv = otra.tra_backward(f64(q), f64(k), f64(v), f64(do), beta, p)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        got = f64(got)
        err = float(np.abs(got - ref).max()) / max(float(np.abs(ref).max()), 1e-30)
        assert err <= TOL, f"{name}: max err {err:.3e} of max|ref|"


def test_tra_backward_full_workload_sampled_heads():
    # The bench's backward workload (B4 H16 T4096 D128, p=2) in the same
    # launch configuration; three (b, h) heads checked in full against the
    # float64 oracle (each head is independent).
    w = workloads.TRA_WORKLOADS["tra_bf16_B4_H16_T4096_D128"]
    q, k, v = workloads.workload_inputs(w)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    grads = bsa.tra_backward(q.cuda(), k.cuda(), v.cuda(), do.cuda(), w.beta, w.p)
    torch.cuda.synchronize()
    for b, h in [(0, 0), (1, 7), (3, 15)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        refs = otra.tra_backward(f64(q[sl]), f64(k[sl]), f64(v[sl]), f64(do[sl]), w.beta, w.p)
        for name, g, ref in zip(("dq", "dk", "dv"), grads, refs):
            gpu = f64(g[sl])
            err = float(np.abs(gpu - ref).max()) / max(float(np.abs(ref).max()), 1e-30)
            assert err <= TOL, f"{name} head ({b},{h}): max err {err:.3e} of max|ref|"


@pytest.mark.parametrize("deterministic", [True, False], ids=["two_kernel", "fused"])
def test_tra_backward_head_groups_cover_every_head(deterministic):
    # At the bench shape the blocks run in head groups of unequal size (64
    # heads in three groups).  Each dk/dv row is computed by one CTA with the
    # same arithmetic whatever the block order, so the full call must equal
    # single-head calls (one group each) bit for bit on every head; so must dq
    # in the two-kernel form.  The fused kernel adds dq's fp32 partials in a
    # run-dependent order: there dq must stay within the bar of the other.
    w = workloads.TRA_WORKLOADS["tra_bf16_B4_H16_T4096_D128"]
    q, k, v = (t.cuda() for t in workloads.workload_inputs(w))
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).cuda()
    full = bsa.tra_backward(q, k, v, do, w.beta, w.p, deterministic=deterministic)
    for b in range(w.B):
        for h in range(w.H):
            sl = (slice(b, b + 1), slice(h, h + 1))
            one = bsa.tra_backward(q[sl], k[sl], v[sl], do[sl], w.beta, w.p, deterministic=deterministic)
            for name, a, c in zip(("dq", "dk", "dv"), full, one):
                if name == "dq" and not deterministic:
                    a, c = f64(a[sl]), f64(c)
                    assert float(np.abs(a - c).max()) <= TOL * max(float(np.abs(c).max()), 1e-30), name
                else:
                    assert torch.equal(a[sl], c), f"{name} head ({b},{h}) differs from its single-head call"


# fp32 inputs: the CUDA-core FFMA kernels, against the oracle at the fp32 bar.
F32_TOL = 1e-4
F32_CASES = [
    # (B, H, T, D, beta, p)
    (1, 2, 256, 64, 1.0, 2.0),
    (2, 1, 200, 128, 0.5, 1.5),   # ragged, general power
    (1, 2, 130, 64, 0.0, 1.0),    # p = 1
    (1, 1, 1, 128, 1.0, 2.0),     # T = 1
    (1, 1, 320, 64, -0.5, 3.7),   # beta < 0 reading, large power
    (1, 2, 150, 32, 1.0, 2.0),    # head dim 32
    (1, 1, 100, 16, 0.5, 1.5),    # head dim 16
    (1, 1, 150, 80, 1.0, 2.0),    # head dims 80, 48
    (1, 2, 100, 48, 0.5, 1.5),
]


@pytest.mark.parametrize("B,H,T,D,beta,p", F32_CASES)
def test_tra_backward_f32(B, H, T, D, beta, p):
    q, k, v = workloads.tra_inputs(B, H, T, D, "f32", seed=T + D)
    do = torch.randn((B, H, T, D), generator=torch.Generator().manual_seed(T + 1))
    dq, dk, dv = bsa.tra_backward(q.cuda(), k.cuda(), v.cuda(), do.cuda(), beta, p)
    torch.cuda.synchronize()
    assert dq.dtype == torch.float32
    rq, rk, rv = otra.tra_backward(f64(q), f64(k), f64(v), f64(do), beta, p)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        err = float(np.abs(f64(got) - ref).max()) / max(float(np.abs(ref).max()), 1e-30)
        assert err <= F32_TOL, f"{name}: max err {err:.3e} of max|ref|"


def _clean_seed(B, H, T, D, beta, gap):
    """First seed whose causal scores all keep |q.k - tau| >= gap (bf16 inputs)."""
    t = otra.tau(T, beta, D)
    keep = np.tril(np.ones((T, T), dtype=bool))
    for seed in range(500):
        q, k, v = workloads.tra_inputs(B, H, T, D, "bf16", seed=seed)
        x = np.einsum("bhid,bhjd->bhij", f64(q), f64(k)) - t[None, None, :, None]
        if np.all(np.abs(x[..., keep]) >= gap):
            return seed, (q, k, v)
    raise AssertionError("no clean seed")


@pytest.mark.parametrize("p", [0.5, 0.75])
def test_tra_backward_power_below_one(p):
    # For p < 1 the derivative p x^(p-1) grows without bound as x -> 0+, so a
    # score that sits within rounding of the threshold makes any two correct
    # evaluations disagree.  The inputs are chosen so that no causal score
    # lies within 5e-4 of tau; there the bf16 bar applies as for every power.
    B, H, T, D, beta = 1, 1, 80, 64, 1.0
    seed, (q, k, v) = _clean_seed(B, H, T, D, beta, 5e-4)
    do = torch.randn((B, H, T, D), generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    dq, dk, dv = bsa.tra_backward(q.cuda(), k.cuda(), v.cuda(), do.cuda(), beta, p)
    torch.cuda.synchronize()
    rq, rk, rv = otra.tra_backward(f64(q), f64(k), f64(v), f64(do), beta, p)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        err = float(np.abs(f64(got) - ref).max()) / max(float(np.abs(ref).max()), 1e-30)
        assert err <= TOL, f"{name}: max err {err:.3e} of max|ref|"


@pytest.mark.parametrize("D", [64, 128])
def test_tra_backward_repeatability(D):
    """The two-kernel form repeats bit for bit; the fused kernel's dk and dv
    do too (each accumulates inside one CTA in a fixed order), and its dq,
    whose fp32 partials are added in a run-dependent order, stays within the
    bar of the two-kernel dq."""
    B, H, T = 1, 4, 1024
    q, k, v = (t.cuda() for t in workloads.tra_inputs(B, H, T, D, "bf16", seed=11 + D))
    g = torch.Generator().manual_seed(5)
    do = torch.randn((B, H, T, D), generator=g).to(torch.bfloat16).cuda()
    det = [bsa.tra_backward(q, k, v, do, 1.0, 2.0, deterministic=True) for _ in range(2)]
    fus = [bsa.tra_backward(q, k, v, do, 1.0, 2.0) for _ in range(2)]
    torch.cuda.synchronize()
    for a, b in zip(det[0], det[1]):
        assert torch.equal(a, b)
    assert torch.equal(fus[0][1], fus[1][1]) and torch.equal(fus[0][2], fus[1][2])
    for a, b in zip(fus[0], det[0]):
        a, b = f64(a), f64(b)
        assert float(np.abs(a - b).max()) <= TOL * max(float(np.abs(b).max()), 1e-30)



def test_tra_backward_concurrent_streams():
    # Two host threads run the fused backward (whose fp32 dq accumulator is a
    # stream-ordered temporary from the library's pool) and the normalised
    # differential forward (pool temporary for the normalised keys) on their
    # own streams at once; the results must equal the same calls made one
    # after the other (dk, dv and the differential output bit for bit, dq
    # within the bar: its partials are added in a run-dependent order).
    import threading

    B, H, T, D = 1, 3, 700, 128
    ins = []
    for s in range(2):
        q, k, v = (t.cuda() for t in workloads.tra_inputs(B, H, T, D, "bf16", seed=60 + s))
        do = torch.randn(q.shape, generator=torch.Generator().manual_seed(s)).to(torch.bfloat16).cuda()
        ins.append((q, k, v, do))
    want = [bsa.tra_backward(q, k, v, do, 1.0, 2.0) for q, k, v, do in ins]
    want_d = [bsa.tra_diff_forward(q, k, v, do, v, 0.5, 0.3, 1.5, normalize=True) for q, k, v, do in ins]
    torch.cuda.synchronize()
    got, got_d, errors = [None, None], [None, None], []

    def worker(i):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                q, k, v, do = ins[i]
                for _ in range(3):
                    got[i] = bsa.tra_backward(q, k, v, do, 1.0, 2.0, stream=st)
                    got_d[i] = bsa.tra_diff_forward(q, k, v, do, v, 0.5, 0.3, 1.5, normalize=True, stream=st)
            st.synchronize()
        except Exception as e:
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    torch.cuda.synchronize()
    assert not errors, errors
    for i in range(2):
        assert torch.equal(got[i][1], want[i][1]) and torch.equal(got[i][2], want[i][2])
        a, b = f64(got[i][0]), f64(want[i][0])
        assert float(np.abs(a - b).max()) <= TOL * max(float(np.abs(b).max()), 1e-30)
        assert torch.equal(got_d[i], want_d[i])


@pytest.mark.parametrize("dtype,D,p", [("bf16", 128, 2.0), ("bf16", 64, 1.5), ("f32", 64, 2.0)])
def test_tra_attention_autograd(dtype, D, p):
    # the autograd form: forward through tra_forward, q/k/v gradients through
    # tra_backward, against the float64 oracle's analytic gradients
    B, H, T = 1, 2, 300
    q, k, v = (t.cuda().requires_grad_(True) for t in workloads.tra_inputs(B, H, T, D, dtype, seed=T + D))
    w = torch.randn((B, H, T, D), generator=torch.Generator().manual_seed(3))
    out = bsa.tra_attention(q, k, v, 1.0, p)
    assert out.dtype == q.dtype
    (out.float() * w.cuda()).sum().backward()
    torch.cuda.synchronize()
    dout = w.to(q.dtype).double().numpy()  # the gradient reaching `out`, in its dtype
    refs = otra.tra_backward(f64(q), f64(k), f64(v), dout, 1.0, p)
    tol = TOL if dtype == "bf16" else F32_TOL
    for name, t, ref in (("dq", q, refs[0]), ("dk", k, refs[1]), ("dv", v, refs[2])):
        err = float(np.abs(f64(t.grad) - ref).max()) / max(float(np.abs(ref).max()), 1e-30)
        assert err <= tol, f"{name}: max err {err:.3e} of max|ref|"
    fwd = otra.tra_forward(f64(q), f64(k), f64(v), 1.0, p)
    assert float(np.abs(f64(out) - fwd).max()) <= tol * float(np.abs(fwd).max())
