"""GPU self tests through the C ABI.

* The expiry branch of the bounded wait every kernel uses: a one-CTA kernel
  waits, with a short limit, on an mbarrier that nothing arrives on.  The
  wait must give up, the library must report code 1 through
  bsa_device_error (and clear it on read), and the context must stay usable:
  a threshold-attention call right after it matches the oracle.
* The FMA-pipe log2 and exp2 of the general-power epilogue against CUDA's
  log2f and exp2f on dense sweeps of float32 inputs.
"""

import numpy as np
import pytest
import torch

from block_sparse_attention_tra_gb300 import bsa, workloads
from oracle import tra as otra

pytestmark = pytest.mark.gpu


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


def test_bounded_wait_expiry_is_reported_and_context_survives():
    assert bsa.device_error() == 0
    assert bsa.selftest_wait_timeout(100000) == 0  # the wait gave up (about 50 us)
    assert bsa.device_error() == 1                 # timeout code recorded ...
    assert bsa.device_error() == 0                 # ... and cleared by the read
    q, k, v = workloads.tra_inputs(1, 2, 300, 64, "bf16", seed=5)
    out = bsa.tra_forward(q.cuda(), k.cuda(), v.cuda(), 2.0, 1.5)
    torch.cuda.synchronize()
    ref = otra.tra_forward(q.double().numpy(), k.double().numpy(), v.double().numpy(), 2.0, 1.5)
    err = float(np.abs(out.double().cpu().numpy() - ref).max()) / float(np.abs(ref).max())
    assert err <= 2e-2
    assert bsa.device_error() == 0


def test_fma_log2_against_cuda_log2f():
    # every binade from 2^-40 to 2^20 with uniformly random mantissas, plus
    # exact powers of two and the neighbourhood of 1
    r = np.random.default_rng(0)
    e = r.integers(-40, 21, size=1 << 20)
    m = 1.0 + r.random(1 << 20)
    x = np.concatenate([np.ldexp(m, e), np.ldexp(1.0, np.arange(-40, 21)), 1.0 + np.linspace(-1e-3, 1e-3, 4097)])
    xt = torch.from_numpy(x.astype(np.float32)).cuda()
    y_fma, y_ref = bsa.selftest_log2(xt)
    torch.cuda.synchronize()
    a, b = y_fma.double().cpu().numpy(), y_ref.double().cpu().numpy()
    exact = np.log2(xt.double().cpu().numpy())
    err_ref = float(np.abs(a - b).max())
    err_exact = float(np.abs(a - exact).max())
    print(f"FMA-pipe log2: max |fma - log2f| = {err_ref:.3e}, max |fma - log2| = {err_exact:.3e}")
    # the polynomial's own bound (1.6e-5 in float32) plus log2f's rounding
    assert err_exact <= 2.0e-5 and err_ref <= 2.5e-5
    # x = 0 (the ReLU's zeros): -127, so exp2(p * it) flushes to 0 for p >= 1
    z, _ = bsa.selftest_log2(torch.zeros(2, dtype=torch.float32, device="cuda"))
    assert float(z.max()) <= -126.99


def test_fma_exp2_against_cuda_exp2f():
    # y over the whole normal range, the neighbourhood of 0 and the integers,
    # then the clamped ends
    r = np.random.default_rng(1)
    y = np.concatenate([r.uniform(-126.0, 127.9, 1 << 20), np.linspace(-4.0, 4.0, 40001),
                        np.arange(-126, 128, dtype=np.float64)]).astype(np.float32)
    yt = torch.from_numpy(y).cuda()
    w_fma, w_ref = bsa.selftest_exp2(yt)
    torch.cuda.synchronize()
    a, b = w_fma.double().cpu().numpy(), w_ref.double().cpu().numpy()
    exact = np.exp2(y.astype(np.float64))
    rel_ref = float(np.max(np.abs(a - b) / b))
    rel_exact = float(np.max(np.abs(a - exact) / exact))
    print(f"FMA-pipe exp2: max rel |fma - exp2f| = {rel_ref:.3e}, max rel |fma - exp2| = {rel_exact:.3e}")
    # the polynomial's own bound (2.9e-6 in float32) plus exp2f's rounding
    assert rel_exact <= 3.5e-6 and rel_ref <= 4e-6
    ends = torch.tensor([-float("inf"), -1e4, -200.0, -127.0, 128.0, 1e4, float("inf")], device="cuda")
    e, _ = bsa.selftest_exp2(ends)
    e = e.cpu()
    assert torch.all(e[:4] == 0.0) and not torch.any(torch.signbit(e[:4]))
    assert torch.all(torch.isinf(e[4:])) and torch.all(e[4:] > 0)
