"""The allocation-free differential entry point (tra_diff_forward_noalloc).

Some callers cannot allocate device memory from inside a library call: their
device memory is owned by their own allocator, or the call sits on a path
that must not wait on the CUDA allocator.  For them the library offers a
variant of the differential forward whose scratch (the row normalisation
factors) lives in a fixed device array held by the library.  These tests call
it through the C ABI, on buffers the test itself owns, and compare its output
with the regular entry point's and the float64 oracle's, on two calls in a
row (the second call reuses the array the first one left filled); without
normalisation the two entry points run the same kernel and must agree bit for
bit.  The file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

from block_sparse_attention_tra_gb300 import bsa, workloads
from oracle import tra as otra

pytestmark = pytest.mark.gpu
TOL = 2e-2  # the bf16 bar used by every parity test here (oracle comparison)


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


def _inputs(B, H, T, D, seed):
    q1, k1, v = workloads.tra_inputs(B, H, T, D, "bf16", seed=seed)
    q2, k2, _ = workloads.tra_inputs(B, H, T, D, "bf16", seed=seed + 1)
    return [t.cuda() for t in (q1, q2, k1, k2, v)]


def _noalloc(ts, out, beta, lam, p, normalize=True):
    B, H, T, D = ts[0].shape
    stream = torch.cuda.current_stream().cuda_stream
    return bsa.tra_diff_forward_noalloc_raw(*(t.data_ptr() for t in ts), out.data_ptr(), B, H, T, D, beta, lam, p,
                                            normalize, bsa.BSA_BF16, stream)


@pytest.mark.parametrize("shape,beta,lam,p", [((1, 2, 384, 128), 0.0, 0.5, 2.0), ((2, 2, 300, 64), 0.1, 0.7, 1.5)])
def test_noalloc_matches_regular_entry_point_twice(shape, beta, lam, p):
    # With normalisation the regular entry point reads keys normalised and
    # rounded to bf16 (from its pool temporary), the allocation-free one folds
    # the key factors into the scores in fp32 (its fixed array holds only the
    # factors): both within the bf16 bar of the float64 oracle and of each
    # other, each bit-repeatable -- on the first call and on the second, which
    # finds the array filled by the first.
    for call, seed in enumerate((11, 12)):  # two calls in a row, different data
        ts = _inputs(*shape, seed=seed + 7 * shape[2])
        want = bsa.tra_diff_forward(*ts, beta, lam, p, normalize=True)
        out = torch.full_like(ts[0], float("nan"))
        assert _noalloc(ts, out, beta, lam, p) == 0
        again = torch.full_like(ts[0], float("nan"))
        assert _noalloc(ts, again, beta, lam, p) == 0
        torch.cuda.synchronize()
        assert torch.equal(out, again), f"call {call}: not repeatable"
        h = [t.double().cpu().numpy() for t in ts]
        ref = otra.tra_diff_forward(*h, beta, lam, p, normalize=True)
        scale = max(float(np.abs(ref).max()), 1e-30)
        for name, got in (("noalloc", out), ("regular", want)):
            err = float(np.abs(got.double().cpu().numpy() - ref).max()) / scale
            assert err <= TOL, f"call {call}, {name}: max err {err:.3e} of max|ref|"
        gap = float((out.double() - want.double()).abs().max()) / scale
        assert gap <= TOL, f"call {call}: the two entry points differ by {gap:.3e} of max|ref|"


def test_noalloc_without_normalisation_and_limit():
    ts = _inputs(1, 1, 256, 64, seed=3)
    want = bsa.tra_diff_forward(*ts, 0.0, 0.5, 2.0, normalize=False)
    out = torch.empty_like(ts[0])
    assert _noalloc(ts, out, 0.0, 0.5, 2.0, normalize=False) == 0
    torch.cuda.synchronize()
    assert torch.equal(out, want)
    # B*H*Tp beyond the fixed array: refused before anything is enqueued
    big = 1 << 20  # rows of the fixed array
    P = ts[0].data_ptr()
    st = bsa.tra_diff_forward_noalloc_raw(P, P, P, P, P, P, 1, 2, big, 64, 0.0, 0.5, 2.0, True, bsa.BSA_BF16, 0)
    assert st == 9 and "scratch" in bsa.status_string(st)
