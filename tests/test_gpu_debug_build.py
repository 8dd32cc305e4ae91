"""GPU: the debug build as a stand-in for a memory sanitizer.

The library compiled with -DBSA_DEBUG checks every gather index (NSA block
indices, split-K list entries, K/V token rows) and every TMA coordinate
against its tensor before the access; a violation records code 3 in the
device error word and the access is clamped into range -- nothing traps.
Each entry point runs here on small, odd and degenerate shapes (T = 1, ragged
tails, empty and future-only selection rows, repeated indices) through the
debug build: no violation may be recorded, and every output must equal the
release build's bit for bit (the checks do not touch the arithmetic).
"""

import numpy as np
import pytest
import torch

from block_sparse_attention_tra_gb300 import bsa, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_attention_tra_gb300 import build

    build.build()
    bsa.load_library()
    torch.cuda.set_device(0)
    path = build.build(debug=True)
    yield path
    assert bsa.device_error() == 0


def both(path, fn):
    """fn() on the release build and on the debug build; the debug build must
    record no violation."""
    a = fn()
    torch.cuda.synchronize()
    with bsa.using_library(path):
        assert bsa.device_error() == 0
        b = fn()
        torch.cuda.synchronize()
        err = bsa.device_error()
    assert err == 0, f"debug build recorded device error {err}"
    return a, b


def same(a, b):
    if isinstance(a, (tuple, list)):
        for x, y in zip(a, b):
            same(x, y)
    else:
        assert torch.equal(a, b)


@pytest.mark.parametrize("B,H,T,D,beta,p,dtype", [
    (1, 1, 1, 64, 1.0, 2.0, "bf16"),
    (1, 2, 300, 128, 1.0, 2.0, "bf16"),
    (2, 3, 333, 64, 2.0, 1.5, "bf16"),
    (1, 2, 129, 128, 0.5, 1.0, "bf16"),
    (1, 2, 130, 64, 1.0, 1.5, "f32"),
    (1, 2, 200, 96, 1.0, 2.0, "bf16"),   # head dim below the tile width 128
    (1, 1, 150, 48, 2.0, 1.5, "bf16"),
])
def test_tra_forward_debug_build(debug_lib, B, H, T, D, beta, p, dtype):
    q, k, v = (t.cuda() for t in workloads.tra_inputs(B, H, T, D, dtype, seed=T))
    same(*both(debug_lib, lambda: bsa.tra_forward(q, k, v, beta, p)))


@pytest.mark.parametrize("T,D,p", [(1, 64, 2.0), (300, 128, 2.0), (257, 64, 1.5), (200, 32, 2.0), (200, 80, 1.5)])
def test_tra_backward_and_diff_debug_build(debug_lib, T, D, p):
    q, k, v = (t.cuda() for t in workloads.tra_inputs(1, 2, T, D, "bf16", seed=T + 1))
    q2, k2, _ = (t.cuda() for t in workloads.tra_inputs(1, 2, T, D, "bf16", seed=T + 2))
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(T)).to(torch.bfloat16).cuda()
    same(*both(debug_lib, lambda: bsa.tra_backward(q, k, v, do, 1.0, p, deterministic=True)))
    # the fused kernel adds dq's fp32 partials in a run-dependent order: dk, dv bit for bit, dq within the bar
    a, b = both(debug_lib, lambda: bsa.tra_backward(q, k, v, do, 1.0, p))
    same(a[1:], b[1:])
    ref = a[0].double()
    assert float((b[0].double() - ref).abs().max()) <= 2e-2 * max(float(ref.abs().max()), 1e-30)
    same(*both(debug_lib, lambda: bsa.tra_diff_forward(q, q2, k, k2, v, 0.1, 0.5, p, normalize=True)))
    # the differential backward: dk1, dk2, dv bit for bit; dq1, dq2 (fused-backward partials) and dlambda
    # (block sums added atomically) within the bar
    a, b = both(debug_lib, lambda: bsa.tra_diff_backward(q, q2, k, k2, v, do, 0.1, 0.5, p, want_dlam=True))
    same(a[2:5], b[2:5])
    for x, y in ((a[0], b[0]), (a[1], b[1]), (a[5], b[5])):
        assert float((y.double() - x.double()).abs().max()) <= 2e-2 * max(float(x.double().abs().max()), 1e-30)


def odd_rows(idx, n_blk):
    """Empty rows, future-only rows, repeats and out-of-range entries."""
    a = idx.clone()
    T = a.shape[2]
    a[:, :, : T // 8] = -1
    a[:, :, T // 8: T // 4, 0] = n_blk - 1          # a future block only (for most rows)
    a[:, :, T // 8: T // 4, 1:] = -1
    a[:, :, T // 2:, -1] = a[:, :, T // 2:, 0]       # a repeat of slot 0
    a[:, :, -3:, 1] = n_blk + 5                      # past the last block: skipped
    return a


@pytest.mark.parametrize("form,D,bs,S", [("tma", 128, 64, 8), ("tma", 64, 64, 16), ("general", 32, 32, 6),
                                         ("general", 128, 128, 4), ("fsa", 128, 64, 8)])
def test_nsa_debug_build(debug_lib, form, D, bs, S):
    B, Hq, Hkv, T = 1, 16, 2, 512
    q, k, v, idx = workloads.nsa_inputs(B, Hq, Hkv, T, D, bs, S, seed=D + bs)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    idx = odd_rows(idx, T // bs).cuda()

    def run():
        lse = torch.empty((B, Hq, T), dtype=torch.float32, device="cuda")
        if form == "fsa":
            out = bsa.nsa_select_forward_fsa(q, k, v, idx, bs, lse=lse)
        else:
            out = bsa.nsa_select_forward(q, k, v, idx, bs, lse=lse)
        return out, lse

    same(*both(debug_lib, run))
