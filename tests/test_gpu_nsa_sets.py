"""GPU: the NSA selection kernels read a query's selected blocks as a set.

Page "nsa_selection_kernel.py", selection_forward_reference: the index row is
scattered one-hot and reduced with ``any``, so a block listed twice counts
once and the order of the slots does not matter.  Every NSA form here (the
TMA kernel for 64-token blocks, the general kernel for the other shapes, and
the block-outer split-K form) is checked against the float64 oracle on index
rows with repeated and permuted entries, and bit for bit against the same
rows with the repeats replaced by -1 padding (the kernels then do exactly the
same work in the same order).  Guard bands around out and lse must stay
untouched.
"""

import numpy as np
import pytest
import torch

from block_sparse_attention_tra_gb300 import bsa, workloads
from oracle import nsa as onsa

pytestmark = pytest.mark.gpu
BF16_TOL = 2e-2
LSE_TOL = 1e-2


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


def with_repeats(idx, bs, T, seed):
    """Copies of live entries written over padding and over other slots, and
    rows shuffled: every row keeps the same set of blocks it had."""
    r = np.random.default_rng(seed)
    a = idx.numpy().copy()
    B, H, TT, S = a.shape
    for b in range(B):
        for h in range(H):
            for i in range(TT):
                row = a[b, h, i]
                live = [x for x in row if x >= 0]
                if not live:
                    continue
                # fill padding slots with repeats of live entries
                for s in range(S):
                    if row[s] < 0 and r.random() < 0.7:
                        row[s] = live[int(r.integers(len(live)))]
                r.shuffle(row)
    return torch.from_numpy(a)


def deduplicated(idx):
    """The same rows with every repeat after its first occurrence set to -1."""
    a = idx.numpy().copy()
    B, H, T, S = a.shape
    for b in range(B):
        for h in range(H):
            for i in range(T):
                seen = set()
                for s in range(S):
                    x = int(a[b, h, i, s])
                    if x >= 0:
                        if x in seen:
                            a[b, h, i, s] = -1
                        seen.add(x)
    return torch.from_numpy(a)


def check(out, lse, ro, rl):
    o, l = f64(out), f64(lse)
    err = float(np.abs(o - ro).max()) / float(np.abs(ro).max())
    assert err <= BF16_TOL, f"out: max err {err:.3e} of max|ref|"
    empty = rl == -1e9
    assert np.all(l[empty] == -1e9)
    if np.any(~empty):
        assert float(np.abs(l[~empty] - rl[~empty]).max()) <= LSE_TOL


def run(form, q, k, v, idx, bs, out=None, lse=None):
    B, Hq, T, D = q.shape
    if lse is None:
        lse = torch.empty((B, Hq, T), dtype=torch.float32, device="cuda")
    if form == "fsa":
        out = bsa.nsa_select_forward_fsa(q, k, v, idx, bs, out=out, lse=lse)
    else:
        out = bsa.nsa_select_forward(q, k, v, idx, bs, out=out, lse=lse)
    torch.cuda.synchronize()
    return out, lse


CASES = [
    # (form, B, Hq, Hkv, T, D, block_size, S)
    ("tma", 1, 16, 1, 512, 128, 64, 8),
    ("tma", 2, 8, 2, 384, 64, 64, 16),
    ("general", 1, 16, 2, 256, 32, 32, 8),
    ("general", 1, 4, 1, 512, 128, 128, 6),
    ("fsa", 1, 16, 1, 512, 128, 64, 8),
    ("fsa", 1, 16, 2, 384, 64, 64, 12),
]


@pytest.mark.parametrize("form,B,Hq,Hkv,T,D,bs,S", CASES)
def test_repeated_and_permuted_indices(form, B, Hq, Hkv, T, D, bs, S):
    q, k, v, idx = workloads.nsa_inputs(B, Hq, Hkv, T, D, bs, S, seed=T + S + D)
    rep = with_repeats(idx, bs, T, seed=S)
    assert not torch.equal(rep, idx)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    out, lse = run(form, q, k, v, rep.cuda(), bs)
    ro, rl = onsa.nsa_select_forward(f64(q), f64(k), f64(v), rep.numpy(), bs)
    check(out, lse, ro, rl)
    # the repeats change nothing at all: the same blocks in the same order
    out2, lse2 = run(form, q, k, v, deduplicated(rep).cuda(), bs)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_row_of_one_block_repeated_everywhere():
    B, Hq, Hkv, T, D, S = 1, 16, 1, 256, 128, 16
    q, k, v, _ = workloads.nsa_inputs(B, Hq, Hkv, T, D, 64, S, seed=4)
    idx = torch.full((B, Hkv, T, S), -1, dtype=torch.int32)
    for i in range(T):
        idx[0, 0, i, :] = i // 64  # the query's own block, sixteen times
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    ro, rl = onsa.nsa_select_forward(f64(q), f64(k), f64(v), idx.numpy(), 64)
    for form in ("tma", "fsa"):
        out, lse = run(form, q, k, v, idx.cuda(), 64)
        check(out, lse, ro, rl)


@pytest.mark.parametrize("form,D,bs", [("tma", 128, 64), ("general", 32, 32), ("fsa", 64, 64)])
def test_nsa_guard_bands_untouched(form, D, bs):
    """Writes only [B, Hq, T, D] of out and [B, Hq, T] of lse."""
    B, Hq, Hkv, T, S = 1, 16, 2, 256, 6
    q, k, v, idx = workloads.nsa_inputs(B, Hq, Hkv, T, D, bs, S, seed=31)
    n, nl, g = B * Hq * T * D, B * Hq * T, 4096
    obuf = torch.full((n + 2 * g,), 7.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((nl + 2 * g,), 7.0, dtype=torch.float32, device="cuda")
    out = obuf[g:g + n].view(B, Hq, T, D)
    lse = lbuf[g:g + nl].view(B, Hq, T)
    run(form, q.cuda(), k.cuda(), v.cuda(), idx.cuda(), bs, out=out, lse=lse)
    assert torch.all(obuf[:g] == 7.0) and torch.all(obuf[g + n:] == 7.0)
    assert torch.all(lbuf[:g] == 7.0) and torch.all(lbuf[g + nl:] == 7.0)
    ro, rl = onsa.nsa_select_forward(f64(q), f64(k), f64(v), idx.numpy(), bs)
    check(out, lse, ro, rl)
