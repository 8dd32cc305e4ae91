"""GPU parity of the NSA selection forward in the block-outer split-K form
(``nsa_select_forward_fsa``) against the float64 oracle of that form, on the
same seeded inputs.

Bars: those of the query-outer NSA path (bf16: max|gpu - ref| <= 2e-2 *
max|ref|; lse within 1e-2 on rows with a valid key, exactly -1e9 and an
exactly-zero output on empty rows).  Small cases compare every output; the
full workloads run in the launch configuration the benchmark times and are
compared on sampled rows.
"""

import numpy as np
import pytest
import torch

from block_sparse_attention_tra_gb300 import bsa, workloads
from oracle import fsa as ofsa
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


def run_fsa(q, k, v, idx, workspace=None):
    out, lse = bsa.nsa_select_forward_fsa(q.cuda(), k.cuda(), v.cuda(), idx.cuda(), 64, return_lse=True,
                                          workspace=workspace)
    torch.cuda.synchronize()
    return f64(out), f64(lse)


def check(gpu_o, gpu_l, ref_o, ref_l):
    err = float(np.abs(gpu_o - ref_o).max()) / max(float(np.abs(ref_o).max()), 1e-30)
    assert err <= BF16_TOL, f"out: max err {err:.3e} of max|ref|"
    empty = ref_l == -1e9
    assert np.all(gpu_l[empty] == -1e9)
    assert np.all(gpu_o[np.broadcast_to(empty[..., None], gpu_o.shape)] == 0.0)
    if np.any(~empty):
        lerr = float(np.abs(gpu_l[~empty] - ref_l[~empty]).max())
        assert lerr <= LSE_TOL, f"lse: max abs err {lerr:.3e}"


FSA_SMALL = [
    # (B, Hq, Hkv, T, D, S)
    (1, 16, 1, 512, 128, 16),   # G = 16: 8 queries per M tile
    (2, 32, 2, 384, 128, 4),
    (1, 32, 2, 1024, 64, 8),    # D = 64
    (1, 8, 2, 256, 128, 4),     # G = 4: 32 queries per M tile
    (1, 4, 4, 192, 64, 3),      # G = 1: 128 queries per M tile
    (1, 6, 2, 256, 128, 5),     # G = 3: 42 queries, rows 126, 127 idle
    (1, 16, 1, 64, 128, 1),     # one block, S = 1
    (1, 16, 4, 320, 64, 32),    # S = 32
    (1, 16, 2, 384, 128, 6),    # G = 8: 16 queries per M tile, TMA stores of 8-row boxes
    (2, 8, 1, 256, 64, 4),      # G = 8, D = 64
]


@pytest.mark.parametrize("B,Hq,Hkv,T,D,S", FSA_SMALL)
def test_fsa_small_full_output(B, Hq, Hkv, T, D, S):
    q, k, v, idx = workloads.nsa_inputs(B, Hq, Hkv, T, D, 64, S, seed=T + S + 1)
    go, gl = run_fsa(q, k, v, idx)
    ro, rl = ofsa.nsa_select_forward_fsa(f64(q), f64(k), f64(v), idx.numpy(), 64)
    check(go, gl, ro, rl)


def test_fsa_items_split_long_block_lists():
    """Every query selects block 0, so block 0's list (T queries) is cut into
    several work items of 32 M tiles; T = 4096 with G = 16 gives 16 items."""
    B, Hq, Hkv, T, D, S = 1, 16, 1, 4096, 128, 3
    q, k, v, idx = workloads.nsa_inputs(B, Hq, Hkv, T, D, 64, S, seed=5)
    idx[..., 0] = torch.arange(T, dtype=torch.int32) // 64
    idx[..., 1] = 0
    idx[0, 0, :64, 1] = -1  # block 0 listed once in its own rows
    idx[..., 2] = torch.where(idx[..., 2] == 0, -1, idx[..., 2])  # keep the entries of a row distinct
    go, gl = run_fsa(q, k, v, idx)
    r = np.random.default_rng(1)
    rows = sorted({0, 63, 64, T - 1} | {int(x) for x in r.integers(0, T, 40)})
    for i in rows:
        toks = onsa.selected_tokens(idx[0, 0, i].numpy(), i, 64)
        ro, rl = onsa.softmax_attend(f64(q[0, :, i]), f64(k[0, 0, toks]), f64(v[0, 0, toks]), D ** -0.5)
        check(go[0, :, i], gl[0, :, i], ro, rl)


def test_fsa_padding_future_and_empty_rows():
    B, Hq, Hkv, T, D, S = 1, 16, 1, 256, 128, 4
    q, k, v, idx = workloads.nsa_inputs(B, Hq, Hkv, T, D, 64, S, seed=21)
    idx[0, 0, 10:20, :] = -1                # empty rows
    idx[0, 0, 30:40, 0] = 3                 # a future block only
    idx[0, 0, 30:40, 1:] = -1
    idx[0, 0, 100:110, 2] = 2               # future block next to valid ones
    go, gl = run_fsa(q, k, v, idx)
    ro, rl = ofsa.nsa_select_forward_fsa(f64(q), f64(k), f64(v), idx.numpy(), 64)
    check(go, gl, ro, rl)
    assert np.all(gl[0, :, 10:20] == -1e9) and np.all(go[0, :, 10:20] == 0)
    assert np.all(gl[0, :, 30:40] == -1e9) and np.all(go[0, :, 30:40] == 0)


def test_fsa_agrees_with_query_outer_kernel_and_is_deterministic():
    """Same selection, the two CUDA paths; and two FSA calls (whose inverted
    lists are filled by atomics in a different order) agree bit for bit."""
    q, k, v, idx = workloads.nsa_inputs(2, 32, 2, 1024, 128, 64, 16, seed=9)
    ws = torch.empty(bsa.nsa_select_fsa_workspace_size(2, 32, 2, 1024, 128, 64, 16), dtype=torch.uint8,
                     device="cuda")
    a_o, a_l = run_fsa(q, k, v, idx, ws)
    b_o, b_l = run_fsa(q, k, v, idx, ws)
    assert np.array_equal(a_o, b_o) and np.array_equal(a_l, b_l)
    qo, ql = bsa.nsa_select_forward(q.cuda(), k.cuda(), v.cuda(), idx.cuda(), 64, return_lse=True)
    torch.cuda.synchronize()
    check(a_o, a_l, f64(qo), f64(ql))


FSA_WORKLOADS = [n for n, w in workloads.NSA_WORKLOADS.items() if w.block_size == 64 and w.D in (64, 128)]


@pytest.mark.parametrize("name", FSA_WORKLOADS)
def test_fsa_full_workload_sampled_rows(name):
    w = workloads.NSA_WORKLOADS[name]
    q, k, v, idx = workloads.workload_inputs(w)
    out, lse = bsa.nsa_select_forward_fsa(q.cuda(), k.cuda(), v.cuda(), idx.cuda(), w.block_size,
                                          return_lse=True)
    torch.cuda.synchronize()
    r = np.random.default_rng(4)
    rows = {(0, 0, 0), (0, 0, 63), (0, 0, 64), (w.B - 1, w.Hkv - 1, w.T - 1), (0, w.Hkv - 1, 1000)}
    while len(rows) < 64:
        rows.add((int(r.integers(w.B)), int(r.integers(w.Hkv)), int(r.integers(w.T))))
    G = w.G
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for (b, g, i) in sorted(rows):
        toks = onsa.selected_tokens(idx[b, g, i].numpy(), i, w.block_size)
        o1, l1 = onsa.softmax_attend(f64(q[b, g * G:(g + 1) * G, i]), f64(k[b, g, toks]), f64(v[b, g, toks]),
                                     w.D ** -0.5)
        ref_o.append(o1)
        ref_l.append(l1)
        got_o.append(f64(out[b, g * G:(g + 1) * G, i]))
        got_l.append(f64(lse[b, g * G:(g + 1) * G, i]))
    check(np.stack(got_o), np.stack(got_l), np.stack(ref_o), np.stack(ref_l))
