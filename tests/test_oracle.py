"""CPU pins of the float64 oracle (no GPU).

Each test checks the oracle against something other than itself: hand-worked
fixtures under ``tests/golden/``, closed forms, textbook special cases computed
with library routines, invariants of the definition, and the scalar brute-force
loops.  The mutation tests at the end plant plausible mistakes in the oracle
(on the CPU) and confirm that the pins catch them.
"""

import math

import numpy as np
import pytest
import torch

from oracle import brute, fsa, nsa, tra
from block_sparse_attention_tra_gb300 import workloads


def rng(seed=0):
    return np.random.default_rng(seed)


def rand_tra(B, H, T, D, seed=0):
    r = rng(seed)
    sc = D ** -0.25
    return (r.standard_normal((B, H, T, D)) * sc, r.standard_normal((B, H, T, D)) * sc,
            r.standard_normal((B, H, T, D)))


# --------------------------------------------------------------------------- TRA

def _golden_tra(golden):
    rows = {r[0]: [float(x) for x in r[1:]] for r in golden("tra_handworked.txt")}
    q = np.array(rows["q"]).reshape(1, 1, 3, 2)
    k = np.array(rows["k"]).reshape(1, 1, 3, 2)
    v = np.array(rows["v"]).reshape(1, 1, 3, 2)
    return q, k, v, rows


def test_tra_handworked_fixture(golden):
    q, k, v, rows = _golden_tra(golden)
    for p, key in ((2.0, "p2"), (1.0, "p1")):
        want = np.array(rows[key]).reshape(1, 1, 3, 2)
        got = tra.tra_forward(q, k, v, 0.0, p)
        np.testing.assert_array_equal(got, want)
        got_b = np.array(brute.tra_forward(q.tolist(), k.tolist(), v.tolist(), 0.0, p))
        np.testing.assert_array_equal(got_b, want)


def test_tra_threshold_handworked_fixture(golden):
    rows = {r[0]: [float(x) for x in r[1:]] for r in golden("tra_threshold_handworked.txt")}
    q = np.array(rows["q"]).reshape(1, 1, 2, 2)
    k = np.array(rows["k"]).reshape(1, 1, 2, 2)
    v = np.array(rows["v"]).reshape(1, 1, 2, 2)
    beta = 1.0 / math.sqrt(math.log(2.0))
    want = np.array(rows["out"]).reshape(1, 1, 2, 2)
    for p in (1.0, 2.0, 1.5, 3.7):
        # tau(1) == 1 up to one rounding, so relu(1 - tau(1))^p is ~1e-16^p
        np.testing.assert_allclose(tra.tra_forward(q, k, v, beta, p), want, atol=1e-12)


def test_tau_inverts_to_row_index():
    """tau(i)^2 * D / (2 beta^2) == ln(i+1): exp of it recovers i+1."""
    for beta, D in ((1.0, 128), (2.0, 64), (0.37, 7)):
        t = tra.tau(10000, beta, D)
        assert t[0] == 0.0
        i = np.arange(10000)
        np.testing.assert_allclose(np.exp(t ** 2 * D / (2 * beta ** 2)), i + 1.0, rtol=1e-10)
        assert np.all(np.diff(t) > 0)


def test_tau_values_at_config_rows():
    # beta=1, D=128, row 4095: sqrt(2 ln 4096 / 128) = sqrt(12 ln 2 / 64)
    assert tra.tau(4096, 1.0, 128)[4095] == pytest.approx(math.sqrt(12 * math.log(2) / 64), rel=1e-14)
    # beta=2, D=64, row 8191: 2 sqrt(2 ln 8192 / 64) = 2 sqrt(13 ln 2 / 32)
    assert tra.tau(8192, 2.0, 64)[8191] == pytest.approx(2 * math.sqrt(13 * math.log(2) / 32), rel=1e-14)


@pytest.mark.parametrize("p", [1.0, 2.0, 1.5, 3.7])
@pytest.mark.parametrize("beta", [0.0, 1.0, 1e6])
def test_tra_row0_closed_form(p, beta):
    """tau(0) = 0, so row 0 is ReLU(q0.k0)^p v0 whatever beta is."""
    q, k, v = rand_tra(2, 3, 20, 16, seed=1)
    out = tra.tra_forward(q, k, v, beta, p)
    for b in range(2):
        for h in range(3):
            s = sum(q[b, h, 0, d] * k[b, h, 0, d] for d in range(16))
            want = (max(s, 0.0) ** p) * v[b, h, 0]
            np.testing.assert_allclose(out[b, h, 0], want, rtol=1e-12, atol=1e-14)


def test_tra_beta0_is_textbook_causal_relu_attention():
    q, k, v = rand_tra(2, 2, 50, 8, seed=2)
    for p in (1.0, 2.0):
        out = tra.tra_forward(q, k, v, 0.0, p)
        for b in range(2):
            for h in range(2):
                w = np.tril(np.maximum(q[b, h] @ k[b, h].T, 0.0)) ** p
                np.testing.assert_allclose(out[b, h], w @ v[b, h], rtol=1e-12, atol=1e-12)


def test_tra_huge_beta_leaves_only_row0():
    q, k, v = rand_tra(1, 2, 40, 16, seed=3)
    out = tra.tra_forward(q, k, v, 1e6, 2.0)
    assert np.all(out[:, :, 1:] == 0.0)
    s = np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    np.testing.assert_allclose(out[:, :, 0], (np.maximum(s, 0) ** 2)[..., None] * v[:, :, 0], rtol=1e-12)


@pytest.mark.parametrize("p", [1.0, 2.0, 1.5])
def test_tra_homogeneity_and_linearity(p):
    """f(c s - c tau) = c^p f(s - tau): scaling q and beta by c scales out by
    c^p; out is linear in v."""
    q, k, v = rand_tra(1, 2, 37, 8, seed=4)
    beta, c = 0.8, 1.7
    base = tra.tra_forward(q, k, v, beta, p)
    np.testing.assert_allclose(tra.tra_forward(c * q, k, v, c * beta, p), c ** p * base, rtol=1e-10, atol=1e-12)
    v2 = rng(5).standard_normal(v.shape)
    np.testing.assert_allclose(tra.tra_forward(q, k, v + 2 * v2, beta, p),
                               base + 2 * tra.tra_forward(q, k, v2, beta, p), rtol=1e-10, atol=1e-10)


def test_tra_causality():
    q, k, v = rand_tra(1, 1, 30, 8, seed=6)
    out = tra.tra_forward(q, k, v, 0.5, 2.0)
    for i in (0, 7, 29):
        k2, v2 = k.copy(), v.copy()
        k2[:, :, i + 1:] += 3.0
        v2[:, :, i + 1:] -= 5.0
        out2 = tra.tra_forward(q, k2, v2, 0.5, 2.0)
        np.testing.assert_array_equal(out2[:, :, : i + 1], out[:, :, : i + 1])


@pytest.mark.parametrize("T,D", [(1, 3), (5, 8), (17, 4), (33, 6)])
@pytest.mark.parametrize("p", [1.0, 2.0, 1.5, 3.7])
@pytest.mark.parametrize("beta", [0.0, 0.7, 2.5, -0.6])
def test_tra_brute_agrees(T, D, p, beta):
    q, k, v = rand_tra(1, 2, T, D, seed=T * 31 + D)
    want = np.array(brute.tra_forward(q.tolist(), k.tolist(), v.tolist(), beta, p))
    got = tra.tra_forward(q, k, v, beta, p, block=7)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_tra_negative_beta_masked_pairs_contribute_nothing():
    """Reading for beta < 0: a future key adds nothing (the page's own comment:
    attend only to positions <= i), so row 0 is still ReLU(q0.k0 - 0)^p v0."""
    q, k, v = rand_tra(1, 1, 10, 4, seed=7)
    out = tra.tra_forward(q, k, v, -1.0, 2.0)
    s = float(q[0, 0, 0] @ k[0, 0, 0])
    np.testing.assert_allclose(out[0, 0, 0], max(s, 0) ** 2 * v[0, 0, 0], rtol=1e-12)


def test_tra_blocking_and_rows_agree():
    q, k, v = rand_tra(2, 2, 300, 16, seed=8)
    a = tra.tra_forward(q, k, v, 1.3, 1.5, block=64)
    b = tra.tra_forward(q, k, v, 1.3, 1.5, block=1000)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    rows = [(1, 0, 0), (0, 1, 299), (1, 1, 128), (0, 0, 63)]
    r = tra.tra_rows(q, k, v, 1.3, 1.5, rows)
    for n, (bb, hh, ii) in enumerate(rows):
        np.testing.assert_allclose(r[n], a[bb, hh, ii], rtol=1e-12, atol=1e-12)


def test_tra_rejects_nonpositive_power():
    with pytest.raises(ValueError):
        tra.relu_power(np.ones(3), 0.0)


def test_tra_flops_count():
    # brute count of causal pairs
    T = 37
    pairs = sum(1 for i in range(T) for j in range(T) if j <= i)
    assert tra.tra_flops(2, 3, T, 8) == 4 * 8 * 6 * pairs
    w = workloads.TRA_WORKLOADS["tra_bf16_B2_H32_T8192_D64"]
    assert w.flops == tra.tra_flops(w.B, w.H, w.T, w.D) == 549_822_922_752


# --------------------------------------------------------------------------- NSA

def rand_nsa(B, Hq, Hkv, T, D, seed=0):
    r = rng(seed)
    return (r.standard_normal((B, Hq, T, D)), r.standard_normal((B, Hkv, T, D)),
            r.standard_normal((B, Hkv, T, D)))


def test_nsa_handworked_fixture(golden):
    rows = golden("nsa_uniform_handworked.txt")
    T, D, bs = 8, 4, 2
    q = np.zeros((1, 2, T, D))
    k = rng(9).standard_normal((1, 1, T, D))
    v = np.array([[j, 2 * j, -j, 1] for j in range(T)], dtype=np.float64).reshape(1, 1, T, D)
    idx = np.array([[int(r[1]), int(r[2])] for r in rows]).reshape(1, 1, T, 2)
    out, lse = nsa.nsa_select_forward(q, k, v, idx, bs)
    bout, blse = brute.nsa_select_forward(q.tolist(), k.tolist(), v.tolist(), idx.tolist(), bs)
    for r in rows:
        i = int(r[0])
        want = np.array([float(x) for x in r[3:7]])
        n = int(r[7])
        want_lse = -1e9 if n == 0 else math.log(n)
        for h in range(2):
            np.testing.assert_allclose(out[0, h, i], want, atol=1e-14)
            np.testing.assert_allclose(bout[0][h][i], want, atol=1e-14)
            assert lse[0, h, i] == pytest.approx(want_lse, abs=1e-14)
            assert blse[0][h][i] == pytest.approx(want_lse, abs=1e-14)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_nsa_full_selection_is_dense_causal_softmax(G):
    """Selecting every causally reachable block reproduces dense causal softmax
    attention with scale D^-0.5 and GQA (torch SDPA, float64, CPU)."""
    import scipy.special

    B, Hkv, T, D, bs = 2, 2, 48, 8, 8
    n_blk = T // bs
    q, k, v = rand_nsa(B, Hkv * G, Hkv, T, D, seed=10 + G)
    idx = -np.ones((B, Hkv, T, n_blk), dtype=np.int64)
    for i in range(T):
        c = i // bs
        idx[:, :, i, : c + 1] = np.arange(c + 1)[::-1]  # any slot order
    out, lse = nsa.nsa_select_forward(q, k, v, idx, bs)
    qt = torch.from_numpy(q)
    kt = torch.from_numpy(k).repeat_interleave(G, dim=1)
    vt = torch.from_numpy(v).repeat_interleave(G, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    s = np.einsum("bhid,bhjd->bhij", q, kt.numpy()) / math.sqrt(D)
    s = np.where(np.tril(np.ones((T, T), dtype=bool)), s, -np.inf)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(s, axis=-1), rtol=1e-12)


def test_nsa_all_padding_is_zero():
    q, k, v = rand_nsa(1, 4, 2, 16, 8, seed=11)
    idx = -np.ones((1, 2, 16, 3), dtype=np.int64)
    out, lse = nsa.nsa_select_forward(q, k, v, idx, 4)
    assert np.all(out == 0.0) and np.all(lse == -1e9)


def test_nsa_future_only_selection_is_empty():
    q, k, v = rand_nsa(1, 2, 1, 16, 8, seed=12)
    idx = -np.ones((1, 1, 16, 2), dtype=np.int64)
    for i in range(16):
        idx[0, 0, i, 0] = i // 4 + 1 if i // 4 + 1 < 4 else -1
    out, lse = nsa.nsa_select_forward(q, k, v, idx, 4)
    assert np.all(out == 0.0) and np.all(lse == -1e9)


def test_nsa_single_key_returns_its_value():
    """Query i = c*bs selecting only block c sees exactly key i."""
    B, Hq, Hkv, T, D, bs = 1, 4, 2, 32, 8, 8
    q, k, v = rand_nsa(B, Hq, Hkv, T, D, seed=13)
    idx = -np.ones((B, Hkv, T, 2), dtype=np.int64)
    idx[..., 0] = (np.arange(T) // bs)[None, None, :]
    out, lse = nsa.nsa_select_forward(q, k, v, idx, bs)
    G = Hq // Hkv
    for i in range(0, T, bs):
        for h in range(Hq):
            np.testing.assert_allclose(out[0, h, i], v[0, h // G, i], rtol=1e-13)
            assert lse[0, h, i] == pytest.approx(float(q[0, h, i] @ k[0, h // G, i]) / math.sqrt(D), rel=1e-12)


def test_nsa_constant_values_pass_through():
    B, Hq, Hkv, T, D, bs = 1, 4, 1, 32, 8, 4
    q, k, _ = rand_nsa(B, Hq, Hkv, T, D, seed=14)
    v = np.broadcast_to(np.arange(D, dtype=np.float64), (B, Hkv, T, D)).copy()
    g = torch.Generator().manual_seed(3)
    idx = workloads.selection_indices(B, Hkv, T, bs, 3, g).numpy()
    out, _ = nsa.nsa_select_forward(q, k, v, idx, bs)
    np.testing.assert_allclose(out, np.broadcast_to(np.arange(D, dtype=np.float64), out.shape), rtol=1e-12)


def test_nsa_slot_order_and_duplicates():
    B, Hq, Hkv, T, D, bs, S = 1, 4, 2, 64, 8, 8, 4
    q, k, v = rand_nsa(B, Hq, Hkv, T, D, seed=15)
    g = torch.Generator().manual_seed(4)
    idx = workloads.selection_indices(B, Hkv, T, bs, S, g).numpy().astype(np.int64)
    base, base_lse = nsa.nsa_select_forward(q, k, v, idx, bs)
    perm = idx[..., ::-1].copy()
    o2, l2 = nsa.nsa_select_forward(q, k, v, perm, bs)
    np.testing.assert_allclose(o2, base, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, base_lse, rtol=1e-12)
    dup = np.concatenate([idx, idx[..., :2]], axis=-1)  # repeat two slots
    o3, l3 = nsa.nsa_select_forward(q, k, v, dup, bs)
    np.testing.assert_allclose(o3, base, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l3, base_lse, rtol=1e-12)


def test_nsa_gather_equals_dense_reading():
    B, Hq, Hkv, T, D, bs, S = 2, 6, 2, 48, 8, 6, 3
    q, k, v = rand_nsa(B, Hq, Hkv, T, D, seed=16)
    g = torch.Generator().manual_seed(5)
    idx = workloads.selection_indices(B, Hkv, T, bs, S, g).numpy().astype(np.int64)
    idx[0, 1, 5:9, 1] = idx[0, 1, 5:9, 0]  # plant duplicates
    idx[1, 0, 20:30, :] = -1  # empty rows
    out, _ = nsa.nsa_select_forward(q, k, v, idx, bs)
    dense = nsa.nsa_select_dense(q, k, v, idx, bs)
    np.testing.assert_allclose(out, dense, rtol=1e-10, atol=1e-12)


def test_nsa_brute_agrees_and_rows():
    B, Hq, Hkv, T, D, bs, S = 1, 4, 2, 24, 5, 4, 3
    q, k, v = rand_nsa(B, Hq, Hkv, T, D, seed=17)
    g = torch.Generator().manual_seed(6)
    idx = workloads.selection_indices(B, Hkv, T, bs, S, g).numpy()
    out, lse = nsa.nsa_select_forward(q, k, v, idx, bs)
    bo, bl = brute.nsa_select_forward(q.tolist(), k.tolist(), v.tolist(), idx.tolist(), bs)
    np.testing.assert_allclose(out, np.array(bo), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, np.array(bl), rtol=1e-12)
    rows = [(0, 0, 0), (0, 1, 23), (0, 1, 9)]
    ro, rl = nsa.nsa_select_rows(q, k, v, idx, bs, rows)
    for n, (b, hk, i) in enumerate(rows):
        np.testing.assert_allclose(ro[n], out[b, hk * 2:(hk + 1) * 2, i], rtol=1e-13)
        np.testing.assert_allclose(rl[n], lse[b, hk * 2:(hk + 1) * 2, i], rtol=1e-13)


def test_nsa_rejects_bad_inputs():
    q, k, v = rand_nsa(1, 2, 1, 16, 4)
    idx = np.zeros((1, 1, 16, 2), dtype=np.int64)
    with pytest.raises(ValueError):
        nsa.nsa_select_forward(q, k, v, idx, 5)  # T % bs != 0
    bad = idx.copy()
    bad[0, 0, 3, 1] = 4  # n_blk = 4 -> out of range
    with pytest.raises(ValueError):
        nsa.nsa_select_forward(q, k, v, bad, 4)
    bad[0, 0, 3, 1] = -2
    with pytest.raises(ValueError):
        nsa.nsa_select_forward(q, k, v, bad, 4)


# -------------------------------------------------- generators (host logic)

def test_selection_generator_structure():
    B, Hkv, T, bs, S = 2, 2, 1024, 64, 16
    g = torch.Generator().manual_seed(0)
    idx = workloads.selection_indices(B, Hkv, T, bs, S, g).numpy()
    assert idx.dtype == np.int32 and idx.shape == (B, Hkv, T, S)
    for b in range(B):
        for h in range(Hkv):
            for i in range(T):
                c = i // bs
                row = idx[b, h, i]
                assert row[0] == c
                kk = min(S - 1, c)
                earlier = row[1:1 + kk]
                assert np.all(earlier < c) and np.all(earlier >= 0)
                assert np.all(np.diff(earlier) > 0)  # distinct, ascending
                assert np.all(row[1 + kk:] == -1)
    g2 = torch.Generator().manual_seed(0)
    assert np.array_equal(idx, workloads.selection_indices(B, Hkv, T, bs, S, g2).numpy())


def test_selection_generator_is_uniform():
    """Each earlier block is picked with probability (S-1)/c."""
    B, Hkv, T, bs, S = 1, 1, 4096, 64, 16
    g = torch.Generator().manual_seed(1)
    idx = workloads.selection_indices(B, Hkv, T, bs, S, g).numpy()
    c = 40
    rows = idx[0, 0, c * bs:(c + 1) * bs, 1:]
    counts = np.bincount(rows.ravel(), minlength=c)[:c]
    expect = bs * 15 / c
    assert counts.sum() == bs * 15
    chi2 = ((counts - expect) ** 2 / expect).sum()
    assert chi2 < 90  # 39 dof; p ~ 1e-5 cut


def test_pairs_count_matches_generated_selection():
    B, Hkv, T, bs, S = 1, 1, 512, 64, 4
    g = torch.Generator().manual_seed(2)
    idx = workloads.selection_indices(B, Hkv, T, bs, S, g).numpy()
    n = sum(len(nsa.selected_tokens(idx[0, 0, i], i, bs)) for i in range(T))
    assert n == nsa.nsa_pairs(T, bs, S)
    w = workloads.NsaWorkload("t", 1, 16, 1, T, 128, bs, S)
    assert w.pairs_per_group == n
    w4 = workloads.NSA_WORKLOADS["nsa_bf16_B2_Hq32_Hkv2_T8192_D128"]
    assert w4.pairs_per_group == nsa.nsa_pairs(8192, 64, 16)
    assert w4.flops == 250_316_062_720


def test_tra_generator_recipe():
    q, k, v = workloads.tra_inputs(1, 2, 4096, 64, "bf16", seed=0)
    assert q.dtype == torch.bfloat16 and q.shape == (1, 2, 4096, 64)
    assert abs(q.float().std().item() - 64 ** -0.25) < 0.01
    assert abs(v.float().std().item() - 1.0) < 0.01
    q2, _, _ = workloads.tra_inputs(1, 2, 4096, 64, "bf16", seed=0)
    assert torch.equal(q, q2)


# ------------------------------------------- planted mistakes must be caught

def _tra_pins_pass(golden):
    try:
        test_tra_handworked_fixture(golden)
        test_tra_threshold_handworked_fixture(golden)
        test_tau_inverts_to_row_index()
        test_tra_beta0_is_textbook_causal_relu_attention()
        test_tra_causality()
        for p in (1.0, 2.0, 1.5):
            test_tra_row0_closed_form(p, 1.0)
    except AssertionError:
        return False
    return True


def test_planted_tra_mistakes_are_caught(golden, monkeypatch):
    assert _tra_pins_pass(golden)
    good_tau, good_relu, good_fwd = tra.tau, tra.relu_power, tra.tra_forward

    mutants = {
        "log10": lambda T, beta, D: beta * np.sqrt(2.0 * np.log10(np.arange(T) + 1.0) / D),
        "no_factor_2": lambda T, beta, D: beta * np.sqrt(np.log(np.arange(T) + 1.0) / D),
        "row_not_shifted": lambda T, beta, D: beta * np.sqrt(2.0 * np.log(np.arange(T) + 2.0) / D),
    }
    for name, bad in mutants.items():
        monkeypatch.setattr(tra, "tau", bad)
        assert not _tra_pins_pass(golden), name
        monkeypatch.setattr(tra, "tau", good_tau)

    monkeypatch.setattr(tra, "relu_power", lambda x, p: np.abs(x) ** p)  # ReLU dropped
    assert not _tra_pins_pass(golden)
    monkeypatch.setattr(tra, "relu_power", good_relu)

    def no_mask(q, k, v, beta, p, block=256):
        q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
        t = tra.tau(q.shape[2], beta, q.shape[3])
        w = tra.relu_power(np.einsum("bhid,bhjd->bhij", q, k) - t[:, None], p)
        return w @ v

    def swapped(q, k, v, beta, p, block=256):
        return good_fwd(k, q, v, beta, p, block)

    def scaled(q, k, v, beta, p, block=256):
        return good_fwd(np.asarray(q) / math.sqrt(np.asarray(q).shape[3]), k, v, beta, p, block)

    for bad in (no_mask, swapped, scaled):
        monkeypatch.setattr(tra, "tra_forward", bad)
        assert not _tra_pins_pass(golden), bad.__name__
    monkeypatch.setattr(tra, "tra_forward", good_fwd)
    assert _tra_pins_pass(golden)


def test_planted_nsa_mistakes_are_caught(golden, monkeypatch):
    good_sel = nsa.selected_tokens

    def pins():
        try:
            test_nsa_handworked_fixture(golden)
            test_nsa_full_selection_is_dense_causal_softmax(2)
            test_nsa_single_key_returns_its_value()
        except AssertionError:
            return False
        return True

    assert pins()

    def no_causal(sel_row, i, bs):
        blocks = sorted({int(x) for x in sel_row if x >= 0})
        if not blocks:
            return np.zeros(0, dtype=np.int64)
        return np.concatenate([np.arange(x * bs, (x + 1) * bs) for x in blocks])

    def strict_causal(sel_row, i, bs):
        t = good_sel(sel_row, i, bs)
        return t[t < i]

    def multiset(sel_row, i, bs):
        toks = [np.arange(x * bs, (x + 1) * bs) for x in sel_row if x >= 0]
        if not toks:
            return np.zeros(0, dtype=np.int64)
        t = np.concatenate(toks)
        return t[t <= i]

    for bad in (no_causal, strict_causal, multiset):
        monkeypatch.setattr(nsa, "selected_tokens", bad)
        assert not pins(), bad.__name__
    monkeypatch.setattr(nsa, "selected_tokens", good_sel)

    good_one = nsa.softmax_attend

    def no_scale(qg, ks, vs, scale):
        return good_one(qg, ks, vs, 1.0)

    def no_max_shift_lse(qg, ks, vs, scale):
        o, l = good_one(qg, ks, vs, scale)
        return o, l - (np.asarray(qg) @ np.asarray(ks).T * scale).max(axis=1) if len(ks) else l

    for bad in (no_scale, no_max_shift_lse):
        monkeypatch.setattr(nsa, "softmax_attend", bad)
        assert not pins(), bad.__name__
    monkeypatch.setattr(nsa, "softmax_attend", good_one)
    assert pins()


# ------------------------------------------------------------- TRA backward

def _torch_tra(q, k, v, beta, p):
    """TRA forward written with torch fp64 ops, differentiated by autograd."""
    T, D = q.shape[-2], q.shape[-1]
    i = torch.arange(T, dtype=torch.float64)
    tau = beta * torch.sqrt(2.0 * torch.log(i + 1.0) / D)
    x = q @ k.transpose(-1, -2) - tau[:, None]
    keep = torch.tril(torch.ones(T, T, dtype=torch.bool))
    w = torch.where(keep & (x > 0), torch.relu(x) ** p, torch.zeros_like(x))
    return w @ v


@pytest.mark.parametrize("p", [1.0, 2.0, 1.5, 3.7])
@pytest.mark.parametrize("beta", [0.0, 0.8])
def test_tra_backward_matches_torch_autograd(p, beta):
    q, k, v = rand_tra(2, 2, 37, 8, seed=20)
    do = rng(21).standard_normal(q.shape)
    dq, dk, dv = tra.tra_backward(q, k, v, do, beta, p, block=16)
    qt, kt, vt = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    out = _torch_tra(qt, kt, vt, beta, p)
    gq, gk, gv = torch.autograd.grad((out * torch.tensor(do)).sum(), (qt, kt, vt))
    np.testing.assert_allclose(dq, gq.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, gk.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, gv.numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("p", [2.0, 1.5, 3.7])
def test_tra_backward_finite_differences(p):
    """Central differences of L = sum(out * dout) (p > 1: L is C^1)."""
    q, k, v = rand_tra(1, 1, 9, 4, seed=22)
    do = rng(23).standard_normal(q.shape)
    beta = 0.3
    dq, dk, dv = tra.tra_backward(q, k, v, do, beta, p)

    def L(qq, kk, vv):
        return float((tra.tra_forward(qq, kk, vv, beta, p) * do).sum())

    h = 1e-6
    r = rng(24)
    for grad, which in ((dq, 0), (dk, 1), (dv, 2)):
        for _ in range(12):
            idx = tuple(int(r.integers(n)) for n in q.shape)
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = L(*args)
            args[which][idx] -= 2 * h
            lm = L(*args)
            assert grad[idx] == pytest.approx((lp - lm) / (2 * h), rel=1e-5, abs=1e-7)


def test_tra_backward_brute_agrees():
    q, k, v = rand_tra(1, 2, 11, 3, seed=25)
    do = rng(26).standard_normal(q.shape)
    for p, beta in ((2.0, 0.5), (1.5, 0.0), (1.0, -0.4)):
        got = tra.tra_backward(q, k, v, do, beta, p, block=4)
        want = brute.tra_backward(q.tolist(), k.tolist(), v.tolist(), do.tolist(), beta, p)
        for g, w_ in zip(got, want):
            np.testing.assert_allclose(g, np.array(w_), rtol=1e-11, atol=1e-12)


def test_tra_backward_textbook_beta0_p1():
    """beta = 0, p = 1: W = tril(ReLU(QK^T)), dV = W^T dO,
    dS = (dO V^T) * tril(QK^T > 0), dQ = dS K, dK = dS^T Q."""
    q, k, v = rand_tra(1, 1, 30, 6, seed=27)
    do = rng(28).standard_normal(q.shape)
    dq, dk, dv = tra.tra_backward(q, k, v, do, 0.0, 1.0)
    s = q[0, 0] @ k[0, 0].T
    w = np.tril(np.maximum(s, 0))
    ds = np.tril((s > 0).astype(float)) * (do[0, 0] @ v[0, 0].T)
    np.testing.assert_allclose(dv[0, 0], w.T @ do[0, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dq[0, 0], ds @ k[0, 0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dk[0, 0], ds.T @ q[0, 0], rtol=1e-12, atol=1e-12)


def test_tra_backward_flops_count():
    assert tra.tra_backward_flops(1, 1, 3, 2) == 10 * 2 * 6


# ----------------------------------------------------------- differential TRA

def test_l2_normalize_matches_torch():
    x = rng(30).standard_normal((2, 3, 7, 5))
    x[0, 0, 0] = 0.0  # zero row stays zero (eps)
    want = torch.nn.functional.normalize(torch.from_numpy(x), p=2, dim=-1).numpy()
    np.testing.assert_allclose(tra.l2_normalize(x), want, rtol=1e-14, atol=1e-300)


def test_tra_diff_special_cases():
    q1, k1, v = rand_tra(1, 2, 40, 8, seed=31)
    q2, k2, _ = rand_tra(1, 2, 40, 8, seed=32)
    beta, p = 0.2, 2.0
    base = tra.tra_forward(tra.l2_normalize(q1), tra.l2_normalize(k1), v, beta, p)
    # lambda = 0 (and below 0, clamped) leaves the first term
    np.testing.assert_allclose(tra.tra_diff_forward(q1, q2, k1, k2, v, beta, 0.0, p), base, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(tra.tra_diff_forward(q1, q2, k1, k2, v, beta, -3.0, p), base, rtol=1e-13, atol=1e-13)
    # lambda >= 1 clamps to 1; equal streams cancel
    np.testing.assert_allclose(tra.tra_diff_forward(q1, q1, k1, k1, v, beta, 1.0, p), 0.0, atol=1e-12)
    np.testing.assert_allclose(tra.tra_diff_forward(q1, q2, k1, k2, v, beta, 7.0, p),
                               tra.tra_diff_forward(q1, q2, k1, k2, v, beta, 1.0, p), rtol=1e-13, atol=1e-13)
    # normalisation: positive row scalings of q or k change nothing
    sc = np.abs(rng(33).standard_normal(q1.shape[:-1] + (1,))) + 0.1
    np.testing.assert_allclose(tra.tra_diff_forward(q1 * sc, q2, k1, k2 / sc, v, beta, 0.4, p),
                               tra.tra_diff_forward(q1, q2, k1, k2, v, beta, 0.4, p), rtol=1e-11, atol=1e-12)
    # without normalisation it is the plain difference of two TRAs
    want = tra.tra_forward(q1, k1, v, beta, p) - 0.4 * tra.tra_forward(q2, k2, v, beta, p)
    np.testing.assert_allclose(tra.tra_diff_forward(q1, q2, k1, k2, v, beta, 0.4, p, normalize=False), want,
                               rtol=1e-13, atol=1e-13)


def test_tra_diff_normalised_scores_are_cosines():
    """With normalisation and beta = 0, p = 1, row 0 is max(cos(q1_0, k1_0), 0) v_0
    minus lambda times the same for stream 2."""
    q1, k1, v = rand_tra(1, 1, 5, 6, seed=34)
    q2, k2, _ = rand_tra(1, 1, 5, 6, seed=35)
    out = tra.tra_diff_forward(q1, q2, k1, k2, v, 0.0, 0.25, 1.0)

    def cos(a, b):
        return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))

    want = max(cos(q1[0, 0, 0], k1[0, 0, 0]), 0) * v[0, 0, 0] - 0.25 * max(cos(q2[0, 0, 0], k2[0, 0, 0]), 0) * v[0, 0, 0]
    np.testing.assert_allclose(out[0, 0, 0], want, rtol=1e-12, atol=1e-14)


# ------------------------------------------- NSA block-outer (FSA) split-K form

def _fsa_handworked_inputs(golden):
    rows = golden("nsa_uniform_handworked.txt")
    T, D, bs = 8, 4, 2
    q = np.zeros((1, 2, T, D))
    k = rng(9).standard_normal((1, 1, T, D))
    v = np.array([[j, 2 * j, -j, 1] for j in range(T)], dtype=np.float64).reshape(1, 1, T, D)
    idx = np.array([[int(r[1]), int(r[2])] for r in rows]).reshape(1, 1, T, 2)
    return q, k, v, idx, bs


def test_fsa_partials_handworked_fixture(golden):
    q, k, v, idx, bs = _fsa_handworked_inputs(golden)
    want = {(int(r[0]), int(r[1])): (float(r[2]), [float(x) for x in r[3:7]])
            for r in golden("fsa_partials_handworked.txt")}
    parts = fsa.fsa_partials(q, k, v, idx, bs)
    assert {(i, j) for (_, _, i, j) in parts} == set(want)
    for (b, h, i, j), (m, l, acc) in parts.items():
        n, a = want[(i, j)]
        np.testing.assert_array_equal(m, 0.0)
        np.testing.assert_allclose(l, n, rtol=0, atol=1e-15)
        for g in range(2):
            np.testing.assert_allclose(acc[g], a, rtol=0, atol=1e-14)
    lists = fsa.block_query_lists(idx, bs)
    assert lists[(0, 0, 1)] == [(2, 0), (3, 0), (7, 1)]  # i=3 lists block 1 twice: first slot
    out, lse = fsa.nsa_select_forward_fsa(q, k, v, idx, bs)
    for r in golden("nsa_uniform_handworked.txt"):
        i, n = int(r[0]), int(r[7])
        np.testing.assert_allclose(out[0, :, i], np.broadcast_to([float(x) for x in r[3:7]], (2, 4)), atol=1e-14)
        assert np.all(lse[0, :, i] == pytest.approx(-1e9 if n == 0 else math.log(n), abs=1e-14))


def test_fsa_single_token_partial_is_the_key():
    """The pair (i = j*bs, block j) sees one token: m = its score, l = 1, acc = its v."""
    B, Hq, Hkv, T, D, bs = 1, 4, 2, 32, 8, 8
    q, k, v = rand_nsa(B, Hq, Hkv, T, D, seed=31)
    idx = -np.ones((B, Hkv, T, 1), dtype=np.int64)
    idx[..., 0] = (np.arange(T) // bs)[None, None, :]
    parts = fsa.fsa_partials(q, k, v, idx, bs)
    for (b, h, i, j), (m, l, acc) in parts.items():
        if i % bs:
            continue
        for g in range(2):
            np.testing.assert_allclose(m[g], q[b, 2 * h + g, i] @ k[b, h, i] / math.sqrt(D), rtol=1e-13)
            np.testing.assert_allclose(acc[g], v[b, h, i], rtol=1e-13)
        np.testing.assert_allclose(l, 1.0, rtol=0, atol=0)


@pytest.mark.parametrize("G,D,bs,S", [(1, 8, 4, 3), (2, 6, 8, 4), (4, 8, 6, 5)])
def test_fsa_equals_query_outer_oracle(G, D, bs, S):
    """The split-K partials + log-sum-exp combine equal one softmax over the
    union of the selected causal tokens (query-outer oracle), including
    padding, duplicates, future-only rows and empty rows."""
    B, Hkv, T = 2, 2, 6 * bs
    q, k, v = rand_nsa(B, Hkv * G, Hkv, T, D, seed=40 + G)
    g = torch.Generator().manual_seed(7 + G)
    idx = workloads.selection_indices(B, Hkv, T, bs, S, g).numpy().astype(np.int64)
    idx[0, 1, 3:7, 1] = idx[0, 1, 3:7, 0]  # duplicates
    idx[1, 0, bs:2 * bs, :] = -1  # empty rows
    idx[1, 1, 2, 0] = 5  # a wholly future block next to valid ones
    idx[1, 1, 3, :] = -1
    idx[1, 1, 3, 0] = 4  # future-only row
    out, lse = fsa.nsa_select_forward_fsa(q, k, v, idx, bs)
    ref, ref_lse = nsa.nsa_select_forward(q, k, v, idx, bs)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12)
    dense = nsa.nsa_select_dense(q, k, v, idx, bs)
    np.testing.assert_allclose(out, dense, rtol=1e-10, atol=1e-12)


def test_fsa_combine_is_shift_invariant():
    """Adding a constant to one pair's local max and scaling its l and acc by
    exp(-constant) describes the same softmax: the combine must not change."""
    B, Hq, Hkv, T, D, bs, S = 1, 2, 1, 32, 8, 8, 3
    q, k, v = rand_nsa(B, Hq, Hkv, T, D, seed=33)
    g = torch.Generator().manual_seed(8)
    idx = workloads.selection_indices(B, Hkv, T, bs, S, g).numpy()
    parts = fsa.fsa_partials(q, k, v, idx, bs)
    rows = {}
    for (b, h, i, j), p in parts.items():
        rows.setdefault((b, h, i), []).append(p)
    for (b, h, i), ps in rows.items():
        def combine(ps):
            m = np.stack([p[0] for p in ps])
            w = np.exp(m - m.max(axis=0))
            L = (w * np.stack([p[1] for p in ps])).sum(axis=0)
            return (w[:, :, None] * np.stack([p[2] for p in ps])).sum(axis=0) / L[:, None]
        c = 3.25
        shifted = [(ps[0][0] + c, ps[0][1] * math.exp(-c), ps[0][2] * math.exp(-c))] + ps[1:]
        np.testing.assert_allclose(combine(shifted), combine(ps), rtol=1e-12, atol=1e-14)


def test_planted_fsa_mistakes_are_caught(golden, monkeypatch):
    good = fsa.fsa_partials

    def pins():
        try:
            test_fsa_partials_handworked_fixture(golden)
            test_fsa_equals_query_outer_oracle(2, 6, 8, 4)
        except AssertionError:
            return False
        return True

    assert pins()

    def no_causal(q, k, v, block_idx, block_size):
        q, k, v, idx = nsa._check(q, k, v, block_idx, block_size)
        G = q.shape[1] // k.shape[1]
        scale = q.shape[-1] ** -0.5
        parts = {}
        for (b, h, j), pairs in fsa.block_query_lists(idx, block_size).items():
            toks = np.arange(j * block_size, (j + 1) * block_size)
            for i, _ in pairs:
                sc = (q[b, h * G:(h + 1) * G, i] @ k[b, h, toks].T) * scale
                m = sc.max(axis=1)
                p = np.exp(sc - m[:, None])
                parts[(b, h, i, j)] = (m, p.sum(axis=1), p @ v[b, h, toks])
        return parts

    def unshifted_l(*a):
        return {key: (m, l * np.exp(m), acc) for key, (m, l, acc) in good(*a).items()}

    for bad in (no_causal, unshifted_l):
        monkeypatch.setattr(fsa, "fsa_partials", bad)
        assert not pins(), bad.__name__
    monkeypatch.setattr(fsa, "fsa_partials", good)
    assert pins()


def _torch_diff(q1, q2, k1, k2, v, beta, lam, p, normalize):
    """The page's differential_threshold_rela_triton, written with torch
    autograd ops on the textbook TRA (for the gradient pin)."""
    if normalize:
        q1, q2, k1, k2 = (torch.nn.functional.normalize(t, p=2, dim=-1) for t in (q1, q2, k1, k2))
    return _torch_tra(q1, k1, v, beta, p) - torch.clamp(lam, 0.0, 1.0) * _torch_tra(q2, k2, v, beta, p)


@pytest.mark.parametrize("normalize", [True, False])
@pytest.mark.parametrize("p,lam", [(2.0, 0.4), (1.5, 0.7), (3.0, 1.3), (1.0, -0.2)])
def test_tra_diff_backward_matches_torch_autograd(normalize, p, lam):
    q1, k1, v = rand_tra(2, 2, 23, 6, seed=40)
    q2, k2, _ = rand_tra(2, 2, 23, 6, seed=41)
    do = rng(42).standard_normal(q1.shape)
    beta = 0.3 if normalize else 0.8
    got = tra.tra_diff_backward(q1, q2, k1, k2, v, do, beta, lam, p, normalize=normalize)
    ts = [torch.tensor(a, requires_grad=True) for a in (q1, q2, k1, k2, v)]
    lt = torch.tensor(float(lam), dtype=torch.float64, requires_grad=True)
    out = _torch_diff(*ts, beta, lt, p, normalize)
    want = torch.autograd.grad((out * torch.tensor(do)).sum(), ts + [lt])
    for g, w in zip(got[:5], want[:5]):
        np.testing.assert_allclose(g, w.numpy(), rtol=1e-9, atol=1e-11)
    assert got[5] == pytest.approx(float(want[5]), rel=1e-9, abs=1e-11)


def test_tra_diff_backward_finite_differences():
    """Central differences of L = sum(out * dout) of the oracle's own forward."""
    q1, k1, v = rand_tra(1, 1, 8, 4, seed=43)
    q2, k2, _ = rand_tra(1, 1, 8, 4, seed=44)
    do = rng(45).standard_normal(q1.shape)
    beta, lam, p = 0.1, 0.35, 2.0
    grads = tra.tra_diff_backward(q1, q2, k1, k2, v, do, beta, lam, p)

    def L(args, lm=lam):
        return float((tra.tra_diff_forward(*args, beta, lm, p) * do).sum())

    base = [q1, q2, k1, k2, v]
    h = 1e-6
    r = rng(46)
    for which in range(5):
        for _ in range(6):
            idx = tuple(int(r.integers(n)) for n in q1.shape)
            a = [t.copy() for t in base]
            a[which][idx] += h
            lp = L(a)
            a[which][idx] -= 2 * h
            lm_ = L(a)
            assert grads[which][idx] == pytest.approx((lp - lm_) / (2 * h), rel=1e-5, abs=1e-7)
    assert grads[5] == pytest.approx((L(base, lam + h) - L(base, lam - h)) / (2 * h), rel=1e-5, abs=1e-7)


def test_l2_normalize_backward_matches_torch():
    x = rng(47).standard_normal((2, 3, 7, 5))
    x[0, 0, 0] = 0.0  # below eps: the map is x / eps there
    g = rng(48).standard_normal(x.shape)
    xt = torch.tensor(x, requires_grad=True)
    (want,) = torch.autograd.grad((torch.nn.functional.normalize(xt, p=2, dim=-1) * torch.tensor(g)).sum(), xt)
    np.testing.assert_allclose(tra.l2_normalize_backward(x, g), want.numpy(), rtol=1e-10, atol=1e-12)
