"""CPU checks of the C ABI: the library loads, exports every entry point that
``include/bsa.h`` declares, and rejects bad arguments on the host before any
device work (no compute call is made here)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_attention_tra_gb300 import build, bsa

    build.build()
    return bsa.load_library()


def header_functions():
    txt = open(os.path.join(ROOT, "include", "bsa.h")).read()
    return re.findall(r"^BSA_API\s+[\w\s\*]+?\b(\w+)\(", txt, flags=re.M)


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ("tra_forward", "nsa_select_forward", "bsa_status_string", "bsa_version", "bsa_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    from block_sparse_attention_tra_gb300 import bsa

    for code in range(8):
        s = bsa.status_string(code)
        assert s and s != "unknown bsa_status"
    assert bsa.status_string(99) == "unknown bsa_status"
    assert lib.bsa_version() >= 100


P = 4096  # a fake, 16-byte aligned "device" address: validation must reject before using it


def tra(lib, q=P, k=P, v=P, o=P, B=1, H=1, T=16, D=64, beta=1.0, p=2.0, dtype=1):
    from block_sparse_attention_tra_gb300 import bsa

    return bsa.tra_forward_raw(q, k, v, o, B, H, T, D, beta, p, dtype, 0)


def nsa(lib, q=P, k=P, v=P, idx=P, o=P, lse=None, B=1, Hq=16, Hkv=1, T=128, D=128, bs=64, S=4):
    from block_sparse_attention_tra_gb300 import bsa

    return bsa.nsa_select_forward_raw(q, k, v, idx, o, lse, B, Hq, Hkv, T, D, bs, S, 0)


def test_tra_argument_errors(lib):
    assert tra(lib, q=None) == 1
    assert tra(lib, o=None) == 1
    assert tra(lib, dtype=7) == 3
    assert tra(lib, B=0) == 2
    assert tra(lib, T=0) == 2
    assert tra(lib, T=-5) == 2
    assert tra(lib, D=100) == 4  # head dims: multiples of 16 up to 128
    assert tra(lib, D=40) == 4
    assert tra(lib, D=8) == 4
    assert tra(lib, D=144) == 4
    assert tra(lib, D=256) == 4
    assert tra(lib, p=0.0) == 4
    assert tra(lib, p=-1.0) == 4
    assert tra(lib, p=float("nan")) == 4
    assert tra(lib, beta=float("inf")) == 4
    assert tra(lib, q=P + 8) == 7
    assert tra(lib, B=1 << 20, H=1 << 12, T=1 << 10, D=128) == 2  # B*H*T*D >= 2^40


def test_nsa_argument_errors(lib):
    assert nsa(lib, idx=None) == 1
    assert nsa(lib, v=None) == 1
    assert nsa(lib, Hq=24, Hkv=16) == 2  # not a multiple
    assert nsa(lib, T=100) == 2  # T % block_size
    assert nsa(lib, S=0) == 2
    assert nsa(lib, S=33) == 2
    assert nsa(lib, D=96) == 4
    assert nsa(lib, D=8) == 4
    assert nsa(lib, bs=48, T=192) == 4  # block sizes 16, 32, 64, 128 only
    assert nsa(lib, bs=256, T=256) == 4
    assert nsa(lib, Hq=32, Hkv=1) == 4  # group of 32 heads
    assert nsa(lib, k=P + 4) == 7
    assert nsa(lib, idx=P + 2) == 7


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-device path")
def test_valid_arguments_without_a_device_report_device_error(lib):
    assert tra(lib) == 6
    assert nsa(lib) == 6
    for D in (16, 32, 64, 128):
        for bs in (16, 32, 64, 128):
            assert nsa(lib, D=D, bs=bs, T=256) == 6


def test_binding_has_no_cpu_path():
    import torch

    from block_sparse_attention_tra_gb300 import BsaError, nsa_select_forward, tra_forward

    x = torch.zeros(1, 1, 8, 64)
    with pytest.raises(BsaError):
        tra_forward(x, x, x, 1.0, 2.0)
    idx = torch.zeros(1, 1, 64, 1, dtype=torch.int32)
    xb = torch.zeros(1, 16, 64, 64, dtype=torch.bfloat16)
    with pytest.raises(BsaError):
        nsa_select_forward(xb, xb[:, :1], xb[:, :1], idx)


def test_backward_and_diff_argument_errors(lib):
    from block_sparse_attention_tra_gb300 import bsa

    assert bsa.tra_backward_raw(P, P, P, None, P, P, P, 1, 1, 16, 64, 1.0, 2.0, 1, 0) == 1
    assert bsa.tra_backward_raw(P, P, P, P, P, P, P, 1, 1, 16, 64, 1.0, 2.0, 7, 0) == 3  # not a bsa_dtype
    assert bsa.tra_backward_raw(P, P, P, P, P, P, P, 1, 1, 16, 100, 1.0, 2.0, 0, 0) == 4  # f32, D = 100
    assert bsa.tra_backward_raw(P, P, P, P, P, P, P, 1, 1, 16, 100, 1.0, 2.0, 1, 0) == 4
    assert bsa.tra_backward_raw(P, P, P, P, P, P, P, 1, 1, 16, 40, 1.0, 2.0, 1, 0) == 4
    assert bsa.tra_backward_raw(P, P, P, P, P, P, P, 1, 1, 16, 8, 1.0, 2.0, 1, 0) == 4
    assert bsa.tra_backward_raw(P, P, P, P, P + 2, P, P, 1, 1, 16, 64, 1.0, 2.0, 1, 0) == 7
    assert bsa.tra_backward_ex_raw(P, P, P, P, P, P, P, 1, 1, 16, 64, 1.0, 2.0, 1, 2, 0) == 4  # unknown flag bit
    assert bsa.tra_backward_ex_raw(P, P, P, None, P, P, P, 1, 1, 16, 64, 1.0, 2.0, 1, 1, 0) == 1
    assert bsa.tra_diff_forward_raw(P, P, None, P, P, P, 1, 1, 16, 64, 1.0, 0.5, 2.0, 1, 1, 0) == 1
    assert bsa.tra_diff_forward_raw(P, P, P, P, P, P, 0, 1, 16, 64, 1.0, 0.5, 2.0, 1, 1, 0) == 2
    assert bsa.tra_diff_forward_raw(P, P, P, P, P, P, 1, 1, 16, 64, 1.0, float("nan"), 2.0, 1, 1, 0) == 4
    assert bsa.tra_diff_forward_raw(P, P, P, P, P, P, 1, 1, 16, 64, 1.0, 0.5, -2.0, 1, 1, 0) == 4


def test_fsa_workspace_size_and_argument_errors(lib):
    from block_sparse_attention_tra_gb300 import bsa

    ws = bsa.nsa_select_fsa_workspace_size
    B, Hq, Hkv, T, D, S = 2, 32, 2, 8192, 128, 16
    need = ws(B, Hq, Hkv, T, D, 64, S)
    partials = B * Hq * T * S * (D + 2) * 4
    assert partials <= need <= partials + B * Hkv * T * S * 4 + (1 << 22)
    assert need % 256 == 0
    assert ws(B, Hq, Hkv, T, 64, 64, S) < need
    assert ws(B, Hq, Hkv, T, 96, 64, S) == 0  # head dim
    assert ws(B, Hq, Hkv, 100, D, 64, S) == 0  # T % block_size
    assert ws(B, 24, 16, T, D, 64, S) == 0  # Hq % Hkv
    assert ws(B, Hq, Hkv, T, D, 64, 33) == 0
    assert ws(64, 64, 4, 32768, D, 64, 32) == 0  # B*Hq*T*S >= 2^31: 32-bit partial rows

    def fsa(q=P, idx=P, lse=None, work=P * 64, nbytes=1 << 40, B=1, Hq=16, Hkv=1, T=128, D=128, bs=64, S=4):
        return bsa.nsa_select_forward_fsa_raw(q, P, P, idx, P, lse, B, Hq, Hkv, T, D, bs, S, work, nbytes, 0)

    assert fsa(q=None) == 1
    assert fsa(work=None) == 1
    assert fsa(work=P * 64 + 16) == 7  # workspace not 256-byte aligned
    assert fsa(idx=P + 2) == 7
    assert fsa(T=100) == 2
    assert fsa(D=96) == 4
    assert fsa(D=32) == 4  # the split-K form is built for 64-token blocks of 64 or 128 dims
    assert fsa(bs=32) == 4
    assert ws(B, Hq, Hkv, T, 32, 64, S) == 0
    assert fsa(Hq=32, Hkv=1) == 4
    assert fsa(nbytes=ws(1, 16, 1, 128, 128, 64, 4) - 1) == 9  # workspace too small
    if not __import__("torch").cuda.is_available():
        assert fsa(nbytes=ws(1, 16, 1, 128, 128, 64, 4)) == 6  # valid: no device here


def test_tra_forward_ex_flags(lib):
    from block_sparse_attention_tra_gb300 import bsa

    def ex(flags, p=1.5, D=64):
        return bsa.tra_forward_ex_raw(P, P, P, P, 1, 1, 16, D, 1.0, p, 1, flags, 0)

    assert ex(2) == 4 and ex(-1) == 4  # unknown flag bits
    assert ex(1, D=100) == 4
    assert ex(1, p=0.0) == 4
    assert bsa.tra_forward_ex_raw(None, P, P, P, 1, 1, 16, 64, 1.0, 1.5, 1, 1, 0) == 1
    if not __import__("torch").cuda.is_available():
        assert ex(0) == 6 and ex(1) == 6 and ex(1, p=2.0) == 6
        assert ex(0, D=96) == 6 and ex(0, D=48) == 6 and ex(1, D=112) == 6  # other multiples of 16: valid


def test_tra_forward_host_workspace_and_argument_errors(lib):
    from block_sparse_attention_tra_gb300 import bsa

    # three stages of q, k, v, out for one chunk of ceil(B*H / 8) heads
    assert bsa.tra_forward_host_workspace_size(4, 16, 4096, 128, 1) == 3 * 4 * 8 * 4096 * 128 * 2
    assert bsa.tra_forward_host_workspace_size(1, 3, 100, 64, 0) == 3 * 4 * ((1 * 100 * 64 * 4 + 255) // 256 * 256)
    assert bsa.tra_forward_host_workspace_size(1, 1, 16, 40, 1) == 0     # D
    assert bsa.tra_forward_host_workspace_size(1, 1, 16, 64, 7) == 0     # dtype
    assert bsa.tra_forward_host_workspace_size(0, 1, 16, 64, 1) == 0     # B
    ws, need = 1 << 20, bsa.tra_forward_host_workspace_size(1, 1, 16, 64, 1)

    def call(q=P, k=P, v=P, o=P, B=1, H=1, T=16, D=64, beta=1.0, p=2.0, dtype=1, w=ws, nbytes=need):
        return bsa.tra_forward_host_raw(q, k, v, o, B, H, T, D, beta, p, dtype, w, nbytes, 0)

    assert call(q=None) == 1 and call(w=None) == 1
    assert call(dtype=5) == 3
    assert call(B=0) == 2 and call(T=0) == 2
    assert call(D=100) == 4 and call(p=0.0) == 4 and call(beta=float("nan")) == 4
    assert call(w=ws + 16) == 7                      # workspace not 256-byte aligned
    assert call(nbytes=need - 1) == 9                # workspace too small
    if not __import__("torch").cuda.is_available():  # (with a device it would copy from the fake host pointers)
        assert call() == 6                           # valid arguments, no device here


def test_selftest_argument_errors(lib):
    # the self-test entry points validate their arguments on the host too
    assert lib.bsa_selftest_log2(None, P, P, 4, None) == 1
    assert lib.bsa_selftest_exp2(P, None, P, 4, None) == 1
    assert lib.bsa_selftest_exp2(P, P, P, 0, None) == 2
    assert lib.bsa_selftest_log2(P, P, P, -3, None) == 2
    assert lib.bsa_selftest_exp2(P + 2, P, P, 4, None) == 7
    assert lib.bsa_selftest_wait_timeout(0, P, None) == 2       # limit out of range
    assert lib.bsa_selftest_wait_timeout(1000, None, None) == 1
    if not __import__("torch").cuda.is_available():
        assert lib.bsa_selftest_exp2(P, P, P, 4, None) == 6


def test_diff_backward_argument_errors(lib):
    from block_sparse_attention_tra_gb300 import bsa

    def call(dout=P, dq1=P, dv=P, dlam=None, D=64, lam=0.5, dtype=1):
        return bsa.tra_diff_backward_raw(P, P, P, P, P, dout, dq1, P, P, P, dv, dlam, 1, 1, 16, D, 1.0, lam, 2.0, 1,
                                         dtype, 0)

    assert call(dout=None) == 1 and call(dq1=None) == 1 and call(dv=None) == 1
    assert call(dv=P + 8) == 7
    assert call(dlam=P + 2) == 7
    assert call(D=100) == 4 and call(lam=float("nan")) == 4
    assert call(dtype=5) == 3
    if not __import__("torch").cuda.is_available():
        assert call() == 6 and call(dlam=P, dtype=0) == 6
