"""ctypes binding of ``libbsa.so`` (declared in ``include/bsa.h``).

Argument marshalling only: every step of both forwards runs in the CUDA
library.  PyTorch is used for device memory and streams.  There is no CPU
fallback: if the library is missing or the device is not usable, the calls
raise.
"""

from __future__ import annotations

import contextlib
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

BSA_F32 = 0
BSA_BF16 = 1
BSA_TRA_SQRT_HALF_POWERS = 1  # tra_forward_ex flag: p = k + 1/2 as x^k sqrt(x)
BSA_TRA_BWD_DETERMINISTIC = 1  # tra_backward_ex flag: the two-kernel bf16 backward (no scratch, bit-repeatable)

_STATUS = {
    0: "BSA_OK",
    1: "BSA_ERR_NULLPTR",
    2: "BSA_ERR_SHAPE",
    3: "BSA_ERR_DTYPE",
    4: "BSA_ERR_UNSUPPORTED",
    5: "BSA_ERR_LAUNCH",
    6: "BSA_ERR_DEVICE",
    7: "BSA_ERR_ALIGN",
    8: "BSA_ERR_MEMORY",
    9: "BSA_ERR_SCRATCH_LIMIT",
}


class BsaError(RuntimeError):
    """A libbsa call returned a non-zero bsa_status, or the library is absent."""

    def __init__(self, msg, status=None):
        super().__init__(msg)
        self.status = status


def library_path() -> str:
    return os.path.join(_HERE, "libbsa.so")


def load_library():
    """Load ``libbsa.so`` once and declare its C signatures."""
    global _LIB
    if _LIB is not None:
        return _LIB
    _LIB = open_library(library_path())
    return _LIB


@contextlib.contextmanager
def using_library(path):
    """Route every call of this module, inside the ``with`` block, to the
    library at ``path`` (e.g. the debug build, ``libbsa_debug.so``)."""
    global _LIB
    saved = load_library()
    _LIB = open_library(path)
    try:
        yield _LIB
    finally:
        _LIB = saved


def open_library(path):
    """Open a build of the library at ``path`` and declare its C signatures."""
    if not os.path.exists(path):
        raise BsaError(f"{path} is not built; run block_sparse_attention_tra_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.tra_forward.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, i32, vp]
    lib.tra_forward.restype = i32
    lib.tra_forward_ex.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, i32, i32, vp]
    lib.tra_forward_ex.restype = i32
    lib.tra_forward_host_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.tra_forward_host_workspace_size.restype = ctypes.c_size_t
    lib.tra_forward_host.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, i32, vp, ctypes.c_size_t, vp]
    lib.tra_forward_host.restype = i32
    lib.nsa_select_forward.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp]
    lib.nsa_select_forward.restype = i32
    lib.tra_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, i32, vp]
    lib.tra_backward.restype = i32
    lib.tra_backward_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, i32, i32, vp]
    lib.tra_backward_ex.restype = i32
    lib.tra_diff_forward.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, f32, i32, i32, vp]
    lib.tra_diff_forward.restype = i32
    lib.tra_diff_backward.argtypes = [vp] * 12 + [i32, i32, i32, i32, f32, f32, f32, i32, i32, vp]
    lib.tra_diff_backward.restype = i32
    lib.tra_diff_forward_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, f32, i32, i32,
                                             vp]
    lib.tra_diff_forward_noalloc.restype = i32
    lib.nsa_select_fsa_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    lib.nsa_select_fsa_workspace_size.restype = ctypes.c_size_t
    lib.nsa_select_forward_fsa.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp,
                                           ctypes.c_size_t, vp]
    lib.nsa_select_forward_fsa.restype = i32
    lib.bsa_status_string.argtypes = [i32]
    lib.bsa_status_string.restype = ctypes.c_char_p
    lib.bsa_version.argtypes = []
    lib.bsa_version.restype = i32
    lib.bsa_device_error.argtypes = []
    lib.bsa_device_error.restype = i32
    lib.bsa_selftest_wait_timeout.argtypes = [ctypes.c_longlong, vp, vp]
    lib.bsa_selftest_wait_timeout.restype = i32
    lib.bsa_selftest_log2.argtypes = [vp, vp, vp, i32, vp]
    lib.bsa_selftest_log2.restype = i32
    lib.bsa_selftest_exp2.argtypes = [vp, vp, vp, i32, vp]
    lib.bsa_selftest_exp2.restype = i32
    lib.bsa_read_probe.argtypes = [vp, ctypes.c_size_t, i32, vp, vp]
    lib.bsa_read_probe.restype = i32
    return lib


def status_string(status: int) -> str:
    return load_library().bsa_status_string(int(status)).decode()


def device_error() -> int:
    """Read and clear the library's device error words (0 = none, 1 = a
    bounded wait inside a kernel timed out, -1 = could not be read)."""
    return int(load_library().bsa_device_error())


def _check(status: int, what: str):
    if status != 0:
        raise BsaError(f"{what} failed: {_STATUS.get(status, status)} ({status_string(status)})", status)


def tra_forward_raw(q, k, v, out, B, H, T, D, beta, p, dtype, stream=0) -> int:
    """Direct C call with integer device pointers; returns the bsa_status."""
    return load_library().tra_forward(q, k, v, out, B, H, T, D, float(beta), float(p), int(dtype), stream)


def tra_forward_ex_raw(q, k, v, out, B, H, T, D, beta, p, dtype, flags, stream=0) -> int:
    """Direct C call of tra_forward_ex with integer device pointers."""
    return load_library().tra_forward_ex(q, k, v, out, B, H, T, D, float(beta), float(p), int(dtype), int(flags),
                                         stream)


def tra_forward_host_workspace_size(B, H, T, D, dtype) -> int:
    """Device bytes tra_forward_host needs for its workspace (0 if the arguments are rejected)."""
    return int(load_library().tra_forward_host_workspace_size(B, H, T, D, int(dtype)))


def tra_forward_host_raw(q, k, v, out, B, H, T, D, beta, p, dtype, workspace, workspace_bytes, stream=0) -> int:
    """Direct C call of tra_forward_host: integer HOST pointers for q, k, v, out and a device workspace."""
    return load_library().tra_forward_host(q, k, v, out, B, H, T, D, float(beta), float(p), int(dtype), workspace,
                                           int(workspace_bytes), stream)


def tra_backward_raw(q, k, v, dout, dq, dk, dv, B, H, T, D, beta, p, dtype, stream=0) -> int:
    """Direct C call with integer device pointers; returns the bsa_status."""
    return load_library().tra_backward(q, k, v, dout, dq, dk, dv, B, H, T, D, float(beta), float(p), int(dtype),
                                       stream)


def tra_backward_ex_raw(q, k, v, dout, dq, dk, dv, B, H, T, D, beta, p, dtype, flags, stream=0) -> int:
    """Direct C call of tra_backward_ex with integer device pointers; returns the bsa_status."""
    return load_library().tra_backward_ex(q, k, v, dout, dq, dk, dv, B, H, T, D, float(beta), float(p), int(dtype),
                                          int(flags), stream)


def tra_diff_forward_raw(q1, q2, k1, k2, v, out, B, H, T, D, beta, lam, p, normalize, dtype, stream=0) -> int:
    """Direct C call with integer device pointers; returns the bsa_status."""
    return load_library().tra_diff_forward(q1, q2, k1, k2, v, out, B, H, T, D, float(beta), float(lam), float(p),
                                           int(bool(normalize)), int(dtype), stream)


def tra_diff_backward_raw(q1, q2, k1, k2, v, dout, dq1, dq2, dk1, dk2, dv, dlam, B, H, T, D, beta, lam, p,
                          normalize, dtype, stream=0) -> int:
    """Direct C call of tra_diff_backward with integer device pointers (dlam
    may be None); returns the bsa_status."""
    return load_library().tra_diff_backward(q1, q2, k1, k2, v, dout, dq1, dq2, dk1, dk2, dv, dlam, B, H, T, D,
                                            float(beta), float(lam), float(p), int(bool(normalize)), int(dtype),
                                            stream)


def tra_diff_forward_noalloc_raw(q1, q2, k1, k2, v, out, B, H, T, D, beta, lam, p, normalize, dtype,
                                 stream=0) -> int:
    """Direct call of the allocation-free differential entry point (for
    callers that cannot allocate device memory during the call: scratch lives
    in a fixed library-held device array); returns the bsa_status."""
    return load_library().tra_diff_forward_noalloc(q1, q2, k1, k2, v, out, B, H, T, D, float(beta), float(lam),
                                                   float(p), int(bool(normalize)), int(dtype), stream)


def nsa_select_forward_raw(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, D, block_size, S,
                           stream=0) -> int:
    """Direct C call with integer device pointers; returns the bsa_status."""
    return load_library().nsa_select_forward(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, D,
                                             block_size, S, stream)


def nsa_select_fsa_workspace_size(B, Hq, Hkv, T, D, block_size, S) -> int:
    """Bytes of workspace ``nsa_select_forward_fsa`` needs (0 = sizes not accepted)."""
    return int(load_library().nsa_select_fsa_workspace_size(B, Hq, Hkv, T, D, block_size, S))


def nsa_select_forward_fsa_raw(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, D, block_size, S, workspace,
                               workspace_bytes, stream=0) -> int:
    """Direct C call with integer device pointers; returns the bsa_status."""
    return load_library().nsa_select_forward_fsa(q, k, v, block_idx, out, lse, B, Hq, Hkv, T, D, block_size, S,
                                                 workspace, int(workspace_bytes), stream)


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t):
    import torch

    if t.dtype == torch.float32:
        return BSA_F32
    if t.dtype == torch.bfloat16:
        return BSA_BF16
    raise BsaError(f"unsupported dtype {t.dtype}", 3)


def tra_forward(q, k, v, beta: float, p: float = 2.0, out=None, stream=None, sqrt_half_powers: bool = False):
    """Threshold rectified attention forward on CUDA tensors ``[B, H, T, D]``.

    ``out = ReLU(q k^T - tau(i))^p v`` with ``tau(i) = beta sqrt(2 ln(i+1)/D)``,
    causal, unnormalised; float32 or bfloat16 in, same dtype out.  Runs on
    ``stream`` (default: torch's current stream) without synchronising.
    ``sqrt_half_powers``: evaluate p = 0.5, 1.5, 2.5, 3.5 as x^k sqrt(x)
    (``tra_forward_ex`` with ``BSA_TRA_SQRT_HALF_POWERS``).
    """
    if q.device.type != "cuda":
        raise BsaError("tra_forward takes CUDA tensors (no CPU path)")
    if not (q.shape == k.shape == v.shape) or q.dim() != 4:
        raise BsaError("q, k, v must share one shape [B, H, T, D]", 2)
    if not (q.dtype == k.dtype == v.dtype):
        raise BsaError("q, k, v must share one dtype", 3)
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    if out is None:
        import torch

        out = torch.empty_like(q)
    B, H, T, D = q.shape
    if sqrt_half_powers:
        st = tra_forward_ex_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, T, D, beta, p,
                                _dtype_code(q), BSA_TRA_SQRT_HALF_POWERS, _stream_handle(stream))
    else:
        st = tra_forward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, T, D,
                             beta, p, _dtype_code(q), _stream_handle(stream))
    _check(st, "tra_forward")
    return out


def tra_forward_host(q, k, v, beta: float, p: float = 2.0, out=None, workspace=None, stream=None):
    """Threshold rectified attention forward on CPU tensors ``[B, H, T, D]``
    (float32 or bfloat16; page-locked tensors, e.g. ``t.pin_memory()``, let the
    copies overlap the kernels).  The library streams chunks of heads through
    the GPU (``tra_forward_host``); ``workspace`` is a uint8 CUDA tensor of at
    least ``tra_forward_host_workspace_size`` bytes (allocated if None).  The
    call is asynchronous on ``stream`` (default: torch's current stream):
    keep q, k, v, out and the workspace alive, and synchronise ``stream``,
    before reading ``out`` or releasing them (the library's copies run on
    its own streams, which torch's allocators do not see)."""
    import torch

    if q.device.type != "cpu" or k.device.type != "cpu" or v.device.type != "cpu":
        raise BsaError("tra_forward_host takes host (CPU) tensors")
    if not (q.shape == k.shape == v.shape) or q.dim() != 4:
        raise BsaError("q, k, v must share one shape [B, H, T, D]", 2)
    if not (q.dtype == k.dtype == v.dtype):
        raise BsaError("q, k, v must share one dtype", 3)
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if out.device.type != "cpu" or out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise BsaError("out must be a contiguous CPU tensor shaped and typed like q", 2)
    B, H, T, D = q.shape
    dt = _dtype_code(q)
    need = tra_forward_host_workspace_size(B, H, T, D, dt)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        if isinstance(stream, torch.cuda.Stream):
            workspace.record_stream(stream)  # not reused before `stream` passes this call
    st = tra_forward_host_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, T, D, beta, p, dt,
                              workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                              _stream_handle(stream))
    _check(st, "tra_forward_host")
    return out


_TRA_FUNCTION = None


def _tra_function():
    """The autograd function of the threshold attention (page
    "triton_threshold_attention.py", ThresholdRelaFunction): forward through
    ``tra_forward``, backward through ``tra_backward``; both on torch's
    current stream."""
    global _TRA_FUNCTION
    if _TRA_FUNCTION is None:
        import torch

        class TraFunction(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, beta, p):
                ctx.save_for_backward(q, k, v)
                ctx.beta, ctx.p = float(beta), float(p)
                return tra_forward(q, k, v, beta, p)

            @staticmethod
            def backward(ctx, dout):
                q, k, v = ctx.saved_tensors
                dq, dk, dv = tra_backward(q, k, v, dout.to(q.dtype).contiguous(), ctx.beta, ctx.p)
                return dq, dk, dv, None, None

        _TRA_FUNCTION = TraFunction
    return _TRA_FUNCTION


def tra_attention(q, k, v, beta: float, p: float = 2.0):
    """Threshold rectified attention with autograd: ``tra_forward`` whose
    gradients with respect to q, k and v come from ``tra_backward`` (CUDA
    tensors ``[B, H, T, D]``, bfloat16 or float32)."""
    return _tra_function().apply(q, k, v, beta, p)


def tra_backward(q, k, v, dout, beta: float, p: float = 2.0, stream=None, deterministic: bool = False):
    """Gradients ``(dq, dk, dv)`` of the threshold rectified attention
    forward for the upstream gradient ``dout``; bf16 or fp32 CUDA tensors
    ``[B, H, T, D]``.  Scores are recomputed; runs on ``stream`` (default:
    torch's current stream) without synchronising.  bf16 runs the fused
    kernel (dq summed in fp32 in a run-dependent order) unless
    ``deterministic`` asks for the two-kernel form."""
    import torch

    if q.device.type != "cuda":
        raise BsaError("tra_backward takes CUDA tensors (no CPU path)")
    if not (q.shape == k.shape == v.shape == dout.shape) or q.dim() != 4:
        raise BsaError("q, k, v, dout must share one shape [B, H, T, D]", 2)
    if not (q.dtype == k.dtype == v.dtype == dout.dtype):
        raise BsaError("q, k, v, dout must share one dtype", 3)
    q, k, v, dout = q.contiguous(), k.contiguous(), v.contiguous(), dout.contiguous()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    B, H, T, D = q.shape
    st = tra_backward_ex_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(), dq.data_ptr(),
                             dk.data_ptr(), dv.data_ptr(), B, H, T, D, beta, p, _dtype_code(q),
                             BSA_TRA_BWD_DETERMINISTIC if deterministic else 0, _stream_handle(stream))
    _check(st, "tra_backward")
    return dq, dk, dv


def tra_diff_forward(q1, q2, k1, k2, v, beta: float, lam: float, p: float = 2.0, normalize: bool = True,
                     out=None, stream=None):
    """Threshold differential attention on bf16 CUDA tensors ``[B, H, T, D]``:
    ``TRA(n(q1), n(k1), v) - clamp(lam, 0, 1) * TRA(n(q2), n(k2), v)`` with
    ``n`` the row-wise L2 normalisation when ``normalize``."""
    import torch

    ts = (q1, q2, k1, k2, v)
    if q1.device.type != "cuda":
        raise BsaError("tra_diff_forward takes CUDA tensors (no CPU path)")
    if any(t.shape != q1.shape for t in ts) or q1.dim() != 4:
        raise BsaError("q1, q2, k1, k2, v must share one shape [B, H, T, D]", 2)
    if any(t.dtype != q1.dtype for t in ts):
        raise BsaError("q1, q2, k1, k2, v must share one dtype", 3)
    q1, q2, k1, k2, v = (t.contiguous() for t in ts)
    if out is None:
        out = torch.empty_like(q1)
    B, H, T, D = q1.shape
    st = tra_diff_forward_raw(q1.data_ptr(), q2.data_ptr(), k1.data_ptr(), k2.data_ptr(), v.data_ptr(),
                              out.data_ptr(), B, H, T, D, beta, lam, p, normalize, _dtype_code(q1),
                              _stream_handle(stream))
    _check(st, "tra_diff_forward")
    return out



def tra_diff_backward(q1, q2, k1, k2, v, dout, beta: float, lam: float, p: float = 2.0, normalize: bool = True,
                      want_dlam: bool = False, stream=None):
    """Gradients ``(dq1, dq2, dk1, dk2, dv, dlam)`` of ``tra_diff_forward`` for
    the upstream gradient ``dout`` (bf16 or fp32 CUDA tensors ``[B, H, T,
    D]``); ``dlam`` is a 1-element float32 CUDA tensor when ``want_dlam``,
    else None."""
    import torch

    ts = (q1, q2, k1, k2, v, dout)
    if q1.device.type != "cuda":
        raise BsaError("tra_diff_backward takes CUDA tensors (no CPU path)")
    if any(t.shape != q1.shape for t in ts) or q1.dim() != 4:
        raise BsaError("q1, q2, k1, k2, v, dout must share one shape [B, H, T, D]", 2)
    if any(t.dtype != q1.dtype for t in ts):
        raise BsaError("q1, q2, k1, k2, v, dout must share one dtype", 3)
    ts = tuple(t.contiguous() for t in ts)
    grads = tuple(torch.empty_like(q1) for _ in range(5))
    dlam = torch.empty(1, dtype=torch.float32, device=q1.device) if want_dlam else None
    B, H, T, D = q1.shape
    st = tra_diff_backward_raw(*(t.data_ptr() for t in ts), *(g.data_ptr() for g in grads),
                               dlam.data_ptr() if dlam is not None else None, B, H, T, D, beta, lam, p, normalize,
                               _dtype_code(q1), _stream_handle(stream))
    _check(st, "tra_diff_backward")
    return grads + (dlam,)


_TRA_DIFF_FUNCTION = None


def _tra_diff_function():
    """The autograd function of the differential form (page
    "triton_threshold_attention.py", differential_threshold_rela_triton):
    forward through ``tra_diff_forward``, backward through
    ``tra_diff_backward``; lambda may be a float or a 0-d / 1-element tensor
    (its gradient is returned when it requires one)."""
    global _TRA_DIFF_FUNCTION
    if _TRA_DIFF_FUNCTION is None:
        import torch

        class TraDiffFunction(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q1, q2, k1, k2, v, beta, lam, p, normalize):
                lam_f = float(lam)
                ctx.save_for_backward(q1, q2, k1, k2, v)
                ctx.args = (float(beta), lam_f, float(p), bool(normalize))
                ctx.lam_tensor = isinstance(lam, torch.Tensor)
                return tra_diff_forward(q1, q2, k1, k2, v, beta, lam_f, p, normalize=normalize)

            @staticmethod
            def backward(ctx, dout):
                q1, q2, k1, k2, v = ctx.saved_tensors
                beta, lam, p, normalize = ctx.args
                want = ctx.lam_tensor and ctx.needs_input_grad[6]
                dq1, dq2, dk1, dk2, dv, dlam = tra_diff_backward(q1, q2, k1, k2, v, dout.to(q1.dtype), beta, lam, p,
                                                                 normalize, want_dlam=want)
                dl = dlam.reshape(()) if want else None
                return dq1, dq2, dk1, dk2, dv, None, dl, None, None

        _TRA_DIFF_FUNCTION = TraDiffFunction
    return _TRA_DIFF_FUNCTION


def tra_diff_attention(q1, q2, k1, k2, v, beta: float, lam, p: float = 2.0, normalize: bool = True):
    """Threshold differential attention with autograd: ``tra_diff_forward``
    whose gradients with respect to q1, q2, k1, k2, v (and lambda, when it is
    a tensor that requires one) come from ``tra_diff_backward``."""
    return _tra_diff_function().apply(q1, q2, k1, k2, v, beta, lam, p, normalize)

def nsa_select_forward(q, k, v, block_idx, block_size: int = 64, out=None, lse=None,
                       return_lse: bool = False, stream=None):
    """NSA selection-branch forward on CUDA tensors.

    q ``[B, Hq, T, D]``, k/v ``[B, Hkv, T, D]`` bf16, ``block_idx [B, Hkv, T,
    S]`` int32 (-1 = padding).  Returns ``out`` (and ``lse [B, Hq, T]`` fp32
    when ``return_lse``).
    """
    import torch

    if q.device.type != "cuda":
        raise BsaError("nsa_select_forward takes CUDA tensors (no CPU path)")
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape or block_idx.dim() != 4:
        raise BsaError("q [B,Hq,T,D], k/v [B,Hkv,T,D], block_idx [B,Hkv,T,S] expected", 2)
    if not (q.dtype == k.dtype == v.dtype == torch.bfloat16):
        raise BsaError("nsa_select_forward takes bfloat16 q, k, v", 3)
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    S = block_idx.shape[-1]
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    idx = block_idx.to(torch.int32).contiguous()
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, T), device=q.device, dtype=torch.float32)
    st = nsa_select_forward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), idx.data_ptr(),
                                out.data_ptr(), lse.data_ptr() if lse is not None else None,
                                B, Hq, Hkv, T, D, block_size, S, _stream_handle(stream))
    _check(st, "nsa_select_forward")
    return (out, lse) if return_lse else out


def nsa_select_forward_fsa(q, k, v, block_idx, block_size: int = 64, out=None, lse=None,
                           return_lse: bool = False, workspace=None, stream=None):
    """NSA selection forward in the block-outer split-K form (same arguments
    and result as ``nsa_select_forward``).  ``workspace`` is a uint8 CUDA
    tensor of at least ``nsa_select_fsa_workspace_size(...)`` bytes; one is
    allocated when it is None.  It stays in use until the stream's work is
    done."""
    import torch

    if q.device.type != "cuda":
        raise BsaError("nsa_select_forward_fsa takes CUDA tensors (no CPU path)")
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape or block_idx.dim() != 4:
        raise BsaError("q [B,Hq,T,D], k/v [B,Hkv,T,D], block_idx [B,Hkv,T,S] expected", 2)
    if not (q.dtype == k.dtype == v.dtype == torch.bfloat16):
        raise BsaError("nsa_select_forward_fsa takes bfloat16 q, k, v", 3)
    B, Hq, T, D = q.shape
    Hkv = k.shape[1]
    S = block_idx.shape[-1]
    q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
    idx = block_idx.to(torch.int32).contiguous()
    need = nsa_select_fsa_workspace_size(B, Hq, Hkv, T, D, block_size, S)
    if need == 0:
        raise BsaError("nsa_select_forward_fsa: sizes not accepted", 2)
    if workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, T), device=q.device, dtype=torch.float32)
    st = nsa_select_forward_fsa_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), idx.data_ptr(), out.data_ptr(),
                                    lse.data_ptr() if lse is not None else None, B, Hq, Hkv, T, D, block_size, S,
                                    workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    _check(st, "nsa_select_forward_fsa")
    return (out, lse) if return_lse else out


def selftest_wait_timeout(limit_cycles: int = 100000, stream=None) -> int:
    """Run the bounded-wait expiry self test (a wait on an mbarrier nothing
    arrives on, with a short limit).  Returns the kernel's result word: 0 when
    the wait gave up as designed.  The timeout is also recorded in the device
    error word that ``device_error()`` reads and clears."""
    import torch

    res = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _check(load_library().bsa_selftest_wait_timeout(int(limit_cycles), res.data_ptr(), _stream_handle(stream)),
           "bsa_selftest_wait_timeout")
    return int(res.item())


def selftest_log2(x, stream=None):
    """The epilogue's FMA-pipe log2 and CUDA's log2f on the same float32
    device tensor; returns ``(y_fma, y_ref)``."""
    import torch

    if not (x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()):
        raise BsaError("selftest_log2 needs a contiguous float32 CUDA tensor")
    y_fma, y_ref = torch.empty_like(x), torch.empty_like(x)
    _check(load_library().bsa_selftest_log2(x.data_ptr(), y_fma.data_ptr(), y_ref.data_ptr(), x.numel(),
                                            _stream_handle(stream)), "bsa_selftest_log2")
    return y_fma, y_ref


def selftest_exp2(y, stream=None):
    """The epilogue's FMA-pipe exp2 (fp32, before the bf16 rounding) and
    CUDA's exp2f on the same float32 device tensor; returns ``(w_fma, w_ref)``."""
    import torch

    if not (y.is_cuda and y.dtype == torch.float32 and y.is_contiguous()):
        raise BsaError("selftest_exp2 needs a contiguous float32 CUDA tensor")
    w_fma, w_ref = torch.empty_like(y), torch.empty_like(y)
    _check(load_library().bsa_selftest_exp2(y.data_ptr(), w_fma.data_ptr(), w_ref.data_ptr(), y.numel(),
                                            _stream_handle(stream)), "bsa_selftest_exp2")
    return w_fma, w_ref


def read_probe(buf, reps: int, sink, stream=None):
    """Enqueue the streaming-read probe over the bytes of CUDA tensor ``buf``
    (``reps`` passes); ``sink`` is a 1-element int32 CUDA tensor."""
    nbytes = buf.numel() * buf.element_size()
    _check(load_library().bsa_read_probe(buf.data_ptr(), nbytes - nbytes % 16, int(reps), sink.data_ptr(),
                                         _stream_handle(stream)), "bsa_read_probe")
