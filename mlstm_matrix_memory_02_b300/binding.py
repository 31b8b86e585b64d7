"""Thin Python binding of the mLSTM C ABI (include/mlstm.h) -- argument marshalling only.

Every function has the name of the C entry point it calls, takes torch CUDA tensors,
checks dtype/shape/contiguity, passes raw device pointers and the current torch stream to
the library, and raises :class:`MlstmError` on a non-OK status.  All computation happens in
the library's CUDA kernels; there is no fallback of any kind: if the compiled library is
missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmlstm_b300.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -m mlstm_matrix_memory_02_b300.build)")

_lib = ctypes.CDLL(LIB_PATH)

F32, BF16 = 0, 1
_DT = {torch.float32: F32, torch.bfloat16: BF16}

_vp, _fp, _i, _sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_lib.mlstm_status_str.restype = ctypes.c_char_p
_lib.mlstm_status_str.argtypes = [_i]
_lib.mlstm_last_cuda_error.restype = _i
_lib.mlstm_last_cuda_error.argtypes = []
_lib.mlstm_wait_selftest.restype = _i
_lib.mlstm_wait_selftest.argtypes = [_vp, _sz, _i, _i, _i, _i, _i, _i, _i, _vp]
_lib.mlstm_groupnorm_gate.restype = _i
_lib.mlstm_groupnorm_gate.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, _vp, _i, _i, _i, _i, _i, _i, _i, _vp]
_lib.mlstm_kernel_launches.restype = ctypes.c_ulonglong
_lib.mlstm_kernel_launches.argtypes = []
_lib.mlstm_fwd_from_gates.restype = _i
_lib.mlstm_fwd_from_gates.argtypes = [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _fp, _fp, _vp, _i,
                                      _fp, _fp, _fp, _vp, _sz, _vp]
_lib.mlstm_fwd_workspace_bytes.restype = _sz
_lib.mlstm_fwd_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i]
_lib.mlstm_fwd_chunkwise.restype = _i
_lib.mlstm_fwd_chunkwise.argtypes = [_vp, _vp, _vp, _fp, _fp, _i, _i, _i, _i, _i, _i, _i,
                                     _fp, _fp, _fp, _vp, _i, _fp, _fp, _fp, _vp, _sz, _vp]
_lib.mlstm_fwd_chunk_states.restype = _i
_lib.mlstm_fwd_chunk_states.argtypes = [_vp, _vp, _fp, _fp, _i, _i, _i, _i, _i, _i, _i,
                                        _fp, _fp, _fp, _fp, _fp, _fp, _vp, _sz, _vp]
_lib.mlstm_fwd_gates.restype = _i
_lib.mlstm_fwd_gates.argtypes = [_fp, _fp, _i, _i, _i, _i, _fp, _fp, _fp, _vp, _sz, _vp]
_lib.mlstm_fwd_path.restype = _i
_lib.mlstm_fwd_path.argtypes = [_i, _i, _i, _i, _i, _i, _i]
_lib.mlstm_fwd_workspace_min_bytes.restype = _sz
_lib.mlstm_fwd_workspace_min_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i]
_lib.mlstm_fwd_segments.restype = _i
_lib.mlstm_fwd_segments.argtypes = [_i, _i, _i, _i, _i, _i, _i, _sz]
_lib.mlstm_bwd_workspace_bytes.restype = _sz
_lib.mlstm_bwd_workspace_bytes.argtypes = [_i, _i, _i, _i, _i, _i, _i]
_lib.mlstm_bwd_chunkwise.restype = _i
_lib.mlstm_bwd_chunkwise.argtypes = [_vp, _vp, _vp, _fp, _fp, _vp, _i, _i, _i, _i, _i, _i, _i, _fp, _fp, _fp,
                                     _vp, _vp, _vp, _fp, _fp, _fp, _fp, _fp, _vp, _sz, _vp]
_lib.mlstm_fwd_check.restype = _i
_lib.mlstm_fwd_check.argtypes = [_vp, _sz, _i, _i, _i, _i, _i, _i, _i, _vp]
_lib.mlstm_step.restype = _i
_lib.mlstm_step.argtypes = [_vp, _vp, _vp, _fp, _fp, _fp, _fp, _fp, _vp, _i, _i, _i, _i,
                            _i, _i, _vp]

_lib.mlstm_step_multi.restype = _i
_lib.mlstm_step_multi.argtypes = [_vp, _vp, _vp, _fp, _fp, _fp, _fp, _fp, _vp, _i, _i, _i, _i, _i,
                                  _i, _i, _vp]
_lib.mlstm_fwd_chunkwise_noalloc.restype = _i
_lib.mlstm_fwd_chunkwise_noalloc.argtypes = [_vp, _vp, _vp, _fp, _fp, _i, _i, _i, _i, _i, _i, _i,
                                             _fp, _fp, _fp, _vp, _i, _fp, _fp, _fp, _vp]
_lib.mlstm_fwd_check_noalloc.restype = _i
_lib.mlstm_fwd_check_noalloc.argtypes = [_vp]
_lib.mlstm_noalloc_scratch.restype = _i
_lib.mlstm_noalloc_scratch.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(_sz)]

EXPORTED = ["mlstm_status_str", "mlstm_last_cuda_error", "mlstm_kernel_launches",
            "mlstm_fwd_workspace_bytes", "mlstm_fwd_chunkwise", "mlstm_fwd_from_gates",
            "mlstm_fwd_chunk_states", "mlstm_fwd_gates", "mlstm_fwd_check", "mlstm_fwd_path",
            "mlstm_step", "mlstm_step_multi", "mlstm_fwd_chunkwise_noalloc", "mlstm_groupnorm_gate",
            "mlstm_wait_selftest", "mlstm_fwd_check_noalloc", "mlstm_noalloc_scratch",
            "mlstm_fwd_workspace_min_bytes", "mlstm_fwd_segments", "mlstm_bwd_workspace_bytes",
            "mlstm_bwd_chunkwise"]
SELFTEST_WAIT_CODE = 90

# Bytes of the fixed scratch array behind mlstm_fwd_chunkwise_noalloc (include/mlstm.h).
NOALLOC_SCRATCH_BYTES = 8 << 20

# Forget-gate variants: "sigmoid" (f = sigmoid(f~), the default) or "exp" (f = exp(f~)); the
# variant is passed to the library OR-ed into the dtype code.
FORGET_EXP = 0x100
FORGET_GATES = ("sigmoid", "exp")


def _dt_code(dtype, forget="sigmoid"):
    if forget not in FORGET_GATES:
        raise ValueError(f"forget must be one of {FORGET_GATES}")
    return _DT[dtype] | (FORGET_EXP if forget == "exp" else 0)


class MlstmError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = _lib.mlstm_status_str(code).decode()
        if code == 6:
            msg += f" (cudaError {_lib.mlstm_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")
        self.code = code


def library():
    """The loaded ctypes handle (for tests that check the exported symbols)."""
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code, where):
    if code != 0:
        raise MlstmError(code, where)


def _dev(t, name, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def mlstm_fwd_workspace_bytes(B, NH, S, DQK, DV, chunk, dtype=torch.bfloat16) -> int:
    return int(_lib.mlstm_fwd_workspace_bytes(B, NH, S, DQK, DV, chunk, _DT[dtype]))


def mlstm_fwd_workspace_min_bytes(B, NH, S, DQK, DV, chunk, dtype=torch.bfloat16) -> int:
    return int(_lib.mlstm_fwd_workspace_min_bytes(B, NH, S, DQK, DV, chunk, _DT[dtype]))


def mlstm_fwd_segments(B, NH, S, DQK, DV, chunk, dtype=torch.bfloat16, ws_bytes=None) -> int:
    """Segments of each head's sequence the forward runs in parallel with a workspace of
    `ws_bytes` (default: mlstm_fwd_workspace_bytes for these sizes); 1 = none, -1 = unsupported."""
    if ws_bytes is None:
        ws_bytes = mlstm_fwd_workspace_bytes(B, NH, S, DQK, DV, chunk, dtype)
    return int(_lib.mlstm_fwd_segments(B, NH, S, DQK, DV, chunk, _DT[dtype], ws_bytes))


def mlstm_fwd_path(B, NH, S, DQK, DV, chunk, dtype=torch.bfloat16) -> int:
    """Kernels mlstm_fwd_chunkwise runs for these sizes: 1 = the fused tensor-core kernel,
    2 = the same with each head's d_qk split over a CTA pair, 0 = the CUDA-core kernels,
    -1 = unsupported sizes or dtype."""
    return int(_lib.mlstm_fwd_path(B, NH, S, DQK, DV, chunk, _DT[dtype]))


def alloc_workspace(B, NH, S, DQK, DV, chunk, dtype=torch.bfloat16, device=None):
    n = mlstm_fwd_workspace_bytes(B, NH, S, DQK, DV, chunk, dtype)
    if n == 0:
        raise ValueError("unsupported sizes for the mLSTM forward")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def mlstm_fwd_chunkwise(q, k, v, igate_pre, fgate_pre, chunk, h_dtype=None, C_init=None,
                        n_init=None, m_init=None, out=None, workspace=None, stream=None,
                        forget="sigmoid"):
    """Chunkwise forward.  q, k [B,NH,S,DQK], v [B,NH,S,DV] (fp32 or bf16), gates [B,NH,S]
    fp32.  Returns (h, C_last, n_last, m_last); ``out`` may supply those four tensors.
    ``forget`` is the forget-gate variant ("sigmoid" or "exp")."""
    B, NH, S, DQK = q.shape
    DV = v.shape[-1]
    dt = q.dtype
    _dev(q, "q", dt)
    _dev(k, "k", dt, (B, NH, S, DQK))
    _dev(v, "v", dt, (B, NH, S, DV))
    _dev(igate_pre, "igate_pre", torch.float32, (B, NH, S))
    _dev(fgate_pre, "fgate_pre", torch.float32, (B, NH, S))
    if dt not in _DT:
        raise TypeError("q, k, v must be float32 or bfloat16")
    h_dtype = h_dtype or dt
    init = (C_init, n_init, m_init)
    if any(x is not None for x in init):
        _dev(C_init, "C_init", torch.float32, (B, NH, DV, DQK))
        _dev(n_init, "n_init", torch.float32, (B, NH, DQK))
        _dev(m_init, "m_init", torch.float32, (B, NH))
    if out is None:
        h = torch.empty((B, NH, S, DV), dtype=h_dtype, device=q.device)
        C_last = torch.empty((B, NH, DV, DQK), dtype=torch.float32, device=q.device)
        n_last = torch.empty((B, NH, DQK), dtype=torch.float32, device=q.device)
        m_last = torch.empty((B, NH), dtype=torch.float32, device=q.device)
    else:
        h, C_last, n_last, m_last = out
        _dev(h, "h", h_dtype, (B, NH, S, DV))
        _dev(C_last, "C_last", torch.float32, (B, NH, DV, DQK))
        _dev(n_last, "n_last", torch.float32, (B, NH, DQK))
        _dev(m_last, "m_last", torch.float32, (B, NH))
    if workspace is None:
        workspace = alloc_workspace(B, NH, S, DQK, DV, chunk, dt, q.device)
    code = _lib.mlstm_fwd_chunkwise(
        _ptr(q), _ptr(k), _ptr(v), _ptr(igate_pre), _ptr(fgate_pre), B, NH, S, DQK, DV, chunk,
        _dt_code(dt, forget), _ptr(C_init), _ptr(n_init), _ptr(m_init), _ptr(h), _DT[h_dtype],
        _ptr(C_last), _ptr(n_last), _ptr(m_last), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(code, "mlstm_fwd_chunkwise")
    return h, C_last, n_last, m_last


def mlstm_bwd_workspace_bytes(B, NH, S, DQK, DV, chunk, dtype=torch.bfloat16) -> int:
    return int(_lib.mlstm_bwd_workspace_bytes(B, NH, S, DQK, DV, chunk, _DT[dtype]))


def mlstm_bwd_chunkwise(q, k, v, igate_pre, fgate_pre, dh, chunk, C_init=None, n_init=None, m_init=None,
                        init_grads=None, workspace=None, stream=None, forget="sigmoid"):
    """Backward of mlstm_fwd_chunkwise for the loss sum(dh * h).  Returns a dict with dq, dk, dv
    (dtype of q), dig, dfg (fp32) and, when ``init_grads`` is true (default: when an initial
    state is given), dC_init, dn_init, dm_init."""
    B, NH, S, DQK = q.shape
    DV = v.shape[-1]
    dt = q.dtype
    if dt not in _DT:
        raise TypeError("q, k, v must be float32 or bfloat16")
    _dev(q, "q", dt)
    _dev(k, "k", dt, (B, NH, S, DQK))
    _dev(v, "v", dt, (B, NH, S, DV))
    _dev(dh, "dh", dt, (B, NH, S, DV))
    _dev(igate_pre, "igate_pre", torch.float32, (B, NH, S))
    _dev(fgate_pre, "fgate_pre", torch.float32, (B, NH, S))
    given = any(x is not None for x in (C_init, n_init, m_init))
    if given:
        _dev(C_init, "C_init", torch.float32, (B, NH, DV, DQK))
        _dev(n_init, "n_init", torch.float32, (B, NH, DQK))
        _dev(m_init, "m_init", torch.float32, (B, NH))
    if init_grads is None:
        init_grads = given
    out = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
           "dig": torch.empty_like(igate_pre), "dfg": torch.empty_like(fgate_pre)}
    if init_grads:
        out["dC_init"] = torch.empty((B, NH, DV, DQK), dtype=torch.float32, device=q.device)
        out["dn_init"] = torch.empty((B, NH, DQK), dtype=torch.float32, device=q.device)
        out["dm_init"] = torch.empty((B, NH), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = mlstm_bwd_workspace_bytes(B, NH, S, DQK, DV, chunk, dt)
        if n == 0:
            raise ValueError("unsupported sizes for the mLSTM backward")
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    code = _lib.mlstm_bwd_chunkwise(
        _ptr(q), _ptr(k), _ptr(v), _ptr(igate_pre), _ptr(fgate_pre), _ptr(dh), B, NH, S, DQK, DV, chunk,
        _dt_code(dt, forget), _ptr(C_init), _ptr(n_init), _ptr(m_init), _ptr(out["dq"]), _ptr(out["dk"]),
        _ptr(out["dv"]), _ptr(out["dig"]), _ptr(out["dfg"]), _ptr(out.get("dC_init")), _ptr(out.get("dn_init")),
        _ptr(out.get("dm_init")), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(code, "mlstm_bwd_chunkwise")
    return out


def mlstm_step_multi(q, k, v, ig, fg, C, n, m, h=None, h_dtype=None, stream=None, forget="sigmoid"):
    """T consecutive decode steps in one launch, in place on (C, n, m).  q, k [B,NH,T,DQK],
    v [B,NH,T,DV], ig, fg [B,NH,T]; returns h [B,NH,T,DV]."""
    B, NH, T, DQK = q.shape
    DV = v.shape[-1]
    dt = q.dtype
    _dev(q, "q", dt)
    _dev(k, "k", dt, (B, NH, T, DQK))
    _dev(v, "v", dt, (B, NH, T, DV))
    _dev(ig, "ig", torch.float32, (B, NH, T))
    _dev(fg, "fg", torch.float32, (B, NH, T))
    _dev(C, "C", torch.float32, (B, NH, DV, DQK))
    _dev(n, "n", torch.float32, (B, NH, DQK))
    _dev(m, "m", torch.float32, (B, NH))
    h_dtype = h_dtype or (h.dtype if h is not None else dt)
    if h is None:
        h = torch.empty((B, NH, T, DV), dtype=h_dtype, device=q.device)
    _dev(h, "h", h_dtype, (B, NH, T, DV))
    code = _lib.mlstm_step_multi(_ptr(q), _ptr(k), _ptr(v), _ptr(ig), _ptr(fg), _ptr(C), _ptr(n),
                                 _ptr(m), _ptr(h), B, NH, T, DQK, DV, _dt_code(dt, forget),
                                 _DT[h_dtype], _stream(stream))
    _check(code, "mlstm_step_multi")
    return h


def mlstm_fwd_chunkwise_noalloc(q, k, v, igate_pre, fgate_pre, chunk, out, C_init=None, n_init=None,
                                m_init=None, stream=None, forget="sigmoid"):
    """The chunkwise forward without any device allocation, for callers that cannot allocate
    (a host application that owns all device memory, a serving loop where cudaMalloc could
    synchronise the device): the library uses its own fixed scratch array.  The four outputs
    (h, C_last, n_last, m_last) must be supplied in ``out`` -- this wrapper allocates nothing
    either; h's dtype is taken from ``out``."""
    B, NH, S, DQK = q.shape
    DV = v.shape[-1]
    dt = q.dtype
    if dt not in _DT:
        raise TypeError("q, k, v must be float32 or bfloat16")
    _dev(q, "q", dt)
    _dev(k, "k", dt, (B, NH, S, DQK))
    _dev(v, "v", dt, (B, NH, S, DV))
    _dev(igate_pre, "igate_pre", torch.float32, (B, NH, S))
    _dev(fgate_pre, "fgate_pre", torch.float32, (B, NH, S))
    if any(x is not None for x in (C_init, n_init, m_init)):
        _dev(C_init, "C_init", torch.float32, (B, NH, DV, DQK))
        _dev(n_init, "n_init", torch.float32, (B, NH, DQK))
        _dev(m_init, "m_init", torch.float32, (B, NH))
    h, C_last, n_last, m_last = out
    if h.dtype not in _DT:
        raise TypeError("h must be float32 or bfloat16")
    _dev(h, "h", h.dtype, (B, NH, S, DV))
    _dev(C_last, "C_last", torch.float32, (B, NH, DV, DQK))
    _dev(n_last, "n_last", torch.float32, (B, NH, DQK))
    _dev(m_last, "m_last", torch.float32, (B, NH))
    code = _lib.mlstm_fwd_chunkwise_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(igate_pre), _ptr(fgate_pre), B, NH, S, DQK, DV, chunk,
        _dt_code(dt, forget), _ptr(C_init), _ptr(n_init), _ptr(m_init), _ptr(h), _DT[h.dtype],
        _ptr(C_last), _ptr(n_last), _ptr(m_last), _stream(stream))
    _check(code, "mlstm_fwd_chunkwise_noalloc")
    return h, C_last, n_last, m_last


def mlstm_fwd_check_noalloc(stream=None):
    """Synchronises the stream and raises MlstmError (MLSTM_ERR_TIMEOUT) if a bounded
    device-side wait of the last forward without allocation on this device gave up."""
    _check(_lib.mlstm_fwd_check_noalloc(_stream(stream)), "mlstm_fwd_check_noalloc")


def mlstm_noalloc_scratch():
    """(device address, bytes) of the library's fixed scratch array on the current device."""
    ptr, n = ctypes.c_void_p(), _sz()
    _check(_lib.mlstm_noalloc_scratch(ctypes.byref(ptr), ctypes.byref(n)), "mlstm_noalloc_scratch")
    return int(ptr.value), int(n.value)


def mlstm_kernel_launches() -> int:
    """Kernels launched by the library in this process so far."""
    return int(_lib.mlstm_kernel_launches())


def mlstm_fwd_from_gates(q, k, v, chunk, workspace, out, C_init=None, n_init=None, stream=None):
    """Second stage of the forward on a workspace prepared by :func:`mlstm_fwd_gates` (same
    sizes, chunk and m_init).  ``out`` = (h, C_last, n_last, m_last), written in place."""
    B, NH, S, DQK = q.shape
    DV = v.shape[-1]
    dt = q.dtype
    h, C_last, n_last, m_last = out
    _dev(q, "q", dt)
    _dev(k, "k", dt, (B, NH, S, DQK))
    _dev(v, "v", dt, (B, NH, S, DV))
    _dev(h, "h", None, (B, NH, S, DV))
    _dev(C_last, "C_last", torch.float32, (B, NH, DV, DQK))
    _dev(n_last, "n_last", torch.float32, (B, NH, DQK))
    _dev(m_last, "m_last", torch.float32, (B, NH))
    code = _lib.mlstm_fwd_from_gates(
        _ptr(q), _ptr(k), _ptr(v), B, NH, S, DQK, DV, chunk, _DT[dt], _ptr(C_init), _ptr(n_init),
        _ptr(h), _DT[h.dtype], _ptr(C_last), _ptr(n_last), _ptr(m_last), _ptr(workspace),
        workspace.numel(), _stream(stream))
    _check(code, "mlstm_fwd_from_gates")
    return out


def mlstm_fwd_chunk_states(k, v, igate_pre, fgate_pre, chunk, C_init=None, n_init=None,
                           m_init=None, workspace=None, stream=None, forget="sigmoid"):
    """Boundary states after every chunk: (C_states [B,NH,NC+1,DV,DQK], n_states
    [B,NH,NC+1,DQK], m_states [B,NH,NC+1])."""
    B, NH, S, DQK = k.shape
    DV = v.shape[-1]
    dt = k.dtype
    _dev(k, "k", dt)
    _dev(v, "v", dt, (B, NH, S, DV))
    _dev(igate_pre, "igate_pre", torch.float32, (B, NH, S))
    _dev(fgate_pre, "fgate_pre", torch.float32, (B, NH, S))
    NC = S // chunk
    Cs = torch.empty((B, NH, NC + 1, DV, DQK), dtype=torch.float32, device=k.device)
    ns = torch.empty((B, NH, NC + 1, DQK), dtype=torch.float32, device=k.device)
    ms = torch.empty((B, NH, NC + 1), dtype=torch.float32, device=k.device)
    if workspace is None:
        workspace = alloc_workspace(B, NH, S, DQK, DV, chunk, dt, k.device)
    code = _lib.mlstm_fwd_chunk_states(
        _ptr(k), _ptr(v), _ptr(igate_pre), _ptr(fgate_pre), B, NH, S, DQK, DV, chunk,
        _dt_code(dt, forget), _ptr(C_init), _ptr(n_init), _ptr(m_init), _ptr(Cs), _ptr(ns), _ptr(ms),
        _ptr(workspace),
        workspace.numel(), _stream(stream))
    _check(code, "mlstm_fwd_chunk_states")
    return Cs, ns, ms


def mlstm_fwd_gates(igate_pre, fgate_pre, chunk, m_init=None, workspace=None, stream=None,
                    outputs=True):
    """Gate preprocessing into ``workspace``; returns the stabiliser per token and per chunk
    boundary (m_tok [B,NH,S], m_states [B,NH,NC+1]), or (None, None) if ``outputs`` is False."""
    B, NH, S = igate_pre.shape
    _dev(igate_pre, "igate_pre", torch.float32)
    _dev(fgate_pre, "fgate_pre", torch.float32, (B, NH, S))
    NC = S // chunk
    m_tok = m_states = None
    if outputs:
        m_tok = torch.empty((B, NH, S), dtype=torch.float32, device=igate_pre.device)
        m_states = torch.empty((B, NH, NC + 1), dtype=torch.float32, device=igate_pre.device)
    if workspace is None:
        workspace = alloc_workspace(B, NH, S, 32, 32, chunk, torch.float32, igate_pre.device)
    code = _lib.mlstm_fwd_gates(_ptr(igate_pre), _ptr(fgate_pre), B, NH, S, chunk, _ptr(m_init),
                                _ptr(m_tok), _ptr(m_states), _ptr(workspace), workspace.numel(),
                                _stream(stream))
    _check(code, "mlstm_fwd_gates")
    return m_tok, m_states


def mlstm_fwd_check(workspace, B, NH, S, DQK, DV, chunk, dtype=torch.bfloat16, stream=None):
    """Synchronise and raise MlstmError if the last forward on ``workspace`` reported a
    device-side wait that gave up."""
    code = _lib.mlstm_fwd_check(_ptr(workspace), workspace.numel(), B, NH, S, DQK, DV, chunk,
                                _DT[dtype], _stream(stream))
    _check(code, "mlstm_fwd_check")


def mlstm_step(q, k, v, ig, fg, C, n, m, h=None, h_dtype=None, stream=None, forget="sigmoid"):
    """One decode step, in place on (C, n, m).  q, k [B,NH,DQK], v [B,NH,DV]; returns h."""
    B, NH, DQK = q.shape
    DV = v.shape[-1]
    dt = q.dtype
    _dev(q, "q", dt)
    _dev(k, "k", dt, (B, NH, DQK))
    _dev(v, "v", dt, (B, NH, DV))
    _dev(ig, "ig", torch.float32, (B, NH))
    _dev(fg, "fg", torch.float32, (B, NH))
    _dev(C, "C", torch.float32, (B, NH, DV, DQK))
    _dev(n, "n", torch.float32, (B, NH, DQK))
    _dev(m, "m", torch.float32, (B, NH))
    h_dtype = h_dtype or (h.dtype if h is not None else dt)
    if h is None:
        h = torch.empty((B, NH, DV), dtype=h_dtype, device=q.device)
    _dev(h, "h", h_dtype, (B, NH, DV))
    code = _lib.mlstm_step(_ptr(q), _ptr(k), _ptr(v), _ptr(ig), _ptr(fg), _ptr(C), _ptr(n),
                           _ptr(m), _ptr(h), B, NH, DQK, DV, _dt_code(dt, forget), _DT[h_dtype],
                           _stream(stream))
    _check(code, "mlstm_step")
    return h


def mlstm_groupnorm_gate(h, o_pre, gamma, beta, eps=1e-5, out=None, y_dtype=None, stream=None):
    """The block step after the cell: per-head group normalisation of h [B,NH,S,DV] and the
    output gate, y = sigmoid(o_pre) * (gamma * (h - mean) / sqrt(var + eps) + beta), with
    gamma, beta [NH, DV] float32.  ``out`` may be h itself (same dtype) for an in-place pass."""
    B, NH, S, DV = h.shape
    if h.dtype not in _DT or o_pre.dtype not in _DT:
        raise TypeError("h and o_pre must be float32 or bfloat16")
    _dev(h, "h", h.dtype)
    _dev(o_pre, "o_pre", o_pre.dtype, (B, NH, S, DV))
    _dev(gamma, "gamma", torch.float32, (NH, DV))
    _dev(beta, "beta", torch.float32, (NH, DV))
    if out is None:
        out = torch.empty((B, NH, S, DV), dtype=y_dtype or h.dtype, device=h.device)
    if out.dtype not in _DT:
        raise TypeError("the output must be float32 or bfloat16")
    _dev(out, "out", out.dtype, (B, NH, S, DV))
    code = _lib.mlstm_groupnorm_gate(_ptr(h), _ptr(o_pre), _ptr(gamma), _ptr(beta), float(eps), _ptr(out),
                                     B, NH, S, DV, _DT[h.dtype], _DT[o_pre.dtype], _DT[out.dtype],
                                     _stream(stream))
    _check(code, "mlstm_groupnorm_gate")
    return out


def mlstm_wait_selftest(workspace, B, NH, S, DQK, DV, chunk, dtype=torch.bfloat16, stream=None):
    """Run one bounded device-side wait that nothing completes (about a second); it records
    SELFTEST_WAIT_CODE in ``workspace``'s error word, so that mlstm_fwd_check on the same
    workspace raises MlstmError with code 7 (MLSTM_ERR_TIMEOUT)."""
    code = _lib.mlstm_wait_selftest(_ptr(workspace), workspace.numel(), B, NH, S, DQK, DV, chunk, _DT[dtype],
                                    _stream(stream))
    _check(code, "mlstm_wait_selftest")

