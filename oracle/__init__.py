"""fp64 CPU oracle for the mLSTM matrix-memory cell -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The product path (the CUDA library and its Python binding) never
imports, links or calls it, and it shares no code with them: the two meet only through the
seeded input generator in ``mlstm_matrix_memory_02_b300.workloads``, which holds none of the
method's arithmetic.

The arithmetic lives in ``mlstm_oracle.c`` (plain C, fp64, one POSIX thread per
(batch, head) pair at a time).  It follows "xLSTM: How Exponential Gating and Matrix Memory
Scale Recurrent Neural Networks" (llms.blog): section 2 "The Normalizer State and Numerical
Stabilization" for the log-space max stabiliser, section 3 "Associative Matrix Cell State"
for the key scale, the C_t / n_t updates and the retrieval, and section 3 "The Parallel
Dual Form" for the quadratic form.  ``groupnorm_gate`` (numpy) is the block step after the
cell: per-head group normalisation and the output gate.  ``recurrent_backward`` (numpy) gives
the gradients of the forward, walked backwards in time.  Pins against closed forms, exact
rational arithmetic and library routines are in ``tests/test_oracle_pins.py``.

Parity pinning: every routine here is pinned (no routine is "parity unpinned").
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mlstm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_mlstm.so")
_lib = None

# -ffp-contract=off: no fused multiply-adds, so every product and sum rounds as written.
CFLAGS = ["-O2", "-fPIC", "-shared", "-pthread", "-ffp-contract=off", "-std=c11"]


def build(src: str = _SRC, out: str = _LIB_PATH, quiet: bool = True) -> str:
    """Compile the oracle with gcc into a shared library; returns its path."""
    cmd = ["gcc", *CFLAGS, "-o", out, src, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"oracle build failed: {' '.join(cmd)}\n{res.stderr}")
    if not quiet and res.stderr:
        print(res.stderr)
    return out


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    dp = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.oracle_mlstm_recurrent.restype = i
    lib.oracle_mlstm_recurrent.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, dp, dp, dp,
                                           dp, dp, dp, dp, dp, dp, dp, i, dp, dp, dp, i, i]
    lib.oracle_mlstm_unstabilised.restype = i
    lib.oracle_mlstm_unstabilised.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, dp, dp, dp, i, i]
    lib.oracle_mlstm_parallel.restype = i
    lib.oracle_mlstm_parallel.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, dp, i, i]
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the compiled oracle (building it first if the library is missing or stale)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        if (not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            build()
        _lib = _declare(ctypes.CDLL(_LIB_PATH))
    return _lib


def _f64(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shapes(q, k, v, ig, fg):
    if q.ndim != 4 or k.shape != q.shape or v.ndim != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("q,k must be [B,NH,S,DQK] and v [B,NH,S,DV]")
    if ig.shape != q.shape[:3] or fg.shape != q.shape[:3]:
        raise ValueError("gate pre-activations must be [B,NH,S]")
    B, NH, S, DQK = q.shape
    return B, NH, S, DQK, v.shape[3]


FORGET_GATES = ("sigmoid", "exp")


def _forget(forget):
    if forget not in FORGET_GATES:
        raise ValueError(f"forget gate must be one of {FORGET_GATES}")
    return int(forget == "exp")


def recurrent(q, k, v, ig, fg, C0=None, n0=None, m0=None, snap_every=0, want_h=True,
              want_m_tok=False, want_den=False, nthreads=0, lib=None, forget="sigmoid"):
    """Stabilised step-by-step mLSTM in fp64.

    ``forget`` selects the forget gate: "sigmoid" (f = sigmoid(f~), log f = log sigmoid(f~))
    or "exp" (f = exp(f~), log f = f~).

    Returns a dict with ``h`` [B,NH,S,DV] (unless want_h is False), the final state ``C``
    [B,NH,DV,DQK], ``n`` [B,NH,DQK], ``m`` [B,NH]; ``m_tok`` [B,NH,S] if asked; and, when
    ``snap_every`` > 0, ``C_snap``/``n_snap``/``m_snap`` holding the state at
    t = 0, snap_every, ..., S (the state entering each chunk, then the final one).
    ``want_den`` adds ``den_tok`` (n_t.q_t) and ``dabs_tok`` (sum_c |q_c| nabs_c) [B,NH,S].
    """
    lib = lib or load()
    q, k, v, ig, fg = (_f64(x) for x in (q, k, v, ig, fg))
    B, NH, S, DQK, DV = _shapes(q, k, v, ig, fg)
    C0 = None if C0 is None else _f64(C0).reshape(B, NH, DV, DQK)
    n0 = None if n0 is None else _f64(n0).reshape(B, NH, DQK)
    m0 = None if m0 is None else _f64(m0).reshape(B, NH)
    out = {
        "C": np.empty((B, NH, DV, DQK)),
        "n": np.empty((B, NH, DQK)),
        "m": np.empty((B, NH)),
    }
    if want_h:
        out["h"] = np.empty((B, NH, S, DV))
    if want_m_tok:
        out["m_tok"] = np.empty((B, NH, S))
    if want_den:
        out["den_tok"] = np.empty((B, NH, S))
        out["dabs_tok"] = np.empty((B, NH, S))
    if snap_every > 0:
        if S % snap_every:
            raise ValueError("snap_every must divide S")
        ns = S // snap_every + 1
        out["C_snap"] = np.empty((B, NH, ns, DV, DQK))
        out["n_snap"] = np.empty((B, NH, ns, DQK))
        out["m_snap"] = np.empty((B, NH, ns))
    rc = lib.oracle_mlstm_recurrent(
        _ptr(q), _ptr(k), _ptr(v), _ptr(ig), _ptr(fg), B, NH, S, DQK, DV,
        _ptr(C0), _ptr(n0), _ptr(m0), _ptr(out.get("h")), _ptr(out["C"]), _ptr(out["n"]),
        _ptr(out["m"]), _ptr(out.get("m_tok")), _ptr(out.get("den_tok")),
        _ptr(out.get("dabs_tok")), int(snap_every), _ptr(out.get("C_snap")),
        _ptr(out.get("n_snap")), _ptr(out.get("m_snap")), int(nthreads), _forget(forget))
    if rc != 0:
        raise ValueError(f"oracle_mlstm_recurrent rejected its arguments (code {rc})")
    return out


def unstabilised(q, k, v, ig, fg, nthreads=0, lib=None, forget="sigmoid"):
    """Unstabilised recurrent mLSTM (f = sigmoid or exp, i = exp, floor 1) in fp64."""
    lib = lib or load()
    q, k, v, ig, fg = (_f64(x) for x in (q, k, v, ig, fg))
    B, NH, S, DQK, DV = _shapes(q, k, v, ig, fg)
    out = {"h": np.empty((B, NH, S, DV)), "C": np.empty((B, NH, DV, DQK)),
           "n": np.empty((B, NH, DQK))}
    rc = lib.oracle_mlstm_unstabilised(_ptr(q), _ptr(k), _ptr(v), _ptr(ig), _ptr(fg), B, NH, S,
                                       DQK, DV, _ptr(out["h"]), _ptr(out["C"]), _ptr(out["n"]),
                                       int(nthreads), _forget(forget))
    if rc != 0:
        raise ValueError(f"oracle_mlstm_unstabilised rejected its arguments (code {rc})")
    return out


def parallel(q, k, v, ig, fg, nthreads=0, lib=None, forget="sigmoid"):
    """Fully parallel quadratic (dual) form from the zero state, fp64, O(S^2) per head."""
    lib = lib or load()
    q, k, v, ig, fg = (_f64(x) for x in (q, k, v, ig, fg))
    B, NH, S, DQK, DV = _shapes(q, k, v, ig, fg)
    h = np.empty((B, NH, S, DV))
    rc = lib.oracle_mlstm_parallel(_ptr(q), _ptr(k), _ptr(v), _ptr(ig), _ptr(fg), B, NH, S, DQK,
                                   DV, _ptr(h), int(nthreads), _forget(forget))
    if rc != 0:
        raise ValueError(f"oracle_mlstm_parallel rejected its arguments (code {rc})")
    return h


def groupnorm_gate(h, o_pre, gamma, beta, eps=1e-5):
    """The block's step after the cell (page section 4 "xLSTM Block Architecture and Residual
    Stacking", the mLSTM block's item 5 "Group Normalization and Output Gating"; section 3
    "Associative Matrix Cell State": h_t = o_t (.) h~_t), in fp64 with numpy.

    h, o_pre: [B, NH, S, DV] (the cell output h~ and the output-gate pre-activation);
    gamma, beta: [NH, DV].  Each head is one group: for every (b, head, t),
        mu = mean_c h~_c,  var = mean_c (h~_c - mu)^2,
        y_c = sigmoid(o~_c) * (gamma_c (h~_c - mu) / sqrt(var + eps) + beta_c).
    Readings: the output gate is the LSTM sigmoid gate o = sigmoid(o~); the normalisation is
    applied before the gate; the variance is the biased one (divide by DV)."""
    h = np.asarray(h, np.float64)
    o = np.asarray(o_pre, np.float64)
    g = np.asarray(gamma, np.float64)[None, :, None, :]
    b = np.asarray(beta, np.float64)[None, :, None, :]
    mu = h.mean(axis=-1, keepdims=True)
    var = ((h - mu) ** 2).mean(axis=-1, keepdims=True)
    norm = (h - mu) / np.sqrt(var + eps)
    gate = 1.0 / (1.0 + np.exp(-o))
    return gate * (g * norm + b)


def _log_forget_np(fg, forget):
    return fg if forget == "exp" else -np.logaddexp(0.0, -fg)


def recurrent_backward(q, k, v, ig, fg, dh, C0=None, n0=None, m0=None, forget="sigmoid"):
    """Gradients of L = sum_t dh_t . h_t through the stabilised recurrent cell, fp64, numpy.

    The cell's h_t = C_t q_t / max(|n_t^T q_t|, exp(-m_t)) equals the unstabilised
    C~_t q_t / max(|n~_t^T q_t|, 1) (page section 2: the stabiliser rescales C and n by
    exp(-m_t)), so its gradients are those of the unstabilised recurrence of section 3
    (C~_t = f_t C~_{t-1} + i_t v_t k^_t^T, n~_t = f_t n~_{t-1} + i_t k^_t), walked backwards
    in time.  They are carried here in the stabilised frame: G_t = dL/dC~_t * exp(m_t) and
    N_t = dL/dn~_t * exp(m_t), so that every factor is the forward's alpha_t or w_t:
        G_t += dh_t q_t^T / D_t,  N_t += -(dh_t . h_t) / D_t * s_t q_t,
        (D_t = max(|n_t^T q_t|, exp(-m_t)), s_t = sign(n_t^T q_t) where |n_t^T q_t| > exp(-m_t),
         else 0: the floor does not depend on q or n)
        dq_t = C_t^T dh_t / D_t - (dh_t . h_t) / D_t * s_t n_t
        dv_t = w_t G_t k^_t,   dk_t = w_t (G_t^T v_t + N_t) / sqrt(d),
        di~_t = w_t (v_t^T G_t k^_t + N_t . k^_t),
        df~_t = alpha_t (<G_t, C_{t-1}> + N_t . n_{t-1}) * (1 - f_t)   (sigmoid gate; f = exp: * 1)
        G_{t-1} += alpha_t G_t,  N_{t-1} += alpha_t N_t.
    With an initial state (C0, n0, m0) (stabilised), also dC0 = G_0, dn0 = N_0 and
    dm0 = <G_0, C0> + N_0 . n0.  Returns a dict of those arrays.  Where |n_t^T q_t| equals
    exp(-m_t) exactly the function has a kink and this is one of its one-sided derivatives."""
    q, k, v, ig, fg, dh = (np.asarray(x, np.float64) for x in (q, k, v, ig, fg, dh))
    B, NH, S, DQK, DV = _shapes(q, k, v, ig, fg)
    scale = 1.0 / np.sqrt(DQK)
    out = {x: np.zeros_like(y) for x, y in (("dq", q), ("dk", k), ("dv", v), ("dig", ig), ("dfg", fg))}
    init = C0 is not None
    if init:
        C0 = np.asarray(C0, np.float64).reshape(B, NH, DV, DQK)
        n0 = np.asarray(n0, np.float64).reshape(B, NH, DQK)
        m0 = np.asarray(m0, np.float64).reshape(B, NH)
        out["dC0"] = np.zeros_like(C0)
        out["dn0"] = np.zeros_like(n0)
        out["dm0"] = np.zeros_like(m0)
    for b in range(B):
        for hh in range(NH):
            # forward, keeping every state and the per-token factors
            C = C0[b, hh].copy() if init else np.zeros((DV, DQK))
            n = n0[b, hh].copy() if init else np.zeros(DQK)
            m = float(m0[b, hh]) if init else 0.0
            Cs, ns, al, ws, fs, ms = [C.copy()], [n.copy()], [], [], [], []
            for t in range(S):
                lf = _log_forget_np(fg[b, hh, t], forget)
                m_new = max(lf + m, ig[b, hh, t])
                a_t = np.exp(lf + m - m_new)
                w_t = np.exp(ig[b, hh, t] - m_new)
                kh = k[b, hh, t] * scale
                C = a_t * C + w_t * np.outer(v[b, hh, t], kh)
                n = a_t * n + w_t * kh
                m = m_new
                Cs.append(C.copy()); ns.append(n.copy())
                al.append(a_t); ws.append(w_t); fs.append(np.exp(lf)); ms.append(m)
            G = np.zeros((DV, DQK))
            N = np.zeros(DQK)
            for t in range(S - 1, -1, -1):
                Ct, nt, qt = Cs[t + 1], ns[t + 1], q[b, hh, t]
                a = float(nt @ qt)
                floor_ = np.exp(-ms[t])
                D = max(abs(a), floor_)
                h = Ct @ qt / D
                g_h = dh[b, hh, t]
                s_t = np.sign(a) if abs(a) > floor_ else 0.0
                dD_scaled = -float(g_h @ h) / D
                out["dq"][b, hh, t] = Ct.T @ g_h / D + dD_scaled * s_t * nt
                G += np.outer(g_h, qt) / D
                N += dD_scaled * s_t * qt
                kh = k[b, hh, t] * scale
                vt = v[b, hh, t]
                out["dv"][b, hh, t] = ws[t] * (G @ kh)
                out["dk"][b, hh, t] = ws[t] * (G.T @ vt + N) * scale
                out["dig"][b, hh, t] = ws[t] * (float(vt @ G @ kh) + float(N @ kh))
                gate = (1.0 - fs[t]) if forget != "exp" else 1.0
                out["dfg"][b, hh, t] = al[t] * (float(np.sum(G * Cs[t])) + float(N @ ns[t])) * gate
                G = al[t] * G
                N = al[t] * N
            if init:
                out["dC0"][b, hh] = G
                out["dn0"][b, hh] = N
                out["dm0"][b, hh] = float(np.sum(G * C0[b, hh])) + float(N @ n0[b, hh])
    return out
