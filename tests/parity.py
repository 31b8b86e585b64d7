"""Comparison helpers and tolerances for GPU-vs-oracle parity.

Tolerances (max-abs error relative to the oracle output's RMS):
  * fp32 q/k/v, fp32 h:              1e-4
  * bf16 q/k/v, fp32 h:              2e-2
  * bf16 h output:                   2e-2 * RMS + 2^-8 * |h_oracle|  (the output's own rounding:
                                     bf16 keeps 8 significant bits)
  * states C, n (rescaled to the oracle's stabiliser): same tolerance as h for the input dtype
  * stabiliser m:                    |dm| <= 1e-4 * (1 + |m|)
On rows whose denominator n_t^T q_t cancels (the long-context stress workload), the error of
any fixed-precision evaluation grows with the denominator's condition number
kappa_t = sum_c |q_c| nabs_c / max(|n_t^T q_t|, e^{-m_t}); those rows are held to
    |dh| <= tol * RMS + kappa_t * (u_num * max|v| + u_den * |h_oracle|),
the first-order bound for a numerator and a denominator computed with relative errors u_num,
u_den per summed term.
"""
from __future__ import annotations

import numpy as np

TOL_F32 = 1e-4
TOL_BF16 = 2e-2
BF16_OUT_REL = 2.0 ** -8
M_TOL = 1e-4


def rms(x):
    x = np.asarray(x, np.float64)
    return float(np.sqrt(np.mean(x * x))) if x.size else 0.0


def rel_err(x, ref):
    """max |x - ref| / RMS(ref)."""
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    r = rms(ref)
    return float(np.max(np.abs(x - ref)) / (r if r > 0 else 1.0))


def state_errs(C, n, m, ora_C, ora_n, ora_m):
    """Errors of a GPU state against the oracle's, after rescaling the GPU state to the
    oracle's stabiliser (both are stored relative to their own m)."""
    C = np.asarray(C, np.float64)
    n = np.asarray(n, np.float64)
    m = np.asarray(m, np.float64)
    s = np.exp(m - ora_m)
    eC = rel_err(C * s[..., None, None], ora_C)
    en = rel_err(n * s[..., None], ora_n)
    em = float(np.max(np.abs(m - ora_m) / (1.0 + np.abs(ora_m)))) if m.size else 0.0
    return eC, en, em


def bf16_out_ok(h, ora_h, tol=TOL_BF16):
    """Elementwise bound for a bf16 h output (see module docstring); returns (ok, worst)."""
    h = np.asarray(h, np.float64)
    ora_h = np.asarray(ora_h, np.float64)
    bound = tol * rms(ora_h) + BF16_OUT_REL * np.abs(ora_h)
    excess = np.abs(h - ora_h) / bound
    return bool(np.all(excess <= 1.0)), float(np.max(excess))


def conditioned_ok(h, ora, v, tol, u_num, u_den):
    """Row-wise conditioned bound for workloads with cancelling denominators.

    ``ora`` must hold h, m_tok, den_tok and dabs_tok.  Returns (ok, worst_excess, stats)."""
    h = np.asarray(h, np.float64)
    oh = ora["h"]
    den_eff = np.maximum(np.abs(ora["den_tok"]), np.exp(-ora["m_tok"]))
    kappa = ora["dabs_tok"] / den_eff
    vmax = float(np.max(np.abs(v)))
    bound = tol * rms(oh) + kappa[..., None] * (u_num * vmax + u_den * np.abs(oh))
    excess = np.abs(h - oh) / bound
    stats = {
        "kappa_max": float(np.max(kappa)),
        "rows_kappa_gt_1e3": int(np.sum(kappa > 1e3)),
        "rel_err_all_rows": rel_err(h, oh),
        "rel_err_kappa_le_100": rel_err(h[kappa <= 100], oh[kappa <= 100]),
    }
    return bool(np.all(excess <= 1.0)), float(np.max(excess)), stats


def u_fp32(dqk, chunk):
    """Relative error per summed term of an fp32 evaluation of nᵀq or C q: the sums run over
    d_qk products (the inter-chunk part) and L (the intra-chunk part), each rounding at 2^-24."""
    return (dqk + chunk) * 2.0 ** -24


def u_tc(dqk):
    """The fused tensor-core kernel's allowance: twice that of fp32 sums at its chunk of 64.
    Its operands are rounded to fp16 but its sums run in fp32; on the long-context stress
    workload its worst error per condition-number bin (kappa > 100) is measured to stay within
    twice the fp32 CUDA-core path's on the same values
    (test_stress_tensor_core_vs_fp32_path_per_kappa_bin), which is what this factor rests on."""
    return 2.0 * u_fp32(dqk, 64)


KAPPA_BINS = ((0.0, 1e2), (1e2, 1e3), (1e3, 1e4), (1e4, np.inf))


def kappa_bin_errors(h, ora, bins=KAPPA_BINS):
    """max |h - h_oracle| / RMS(h_oracle) over the rows whose condition number kappa_t (module
    docstring) lies in each (lo, hi] bin; returns [(rows, error or None)] per bin."""
    h = np.asarray(h, np.float64)
    oh = ora["h"]
    kappa = ora["dabs_tok"] / np.maximum(np.abs(ora["den_tok"]), np.exp(-ora["m_tok"]))
    err = np.max(np.abs(h - oh), axis=-1) / rms(oh)
    out = []
    for lo, hi in bins:
        sel = (kappa > lo) & (kappa <= hi)
        out.append((int(sel.sum()), float(err[sel].max()) if sel.any() else None))
    return out

