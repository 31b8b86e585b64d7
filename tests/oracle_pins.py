"""Pins for the fp64 oracle: properties fixed by the mathematics of the mLSTM cell, each
computed by a route other than the oracle's own loop.

Page: "xLSTM: How Exponential Gating and Matrix Memory Scale Recurrent Neural Networks"
(llms.blog).  Section 2 "The Normalizer State and Numerical Stabilization" (max
stabiliser), section 3 "Associative Matrix Cell State" (updates, retrieval, key scale) and
"The Parallel Dual Form" (unrolled sum, causal decay matrix).

Each pin takes the loaded oracle library so that the mutation test can run the same pins
against deliberately broken copies of the oracle.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

import oracle
from golden.exact_case import exact_rational_case

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rand_inputs(B, NH, S, DQK, DV, seed, ig=(0.0, 1.0), fg=(1.0, 1.5)):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, NH, S, DQK))
    k = rng.standard_normal((B, NH, S, DQK))
    v = rng.standard_normal((B, NH, S, DV))
    igp = ig[0] + ig[1] * rng.standard_normal((B, NH, S))
    fgp = fg[0] + fg[1] * rng.standard_normal((B, NH, S))
    return q, k, v, igp, fgp


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def log_sigmoid_np(x):
    # library route: log sigma(x) = -log(1 + e^{-x}) via numpy's logaddexp
    return -np.logaddexp(0.0, -np.asarray(x, np.float64))


# ---------------------------------------------------------------- the pins
def pin_recurrent_equals_parallel(lib):
    """Recurrent form == the parallel dual form H = ((Q K^T) o S) V, row-normalised
    (section 3 "The Parallel Dual Form"); DQK != DV so a transposed operand shows."""
    worst = 0.0
    for seed, fg in ((1, (1.0, 1.5)), (2, (-1.0, 2.0)), (3, (4.0, 0.5))):
        q, k, v, ig, fgp = rand_inputs(2, 2, 20, 6, 5, seed, fg=fg)
        h_rec = oracle.recurrent(q, k, v, ig, fgp, lib=lib)["h"]
        h_par = oracle.parallel(q, k, v, ig, fgp, lib=lib)
        worst = max(worst, rel(h_rec, h_par))
    return worst <= 1e-11, f"recurrent vs parallel rel err {worst:.3e}"


def pin_stabiliser_is_a_rescaling(lib):
    """The max stabiliser rescales C and n by exp(-m_t) and leaves h unchanged
    (section 2): stabilised h == unstabilised h, C_stab e^m == C_unstab, n likewise."""
    worst = 0.0
    for seed in (4, 5):
        q, k, v, ig, fg = rand_inputs(2, 3, 40, 7, 4, seed, ig=(0.0, 1.5), fg=(0.5, 2.0))
        st = oracle.recurrent(q, k, v, ig, fg, lib=lib)
        un = oracle.unstabilised(q, k, v, ig, fg, lib=lib)
        e = np.exp(st["m"])
        worst = max(worst, rel(st["h"], un["h"]), rel(st["C"] * e[..., None, None], un["C"]),
                    rel(st["n"] * e[..., None], un["n"]))
    return worst <= 1e-11, f"stabilised vs unstabilised rel err {worst:.3e}"


def pin_single_token_closed_form(lib):
    """From the zero state (m_0 = 0) one token gives m_1 = max(log sigma(f~), i~),
    C_1 = e^{i~ - m_1} v k^T/sqrt(d), n_1 = e^{i~ - m_1} k/sqrt(d) and
    h_1 = e^{i~} (k.q/sqrt(d)) v / max(e^{i~} |k.q/sqrt(d)|, 1)."""
    rng = np.random.default_rng(6)
    worst = 0.0
    both_branches = set()
    for trial in range(12):
        d, dv = 8, 3
        q = rng.standard_normal((1, 1, 1, d))
        k = rng.standard_normal((1, 1, 1, d))
        v = rng.standard_normal((1, 1, 1, dv))
        ig = np.array([[[rng.uniform(-4, 4)]]])
        fg = np.array([[[rng.uniform(-4, 4)]]])
        out = oracle.recurrent(q, k, v, ig, fg, lib=lib)
        s = float(k[0, 0, 0] @ q[0, 0, 0]) / np.sqrt(d)
        i = float(np.exp(ig[0, 0, 0]))
        den = max(i * abs(s), 1.0)
        both_branches.add(i * abs(s) >= 1.0)
        h = i * s * v[0, 0, 0] / den
        m1 = max(float(log_sigmoid_np(fg[0, 0, 0])), float(ig[0, 0, 0]))
        w = np.exp(float(ig[0, 0, 0]) - m1)
        C1 = w * np.outer(v[0, 0, 0], k[0, 0, 0] / np.sqrt(d))
        n1 = w * k[0, 0, 0] / np.sqrt(d)
        worst = max(worst, rel(out["h"][0, 0, 0], h), rel(out["C"][0, 0], C1),
                    rel(out["n"][0, 0], n1), abs(float(out["m"][0, 0]) - m1))
    ok = worst <= 1e-12 and both_branches == {True, False}
    return ok, f"single-token closed form err {worst:.3e}, branches {sorted(both_branches)}"


def pin_linear_attention_limit(lib):
    """f~ -> +inf (f = 1) with i~ = 0 reduces the cell to causal linear attention
    (section 3, last paragraph): h_t = sum_{j<=t} (q_t.k_j) v_j / max(|sum_{j<=t} q_t.k_j|, 1),
    evaluated with a masked matrix product."""
    q, k, v, _, _ = rand_inputs(1, 2, 32, 6, 5, 7)
    ig = np.zeros(q.shape[:3])
    fg = np.full(q.shape[:3], 60.0)  # log sigma(60) = -8.8e-27: the decay is 1 to fp64
    h = oracle.recurrent(q, k, v, ig, fg, lib=lib)["h"]
    kh = k / np.sqrt(q.shape[-1])
    A = np.tril(np.einsum("bhtc,bhjc->bhtj", q, kh))
    num = np.einsum("bhtj,bhja->bhta", A, v)
    den = np.maximum(np.abs(A.sum(-1)), 1.0)
    err = rel(h, num / den[..., None])
    return err <= 1e-12, f"linear-attention limit rel err {err:.3e}"


def pin_stabiliser_max_plus_form(lib):
    """Unrolling m_t = max(log f_t + m_{t-1}, i~_t) gives
    m_t = F_t + max(m_0, max_{j<=t}(i~_j - F_j)) with F_t = sum_{tau<=t} log f_tau;
    checked with cumulative sums and running maxima, also from a nonzero m_0."""
    q, k, v, ig, fg = rand_inputs(2, 2, 50, 4, 4, 8, ig=(0.0, 3.0), fg=(0.0, 2.0))
    m0 = np.array([[0.0, 2.5], [-1.0, 7.0]])
    C0 = np.zeros((2, 2, 4, 4))
    n0 = np.zeros((2, 2, 4))
    out = oracle.recurrent(q, k, v, ig, fg, C0=C0, n0=n0, m0=m0, want_m_tok=True, lib=lib)
    F = np.cumsum(log_sigmoid_np(fg), axis=-1)
    run = np.maximum.accumulate(ig - F, axis=-1)
    m_ref = F + np.maximum(m0[..., None], run)
    err = float(np.max(np.abs(out["m_tok"] - m_ref) / (1 + np.abs(m_ref))))
    err = max(err, float(np.max(np.abs(out["m"] - m_ref[..., -1]))))
    return err <= 1e-12, f"max-plus stabiliser err {err:.3e}"


def pin_exact_rational(lib):
    """Exact rational evaluation of the unrolled sum (section 3) on integer inputs;
    the stabiliser stays at m = 0 here, so the stabilised oracle is compared as is."""
    (q, k, v, ig, fg), h, C, n = exact_rational_case()
    out = oracle.recurrent(q, k, v, ig, fg, lib=lib)
    hx = np.array([[float(x) for x in row] for row in h])
    Cx = np.array([[float(x) for x in row] for row in C])
    nx = np.array([float(x) for x in n])
    err = max(rel(out["h"][0, 0], hx), rel(out["C"][0, 0], Cx), rel(out["n"][0, 0], nx),
              abs(float(out["m"][0, 0])))
    # both sides of max(|n.q|, 1) and both signs of n.q must occur in this case
    nq_vals = []
    for t in range(q.shape[2]):
        kk = k[0, 0, : t + 1] / 2.0
        w = 2.0 ** -(t - np.arange(t + 1))
        nq_vals.append(float((w[:, None] * kk).sum(0) @ q[0, 0, t]))
    nq_vals = np.array(nq_vals)
    covered = (np.any(np.abs(nq_vals) < 1) and np.any(np.abs(nq_vals) > 1)
               and np.any(nq_vals < -1))
    return err <= 1e-14 and covered, f"exact rational err {err:.3e}, branches covered {covered}"


def pin_golden_fixture(lib):
    """Stored exact values (tests/golden/exact_rational_case.json, written by
    tests/golden/make_golden.py from the unrolled sum in exact arithmetic)."""
    with open(os.path.join(GOLDEN, "exact_rational_case.json")) as f:
        g = json.load(f)
    q, k, v = (np.array(g[x], np.float64) for x in ("q", "k", "v"))
    ig, fg = np.array(g["ig"], np.float64), np.array(g["fg"], np.float64)
    out = oracle.recurrent(q, k, v, ig, fg, lib=lib)
    hx = np.array([[float(Fraction(x)) for x in row] for row in g["h"]])
    Cx = np.array([[float(Fraction(x)) for x in row] for row in g["C_last"]])
    err = max(rel(out["h"][0, 0], hx), rel(out["C"][0, 0], Cx))
    return err <= 1e-14, f"golden fixture err {err:.3e}"


def pin_split_sequence(lib):
    """The state (C, n, m) carries everything (section 5 "Inference Memory and Throughput
    Trade-Offs"): running S1 tokens, then S2 more from that state, equals running S1+S2."""
    q, k, v, ig, fg = rand_inputs(2, 2, 36, 5, 6, 10, ig=(0.0, 2.0), fg=(1.0, 2.0))
    full = oracle.recurrent(q, k, v, ig, fg, lib=lib)
    s1 = 13
    a = oracle.recurrent(q[:, :, :s1], k[:, :, :s1], v[:, :, :s1], ig[:, :, :s1], fg[:, :, :s1],
                         lib=lib)
    b = oracle.recurrent(q[:, :, s1:], k[:, :, s1:], v[:, :, s1:], ig[:, :, s1:], fg[:, :, s1:],
                         C0=a["C"], n0=a["n"], m0=a["m"], lib=lib)
    err = max(rel(np.concatenate([a["h"], b["h"]], axis=2), full["h"]), rel(b["C"], full["C"]),
              rel(b["n"], full["n"]), float(np.max(np.abs(b["m"] - full["m"]))))
    return err <= 1e-12, f"split-sequence err {err:.3e}"


def pin_snapshots(lib):
    """Chunk-boundary snapshots equal the final state of the prefix runs."""
    q, k, v, ig, fg = rand_inputs(1, 2, 24, 4, 3, 11)
    out = oracle.recurrent(q, k, v, ig, fg, snap_every=8, lib=lib)
    err = float(np.max(np.abs(out["C_snap"][:, :, 0]))) + float(np.max(np.abs(out["m_snap"][:, :, 0])))
    for s, t in enumerate((8, 16, 24), start=1):
        pre = oracle.recurrent(q[:, :, :t], k[:, :, :t], v[:, :, :t], ig[:, :, :t], fg[:, :, :t],
                               lib=lib)
        err = max(err, rel(out["C_snap"][:, :, s], pre["C"]), rel(out["n_snap"][:, :, s], pre["n"]),
                  float(np.max(np.abs(out["m_snap"][:, :, s] - pre["m"]))))
    return err <= 1e-13, f"snapshot err {err:.3e}"


def pin_causality_and_linearity(lib):
    """Causal decay matrix: S_ij = 0 for i < j (token t' cannot change h_t, t < t');
    H = ((Q K^T) o S) V is linear in V."""
    q, k, v, ig, fg = rand_inputs(1, 2, 30, 4, 4, 12)
    base = oracle.recurrent(q, k, v, ig, fg, lib=lib)
    tp = 17
    q2, k2, v2, ig2, fg2 = (x.copy() for x in (q, k, v, ig, fg))
    q2[:, :, tp] += 1.0; k2[:, :, tp] -= 2.0; v2[:, :, tp] *= 3.0; ig2[:, :, tp] += 5.0; fg2[:, :, tp] -= 1.0
    pert = oracle.recurrent(q2, k2, v2, ig2, fg2, lib=lib)
    causal = np.array_equal(base["h"][:, :, :tp], pert["h"][:, :, :tp])
    changed = not np.allclose(base["h"][:, :, tp:], pert["h"][:, :, tp:])
    scaled = oracle.recurrent(q, k, 2.5 * v, ig, fg, lib=lib)
    lin = max(rel(scaled["h"], 2.5 * base["h"]), rel(scaled["C"], 2.5 * base["C"]))
    ok = causal and changed and lin <= 1e-14
    return ok, f"causal {causal}, later rows changed {changed}, linearity err {lin:.3e}"


def pin_denominator_brute_force(lib):
    """n_t.q_t and its absolute-term sum, brute force from the unrolled sum (section 3):
    n_t q_t = e^{-m_t} sum_{j<=t} (prod_{tau=j+1..t} f_tau) i_j (q_t . k_j) and the same
    with |q_t| . |k_j|; m_t from the pinned stabiliser output."""
    q, k, v, ig, fg = rand_inputs(1, 2, 18, 5, 3, 13, ig=(0.0, 1.5), fg=(0.5, 1.5))
    out = oracle.recurrent(q, k, v, ig, fg, want_m_tok=True, want_den=True, lib=lib)
    kh = k / np.sqrt(q.shape[-1])
    f = 1.0 / (1.0 + np.exp(-fg))
    err = 0.0
    for h_ in range(2):
        for t in range(q.shape[2]):
            den = dab = 0.0
            for j in range(t + 1):
                w = np.exp(ig[0, h_, j]) * np.prod(f[0, h_, j + 1: t + 1])
                den += w * float(q[0, h_, t] @ kh[0, h_, j])
                dab += w * float(np.abs(q[0, h_, t]) @ np.abs(kh[0, h_, j]))
            e = np.exp(-out["m_tok"][0, h_, t])
            err = max(err, abs(out["den_tok"][0, h_, t] - den * e) / (dab * e),
                      abs(out["dabs_tok"][0, h_, t] - dab * e) / (dab * e))
    return err <= 1e-13, f"denominator brute force err {err:.3e}"


# ---------------------------------------------------------------- exponential forget gate
# Section 2 allows f = exp(f~) as well as sigmoid(f~); then log f = f~ and the stabiliser is
# the printed m_t = max(f~_t + m_{t-1}, i~_t).
def pin_exp_forget_is_a_rescaling(lib):
    """Exponential forget gate: stabilised h == unstabilised h (f = exp(f~), i = exp(i~),
    floor 1), C_stab e^m == C_unstab, n likewise.  f~ around -0.1 keeps the unstabilised
    products finite; i~ spread keeps the stabiliser moving."""
    worst = 0.0
    for seed in (21, 22):
        q, k, v, ig, fg = rand_inputs(2, 2, 40, 6, 5, seed, ig=(0.0, 1.5), fg=(-0.1, 0.2))
        st = oracle.recurrent(q, k, v, ig, fg, lib=lib, forget="exp")
        un = oracle.unstabilised(q, k, v, ig, fg, lib=lib, forget="exp")
        e = np.exp(st["m"])
        worst = max(worst, rel(st["h"], un["h"]), rel(st["C"] * e[..., None, None], un["C"]),
                    rel(st["n"] * e[..., None], un["n"]))
    return worst <= 1e-11, f"exp forget: stabilised vs unstabilised rel err {worst:.3e}"


def pin_exp_forget_dual_form(lib):
    """Exponential forget gate: recurrent == parallel dual form with S_tj = prod exp(f~) i_j."""
    worst = 0.0
    for seed in (23, 24):
        q, k, v, ig, fg = rand_inputs(1, 2, 18, 6, 5, seed, fg=(-0.2, 0.3))
        worst = max(worst, rel(oracle.recurrent(q, k, v, ig, fg, lib=lib, forget="exp")["h"],
                               oracle.parallel(q, k, v, ig, fg, lib=lib, forget="exp")))
    return worst <= 1e-11, f"exp forget: recurrent vs parallel rel err {worst:.3e}"


def pin_exp_forget_equals_sigmoid_in_log_space(lib):
    """The two variants differ only in log f: the exponential gate fed f~' = log sigmoid(f~)
    (computed by numpy's logaddexp) gives the sigmoid gate's outputs at f~, state included."""
    q, k, v, ig, fg = rand_inputs(2, 2, 30, 5, 4, 25, ig=(0.0, 2.0), fg=(1.0, 2.0))
    a = oracle.recurrent(q, k, v, ig, fg, lib=lib)
    b = oracle.recurrent(q, k, v, ig, log_sigmoid_np(fg), lib=lib, forget="exp")
    err = max(rel(b["h"], a["h"]), rel(b["C"], a["C"]), rel(b["n"], a["n"]),
              float(np.max(np.abs(b["m"] - a["m"]))))
    # and the variants are not the same map: the exponential gate at f~ itself differs
    c = oracle.recurrent(q, k, v, ig, fg, lib=lib, forget="exp")
    differs = rel(c["h"], a["h"]) > 1e-3
    return err <= 1e-12 and differs, f"exp(log sigmoid) vs sigmoid err {err:.3e}, distinct {differs}"


def pin_exp_forget_two_token_scalar(lib):
    """d_qk = d_v = 1, two tokens, written out by hand: C_1 = i_1 v_1 k_1, n_1 = i_1 k_1,
    C_2 = f_2 C_1 + i_2 v_2 k_2, n_2 = f_2 n_1 + i_2 k_2 with f_2 = e^{f~_2}, i_t = e^{i~_t};
    h_t = C_t q_t / max(|n_t q_t|, 1); m_1 = max(f~_1, i~_1), m_2 = max(f~_2 + m_1, i~_2).
    Cases cover both sides of the max in the denominator and in the stabiliser."""
    worst = 0.0
    cases = [((0.7, -1.3), (1.5, 0.4), (-0.8, 2.0), (0.3, -0.2), (-0.5, 0.6)),
             ((2.0, 0.5), (-1.0, 3.0), (0.9, -0.4), (1.2, -2.5), (0.1, -1.7)),
             ((-0.3, 1.1), (0.6, 0.8), (1.4, 1.9), (-1.5, 0.2), (2.2, 0.05))]
    for qq, kk, vv, ii, ff in cases:
        q = np.array(qq).reshape(1, 1, 2, 1); k = np.array(kk).reshape(1, 1, 2, 1)
        v = np.array(vv).reshape(1, 1, 2, 1)
        ig = np.array(ii).reshape(1, 1, 2); fg = np.array(ff).reshape(1, 1, 2)
        i1, i2 = np.exp(ii[0]), np.exp(ii[1])
        f2 = np.exp(ff[1])
        C1, n1 = i1 * vv[0] * kk[0], i1 * kk[0]
        C2, n2 = f2 * C1 + i2 * vv[1] * kk[1], f2 * n1 + i2 * kk[1]
        h1 = C1 * qq[0] / max(abs(n1 * qq[0]), 1.0)
        h2 = C2 * qq[1] / max(abs(n2 * qq[1]), 1.0)
        m1 = max(ff[0], ii[0]); m2 = max(ff[1] + m1, ii[1])
        out = oracle.recurrent(q, k, v, ig, fg, lib=lib, forget="exp")
        worst = max(worst, rel(out["h"].ravel(), np.array([h1, h2])),
                    abs(float(out["m"].ravel()[0]) - m2),
                    rel(out["C"].ravel() * np.exp(m2), np.array([C2])))
    return worst <= 1e-13, f"exp forget two-token closed form err {worst:.3e}"


# ---------------------------------------------------------------- group norm and output gate
def _gn_inputs(seed, B=2, NH=3, S=5, DV=40):
    rng = np.random.default_rng(seed)
    h = 2.0 * rng.standard_normal((B, NH, S, DV)) + 0.7
    o = 1.5 * rng.standard_normal((B, NH, S, DV))
    g = 1.0 + 0.3 * rng.standard_normal((NH, DV))
    b = 0.2 * rng.standard_normal((NH, DV))
    return h, o, g, b


def pin_groupnorm_matches_torch(lib):
    """The normalisation is torch's group_norm with one group per head (a library routine,
    fp64 on the CPU): per token, the NH * DV channels split into NH groups of DV."""
    import torch
    h, o, g, b = _gn_inputs(31)
    B, NH, S, DV = h.shape
    big = np.full_like(o, 60.0)  # sigmoid(60) == 1 in fp64: the gate is the identity
    y = oracle.groupnorm_gate(h, big, g, b, eps=1e-5)
    x = torch.from_numpy(np.ascontiguousarray(h.transpose(0, 2, 1, 3).reshape(B * S, NH * DV)))
    ref = torch.nn.functional.group_norm(x, NH, torch.from_numpy(g.reshape(-1)),
                                         torch.from_numpy(b.reshape(-1)), eps=1e-5)
    ref = ref.numpy().reshape(B, S, NH, DV).transpose(0, 2, 1, 3)
    err = rel(y, ref)
    return err <= 1e-13, f"group norm vs torch err {err:.3e}"


def pin_groupnorm_gate_invariants(lib):
    """gamma = 1, beta = 0, open gate: every (b, head, t) row has mean 0 and variance
    var / (var + eps); a shut-half gate (o~ = 0, sigmoid = 1/2) halves the output; a constant
    row normalises to 0, leaving sigmoid(o~) beta."""
    h, o, g, b = _gn_inputs(32)
    NH, DV = g.shape
    ones, zeros = np.ones((NH, DV)), np.zeros((NH, DV))
    y = oracle.groupnorm_gate(h, np.full_like(o, 60.0), ones, zeros, eps=1e-3)
    var = h.var(axis=-1)
    err = max(float(np.max(np.abs(y.mean(axis=-1)))),
              float(np.max(np.abs(y.var(axis=-1) - var / (var + 1e-3)))))
    half = oracle.groupnorm_gate(h, np.zeros_like(o), g, b)
    full = oracle.groupnorm_gate(h, np.full_like(o, 60.0), g, b)
    err = max(err, rel(half, 0.5 * full))
    const = oracle.groupnorm_gate(np.full_like(h, 3.25), o, g, b)
    err = max(err, rel(const, b[None, :, None, :] / (1.0 + np.exp(-o))))
    return err <= 1e-13, f"group norm / gate invariants err {err:.3e}"


# ---------------------------------------------------------------- backward
def _fd_grads(fwd_loss, arrays, eps=1e-6):
    """Central differences of a scalar function of several arrays, element by element."""
    out = []
    for i, arr in enumerate(arrays):
        g = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus = [a.copy() for a in arrays]
            minus = [a.copy() for a in arrays]
            plus[i][idx] += eps
            minus[i][idx] -= eps
            g[idx] = (fwd_loss(*plus) - fwd_loss(*minus)) / (2 * eps)
        out.append(g)
    return out


def _backward_case(lib, forget, seed, init, qscale=1.0):
    rng = np.random.default_rng(seed)
    B, NH, S, DQK, DV = 1, 2, 6, 4, 3
    q = qscale * rng.standard_normal((B, NH, S, DQK))
    k = rng.standard_normal((B, NH, S, DQK))
    v = rng.standard_normal((B, NH, S, DV))
    ig = 1.2 * rng.standard_normal((B, NH, S))
    fg = (rng.normal(1.0, 1.5, (B, NH, S)) if forget == "sigmoid" else rng.normal(-0.1, 0.3, (B, NH, S)))
    dh = rng.standard_normal((B, NH, S, DV))
    arrays = [q, k, v, ig, fg]
    if init:
        arrays += [0.4 * rng.standard_normal((B, NH, DV, DQK)), 0.4 * rng.standard_normal((B, NH, DQK)),
                   rng.uniform(-1.0, 1.5, (B, NH))]

    def loss(*a):
        kw = dict(C0=a[5], n0=a[6], m0=a[7]) if init else {}
        return float(np.sum(oracle.recurrent(*a[:5], lib=lib, forget=forget, **kw)["h"] * dh))

    fd = _fd_grads(loss, arrays)
    kw = dict(C0=arrays[5], n0=arrays[6], m0=arrays[7]) if init else {}
    g = oracle.recurrent_backward(*arrays[:5], dh, forget=forget, **kw)
    names = ["dq", "dk", "dv", "dig", "dfg"] + (["dC0", "dn0", "dm0"] if init else [])
    return max(rel(g[nm], f) for nm, f in zip(names, fd))


def pin_backward_finite_differences(lib):
    """Gradients of sum_t dh_t . h_t w.r.t. q, k, v, i~, f~ and the initial state (C0, n0, m0),
    against central differences of the C oracle's forward (a separate implementation)."""
    err = max(_backward_case(lib, "sigmoid", 51, False), _backward_case(lib, "sigmoid", 52, True))
    return err <= 1e-7, f"backward vs finite differences rel err {err:.3e}"


def pin_backward_exp_forget_finite_differences(lib):
    """The same for the exponential forget gate (df~ = alpha (<G, C_{t-1}> + N . n_{t-1}))."""
    err = max(_backward_case(lib, "exp", 53, False), _backward_case(lib, "exp", 54, True))
    return err <= 1e-7, f"exp-gate backward vs finite differences rel err {err:.3e}"


def pin_backward_floor_branch(lib):
    """Small q: the floor exp(-m_t) decides the denominator on most rows, where it carries no
    gradient to q or n; the analytic gradients still match central differences."""
    err = _backward_case(lib, "sigmoid", 55, False, qscale=0.05)
    return err <= 1e-7, f"floor-branch backward vs finite differences rel err {err:.3e}"


def pin_exp_forget_golden_fixture(lib):
    """The stored exact case (f = sigmoid(0) = 1/2, i = 1) through the exponential gate with
    f~ = log(1/2): the same exact values, to rounding."""
    with open(os.path.join(GOLDEN, "exact_rational_case.json")) as f:
        g = json.load(f)
    q, k, v = (np.array(g[x], np.float64) for x in ("q", "k", "v"))
    ig = np.array(g["ig"], np.float64)
    fg = np.full_like(ig, np.log(0.5))
    out = oracle.recurrent(q, k, v, ig, fg, lib=lib, forget="exp")
    hx = np.array([[float(Fraction(x)) for x in row] for row in g["h"]])
    Cx = np.array([[float(Fraction(x)) for x in row] for row in g["C_last"]])
    err = max(rel(out["h"][0, 0], hx), rel(out["C"][0, 0], Cx))
    return err <= 1e-14, f"exp-gate golden fixture err {err:.3e}"


ALL_PINS = [
    pin_recurrent_equals_parallel,
    pin_stabiliser_is_a_rescaling,
    pin_single_token_closed_form,
    pin_linear_attention_limit,
    pin_stabiliser_max_plus_form,
    pin_exact_rational,
    pin_golden_fixture,
    pin_split_sequence,
    pin_snapshots,
    pin_causality_and_linearity,
    pin_denominator_brute_force,
    pin_exp_forget_is_a_rescaling,
    pin_exp_forget_dual_form,
    pin_exp_forget_equals_sigmoid_in_log_space,
    pin_exp_forget_two_token_scalar,
    pin_exp_forget_golden_fixture,
    pin_groupnorm_matches_torch,
    pin_groupnorm_gate_invariants,
    pin_backward_finite_differences,
    pin_backward_exp_forget_finite_differences,
    pin_backward_floor_branch,
]


def run_all(lib):
    """[(name, ok, message)] for every pin (exceptions count as failures)."""
    res = []
    for pin in ALL_PINS:
        try:
            ok, msg = pin(lib)
        except Exception as e:  # a broken oracle may fail loudly instead of numerically
            ok, msg = False, f"raised {type(e).__name__}: {e}"
        res.append((pin.__name__, bool(ok), msg))
    return res
