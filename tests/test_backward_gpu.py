"""GPU parity of the chunkwise backward (mlstm_bwd_chunkwise, through the C ABI) against the
oracle's fp64 recurrent backward (oracle.recurrent_backward, itself pinned by central
differences in the CPU tests) on the same seeded inputs and the same upstream gradient dh.

Every gradient is compared as max |x - x_oracle| / RMS(x_oracle): 1e-4 for fp32 inputs, 2e-2 for
bf16 inputs (the arithmetic is fp32).  Gradients written in bf16 (dq, dk, dv of bf16 inputs) are
held, like a bf16 h, to 2e-2 RMS + 2^-8 |x_oracle| elementwise: rounding a heavy-tailed array to
bf16 alone costs 2^-9 max|x| / RMS in the max-abs/RMS metric.
Cases whose normaliser cancels on some rows (an initial state, heavy-tailed gates) add the
first-order allowance of fp32 arithmetic on those rows: the gradients divide by D_t once
(through g_t) and twice (through c_t, which also carries h_t), so a row whose denominator has
condition number kappa_t carries about 2 kappa_t times the per-term error of fp32 sums,
(d_qk + L) 2^-24; the allowance adds that for the worst row.
"""
import numpy as np
import pytest
import torch

import oracle
from mlstm_matrix_memory_02_b300 import workloads as W
from parity import TOL_BF16, TOL_F32, bf16_out_ok, rel_err, u_fp32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from mlstm_matrix_memory_02_b300 import binding
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding


def npy(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def upstream(w, seed=21):
    """dh: N(0, 1) draws, rounded to bf16 for bf16 workloads so both sides see the same values."""
    rng = np.random.default_rng(seed)
    dh = rng.standard_normal((w.B, w.NH, w.S, w.DV)).astype(np.float32)
    if w.dtype == "bf16":
        dh = torch.from_numpy(dh).to(torch.bfloat16).float().numpy()
    return dh


def initial_state(w, seed=11):
    rng = np.random.default_rng(seed)
    C0 = (0.3 * rng.standard_normal((w.B, w.NH, w.DV, w.DQK))).astype(np.float32)
    n0 = (0.3 * rng.standard_normal((w.B, w.NH, w.DQK))).astype(np.float32)
    m0 = rng.uniform(-2, 3, (w.B, w.NH)).astype(np.float32)
    return C0, n0, m0


def exp_forget(inp, seed=7):
    """f~ for f = exp(f~): log sigmoid of the workload's draws plus N(0, 0.05) noise."""
    rng = np.random.default_rng(seed)
    out = dict(inp)
    fg = inp["fg"].astype(np.float64)
    out["fg"] = (-np.logaddexp(0.0, -fg) + 0.05 * rng.standard_normal(fg.shape)).astype(np.float32)
    return out


def run_case(B, w, chunk, init=False, forget="sigmoid", tol=None, conditioned=False):
    inp = W.make_inputs(w)
    if forget == "exp":
        inp = exp_forget(inp)
    dh = upstream(w)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    tol = tol or (TOL_BF16 if w.dtype == "bf16" else TOL_F32)
    kw, okw = {}, {}
    if init:
        C0, n0, m0 = initial_state(w)
        okw = dict(C0=C0, n0=n0, m0=m0)
        kw = dict(C_init=torch.from_numpy(C0).cuda(), n_init=torch.from_numpy(n0).cuda(),
                  m_init=torch.from_numpy(m0).cuda())
    ora = oracle.recurrent_backward(inp["q"], inp["k"], inp["v"], inp["ig"], inp["fg"], dh, forget=forget, **okw)
    if conditioned:
        fwd = oracle.recurrent(**inp, **okw, forget=forget, want_m_tok=True, want_den=True)
        kappa = fwd["dabs_tok"] / np.maximum(np.abs(fwd["den_tok"]), np.exp(-fwd["m_tok"]))
        tol += 2.0 * float(kappa.max()) * u_fp32(w.DQK, chunk)
    d = {x: torch.from_numpy(inp[x]).cuda().to(dt).contiguous() for x in ("q", "k", "v")}
    d.update({x: torch.from_numpy(inp[x]).cuda().contiguous() for x in ("ig", "fg")})
    g = B.mlstm_bwd_chunkwise(d["q"], d["k"], d["v"], d["ig"], d["fg"], torch.from_numpy(dh).cuda().to(dt), chunk,
                              forget=forget, **kw)
    torch.cuda.synchronize()
    names = [("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("dig", "dig"), ("dfg", "dfg")]
    if init:
        names += [("dC_init", "dC0"), ("dn_init", "dn0"), ("dm_init", "dm0")]
    errs, bad = {}, {}
    for ours, theirs in names:
        x = npy(g[ours])
        assert np.all(np.isfinite(x)), ours
        errs[ours] = rel_err(x, ora[theirs])
        if dt == torch.bfloat16 and ours in ("dq", "dk", "dv"):
            ok, worst = bf16_out_ok(x, ora[theirs], tol)
            if not ok:
                bad[ours] = worst
        elif errs[ours] > tol:
            bad[ours] = errs[ours]
    assert not bad, (bad, errs)
    return errs


@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_backward_tiny_fp32(B, chunk):
    run_case(B, W.TINY_F32, chunk)


@pytest.mark.parametrize("forget", ["sigmoid", "exp"])
def test_backward_tiny_fp32_with_initial_state(B, forget):
    run_case(B, W.TINY_F32.with_(B=2, NH=2, S=96, DQK=64, DV=32), 32, init=True, forget=forget, conditioned=True)


@pytest.mark.parametrize("dqk,dv,s,chunk", [(96, 160, 64, 16), (64, 32, 128, 128), (32, 64, 48, 16)])
def test_backward_fp32_shapes(B, dqk, dv, s, chunk):
    """d_qk != d_v, chunk 128, and a sequence of three chunks."""
    run_case(B, W.TINY_F32.with_(NH=2, S=s, DQK=dqk, DV=dv), chunk, init=(dqk == 64), conditioned=True)


@pytest.mark.parametrize("init", [False, True])
def test_backward_350m_shape_bf16(B, init):
    """d = 256 heads as in the 350M-style layer (fewer heads and tokens so the fp64 oracle
    finishes in seconds): bf16 inputs, dh and gradients."""
    run_case(B, W.LAYER_350M.with_(B=1, NH=2, S=256), 64, init=init, conditioned=init)


@pytest.mark.parametrize("dqk,dv,s,chunk,init", [(64, 128, 192, 64, False), (128, 256, 256, 128, True),
                                                 (512, 128, 128, 64, True), (256, 384, 384, 128, False)])
def test_backward_bf16_tensor_core_states(B, dqk, dv, s, chunk, init):
    """bf16 shapes whose boundary and adjoint states walk on tensor cores (chunk 64 or 128, d_qk a
    power of two from 64, d_v a multiple of 128), every d_qk variant of that kernel."""
    run_case(B, W.LAYER_350M.with_(B=1, NH=2, S=s, DQK=dqk, DV=dv), chunk, init=init, conditioned=init)


def test_backward_full_size_sampled_heads(B):
    """The 350M-style layer at full size (B=8, NH=4, S=1024, d=256, chunk 64: the configuration
    the benchmark times) through the tensor-core backward; two sampled heads against the fp64
    oracle's backward of those heads alone (heads are independent)."""
    w = W.LAYER_350M
    inp = W.make_inputs(w)
    dh = upstream(w)
    d = {x: torch.from_numpy(inp[x]).cuda().to(torch.bfloat16).contiguous() for x in ("q", "k", "v")}
    d.update({x: torch.from_numpy(inp[x]).cuda().contiguous() for x in ("ig", "fg")})
    g = B.mlstm_bwd_chunkwise(d["q"], d["k"], d["v"], d["ig"], d["fg"], torch.from_numpy(dh).cuda().to(torch.bfloat16),
                              w.chunk)
    torch.cuda.synchronize()
    for (i, j) in ((3, 1), (6, 2)):
        sl = lambda x: x[i:i + 1, j:j + 1]
        ora = oracle.recurrent_backward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["ig"]), sl(inp["fg"]), sl(dh))
        for name in ("dq", "dk", "dv", "dig", "dfg"):
            x = sl(npy(g[name]))
            assert np.all(np.isfinite(x)), name
            if name in ("dq", "dk", "dv"):
                ok, worst = bf16_out_ok(x, ora[name], TOL_BF16)
                assert ok, (i, j, name, worst)
            else:
                assert rel_err(x, ora[name]) <= TOL_BF16, (i, j, name, rel_err(x, ora[name]))


def test_backward_state_paths_agree(B):
    """The same bf16 inputs with chunk 32 (states on CUDA cores) and chunk 64 (states on tensor
    cores): the gradients agree to the bf16 tolerance."""
    w = W.LAYER_350M.with_(B=1, NH=2, S=256, DQK=128, DV=128)
    inp = W.make_inputs(w)
    d = {x: torch.from_numpy(inp[x]).cuda().to(torch.bfloat16).contiguous() for x in ("q", "k", "v")}
    d.update({x: torch.from_numpy(inp[x]).cuda().contiguous() for x in ("ig", "fg")})
    dh = torch.from_numpy(upstream(w)).cuda().to(torch.bfloat16)
    g32, g64 = (B.mlstm_bwd_chunkwise(d["q"], d["k"], d["v"], d["ig"], d["fg"], dh, c) for c in (32, 64))
    torch.cuda.synchronize()
    for name in ("dq", "dk", "dv", "dig", "dfg"):
        a, b = npy(g64[name]), npy(g32[name])
        if name in ("dq", "dk", "dv"):
            # both sides are rounded to bf16: twice the one-sided bound
            bound = 2 * (TOL_BF16 * np.sqrt(np.mean(b * b)) + 2.0 ** -8 * np.abs(b))
            assert np.all(np.abs(a - b) <= bound), (name, float(np.max(np.abs(a - b) / bound)))
        else:
            assert rel_err(a, b) <= TOL_BF16, name


def test_backward_stress_gates_fp32(B):
    """Heavy-tailed input gates and weak forget gates (the long-context workload's gate
    distributions) at a small size, fp32."""
    w = W.TINY_F32.with_(B=1, NH=2, S=128, DQK=64, DV=64, ig=("student_t", 4.0, 3.0), fg=("normal", 0.0, 2.0))
    run_case(B, w, 32, conditioned=True)


def test_backward_empty_sequence(B):
    """S = 0: no token gradients; the initial state's gradients are zero."""
    w = W.TINY_F32.with_(S=0)
    C0, n0, m0 = initial_state(w)
    z = torch.zeros((w.B, w.NH, 0, w.DQK), device="cuda")
    zv = torch.zeros((w.B, w.NH, 0, w.DV), device="cuda")
    zg = torch.zeros((w.B, w.NH, 0), device="cuda")
    g = B.mlstm_bwd_chunkwise(z, z.clone(), zv, zg, zg.clone(), zv.clone(), 16, C_init=torch.from_numpy(C0).cuda(),
                              n_init=torch.from_numpy(n0).cuda(), m_init=torch.from_numpy(m0).cuda())
    torch.cuda.synchronize()
    for name in ("dC_init", "dn_init", "dm_init"):
        assert torch.count_nonzero(g[name]) == 0, name


def test_backward_is_linear_in_dh(B):
    """The backward is linear in the upstream gradient: grads(2 dh1 - dh2) = 2 grads(dh1) - grads(dh2)."""
    w = W.TINY_F32.with_(NH=2, S=64, DQK=32, DV=32)
    inp = W.make_inputs(w)
    d = {x: torch.from_numpy(inp[x]).cuda().contiguous() for x in ("q", "k", "v", "ig", "fg")}
    g1 = torch.from_numpy(upstream(w, 1)).cuda()
    g2 = torch.from_numpy(upstream(w, 2)).cuda()
    r1, r2, r3 = (B.mlstm_bwd_chunkwise(d["q"], d["k"], d["v"], d["ig"], d["fg"], x, 16) for x in (g1, g2, 2 * g1 - g2))
    torch.cuda.synchronize()
    for name in ("dq", "dk", "dv", "dig", "dfg"):
        ref = 2 * npy(r1[name]) - npy(r2[name])
        assert rel_err(npy(r3[name]), ref) <= 1e-5, name


def test_backward_argument_errors(B):
    w = W.TINY_F32
    inp = W.make_inputs(w)
    d = {x: torch.from_numpy(inp[x]).cuda().contiguous() for x in ("q", "k", "v", "ig", "fg")}
    dh = torch.zeros((w.B, w.NH, w.S, w.DV), device="cuda")
    ws = torch.empty(B.mlstm_bwd_workspace_bytes(w.B, w.NH, w.S, w.DQK, w.DV, 16, torch.float32), dtype=torch.uint8,
                     device="cuda")
    with pytest.raises(B.MlstmError) as e:  # chunk not in {16, 32, 64, 128}
        B.mlstm_bwd_chunkwise(d["q"], d["k"], d["v"], d["ig"], d["fg"], dh, 48, workspace=ws)
    assert e.value.code == 3
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.MlstmError) as e:
        B.mlstm_bwd_chunkwise(d["q"], d["k"], d["v"], d["ig"], d["fg"], dh, 16, workspace=ws)
    assert e.value.code == 5
