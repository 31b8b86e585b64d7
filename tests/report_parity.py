"""Parity report (not a test: prints the measured errors that the GPU tests bound).

    python tests/report_parity.py

Runs every workload once through the C ABI on cuda:0 and through the fp64 oracle on the same
seeded inputs, and prints one Markdown row per workload: the kernel path, max-abs error over
the oracle output's RMS for h, C_last and n_last (states compared after rescaling to the
oracle's stabiliser), the largest relative error of m_last, and NaN/Inf counts.  The decode
row covers 64 steps of B=256, NH=8, d=256 on 12 sampled heads (the oracle builds their state
from 512 prior tokens); the multi-token row the same heads with 16 tokens per launch.
"""
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

import oracle  # noqa: E402
from mlstm_matrix_memory_02_b300 import binding as B  # noqa: E402
from mlstm_matrix_memory_02_b300 import workloads as W  # noqa: E402
from parity import rel_err, state_errs  # noqa: E402

PATHS = {0: "CUDA cores", 1: "tensor cores", 2: "tensor cores, CTA pair"}


def dev(inp, dtype):
    out = {k: torch.from_numpy(inp[k]).cuda().to(dtype).contiguous() for k in ("q", "k", "v")}
    out.update({k: torch.from_numpy(inp[k]).cuda().contiguous() for k in ("ig", "fg")})
    return out


def npy(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def fwd_row(name):
    w = W.WORKLOADS[name]
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    inp = W.make_inputs(w)
    ora = oracle.recurrent(**inp)
    d = dev(inp, dt)
    h, C, n, m = B.mlstm_fwd_chunkwise(d["q"], d["k"], d["v"], d["ig"], d["fg"], w.chunk, h_dtype=torch.float32)
    torch.cuda.synchronize()
    h, C, n, m = npy(h), npy(C), npy(n), npy(m)
    eC, en, em = state_errs(C, n, m, ora["C"], ora["n"], ora["m"])
    path = PATHS[B.mlstm_fwd_path(w.B, w.NH, w.S, w.DQK, w.DV, w.chunk, dt)]
    bad = int(np.sum(~np.isfinite(h)))
    return f"| {w.name} | {path} | {rel_err(h, ora['h']):.2e} | {eC:.2e} | {en:.2e} | {em:.1e} | {bad} |"


def decode_rows():
    w = W.DECODE
    prior, steps = W.make_decode_inputs(w)
    P = w.B * w.NH
    rng = np.random.default_rng(123)
    sample = np.sort(rng.choice(P, 12, replace=False))
    bi, hi = sample // w.NH, sample % w.NH

    def pick(x):
        return x[bi, hi][:, None]

    o_prior = oracle.recurrent(**{k: pick(v) for k, v in prior.items()}, want_h=False)
    o_steps = oracle.recurrent(**{k: pick(v) for k, v in steps.items()},
                               C0=o_prior["C"], n0=o_prior["n"], m0=o_prior["m"])
    rows = []
    for multi in (False, True):
        d = dev(prior, torch.bfloat16)
        _, C, n, m = B.mlstm_fwd_chunkwise(d["q"], d["k"], d["v"], d["ig"], d["fg"], 64)
        bt, ht = torch.from_numpy(bi).cuda(), torch.from_numpy(hi).cuda()
        C[bt, ht] = torch.from_numpy(o_prior["C"][:, 0].astype(np.float32)).cuda()
        n[bt, ht] = torch.from_numpy(o_prior["n"][:, 0].astype(np.float32)).cuda()
        m[bt, ht] = torch.from_numpy(o_prior["m"][:, 0].astype(np.float32)).cuda()
        s = dev(steps, torch.bfloat16)
        hs = []
        if multi:
            for t0 in range(0, w.S, 16):
                part = [s[k][:, :, t0:t0 + 16].contiguous() for k in ("q", "k", "v", "ig", "fg")]
                hs.append(B.mlstm_step_multi(*part, C, n, m, h_dtype=torch.float32)[bt, ht])
            h = npy(torch.cat(hs, dim=1))
        else:
            for t in range(w.S):
                hs.append(B.mlstm_step(*(s[k][:, :, t].contiguous() for k in ("q", "k", "v", "ig", "fg")),
                                       C, n, m, h_dtype=torch.float32)[bt, ht])
            h = npy(torch.stack(hs, dim=1))
        torch.cuda.synchronize()
        eC, en, em = state_errs(npy(C[bt, ht]), npy(n[bt, ht]), npy(m[bt, ht]), o_steps["C"][:, 0],
                                o_steps["n"][:, 0], o_steps["m"][:, 0])
        label = "decode, 16 tokens per launch (mlstm_step_multi)" if multi else "decode, one token per launch"
        rows.append(f"| {label} | CUDA cores | {rel_err(h, o_steps['h'][:, 0]):.2e} | {eC:.2e} | {en:.2e} | "
                    f"{em:.1e} | {int(np.sum(~np.isfinite(h)))} |")
    return rows


def main():
    print("| workload | path | h | C_last | n_last | m_last | NaN/Inf in h |")
    print("|---|---|---|---|---|---|---|")
    for name in ("tiny", "350m", "1p3b", "stress"):
        print(fwd_row(name), flush=True)
    for row in decode_rows():
        print(row, flush=True)


if __name__ == "__main__":
    main()
