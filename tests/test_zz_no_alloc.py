"""The forward entry point that allocates nothing (mlstm_fwd_chunkwise_noalloc), for callers
that cannot allocate device memory -- a plugin inside an application that owns all device
memory through its own pool, or a serving loop where cudaMalloc could synchronise the device.
It works from a fixed scratch array inside the library, so it must give the same outputs as
the regular workspace entry point, call after call (the array keeps the previous call's
contents), and refuse sizes its array cannot hold before launching anything.

This file is collected last on purpose; it needs nothing from the other test files and passes
alone in a fresh process as well as after them.
"""
import numpy as np
import pytest
import torch

from parity import TOL_BF16, TOL_F32, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from mlstm_matrix_memory_02_b300 import binding
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding


def _inputs(w, dtype):
    from mlstm_matrix_memory_02_b300 import workloads as W
    inp = W.make_inputs(w)
    d = {key: torch.from_numpy(inp[key]).cuda().to(dtype).contiguous() for key in ("q", "k", "v")}
    d.update({key: torch.from_numpy(inp[key]).cuda().contiguous() for key in ("ig", "fg")})
    return d


def _outputs(w, h_dtype):
    dev = "cuda"
    return (torch.full((w.B, w.NH, w.S, w.DV), float("nan"), dtype=h_dtype, device=dev),
            torch.full((w.B, w.NH, w.DV, w.DQK), float("nan"), device=dev),
            torch.full((w.B, w.NH, w.DQK), float("nan"), device=dev),
            torch.full((w.B, w.NH), float("nan"), device=dev))


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("case", ["tensor_core_pair", "cuda_core_fp32_with_init"])
def test_no_alloc_forward_matches_workspace_forward(B, case):
    from mlstm_matrix_memory_02_b300 import workloads as W
    if case == "tensor_core_pair":
        w = W.LAYER_350M.with_(B=2, NH=2, S=256, DQK=512, DV=256)
        dtype, tol, chunk, init = torch.bfloat16, TOL_BF16, 64, None
        assert B.mlstm_fwd_path(w.B, w.NH, w.S, w.DQK, w.DV, chunk) >= 1
    else:
        w = W.TINY_F32.with_(B=2, NH=3, S=96, DQK=64, DV=32)
        dtype, tol, chunk = torch.float32, TOL_F32, 32
        g = torch.Generator(device="cuda").manual_seed(3)
        init = (0.3 * torch.randn((w.B, w.NH, w.DV, w.DQK), device="cuda", generator=g),
                0.3 * torch.randn((w.B, w.NH, w.DQK), device="cuda", generator=g),
                torch.randn((w.B, w.NH), device="cuda", generator=g))
    d = _inputs(w, dtype)
    kw = {} if init is None else dict(C_init=init[0], n_init=init[1], m_init=init[2])
    ref = B.mlstm_fwd_chunkwise(d["q"], d["k"], d["v"], d["ig"], d["fg"], chunk, h_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    ref = [_np(x) for x in ref]
    for call in range(2):  # the second call starts from the first call's scratch contents
        out = _outputs(w, torch.float32)
        B.mlstm_fwd_chunkwise_noalloc(d["q"], d["k"], d["v"], d["ig"], d["fg"], chunk, out, **kw)
        torch.cuda.synchronize()
        got = [_np(x) for x in out]
        for name, a, b in zip(("h", "C_last", "n_last", "m_last"), got, ref):
            assert np.all(np.isfinite(a)), (call, name)
            assert rel_err(a, b) <= tol, (call, name, rel_err(a, b))


def test_no_alloc_forward_refuses_sizes_beyond_its_scratch(B):
    from mlstm_matrix_memory_02_b300 import workloads as W
    # fp32 inputs take the CUDA-core path, whose workspace holds every boundary state
    w = W.TINY_F32.with_(B=1, NH=2, S=1024, DQK=256, DV=256, chunk=16)
    assert B.mlstm_fwd_workspace_bytes(w.B, w.NH, w.S, w.DQK, w.DV, w.chunk, torch.float32) \
        > B.NOALLOC_SCRATCH_BYTES
    d = _inputs(w, torch.float32)
    out = _outputs(w, torch.float32)
    with pytest.raises(B.MlstmError) as e:
        B.mlstm_fwd_chunkwise_noalloc(d["q"], d["k"], d["v"], d["ig"], d["fg"], w.chunk, out)
    assert e.value.code == 5  # MLSTM_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(out[0]).all() and torch.isnan(out[1]).all()  # nothing ran
