"""The forward entry point that allocates nothing (mlstm_fwd_chunkwise_noalloc), for callers
that cannot allocate device memory -- a plugin inside an application that owns all device
memory through its own pool, or a serving loop where cudaMalloc could synchronise the device.
It works from a fixed scratch array inside the library and runs the same kernels on the same
inputs as the regular workspace entry point, so its outputs must be bit-identical to that
entry point's, call after call (the array keeps the previous call's contents).  It must refuse
sizes its array cannot hold before launching anything, and a device-side wait that gives up in
it must be visible through mlstm_fwd_check_noalloc.

This file is collected last on purpose; it needs nothing from the other test files and passes
alone in a fresh process as well as after them.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from parity import TOL_BF16, TOL_F32, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    from mlstm_matrix_memory_02_b300 import binding
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding


def _inputs(inp, dtype):
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


def _case(case):
    from mlstm_matrix_memory_02_b300 import workloads as W
    if case == "tensor_core_pair":
        w = W.LAYER_350M.with_(B=2, NH=2, S=256, DQK=512, DV=256)
        return w, torch.bfloat16, TOL_BF16, 64, None
    if case == "tensor_core_chunk128":
        # asked for chunk 128, the fused kernel runs (in its own chunks of 64) on a small workspace
        w = W.LAYER_350M.with_(B=1, NH=2, S=512, chunk=128)
        return w, torch.bfloat16, TOL_BF16, 128, None
    w = W.TINY_F32.with_(B=2, NH=3, S=96, DQK=64, DV=32)
    g = torch.Generator(device="cuda").manual_seed(3)
    init = (0.3 * torch.randn((w.B, w.NH, w.DV, w.DQK), device="cuda", generator=g),
            0.3 * torch.randn((w.B, w.NH, w.DQK), device="cuda", generator=g),
            torch.randn((w.B, w.NH), device="cuda", generator=g))
    return w, torch.float32, TOL_F32, 32, init


@pytest.mark.parametrize("case", ["tensor_core_pair", "tensor_core_chunk128", "cuda_core_fp32_with_init"])
def test_no_alloc_forward_matches_workspace_forward(B, case):
    from mlstm_matrix_memory_02_b300 import workloads as W
    w, dtype, tol, chunk, init = _case(case)
    if dtype == torch.bfloat16:
        assert B.mlstm_fwd_path(w.B, w.NH, w.S, w.DQK, w.DV, chunk) >= 1
        assert B.mlstm_fwd_workspace_bytes(w.B, w.NH, w.S, w.DQK, w.DV, chunk) <= B.NOALLOC_SCRATCH_BYTES
    inp = W.make_inputs(w)
    d = _inputs(inp, dtype)
    kw = {} if init is None else dict(C_init=init[0], n_init=init[1], m_init=init[2])
    ref = B.mlstm_fwd_chunkwise(d["q"], d["k"], d["v"], d["ig"], d["fg"], chunk, h_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    for call in range(2):  # the second call starts from the first call's scratch contents
        out = _outputs(w, torch.float32)
        B.mlstm_fwd_chunkwise_noalloc(d["q"], d["k"], d["v"], d["ig"], d["fg"], chunk, out, **kw)
        B.mlstm_fwd_check_noalloc()
        for name, a, b in zip(("h", "C_last", "n_last", "m_last"), out, ref):
            assert torch.equal(a, b), (call, name)
    if init is None:  # the outputs themselves against the oracle
        assert rel_err(_np(out[0]), oracle.recurrent(**inp)["h"]) <= tol


def test_no_alloc_wait_failure_is_reported(B):
    """A bounded device-side wait that gives up in the fixed scratch array's error word is
    reported by mlstm_fwd_check_noalloc (the wait self-test stands in for a forward's wait, with
    no fault); the next forward without allocation clears the word and checks clean."""
    from mlstm_matrix_memory_02_b300 import workloads as W
    ptr, nbytes = B.mlstm_noalloc_scratch()
    assert nbytes == B.NOALLOC_SCRATCH_BYTES and ptr % 256 == 0
    lib = B.library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.mlstm_wait_selftest(ctypes.c_void_p(ptr), ctypes.c_size_t(nbytes), 1, 2, 128, 128, 128, 64, 1,
                                   stream) == 0
    with pytest.raises(B.MlstmError) as e:
        B.mlstm_fwd_check_noalloc()
    assert e.value.code == 7
    assert lib.mlstm_last_cuda_error() == B.SELFTEST_WAIT_CODE
    w, dtype, _, chunk, _ = _case("tensor_core_pair")
    d = _inputs(W.make_inputs(w), dtype)
    out = _outputs(w, torch.float32)
    B.mlstm_fwd_chunkwise_noalloc(d["q"], d["k"], d["v"], d["ig"], d["fg"], chunk, out)
    B.mlstm_fwd_check_noalloc()
    ref = B.mlstm_fwd_chunkwise(d["q"], d["k"], d["v"], d["ig"], d["fg"], chunk, h_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(out[0], ref[0])


def test_no_alloc_forward_refuses_sizes_beyond_its_scratch(B):
    from mlstm_matrix_memory_02_b300 import workloads as W
    # fp32 inputs take the CUDA-core path, whose workspace holds every boundary state
    w = W.TINY_F32.with_(B=1, NH=2, S=1024, DQK=256, DV=256, chunk=16)
    assert B.mlstm_fwd_workspace_bytes(w.B, w.NH, w.S, w.DQK, w.DV, w.chunk, torch.float32) \
        > B.NOALLOC_SCRATCH_BYTES
    d = _inputs(W.make_inputs(w), torch.float32)
    out = _outputs(w, torch.float32)
    with pytest.raises(B.MlstmError) as e:
        B.mlstm_fwd_chunkwise_noalloc(d["q"], d["k"], d["v"], d["ig"], d["fg"], w.chunk, out)
    assert e.value.code == 5  # MLSTM_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(out[0]).all() and torch.isnan(out[1]).all()  # nothing ran
