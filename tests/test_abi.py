"""CPU tests of the C ABI: the library builds for sm_103a, loads, exports every entry point
declared in include/mlstm.h, and rejects bad arguments on the host before any launch.

No GPU is needed and no kernel is launched: every call here fails argument validation,
which runs before the library touches the device.
"""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mlstm.h")

OK, ERR_NULL, ERR_ALIGN, ERR_SHAPE, ERR_DTYPE, ERR_WS, ERR_LAUNCH, ERR_TIMEOUT, ERR_DEVICE = range(9)


@pytest.fixture(scope="module")
def lib():
    from mlstm_matrix_memory_02_b300 import build
    build.build()
    from mlstm_matrix_memory_02_b300 import binding
    return binding.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mlstm_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("mlstm_fwd_chunkwise", "mlstm_step", "mlstm_fwd_workspace_bytes",
                     "mlstm_status_str"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    from mlstm_matrix_memory_02_b300 import binding
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in mlstm.h but not exported"
    assert sorted(binding.EXPORTED) == declared_functions()


def test_status_strings(lib):
    for code in range(9):
        s = lib.mlstm_status_str(code)
        assert s and s.startswith(b"MLSTM_")
    assert lib.mlstm_status_str(99) == b"MLSTM_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    ws = lib.mlstm_fwd_workspace_bytes
    assert ws(4, 4, 2048, 512, 512, 64, 1) > 0
    P, S, NC = 16, 2048, 32
    gates = 3 * P * S * 4 + P * (NC + 1) * 4
    # CUDA-core path (fp32 inputs): gate arrays (3 x P x S fp32) + chunk m + boundary states
    # (P x (NC+1) x DV x DQK fp32)
    need = gates + P * (NC + 1) * 512 * 512 * 4 + P * (NC + 1) * 512 * 4
    assert ws(4, 4, 2048, 512, 512, 64, 0) >= need
    # tensor-core path (bf16, chunk 64): gate arrays, chunk m and a copy of n_init; no states.
    # The full size adds the three-kernel forward's per-chunk operands (beta q and w k in fp16,
    # P in fp16, per-token and per-chunk floats)
    assert lib.mlstm_fwd_path(4, 4, 2048, 512, 512, 64, 1) == 2  # d_qk = 512: CTA pair
    least = lib.mlstm_fwd_workspace_min_bytes(4, 4, 2048, 512, 512, 64, 1)
    assert gates + P * 512 * 4 <= least < need // 100
    assert least + _prepass_bytes(P, S, 512) <= ws(4, 4, 2048, 512, 512, 64, 1) < need // 5
    assert ws(1, 1, 100, 64, 64, 64, 1) == 0      # S % chunk != 0
    assert ws(1, 1, 128, 48, 64, 64, 1) == 0      # DQK not a multiple of 32
    assert ws(1, 1, 128, 64, 1024, 64, 1) == 0    # DV above 512
    assert ws(1, 1, 128, 64, 64, 48, 1) == 0      # chunk not in {16,32,64,128}
    assert ws(1, 1, 128, 64, 64, 64, 7) == 0      # bad dtype code
    assert ws(1, 1, 0, 64, 64, 64, 0) > 0         # empty sequence is allowed


def test_workspace_bytes_follow_the_path_that_runs(lib):
    """The fused kernel walks any asked-for chunk in its own chunks of 64 and keeps no boundary
    state, so a bf16 forward asked for chunk 128 needs only the gate arrays of its chunk (for
    mlstm_fwd_chunk_states and mlstm_fwd_gates) and the fused kernel's own small layout; fp32
    inputs take the CUDA-core path and need every boundary state."""
    ws, ws_min = lib.mlstm_fwd_workspace_bytes, lib.mlstm_fwd_workspace_min_bytes
    P, S = 8, 16384
    assert lib.mlstm_fwd_path(1, 8, S, 256, 256, 128, 1) >= 1
    gates128 = 3 * P * S * 4 + P * (S // 128 + 1) * 4
    assert gates128 <= ws_min(1, 8, S, 256, 256, 128, 1) < 4 << 20
    assert ws(1, 8, S, 256, 256, 128, 0) > P * (S // 128) * 256 * 256 * 4
    assert ws_min(1, 8, S, 256, 256, 128, 0) == ws(1, 8, S, 256, 256, 128, 0)


def _prepass_bytes(P, S, D):
    """Workspace of the three-kernel forward, restated: beta q and w k (fp16, D per token), P
    (fp16, 64 per token), den, 1/den and six gate factors per token (eight floats), the n
    increment (D floats) and two float4 per chunk."""
    NC = S // 64
    return 2 * P * S * D * 2 + P * S * 64 * 2 + P * S * 8 * 4 + P * NC * D * 4 + P * NC * 32


def _prepass_expected(P, S, D):
    """Where the three-kernel forward applies: d_qk = 512 (always a CTA pair), at most 64
    chunks of 64 tokens, and no sequence segments."""
    return D == 512 and 64 <= S <= 4096 and S % 64 == 0


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 148


def _segments_expected(P, S, D, DV):
    """The rule mlstm_fwd_segments follows, restated: the largest power of two G with G times
    the plain grid's CTAs within the SM count, S divisible by 64 G, at least 256 tokens a segment."""
    pair = D == 512 or (D >= 128 and P * (DV // 128) < _sms())
    ctas = P * (DV // 128) * (2 if pair else 1)
    G = 1
    while ctas * 2 * G <= _sms() and S % (64 * 2 * G) == 0 and S // (2 * G) >= 256:
        G *= 2
    return G


@pytest.mark.parametrize("b,nh,s,dqk,dv", [(1, 8, 16384, 256, 256), (4, 4, 2048, 512, 512),
                                           (8, 4, 1024, 256, 256), (1, 2, 1024, 256, 256),
                                           (1, 1, 2048, 512, 256), (2, 1, 1024, 128, 128),
                                           (1, 2, 512, 64, 128), (1, 2, 448, 256, 256)])
def test_sequence_parallel_selection(lib, b, nh, s, dqk, dv):
    """Long sequences over few heads run in G parallel segments when the workspace holds the
    segment buffers (per (head, segment) two fp32 states C, n, m and a float, per token two
    weights, per first-pass chunk a few floats); the least workspace runs them whole, and the
    CUDA-core path never splits."""
    ws, ws_min, seg = lib.mlstm_fwd_workspace_bytes, lib.mlstm_fwd_workspace_min_bytes, lib.mlstm_fwd_segments
    G = _segments_expected(b * nh, s, dqk, dv)
    full, least = ws(b, nh, s, dqk, dv, 64, 1), ws_min(b, nh, s, dqk, dv, 64, 1)
    assert seg(b, nh, s, dqk, dv, 64, 1, full) == G
    assert seg(b, nh, s, dqk, dv, 64, 1, least) == 1
    assert seg(b, nh, s, dqk, dv, 64, 1, full - 1) == (1 if G > 1 else G)
    assert seg(b, nh, s, dqk, dv, 64, 0, 1 << 40) == 1  # fp32 inputs: CUDA-core kernels
    if G > 1:
        # first-pass segments: finer where the GPU has room, at least 128 tokens each
        G1 = G
        while b * nh * (dv // 128) * 2 * G1 <= _sms() and s % (64 * 2 * G1) == 0 and s // (2 * G1) >= 128:
            G1 *= 2
        per_state = (dv * dqk + dqk + 1) * 4  # C, n, m
        per_token = 2 * 4                     # two weights
        least_extra = b * nh * ((G + G1) * per_state + s * per_token)
        slack = b * nh * (3 * 4 * G1 + 4 * G + 4 * (s // 64)) + 14 * 256  # B, m1, chains, round-ups
        assert least_extra <= full - least <= least_extra + slack
    elif _prepass_expected(b * nh, s, dqk):
        extra = _prepass_bytes(b * nh, s, dqk)
        assert extra <= full - least <= extra + 24 * 256  # round-ups
    else:
        assert full == least
    assert seg(1, 2, 100, 64, 64, 64, 1, 1 << 30) == -1  # S % chunk != 0
    assert seg(1, 2, 128, 64, 64, 64, 7, 1 << 30) == -1  # bad dtype code


def test_sequence_parallel_layer_sizes(lib):
    """The long-context layer (B=1 NH=8 S=16384 d=256: 32 CTAs alone) runs in 4 segments on a
    148-SM device; the 1.3B-style layer (128 CTAs) and the 350M-style layer fill the GPU whole."""
    if _sms() != 148:
        pytest.skip("segment counts below are those of a 148-SM device")
    ws, seg = lib.mlstm_fwd_workspace_bytes, lib.mlstm_fwd_segments
    assert seg(1, 8, 16384, 256, 256, 128, 1, ws(1, 8, 16384, 256, 256, 128, 1)) == 4
    assert seg(4, 4, 2048, 512, 512, 64, 1, ws(4, 4, 2048, 512, 512, 64, 1)) == 1
    assert seg(8, 4, 1024, 256, 256, 64, 1, ws(8, 4, 1024, 256, 256, 64, 1)) == 1


def test_noalloc_helpers_argument_errors(lib):
    """mlstm_noalloc_scratch rejects a NULL output before touching the device; without a usable
    device both no-allocation helpers report MLSTM_ERR_DEVICE instead of launching."""
    assert lib.mlstm_noalloc_scratch(None, None) == ERR_NULL
    if not torch.cuda.is_available():
        ptr = ctypes.c_void_p()
        assert lib.mlstm_noalloc_scratch(ctypes.byref(ptr), None) == ERR_DEVICE
        assert lib.mlstm_fwd_check_noalloc(None) == ERR_DEVICE


FAKE = 0x100000  # 16-byte aligned, never dereferenced: every call below fails validation


def _fwd(lib, q=FAKE, ws=FAKE, ws_bytes=1 << 40, S=128, DQK=64, DV=64, chunk=64, dt=1, hdt=0,
         init=(None, None, None), last=(FAKE, FAKE, FAKE)):
    p = ctypes.c_void_p
    return lib.mlstm_fwd_chunkwise(p(q), p(FAKE), p(FAKE), p(FAKE), p(FAKE), 1, 2, S, DQK, DV,
                                   chunk, dt, p(init[0]), p(init[1]), p(init[2]), p(FAKE), hdt,
                                   p(last[0]), p(last[1]), p(last[2]), p(ws),
                                   ctypes.c_size_t(ws_bytes), p(None))


def test_fwd_argument_errors(lib):
    assert _fwd(lib, dt=5) == ERR_DTYPE
    assert _fwd(lib, hdt=9) == ERR_DTYPE
    assert _fwd(lib, S=100) == ERR_SHAPE
    assert _fwd(lib, DQK=40) == ERR_SHAPE
    assert _fwd(lib, chunk=256) == ERR_SHAPE
    assert _fwd(lib, q=None) == ERR_NULL
    assert _fwd(lib, last=(FAKE, None, FAKE)) == ERR_NULL
    assert _fwd(lib, init=(FAKE, None, None)) == ERR_NULL  # all three or none
    assert _fwd(lib, q=FAKE + 4) == ERR_ALIGN
    assert _fwd(lib, init=(FAKE, FAKE + 8, FAKE)) == ERR_ALIGN
    assert _fwd(lib, ws_bytes=16) == ERR_WS
    # the exponential forget-gate flag rides in dt: accepted, and the other checks still apply
    assert _fwd(lib, dt=0x100 | 5) == ERR_DTYPE
    assert _fwd(lib, dt=0x100 | 1, S=100) == ERR_SHAPE
    assert _fwd(lib, dt=0x100 | 1, ws_bytes=16) == ERR_WS


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device status")
def test_fwd_without_device(lib):
    assert _fwd(lib) == ERR_DEVICE


def test_step_argument_errors(lib):
    p = ctypes.c_void_p

    def step(q=FAKE, DQK=64, DV=64, dt=1, hdt=1):
        return lib.mlstm_step(p(q), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE),
                              p(FAKE), 2, 2, DQK, DV, dt, hdt, p(None))

    assert step(dt=3) == ERR_DTYPE
    assert step(dt=0x100 | 3) == ERR_DTYPE
    assert step(dt=0x100 | 1, DQK=16) == ERR_SHAPE
    assert step(DQK=16) == ERR_SHAPE
    assert step(DV=544) == ERR_SHAPE
    assert step(q=None) == ERR_NULL
    assert step(q=FAKE + 2) == ERR_ALIGN


def test_states_and_gates_argument_errors(lib):
    p = ctypes.c_void_p
    r = lib.mlstm_fwd_chunk_states(p(FAKE), p(FAKE), p(FAKE), p(FAKE), 1, 1, 96, 64, 64, 64, 1,
                                   p(None), p(None), p(None), p(FAKE), p(FAKE), p(FAKE), p(FAKE),
                                   ctypes.c_size_t(1 << 40), p(None))
    assert r == ERR_SHAPE
    r = lib.mlstm_fwd_gates(p(FAKE), p(None), 1, 1, 128, 64, p(None), p(FAKE), p(FAKE), p(FAKE),
                            ctypes.c_size_t(1 << 40), p(None))
    assert r == ERR_NULL
    r = lib.mlstm_fwd_gates(p(FAKE), p(FAKE), 1, 1, 128, 64, p(None), p(FAKE), p(FAKE), p(FAKE),
                            ctypes.c_size_t(8), p(None))
    assert r == ERR_WS


def test_binding_rejects_cpu_tensors(lib):
    from mlstm_matrix_memory_02_b300 import binding
    x = torch.zeros(1, 1, 64, 32)
    g = torch.zeros(1, 1, 64)
    with pytest.raises(TypeError):
        binding.mlstm_fwd_chunkwise(x, x, x, g, g, 16)


def test_groupnorm_gate_argument_errors(lib):
    p = ctypes.c_void_p

    def gn(h=FAKE, gamma=FAKE, DV=64, S=4, eps=1e-5, dts=(0, 0, 0)):
        return lib.mlstm_groupnorm_gate(p(h), p(FAKE), p(gamma), p(FAKE), ctypes.c_float(eps), p(FAKE),
                                         2, 2, S, DV, *dts, p(None))

    assert gn(dts=(2, 0, 0)) == ERR_DTYPE
    assert gn(dts=(0, 0, 0x100)) == ERR_DTYPE  # the forget-gate flag has no meaning here
    assert gn(DV=48) == ERR_SHAPE
    assert gn(DV=544) == ERR_SHAPE
    assert gn(S=-1) == ERR_SHAPE
    assert gn(eps=0.0) == ERR_SHAPE
    assert gn(eps=float("nan")) == ERR_SHAPE
    assert gn(h=None) == ERR_NULL
    assert gn(gamma=None, S=0) == ERR_NULL
    assert gn(h=FAKE + 8) == ERR_ALIGN


def test_header_is_plain_c(lib, tmp_path):
    """include/mlstm.h compiles as C99 (no C++ in the boundary) and every declaration links
    against the library."""
    import shutil
    import subprocess
    if not shutil.which("gcc"):
        pytest.skip("gcc not found")
    src = tmp_path / "abi.c"
    names = declared_functions()
    src.write_text('#include "mlstm.h"\n#include <stdio.h>\n'
                   "int main(void) {\n"
                   + "".join(f'  printf("%p\\n", (void *){n});\n' for n in names)
                   + "  return mlstm_status_str(MLSTM_OK)[0] == 'M' ? 0 : 1;\n}\n")
    lib_dir = os.path.join(ROOT, "mlstm_matrix_memory_02_b300")
    exe = tmp_path / "abi"
    res = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                          "-L", lib_dir, "-lmlstm_b300", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


def test_forget_gate_codes():
    from mlstm_matrix_memory_02_b300 import binding as B
    assert B._dt_code(torch.float32) == 0 and B._dt_code(torch.bfloat16) == 1
    assert B._dt_code(torch.bfloat16, "exp") == 1 | B.FORGET_EXP
    with pytest.raises(ValueError):
        B._dt_code(torch.float32, "tanh")


def test_wait_selftest_argument_errors(lib):
    p = ctypes.c_void_p
    st = lib.mlstm_wait_selftest
    assert st(p(None), ctypes.c_size_t(1 << 20), 1, 2, 128, 128, 128, 64, 1, p(None)) == ERR_NULL
    assert st(p(FAKE), ctypes.c_size_t(1 << 20), 1, 2, 128, 128, 128, 64, 5, p(None)) == ERR_DTYPE
    assert st(p(FAKE), ctypes.c_size_t(1 << 20), 1, 2, 100, 128, 128, 64, 1, p(None)) == ERR_SHAPE
    assert st(p(FAKE + 4), ctypes.c_size_t(1 << 20), 1, 2, 128, 128, 128, 64, 1, p(None)) == ERR_ALIGN
    assert st(p(FAKE), ctypes.c_size_t(8), 1, 2, 128, 128, 128, 64, 1, p(None)) == ERR_WS


def test_forward_path_selection(lib):
    """Which kernels mlstm_fwd_chunkwise runs, decided on the host: the fused tensor-core kernel
    for bf16 inputs with S a multiple of 64, d_qk in {64..512} (powers of two) and d_v a
    multiple of 128, whatever chunk is asked for; the CTA pair for d_qk = 512 or when one CTA
    per d_v tile would leave SMs idle; the CUDA-core kernels otherwise."""
    path = lib.mlstm_fwd_path
    assert path(4, 4, 2048, 512, 512, 64, 1) == 2          # 1.3B-style layer
    assert path(8, 4, 1024, 256, 256, 64, 1) == 2          # 350M-style layer: 64 tiles < 148 SMs
    assert path(1, 8, 16384, 256, 256, 128, 1) == 2        # stress layer asks for chunk 128
    assert path(2, 80, 64, 128, 128, 64, 1) == 1           # 160 tiles: one CTA each
    assert path(1, 2, 64, 64, 128, 64, 1) == 1             # d_qk = 64: never split
    assert path(1, 2, 96, 128, 128, 32, 1) == 0            # S not a multiple of 64
    assert path(1, 2, 128, 96, 128, 64, 1) == 0            # d_qk not a power of two
    assert path(1, 2, 128, 128, 96, 64, 1) == 0            # d_v not a multiple of 128
    assert path(4, 4, 2048, 512, 512, 64, 0) == 0          # fp32 inputs
    assert path(4, 4, 2048, 512, 512, 64, 1 | 0x100) == 2  # the forget-gate flag changes nothing
    assert path(1, 2, 100, 64, 64, 64, 1) == -1            # S % chunk != 0

