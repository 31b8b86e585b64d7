"""CPU tests of the seeded input generator shared by the GPU path and the oracle."""
import numpy as np
import torch

from mlstm_matrix_memory_02_b300 import workloads as W


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32),
                        np.array([1.0, -2.5, 3.00390625, 3.005859375, 65504.0, 1e-20], np.float32)])
    ours = W.round_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours, ref)


def test_inputs_are_seeded_and_shaped():
    w = W.TINY_F32
    a = W.make_inputs(w)
    b = W.make_inputs(w)
    for key in ("q", "k", "v", "ig", "fg"):
        assert np.array_equal(a[key], b[key])
        assert a[key].dtype == np.float32
    assert a["q"].shape == (1, 2, 64, 32) and a["v"].shape == (1, 2, 64, 32)
    assert a["ig"].shape == (1, 2, 64)
    c = W.make_inputs(w, seed=1)
    assert not np.array_equal(a["q"], c["q"])


def test_bf16_workload_values_are_bf16():
    w = W.LAYER_350M.with_(B=1, NH=1, S=64)
    a = W.make_inputs(w)
    for key in ("q", "k", "v"):
        assert np.array_equal(a[key], W.round_to_bf16(a[key]))
    # gate pre-activations stay fp32
    assert not np.array_equal(a["fg"], W.round_to_bf16(a["fg"]))


def test_distributions_follow_the_workload():
    w = W.LAYER_350M.with_(B=2, NH=2, S=4096)
    a = W.make_inputs(w)
    assert abs(float(a["fg"].mean()) - 3.0) < 0.05 and abs(float(a["fg"].std()) - 1.5) < 0.05
    assert abs(float(a["ig"].mean())) < 0.05 and abs(float(a["ig"].std()) - 1.0) < 0.05
    s = W.STRESS_16K.with_(NH=2, S=8192)
    b = W.make_inputs(s)
    assert float(np.max(np.abs(b["ig"]))) > 20.0   # heavy tails: spikes of exp(>= 20)
    assert abs(float(b["fg"].std()) - 2.0) < 0.1


def test_decode_inputs():
    w = W.DECODE.with_(B=2, NH=2, S=3, prior=5)
    prior, steps = W.make_decode_inputs(w)
    assert prior["q"].shape == (2, 2, 5, 256) and steps["q"].shape == (2, 2, 3, 256)
    assert not np.array_equal(prior["q"][:, :, :3], steps["q"])
