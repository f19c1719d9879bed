"""The seeded input generator: the tensor SplitMix64 matches the integer
definition, draws are reproducible and have the stated distributions."""
import math

import numpy as np
import torch

import synth


def test_mix64_tensor_matches_integer_definition():
    key = synth.tensor_key(0, synth.TID_W1)
    w = synth.words(key, 0, 64, "cpu").numpy().view(np.uint64)
    for c in range(64):
        z = (key + (c + 1) * 0x9E3779B97F4A7C15) & ((1 << 64) - 1)
        assert int(w[c]) == synth.mix64_int(z)
    # SplitMix64 reference value: seed 1234567 -> first output of the standard generator
    assert synth.mix64_int(1234567 + 0x9E3779B97F4A7C15) == 6457827717110365317


def test_gaussian_reproducible_and_distributed():
    a = synth.gaussian_bf16((1000, 100), 0.5, 0, 3)
    b = synth.gaussian_bf16((1000, 100), 0.5, 0, 3, chunk=777)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    v = a.double()
    assert abs(v.mean().item()) < 0.01
    assert abs(v.std().item() - 0.5) < 0.01
    c = synth.gaussian_bf16((1000, 100), 0.5, 1, 3)
    assert not torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_zipf_bias_is_log_of_a_permutation():
    E, s = 64, 1.0
    b = synth.zipf_bias(E, s, 0).astype(np.float64)
    pi = np.rint(np.exp(-b / s)).astype(int)
    assert sorted(pi.tolist()) == list(range(1, E + 1))
    np.testing.assert_allclose(b, -s * np.log(pi), rtol=1e-6)


def test_configs_match_the_stated_workloads():
    c = synth.CONFIGS
    assert (c["tiny"].T, c["tiny"].d, c["tiny"].E, c["tiny"].k, c["tiny"].F) == (256, 256, 8, 2, 512)
    assert (c["mid"].T, c["mid"].d, c["mid"].E, c["mid"].k, c["mid"].F, c["mid"].zipf_s) == \
        (4096, 2048, 64, 6, 1408, 1.0)
    assert (c["dit"].T, c["dit"].d, c["dit"].E, c["dit"].k, c["dit"].F, c["dit"].S) == \
        (32768, 1152, 16, 2, 4608, 8)
    assert (c["fine"].T, c["fine"].d, c["fine"].E, c["fine"].k, c["fine"].F) == (16384, 4096, 256, 8, 2048)
    assert (c["coarse"].T, c["coarse"].d, c["coarse"].E, c["coarse"].k, c["coarse"].F) == \
        (8192, 4096, 8, 2, 14336)
    assert math.isclose(c["mid"].gemm_flops(), 6 * 4096 * 6 * 2048 * 1408)
