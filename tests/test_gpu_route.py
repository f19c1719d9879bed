"""GPU router (moe_route) against the oracle: top-k indices bit-exact, gates
within 1e-5. The selection is taken on fp32 logits summed in ascending feature
order on both sides, so near-ties are decided identically."""
import json
import os

import numpy as np
import pytest
import torch

import grouped_gemm_softmax_gb300 as moe
import oracle
import synth
from conftest import f32_to_bf16_bits
from gpu_helpers import GATE_ATOL, bits, check_route, custom_cfg, need_gpu

pytestmark = pytest.mark.gpu


def run_route(x, wr, bias, k):
    T, d = x.shape
    E = wr.shape[0]
    s = moe.Shape(T=T, d=d, E=E, top_k=k, ffn=8)
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    gate = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    moe.route(s, x, wr, bias, idx, gate)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), gate.cpu().numpy()


@pytest.mark.parametrize("T,d,E,k,zipf", [
    (256, 256, 8, 2, 0.0), (100, 64, 3, 2, 0.0), (1, 8, 1, 1, 0.0), (333, 136, 33, 5, 1.0),
    (130, 512, 64, 6, 1.0), (64, 1152, 16, 2, 1.2), (70, 256, 256, 8, 0.0), (65, 128, 200, 7, 0.5),
    (17, 32, 100, 4, 0.0), (4096, 2048, 64, 6, 1.0), (1000, 4096, 256, 8, 0.0), (129, 40, 128, 8, 0.0),
    # E > 128 picks its token tile (8 * TM tokens, TM 4..8) from T for the fullest
    # last wave (two blocks per SM); on 152 SMs: 36 -> TM 4, 43 -> 5, 50 -> 6,
    # 57 -> 7, 29 -> 8 (one block each), 12160 -> 5 and 8512 -> 4 (many blocks;
    # the fine layer, T = 16384, takes 7)
    (36, 64, 256, 8, 0.0), (43, 64, 256, 8, 0.0), (50, 64, 256, 8, 0.0), (57, 64, 256, 8, 0.0),
    (29, 64, 256, 8, 0.0), (8512, 64, 256, 8, 0.0), (12160, 64, 256, 8, 0.0),
    # up to 16 experts keep the weights resident per block while they fit: a
    # feature count off the 64-feature chunk, a ragged last task, fewer
    # experts than the logits a lane holds, more tasks than the grid's warps
    # (warps loop over tasks), and weights too large to keep (9..16 experts:
    # d > 2048; up to 8: d > 4992)
    (1000, 200, 16, 3, 1.0), (77, 520, 11, 4, 0.5), (40000, 64, 9, 8, 0.0), (100, 4096, 12, 2, 0.0),
    (500, 2048, 16, 2, 0.0), (500, 2056, 16, 2, 0.0), (1, 8, 12, 2, 0.0),
    (30000, 64, 5, 2, 1.0), (10, 4992, 8, 2, 0.0), (10, 5000, 8, 2, 0.0), (13, 72, 2, 2, 0.0),
])
def test_route_parity(T, d, E, k, zipf):
    need_gpu()
    cfg = custom_cfg(T, d, E, k, 8, zipf_s=zipf)
    inp = synth.make_inputs(cfg, seed=T + E, device="cuda", weights=False)
    idx, gate = run_route(inp.x, inp.wr, inp.bias, k)
    ref = oracle.route(bits(inp.x), bits(inp.wr), None if inp.bias is None else inp.bias.cpu().numpy(), k)
    check_route(idx, gate, ref)
    np.testing.assert_allclose(gate.sum(1), 1.0, atol=1e-5)


def test_route_exact_ties_go_to_the_lower_expert():
    need_gpu()
    rng = np.random.default_rng(11)
    T, d, E, k = 200, 16, 40, 6
    x = rng.integers(-2, 3, size=(T, d))
    wr = rng.integers(-1, 2, size=(E, d))
    xt = synth.bits_to_bf16(f32_to_bf16_bits(x)).cuda()
    wt = synth.bits_to_bf16(f32_to_bf16_bits(wr)).cuda()
    idx, gate = run_route(xt, wt, None, k)
    ref = oracle.route(f32_to_bf16_bits(x), f32_to_bf16_bits(wr), None, k)
    check_route(idx, gate, ref)
    z = x @ wr.T
    assert sum(len(set(row)) < E for row in z) > T // 2  # ties really occur


def test_route_hand_example():
    need_gpu()
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_example.json")))
    x = np.zeros((4, 8))
    x[:, :2] = g["x"]
    wr = np.zeros((3, 8))
    wr[:, :2] = g["w_router"]
    idx, gate = run_route(synth.bits_to_bf16(f32_to_bf16_bits(x)).cuda(),
                          synth.bits_to_bf16(f32_to_bf16_bits(wr)).cuda(), None, 2)
    np.testing.assert_array_equal(idx, g["topk_idx"])
    np.testing.assert_allclose(gate, g["gates"], atol=GATE_ATOL)


def test_route_k1_gate_is_exactly_one():
    need_gpu()
    cfg = custom_cfg(300, 64, 12, 1, 8)
    inp = synth.make_inputs(cfg, seed=5, device="cuda", weights=False)
    idx, gate = run_route(inp.x, inp.wr, None, 1)
    assert np.all(gate == 1.0)
