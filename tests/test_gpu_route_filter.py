"""The layer's filter-then-verify routing against its direct routing and the oracle.

Both routings must give the same bits: the same experts in the same order and
the same gate bits, for every token. Shapes cover one and several candidate
tiles of 128 tokens, ragged feature chunks (d not a multiple of 64), both
exact-kernel ring depths, and the cases that take the full path instead of
the candidate lists: rows of zeros (every expert ties), duplicated expert rows
(exact ties between two experts), near-ties one bf16 ulp apart, and rows so
large that the error bound is not trusted."""
import numpy as np
import pytest
import torch

import grouped_gemm_softmax_gb300 as moe
from gpu_helpers import GpuLayer, check_route, custom_cfg, need_gpu, oracle_route

pytestmark = pytest.mark.gpu

DIRECT = moe.Tuning(router=moe.ROUTER_DIRECT)
FILTER = moe.Tuning(router=moe.ROUTER_FILTER_VERIFY)


def _route_both(layer):
    layer.forward(DIRECT)
    idx_d, gate_d = layer.routing()
    layer.forward(FILTER)
    idx_f, gate_f = layer.routing()
    np.testing.assert_array_equal(idx_f, idx_d)
    np.testing.assert_array_equal(gate_f.view(np.uint32), gate_d.view(np.uint32))
    return idx_f, gate_f


CASES = [
    # T, d, E, k, zipf (bias)
    (1, 4096, 256, 8, 0.0),
    (127, 4096, 256, 8, 1.0),
    (129, 72, 256, 8, 0.0),
    (1000, 4104, 256, 8, 0.0),
    (3000, 2048, 200, 6, 2.0),
    (4100, 1024, 130, 4, 0.0),
    (700, 256, 64, 2, 0.0),
    (333, 8, 17, 3, 0.0),
    (300, 520, 8, 8, 0.0),
    (50, 64, 1, 1, 0.0),
    (20000, 512, 256, 8, 0.0),  # 128 tokens per exact block: the 3-deep ring
]


@pytest.mark.parametrize("T,d,E,k,zipf", CASES, ids=lambda v: str(v))
def test_filter_verify_matches_direct_and_oracle(T, d, E, k, zipf):
    need_gpu()
    layer = GpuLayer(custom_cfg(T, d, E, k, 8, zipf_s=zipf), seed=T + E)
    idx, gate = _route_both(layer)
    check_route(idx, gate, oracle_route(layer))


@pytest.mark.parametrize("E,k", [(256, 8), (130, 2), (40, 4)])
def test_filter_verify_on_ties_and_outliers(E, k):
    """Zero rows, duplicated experts, one-ulp near-ties and huge rows."""
    need_gpu()
    T, d = 1024, 1024
    layer = GpuLayer(custom_cfg(T, d, E, k, 8), seed=7)
    x, wr = layer.inp.x, layer.inp.wr
    with torch.no_grad():
        x[0:40].zero_()                     # every logit 0: all experts tie
        wr[5].copy_(wr[3])                  # experts 3 and 5 tie exactly on every token
        wr[E - 1].copy_(wr[0])              # the first and last expert tie
        near = wr[1].clone()
        bits = near.view(torch.int16)
        bits[d // 2] += 1                   # expert 2 = expert 1 but one ulp in one feature
        wr[2].copy_(near)
        # tokens that prefer expert 1 strongly, so the near-tie is decided at the top
        x[100:140].copy_(wr[1].float().mul(8.0 * d ** 0.5).to(torch.bfloat16).expand(40, d))
        x[200:210].mul_(2.0 ** 100)         # large rows, still inside the trusted range
        x[210:220].mul_(2.0 ** 110)         # |x| |w| beyond the trusted range: the full path
        x[300:310].mul_(2.0 ** -120)        # tiny rows: products near the underflow threshold
    idx, gate = _route_both(layer)
    check_route(idx, gate, oracle_route(layer))
    # the ties went to the lower expert
    assert np.all(idx[0] == np.arange(k))



STANDALONE = [
    (16384, 4096, 256, 8, 0.0),   # the fine-grained workload's router
    (16384, 4096, 256, 8, 1.5),
    (5000, 7168, 256, 8, 0.0),
    (2048, 2048, 160, 6, 0.0),
    (777, 1000, 129, 3, 0.5),
]


@pytest.mark.parametrize("T,d,E,k,zipf", STANDALONE, ids=lambda v: str(v))
def test_route_filtered_matches_route(T, d, E, k, zipf):
    """The standalone entry point against moe_route, every token, bit for bit."""
    need_gpu()
    import synth
    cfg = custom_cfg(T, d, E, k, 8, zipf_s=zipf)
    inp = synth.make_inputs(cfg, seed=11, device="cuda", weights=False)
    s = moe.Shape(T=T, d=d, E=E, top_k=k, ffn=8)
    idx_a = torch.empty(T, k, dtype=torch.int32, device="cuda")
    gate_a = torch.empty(T, k, dtype=torch.float32, device="cuda")
    idx_b, gate_b = torch.empty_like(idx_a), torch.empty_like(gate_a)
    moe.route(s, inp.x, inp.wr, inp.bias, idx_a, gate_a)
    scratch = moe.alloc_route_scratch(s)
    for _ in range(2):  # the second call reuses the scratch
        idx_b.fill_(-1)
        moe.route_filtered(s, inp.x, inp.wr, inp.bias, idx_b, gate_b, scratch)
        assert moe.last_device_status(scratch) == moe.MOE_OK
        assert torch.equal(idx_b, idx_a)
        assert torch.equal(gate_b.view(torch.int32), gate_a.view(torch.int32))
