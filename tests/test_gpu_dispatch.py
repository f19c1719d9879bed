"""GPU dispatch (moe_dispatch) against the oracle's counting sort: counts,
offsets, row_of_slot, slot_of_row bit-exact, x_perm an exact row copy. The
routing fed in comes from the oracle (or is built here), never from the GPU."""
import numpy as np
import pytest
import torch

import grouped_gemm_softmax_gb300 as moe
import oracle
import synth
from gpu_helpers import bits, custom_cfg, need_gpu

pytestmark = pytest.mark.gpu


def run_dispatch(x, idx_np, E):
    T, d = x.shape
    k = idx_np.shape[1]
    s = moe.Shape(T=T, d=d, E=E, top_k=k, ffn=8)
    R = T * k
    idx = torch.from_numpy(np.ascontiguousarray(idx_np, dtype=np.int32)).cuda()
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    ros = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    sor = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    xp = torch.zeros((R, d), dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(s)
    moe.dispatch(s, x, idx, counts, offsets, ros, sor, xp, ws)
    assert moe.last_device_status(ws) == moe.MOE_OK
    return (counts.cpu().numpy(), offsets.cpu().numpy(), ros.cpu().numpy(), sor.cpu().numpy(),
            bits(xp))


def check(x, idx_np, E):
    counts, offsets, ros, sor, xp = run_dispatch(x, idx_np, E)
    ref = oracle.dispatch(idx_np, E)
    np.testing.assert_array_equal(counts, ref.counts)
    np.testing.assert_array_equal(offsets, ref.offsets)
    np.testing.assert_array_equal(ros, ref.row_of_slot)
    np.testing.assert_array_equal(sor, ref.slot_of_row)
    k = idx_np.shape[1]
    np.testing.assert_array_equal(xp, bits(x)[ref.slot_of_row // k])


@pytest.mark.parametrize("T,d,E,k,zipf", [
    (256, 256, 8, 2, 0.0), (1, 8, 1, 1, 0.0), (1000, 2048, 64, 6, 1.0), (4096, 512, 256, 8, 0.0),
    (777, 136, 5, 3, 0.0), (300, 64, 256, 1, 0.0), (32768, 1152, 16, 2, 1.2), (5000, 64, 200, 7, 2.0),
])
def test_dispatch_parity_on_oracle_routing(T, d, E, k, zipf):
    need_gpu()
    cfg = custom_cfg(T, d, E, k, 8, zipf_s=zipf)
    inp = synth.make_inputs(cfg, seed=3, device="cuda", weights=False)
    r = oracle.route(bits(inp.x), bits(inp.wr), None if inp.bias is None else inp.bias.cpu().numpy(), k)
    check(inp.x, r.idx, E)


def test_dispatch_all_tokens_to_one_expert_and_empty_experts():
    need_gpu()
    T, d, E, k = 3000, 64, 16, 2
    x = synth.gaussian_bf16((T, d), 1.0, 0, synth.TID_X, "cuda")
    idx = np.stack([np.full(T, 5), np.full(T, 9)], 1).astype(np.int32)
    check(x, idx, E)


def test_dispatch_many_chunks():
    """More tokens than one rank chunk holds: chunk bases must chain across blocks."""
    need_gpu()
    T, d, E, k = 70000, 8, 256, 8
    rng = np.random.default_rng(0)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    x = synth.gaussian_bf16((T, d), 1.0, 0, synth.TID_X, "cuda")
    check(x, idx, E)


def test_dispatch_reports_expert_ids_out_of_range():
    need_gpu()
    T, d, E, k = 64, 16, 4, 2
    x = synth.gaussian_bf16((T, d), 1.0, 0, synth.TID_X, "cuda")
    idx = np.tile(np.array([[0, 1]], np.int32), (T, 1))
    idx[10, 1] = 4  # outside [0, E)
    s = moe.Shape(T=T, d=d, E=E, top_k=k, ffn=8)
    R = T * k
    dev = dict(dtype=torch.int32, device="cuda")
    counts, offsets = torch.empty(E, **dev), torch.empty(E + 1, **dev)
    ros, sor = torch.empty(R, **dev), torch.full((R,), -1, **dev)
    xp = torch.zeros((R, d), dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(s)
    moe.dispatch(s, x, torch.from_numpy(idx).cuda(), counts, offsets, ros, sor, xp, ws)
    assert moe.last_device_status(ws) == moe.MOE_ERR_INVALID_ARG
    assert ros.cpu().numpy()[21] == -1
    assert counts.cpu().numpy().sum() == R - 1
    assert moe.last_device_status(ws) == moe.MOE_OK  # the status was cleared
