"""GPU combine (moe_combine): identity experts with k = 1 give back x bit for
bit; the gate-weighted sum matches the oracle; owner-aligned segments hold
tokens in rank order."""
import numpy as np
import pytest
import torch

import grouped_gemm_softmax_gb300 as moe
import oracle
import synth
from gpu_helpers import assert_close, bits, custom_cfg, need_gpu, to_f64

pytestmark = pytest.mark.gpu


def dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def run_combine(s, y, gate, ros):
    rows = s.T // s.num_segments
    segs = [torch.full((rows, s.d), float("nan"), dtype=torch.bfloat16, device="cuda")
            for _ in range(s.num_segments)]
    moe.combine(s, y, gate, ros, segs)
    torch.cuda.synchronize()
    return torch.cat(segs, 0)


def test_identity_experts_round_trip_is_exact():
    """k = 1: the gate is exactly 1, so combine(dispatch(x)) reproduces x."""
    need_gpu()
    cfg = custom_cfg(1000, 512, 16, 1, 8)
    inp = synth.make_inputs(cfg, seed=2, device="cuda", weights=False)
    r = oracle.route(bits(inp.x), bits(inp.wr), None, 1)
    disp = oracle.dispatch(r.idx, cfg.E)
    s = moe.Shape(T=cfg.T, d=cfg.d, E=cfg.E, top_k=1, ffn=8)
    xperm = inp.x[torch.from_numpy(disp.slot_of_row.astype(np.int64)).cuda()].contiguous()
    out = run_combine(s, xperm, torch.ones(cfg.T, 1, device="cuda"), dev_i32(disp.row_of_slot))
    assert torch.equal(out.view(torch.int16), inp.x.view(torch.int16))


@pytest.mark.parametrize("T,d,E,k,S", [(256, 256, 8, 2, 1), (512, 1152, 16, 2, 8), (300, 2048, 64, 6, 3),
                                       (64, 4096, 256, 8, 1), (7, 8, 3, 3, 7)])
def test_combine_parity(T, d, E, k, S):
    need_gpu()
    cfg = custom_cfg(T, d, E, k, 8)
    inp = synth.make_inputs(cfg, seed=T, device="cuda", weights=False)
    r = oracle.route(bits(inp.x), bits(inp.wr), None, k)
    disp = oracle.dispatch(r.idx, E)
    y = synth.gaussian_bf16((T * k, d), 1.0, 1, synth.TID_ROWS, "cuda")
    s = moe.Shape(T=T, d=d, E=E, top_k=k, ffn=8, num_segments=S)
    gate32 = torch.from_numpy(r.gate.astype(np.float32)).cuda()
    out = run_combine(s, y, gate32, dev_i32(disp.row_of_slot))
    yb = bits(y)
    ref = oracle.combine((yb.astype(np.uint32) << 16).view(np.float32).astype(np.float64),
                         r.gate.astype(np.float32).astype(np.float64), disp.row_of_slot)
    assert_close(to_f64(out), ref, "combine")
    # rounding only: within one bf16 ulp of the fp64 sum, plus fp32 accumulation noise
    yabs = np.abs((yb.astype(np.uint32) << 16).view(np.float32).astype(np.float64))
    mag = oracle.combine(yabs, r.gate.astype(np.float32).astype(np.float64), disp.row_of_slot)
    err = np.abs(to_f64(out) - ref)
    assert np.all(err <= np.abs(ref) * 2.0 ** -8 + mag * 2.0 ** -20)
