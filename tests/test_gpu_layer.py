"""The fused layer (moe_layer_forward) end to end against the oracle.

Small cases compare every output. The full-size workloads (the bench's
configuration among them, in the launch configuration the bench times)
compare routing for every token bit-exactly, the dispatch permutation
bit-exactly, y_perm on a seeded sample of rows and the layer output on a
seeded sample of tokens within the stated tolerances."""
import json
import os

import numpy as np
import pytest
import torch

import grouped_gemm_softmax_gb300 as moe
import oracle
import synth
from conftest import f32_to_bf16_bits
from gpu_helpers import (GpuLayer, assert_close, bits, check_dispatch, check_route, compact_experts,
                         custom_cfg, need_gpu, oracle_route, sample_tokens, to_f64)
from routing_checks import check_fp64_selection

pytestmark = pytest.mark.gpu


def test_hand_example_on_gpu():
    """The hand-worked example, zero-padded to d = F = 8 (padding changes no output)."""
    need_gpu()
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_example.json")))
    T, E, k, d, F = 4, 3, 2, 8, 8
    x = np.zeros((T, d)); x[:, :2] = g["x"]
    wr = np.zeros((E, d)); wr[:, :2] = g["w_router"]
    w1 = np.zeros((E, F, d)); w1[:, :1, :2] = g["W1"]
    w3 = np.zeros((E, F, d)); w3[:, :1, :2] = g["W3"]
    w2 = np.zeros((E, d, F)); w2[:, :2, :1] = g["W2"]
    dev = lambda a: synth.bits_to_bf16(f32_to_bf16_bits(a)).cuda()
    s = moe.Shape(T=T, d=d, E=E, top_k=k, ffn=F)
    ws = moe.alloc_workspace(s)
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    moe.layer_forward(s, dev(x), dev(wr), None, dev(w1), dev(w3), dev(w2), [out], ws)
    assert moe.last_device_status(ws) == moe.MOE_OK
    got = to_f64(out)
    np.testing.assert_array_equal(got[:, 2:], 0.0)
    # h and y are rounded to bf16 on the GPU: a few bf16 ulps of the closed forms
    np.testing.assert_allclose(got[:, :2], np.array(g["out"]), rtol=2e-2, atol=1e-3)
    idx = moe.ws_view(ws, s, moe.WS.TOPK_IDX, torch.int32, (T, k)).cpu().numpy()
    np.testing.assert_array_equal(idx, g["topk_idx"])
    sor = moe.ws_view(ws, s, moe.WS.SLOT_OF_ROW, torch.int32, (T * k,)).cpu().numpy()
    np.testing.assert_array_equal(sor, g["slot_of_row"])


def _full_compare(layer, out, n_tokens, n_rows, seed=0, every_band=False):
    """Routing and dispatch bit-exact; y_perm on sampled rows and out on sampled
    tokens within the tolerances. every_band: y_perm also on one row of every
    128-row band of every expert (so every scheduler row of the grouped GEMM,
    128 or 256 rows, in either operand orientation) and on each expert's last row;
    and the fp64 selection check on the GPU's indices."""
    cfg = layer.cfg
    ref = oracle_route(layer, keep_logits=every_band)
    idx, gate = layer.routing()
    check_route(idx, gate, ref)
    if every_band:
        sens = check_fp64_selection(idx, bits(layer.inp.x), bits(layer.inp.wr), ref)
        print(f"{cfg.name}: {len(sens)} fp-sensitive tokens {list(sens[:8])}")
    disp = check_dispatch(layer.dispatch_state(), ref.idx, cfg.E)
    # y_perm on sampled rows (first and last row of every expert among them)
    rows = set()
    rng = np.random.default_rng(seed)
    for e in rng.choice(cfg.E, size=min(cfg.E, 8), replace=False):
        a, b = disp.offsets[e], disp.offsets[e + 1]
        if b > a:
            rows.update([a, b - 1, (a + b) // 2])
    if every_band:
        for e in range(cfg.E):
            a, b = int(disp.offsets[e]), int(disp.offsets[e + 1])
            for r0 in range(a, b, 128):
                rows.add(int(rng.integers(r0, min(r0 + 128, b))))
            if b > a:
                rows.add(b - 1)
    rows.update(rng.choice(cfg.R, size=min(cfg.R, n_rows), replace=False).tolist())
    rows = np.array(sorted(rows), np.int64)
    er = np.searchsorted(disp.offsets, rows, side="right") - 1
    tokens = sample_tokens(cfg.T, n_tokens, seed)
    used = set(er.tolist()) | set(ref.idx[tokens].reshape(-1).tolist())
    w1, w3, w2, remap = compact_experts(layer, used)
    xb = bits(layer.inp.x)
    _, yref = oracle.ffn_rows(xb[disp.slot_of_row[rows] // cfg.k], remap[er], w1, w3, w2, len(remap))
    yperm = moe.ws_view(layer.ws, layer.shape, moe.WS.Y_PERM, torch.bfloat16, (cfg.R, cfg.d))
    assert_close(to_f64(yperm[torch.from_numpy(rows).cuda()]), yref, f"{cfg.name} y_perm rows")
    oref = oracle.layer_tokens(xb, remap[ref.idx], ref.gate, w1, w3, w2, tokens, len(remap))
    return assert_close(to_f64(out[torch.from_numpy(tokens.astype(np.int64)).cuda()]), oref,
                        f"{cfg.name} out")


def test_tiny_layer_every_token():
    need_gpu()
    layer = GpuLayer(synth.CONFIGS["tiny"])
    out = layer.forward()
    _full_compare(layer, out, n_tokens=256, n_rows=512)


@pytest.mark.parametrize("cfg", [custom_cfg(1000, 136, 5, 3, 200, S=8, zipf_s=2.0),
                                 custom_cfg(333, 256, 33, 4, 128, S=3, zipf_s=1.0),
                                 custom_cfg(64, 512, 256, 8, 64),
                                 custom_cfg(1, 64, 4, 2, 64),
                                 custom_cfg(50, 16, 6, 2, 24),
                                 # 64 segments (the most allowed); top_k = E; almost every row on one expert
                                 custom_cfg(128, 64, 8, 2, 64, S=64),
                                 custom_cfg(40, 32, 8, 8, 64),
                                 custom_cfg(2000, 64, 16, 1, 64, zipf_s=8.0)],
                         ids=lambda c: f"T{c.T}_E{c.E}_k{c.k}_d{c.d}_S{c.S}")
def test_ragged_layers_every_token(cfg):
    need_gpu()
    layer = GpuLayer(cfg, seed=1)
    out = layer.forward()
    _full_compare(layer, out, n_tokens=cfg.T, n_rows=cfg.R)


def random_shape(E: int):
    """A seeded random layer shape with E experts: T a multiple of S, d and F
    multiples of 8 up to 384 (several K and N tiles, ragged tails), k up to
    min(8, E), Zipf skew 0, 1 or 2."""
    rng = np.random.default_rng(7000 + E)
    k = int(rng.integers(1, min(8, E) + 1))
    S = int(rng.choice([1, 2, 3, 8]))
    T = int(rng.integers(1, 80)) * S
    d = 8 * int(rng.integers(1, 49))
    F = 8 * int(rng.integers(1, 49))
    zipf = float(rng.choice([0.0, 1.0, 2.0]))
    return custom_cfg(T, d, E, k, F, S=S, zipf_s=zipf)


# one expert count per router kernel family (<= 8, 9..16, 17..32, 33..64,
# 65..128, > 128) and their edges
@pytest.mark.parametrize("E", [1, 3, 8, 9, 16, 17, 40, 64, 65, 130, 256])
def test_random_shapes_every_token(E):
    need_gpu()
    cfg = random_shape(E)
    print(f"E={E}: T={cfg.T} d={cfg.d} k={cfg.k} F={cfg.F} S={cfg.S} zipf={cfg.zipf_s}")
    layer = GpuLayer(cfg, seed=E)
    out = layer.forward()
    _full_compare(layer, out, n_tokens=cfg.T, n_rows=cfg.R)


@pytest.mark.parametrize("cfg", [synth.CONFIGS["tiny"], custom_cfg(333, 256, 33, 4, 128, S=3, zipf_s=1.0)],
                         ids=["tiny", "T333_E33"])
def test_layer_replays_from_a_cuda_graph(cfg):
    """The layer only enqueues stream work (no allocation, no synchronisation),
    so it can be captured once and replayed; every replay equals an eager call
    bit for bit."""
    need_gpu()
    layer = GpuLayer(cfg, seed=2)
    eager = layer.forward().clone()  # the eager call also does each launch's one-time setup
    i = layer.inp
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.layer_forward(layer.shape, i.x, i.wr, i.bias, i.w1, i.w3, i.w2, layer.out, layer.ws)
    for _ in range(3):
        for o in layer.out:
            o.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        assert moe.last_device_status(layer.ws) == moe.MOE_OK
        assert torch.equal(torch.cat(layer.out, 0).view(torch.int16), eager.view(torch.int16))


def test_first_calls_from_several_threads_at_once():
    """The one-time per-device launch setup is thread safe and grouped GEMMs of
    different calls may share the GPU: in a fresh process, four threads start
    their first layer calls together (each with its own stream, inputs and
    workspace) and all get the single-threaded result."""
    need_gpu()
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([os.path.dirname(here), here,
                                                       os.environ.get("PYTHONPATH", "")]))
    r = subprocess.run([sys.executable, os.path.join(here, "_concurrent_first_calls.py"), "4"],
                       capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok")


def test_schedules_and_repeat_calls_are_bit_identical():
    need_gpu()
    layer = GpuLayer(synth.CONFIGS["tiny"])
    a = layer.forward().clone()
    b = layer.forward(tuning=moe.Tuning(schedule=moe.SCHEDULE_EXPERT_WAVE)).clone()
    c = layer.forward().clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_layer_with_h_ring_is_bit_identical():
    need_gpu()
    cfg = synth.CONFIGS["tiny"]
    layer = GpuLayer(cfg)
    a = layer.forward().clone()
    t = moe.Tuning(h_ring_rows=33)
    ws = moe.alloc_workspace(layer.shape, tuning=t)
    i = layer.inp
    moe.layer_forward(layer.shape, i.x, i.wr, i.bias, i.w1, i.w3, i.w2, layer.out, ws, tuning=t)
    assert moe.last_device_status(ws) == moe.MOE_OK
    ring_out = torch.cat(layer.out, 0)
    assert torch.equal(ring_out.view(torch.int16), a.view(torch.int16))
    layer.ws = ws  # the ring call's routing, permutation and y_perm, against the oracle
    _full_compare(layer, ring_out, n_tokens=cfg.T, n_rows=cfg.R)


FUSED_CASES = [custom_cfg(1000, 136, 5, 3, 200, S=8, zipf_s=2.0), custom_cfg(333, 256, 33, 4, 128, S=3, zipf_s=1.0),
               custom_cfg(64, 512, 256, 8, 64), custom_cfg(1, 64, 4, 2, 64), custom_cfg(4096, 512, 8, 2, 256, S=4)]
GEMM_MODES = {"m1": dict(cta_group=1, orientation=moe.ORIENT_TOKENS_M),
              "m2": dict(cta_group=2, orientation=moe.ORIENT_TOKENS_M),
              "n1": dict(cta_group=1, orientation=moe.ORIENT_TOKENS_N),
              "n2": dict(cta_group=2, orientation=moe.ORIENT_TOKENS_N)}


@pytest.mark.parametrize("mode", sorted(GEMM_MODES))
@pytest.mark.parametrize("cfg", FUSED_CASES, ids=lambda c: f"T{c.T}_E{c.E}_S{c.S}")
def test_fused_combine_is_bit_identical(cfg, mode):
    """The combine done by consumer warps inside the grouped GEMM, each token
    written once its last expert row is finished, gives the separate combine
    kernel's bits (same fp32 sum in j order), into every owner segment."""
    need_gpu()
    layer = GpuLayer(cfg, seed=2)
    a = layer.forward(tuning=moe.Tuning(**GEMM_MODES[mode])).clone()
    for seg in layer.out:
        seg.fill_(float("nan"))
    b = layer.forward(tuning=moe.Tuning(**GEMM_MODES[mode], fused_combine=1))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    _full_compare(layer, b, n_tokens=min(cfg.T, 512), n_rows=min(cfg.R, 256))


def test_fused_combine_with_h_ring_and_a_timeout():
    """Fused combine over a ring-buffered h is still bit-identical; and when a
    Linear-2 dependency can never be met the consumers give up with the rest
    of the kernel (bounded waits) and the context stays usable."""
    need_gpu()
    cfg = custom_cfg(4096, 256, 8, 2, 256, S=2)
    layer = GpuLayer(cfg, seed=3)
    a = layer.forward().clone()
    t = moe.Tuning(fused_combine=1, h_ring_rows=48)
    ws = moe.alloc_workspace(layer.shape, tuning=t)
    i = layer.inp
    moe.layer_forward(layer.shape, i.x, i.wr, i.bias, i.w1, i.w3, i.w2, layer.out, ws, tuning=t)
    assert moe.last_device_status(ws) == moe.MOE_OK
    assert torch.equal(torch.cat(layer.out, 0).view(torch.int16), a.view(torch.int16))
    ring_ws, layer.ws = layer.ws, ws
    _full_compare(layer, torch.cat(layer.out, 0), n_tokens=512, n_rows=512)
    layer.ws = ring_ws
    bad = moe.Tuning(fused_combine=1, wait_limit_us=20000, unmet_dependency=1)
    moe.layer_forward(layer.shape, i.x, i.wr, i.bias, i.w1, i.w3, i.w2, layer.out, ws, tuning=bad)
    assert moe.last_device_status(ws) == moe.MOE_ERR_TIMEOUT
    moe.layer_forward(layer.shape, i.x, i.wr, i.bias, i.w1, i.w3, i.w2, layer.out, ws, tuning=t)
    assert moe.last_device_status(ws) == moe.MOE_OK
    assert torch.equal(torch.cat(layer.out, 0).view(torch.int16), a.view(torch.int16))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mid", "dit", "fine", "coarse"])
def test_full_size_configs(name):
    need_gpu()
    layer = GpuLayer(synth.CONFIGS[name])
    out = layer.forward()
    out2 = layer.forward(tuning=moe.Tuning(schedule=moe.SCHEDULE_EXPERT_WAVE))
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    out3 = layer.forward(tuning=moe.Tuning(fused_combine=1))
    assert torch.equal(out.view(torch.int16), out3.view(torch.int16))
    for order in (1, 2):
        out4 = layer.forward(tuning=moe.Tuning(row_order=order))
        assert torch.equal(out.view(torch.int16), out4.view(torch.int16))
    maxrel, fro = _full_compare(layer, out, n_tokens=256, n_rows=48, every_band=True)
    print(f"{name}: max err / max|ref| = {maxrel:.2e}, rel Frobenius = {fro:.2e}")
    del layer
    torch.cuda.empty_cache()


def test_tile_timeline_records_every_tile_once():
    """The per-tile timeline (Xian et al., section 5.2.3: per-tile mainloop and
    epilogue spans measured in the kernel) does not change the results, records
    every tile of the layer exactly once in the CTA pair that ran it, with MMA
    start <= last MMA issue <= end of the epilogue stores, and is not truncated
    when sized as the bench sizes it."""
    need_gpu()
    cfg = custom_cfg(3000, 256, 8, 2, 512, zipf_s=1.0)  # tokens on the N side, CTA pairs
    layer = GpuLayer(cfg, seed=4)
    plain = layer.forward().clone()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cap = moe.tile_trace_capacity(layer.shape, sms)
    tt = torch.zeros(sms * cap * moe.TILE_TRACE_WORDS, dtype=torch.int64, device="cuda")
    tr = torch.zeros(sms * moe.TRACE_WORDS, dtype=torch.int64, device="cuda")
    traced = layer.forward(tuning=moe.Tuning(trace=tr, tile_trace=tt, tile_trace_cap=cap))
    assert torch.equal(plain.view(torch.int16), traced.view(torch.int16))
    rec = tt.view(sms, cap, moe.TILE_TRACE_WORDS).cpu().numpy().astype(np.int64)
    assert not (rec[:, -1, 1] > 0).any(), "timeline truncated"
    # the tiles of the layer: 256-token scheduler rows, Linear-1 tiles of 128 h
    # columns and Linear-2 tiles of 256 y columns per row
    counts = np.diff(layer.dispatch_state()["offsets"])
    P = int(sum((int(c) + 255) // 256 for c in counts))
    P1, P2 = (cfg.F + 127) // 128, (cfg.d + 255) // 256
    expected = sorted([(0, r, n) for r in range(P) for n in range(P1)] +
                      [(1, r, n) for r in range(P) for n in range(P2)])
    got = []
    for cta in range(0, sms, 2):  # the first CTA of each pair issues the MMAs
        for w in rec[cta]:
            if w[3] == 0:
                continue
            got.append((int(w[0] & 3), int((w[0] >> 2) & 0xFFFFFFFF), int(w[0] >> 34)))
            assert w[1] > 0 and w[3] <= w[4] <= w[7], w
    assert sorted(got) == expected


def test_overlapping_layers_on_two_streams():
    """Two streams each run layer calls back to back, so their persistent
    grouped GEMMs (one CTA pair per SM each) share the GPU and each grid gets
    only part of the SMs at times; tiles are claimed in order by running CTAs,
    so both complete, with the results of separate calls."""
    need_gpu()
    cfgs = [synth.CONFIGS["mid"], custom_cfg(8192, 1024, 16, 2, 2048, zipf_s=1.0)]
    layers = [GpuLayer(c, seed=5 + i) for i, c in enumerate(cfgs)]
    ref = [layer.forward().clone() for layer in layers]
    streams = [torch.cuda.Stream() for _ in layers]
    torch.cuda.synchronize()
    for _ in range(4):
        for layer in layers:
            for o in layer.out:
                o.fill_(float("nan"))
        torch.cuda.synchronize()
        for rep in range(3):
            for layer, st in zip(layers, streams):
                i = layer.inp
                moe.layer_forward(layer.shape, i.x, i.wr, i.bias, i.w1, i.w3, i.w2, layer.out, layer.ws,
                                  stream=st)
        torch.cuda.synchronize()
        for layer, st, r in zip(layers, streams, ref):
            assert moe.last_device_status(layer.ws, st) == moe.MOE_OK, moe.last_device_detail()
            assert torch.equal(torch.cat(layer.out, 0).view(torch.int16), r.view(torch.int16))
