"""Helpers shared by the GPU parity tests: run the C-ABI steps on torch CUDA
tensors and compare with the fp64 oracle under the stated tolerances."""
import numpy as np
import pytest
import torch

import grouped_gemm_softmax_gb300 as moe
import oracle
import synth
from grouped_gemm_softmax_gb300 import build as moe_build

# Output tolerance for bf16 results against the fp64 oracle (the layer's pass
# criteria): max |err| <= 2e-2 * max |ref|  and  ||err||_F <= 5e-3 * ||ref||_F.
MAX_REL = 2e-2
FRO_REL = 5e-3
GATE_ATOL = 1e-5


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    moe_build.build()
    moe.library()


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t)


def assert_close(out, ref, what=""):
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    assert out.shape == ref.shape, (out.shape, ref.shape)
    assert np.all(np.isfinite(out)), f"{what}: non-finite values"
    err = np.abs(out - ref)
    scale = np.abs(ref).max()
    fro = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)
    assert err.max() <= MAX_REL * scale, f"{what}: max err {err.max():.3e} > {MAX_REL}*{scale:.3e}"
    assert fro <= FRO_REL, f"{what}: relative Frobenius error {fro:.3e} > {FRO_REL}"
    return err.max() / max(scale, 1e-300), fro


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def shape_of(cfg) -> moe.Shape:
    return moe.Shape(T=cfg.T, d=cfg.d, E=cfg.E, top_k=cfg.k, ffn=cfg.F, num_segments=cfg.S)


class GpuLayer:
    """Inputs on the GPU plus the workspace for one shape."""

    def __init__(self, cfg, seed=0, device="cuda"):
        self.cfg = cfg
        self.shape = shape_of(cfg)
        self.inp = synth.make_inputs(cfg, seed=seed, device=device)
        self.ws = moe.alloc_workspace(self.shape, device)
        rows = cfg.T // cfg.S
        self.out = [torch.empty(rows, cfg.d, dtype=torch.bfloat16, device=device) for _ in range(cfg.S)]

    def view(self, region, dtype, dims):
        return moe.ws_view(self.ws, self.shape, region, dtype, dims)

    def forward(self, tuning=None):
        i = self.inp
        moe.layer_forward(self.shape, i.x, i.wr, i.bias, i.w1, i.w3, i.w2, self.out, self.ws,
                          tuning=tuning)
        st = moe.last_device_status(self.ws)
        assert st == moe.MOE_OK, f"device status {st} {moe.last_device_detail()}"
        return torch.cat(self.out, 0)

    def routing(self):
        T, k = self.cfg.T, self.cfg.k
        idx = self.view(moe.WS.TOPK_IDX, torch.int32, (T, k)).cpu().numpy()
        gate = self.view(moe.WS.TOPK_GATE, torch.float32, (T, k)).cpu().numpy()
        return idx, gate

    def dispatch_state(self):
        E, R, d = self.cfg.E, self.cfg.R, self.cfg.d
        return dict(
            counts=self.view(moe.WS.COUNTS, torch.int32, (E,)).cpu().numpy(),
            offsets=self.view(moe.WS.OFFSETS, torch.int32, (E + 1,)).cpu().numpy(),
            row_of_slot=self.view(moe.WS.ROW_OF_SLOT, torch.int32, (R,)).cpu().numpy(),
            slot_of_row=self.view(moe.WS.SLOT_OF_ROW, torch.int32, (R,)).cpu().numpy(),
        )


def oracle_route(layer: GpuLayer, keep_logits: bool = False):
    i, cfg = layer.inp, layer.cfg
    bias = None if i.bias is None else i.bias.cpu().numpy()
    return oracle.route(bits(i.x), bits(i.wr), bias, cfg.k, keep_logits=keep_logits)


def check_route(idx_gpu, gate_gpu, ref):
    np.testing.assert_array_equal(idx_gpu, ref.idx)
    np.testing.assert_allclose(gate_gpu.astype(np.float64), ref.gate, rtol=0, atol=GATE_ATOL)


def check_dispatch(state, idx, E):
    ref = oracle.dispatch(idx, E)
    np.testing.assert_array_equal(state["counts"], ref.counts)
    np.testing.assert_array_equal(state["offsets"], ref.offsets)
    np.testing.assert_array_equal(state["row_of_slot"], ref.row_of_slot)
    np.testing.assert_array_equal(state["slot_of_row"], ref.slot_of_row)
    return ref


def sample_tokens(T, n, seed=0):
    """A seeded sample of token ids that always includes the first and last token."""
    if n >= T:
        return np.arange(T, dtype=np.int32)
    rng = np.random.default_rng(seed)
    pick = rng.choice(T - 2, size=n - 2, replace=False) + 1
    return np.sort(np.concatenate([[0, T - 1], pick])).astype(np.int32)


def compact_experts(layer: GpuLayer, experts):
    """Weights of only the listed experts (host bf16 bits) and the expert -> slot map."""
    experts = sorted(set(int(e) for e in experts))
    i = layer.inp
    if len(experts) == layer.cfg.E:  # all of them: no device-side copy
        w1, w3, w2 = bits(i.w1), bits(i.w3), bits(i.w2)
    else:
        sel = torch.tensor(experts, dtype=torch.long, device=layer.inp.w1.device)
        w1 = bits(i.w1.index_select(0, sel))
        w3 = bits(i.w3.index_select(0, sel))
        w2 = bits(i.w2.index_select(0, sel))
    remap = np.full(layer.cfg.E, -1, np.int32)
    remap[experts] = np.arange(len(experts), dtype=np.int32)
    return w1, w3, w2, remap


def custom_cfg(T, d, E, k, F, S=1, zipf_s=0.0):
    return synth.MoEConfig("custom", T=T, d=d, E=E, k=k, F=F, S=S, zipf_s=zipf_s)
