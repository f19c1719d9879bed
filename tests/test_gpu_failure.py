"""Failure detection without a GPU fault: every wait in the grouped GEMM is
bounded. Here a Linear-2 dependency that nothing satisfies (set from the
host) makes the wait run out; the kernel records MOE_ERR_TIMEOUT and where,
drains, frees its tensor memory and returns, and the context stays usable."""
import time

import numpy as np
import pytest
import torch

import grouped_gemm_softmax_gb300 as moe
import oracle
import synth
from gpu_helpers import assert_close, bits, need_gpu, to_f64

pytestmark = pytest.mark.gpu

# where the timeout is recorded: the producer's wait for the Linear-1 rows, or
# a wait that starves behind it (the MMA thread's wait for the next loaded
# stage, the epilogue's wait for the next accumulator, a wait on the CTA's
# tile-descriptor queue), whichever limit runs out first
WHERE_STARVED = {2, 3, 5, 11}


def _case(counts, d, F):
    counts = np.asarray(counts)
    E, R = len(counts), int(counts.sum())
    off = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)).cuda()
    x = synth.gaussian_bf16((R, d), 1.0, 3, synth.TID_ROWS, "cuda")
    w1 = synth.gaussian_bf16((E, F, d), d ** -0.5, 3, synth.TID_W1, "cuda")
    w3 = synth.gaussian_bf16((E, F, d), d ** -0.5, 3, synth.TID_W3, "cuda")
    w2 = synth.gaussian_bf16((E, d, F), F ** -0.5, 3, synth.TID_W2, "cuda")
    return counts, off, x, w1, w3, w2


MODES = [dict(cta_group=1, orientation=moe.ORIENT_TOKENS_M), dict(cta_group=2, orientation=moe.ORIENT_TOKENS_M),
         dict(cta_group=1, orientation=moe.ORIENT_TOKENS_N), dict(cta_group=2, orientation=moe.ORIENT_TOKENS_N)]


@pytest.mark.parametrize("mode", MODES, ids=["m1", "m2", "n1", "n2"])
def test_unmet_dependency_times_out_and_the_context_survives(mode):
    need_gpu()
    counts, off, x, w1, w3, w2 = _case([300, 40, 0, 513], 256, 384)
    E, R, d, F = len(counts), int(counts.sum()), 256, 384
    s = moe.Shape(T=R, d=d, E=E, top_k=1, ffn=F)
    ws = moe.alloc_workspace(s)
    y = torch.zeros(R, d, dtype=torch.bfloat16, device="cuda")
    t0 = time.time()
    moe.expert_ffn(s, x, off, w1, w3, w2, y, ws,
                   tuning=moe.Tuning(**mode, wait_limit_us=20000, unmet_dependency=1))
    st = moe.last_device_status(ws)
    elapsed = time.time() - t0
    assert st == moe.MOE_ERR_TIMEOUT
    where, block, detail = moe.last_device_detail()
    assert where in WHERE_STARVED
    assert elapsed < 10.0
    assert moe.last_device_status(ws) == moe.MOE_OK  # reading it cleared it

    # the same context runs the normal call correctly afterwards
    moe.expert_ffn(s, x, off, w1, w3, w2, y, ws, tuning=moe.Tuning(**mode))
    assert moe.last_device_status(ws) == moe.MOE_OK
    er = np.repeat(np.arange(E), counts).astype(np.int32)
    _, yref = oracle.ffn_rows(bits(x), er, bits(w1), bits(w3), bits(w2), E)
    assert_close(to_f64(y), yref, "after timeout")
