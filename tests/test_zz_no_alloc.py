"""moe_dispatch_noalloc: the dispatch call for callers that cannot allocate
device memory (its scratch is a fixed array inside the library instead of a
caller workspace). Called through the C ABI and compared with moe_dispatch,
bit for bit (integer and copy work), on two calls in a row so that whatever
the first call leaves in the shared array cannot leak into the second.

This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import grouped_gemm_softmax_gb300 as moe
import oracle
import synth
from gpu_helpers import bits, custom_cfg, need_gpu

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    lib = moe.library()
    f = lib.moe_dispatch_noalloc
    f.argtypes = [ctypes.POINTER(moe._CShape)] + [ctypes.c_void_p] * 8
    f.restype = ctypes.c_int
    return f


def _outputs(T, d, E, k):
    R = T * k
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(counts=torch.full((E,), -1, **i32), offsets=torch.full((E + 1,), -1, **i32),
                ros=torch.full((R,), -1, **i32), sor=torch.full((R,), -1, **i32),
                xp=torch.zeros((R, d), dtype=torch.bfloat16, device="cuda"))


def _case(T, d, E, k, zipf, seed):
    cfg = custom_cfg(T, d, E, k, 8, zipf_s=zipf)
    inp = synth.make_inputs(cfg, seed=seed, device="cuda", weights=False)
    r = oracle.route(bits(inp.x), bits(inp.wr), None if inp.bias is None else inp.bias.cpu().numpy(), k)
    return inp.x, torch.from_numpy(r.idx).cuda()


def test_noalloc_dispatch_matches_workspace_dispatch_twice_in_a_row():
    need_gpu()
    f = _noalloc_fn()
    # different shapes and routings back to back: the second call must not see
    # anything the first one left in the shared scratch
    cases = [(4096, 256, 64, 6, 1.0, 1), (1000, 136, 5, 3, 2.0, 2)]
    for T, d, E, k, zipf, seed in cases:
        x, idx = _case(T, d, E, k, zipf, seed)
        s = moe.Shape(T=T, d=d, E=E, top_k=k, ffn=8)
        ref = _outputs(T, d, E, k)
        moe.dispatch(s, x, idx, ref["counts"], ref["offsets"], ref["ros"], ref["sor"], ref["xp"],
                     moe.alloc_workspace(s))
        got = _outputs(T, d, E, k)
        st = f(ctypes.byref(s.c()), x.data_ptr(), idx.data_ptr(), got["counts"].data_ptr(),
               got["offsets"].data_ptr(), got["ros"].data_ptr(), got["sor"].data_ptr(),
               got["xp"].data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == moe.MOE_OK
        torch.cuda.synchronize()
        for key in ("counts", "offsets", "ros", "sor"):
            assert torch.equal(got[key], ref[key]), key
        assert torch.equal(got["xp"].view(torch.int16), ref["xp"].view(torch.int16))
        # and both equal the oracle's counting sort
        disp = oracle.dispatch(idx.cpu().numpy(), E)
        np.testing.assert_array_equal(got["ros"].cpu().numpy(), disp.row_of_slot)


def test_noalloc_dispatch_rejects_shapes_beyond_its_scratch():
    need_gpu()
    f = _noalloc_fn()
    s = moe.Shape(T=16384, d=64, E=256, top_k=8, ffn=8)  # needs 8192 cells > 4096
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    st = f(ctypes.byref(s.c()), fake, fake, fake, fake, fake, fake, fake, None)
    assert st == moe.MOE_ERR_UNSUPPORTED
