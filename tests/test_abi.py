"""The C-ABI library: it builds, loads without a GPU, exports every entry point
include/moe.h declares, and its host-side argument checks and workspace layout
behave as documented. No call here reaches the GPU."""
import ctypes
import os
import re

import pytest

import grouped_gemm_softmax_gb300 as moe
from grouped_gemm_softmax_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return moe.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_layer_forward",
                     "moe_workspace_bytes", "moe_last_device_status", "moe_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert missing == []


def test_status_strings(lib):
    assert moe._status_string(0) == "ok"
    assert moe._status_string(5) == "device wait timed out"
    assert moe._status_string(99) == "unknown status"


def test_workspace_layout_regions_are_disjoint_and_aligned(lib):
    s = moe.Shape(T=4096, d=2048, E=64, top_k=6, ffn=1408)
    total = moe.workspace_bytes(s)
    R = s.R
    expect = {moe.WS.X_PERM: R * s.d * 2, moe.WS.H: R * s.ffn * 2, moe.WS.Y_PERM: R * s.d * 2,
              moe.WS.TOPK_IDX: R * 4, moe.WS.ROW_OF_SLOT: R * 4, moe.WS.OFFSETS: (s.E + 1) * 4}
    spans = []
    for r in range(13):
        off, nb = moe.workspace_region(s, r)
        assert off % 1024 == 0
        assert off + nb <= total
        spans.append((off, off + nb))
        if r in expect:
            assert nb == expect[r]
    assert moe.workspace_region(s, moe.WS.STATUS)[0] == 0
    spans.sort()
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
    # h dominates: R*F*2 + 2*R*d*2 plus small regions
    assert total < (R * s.ffn * 2 + 2 * R * s.d * 2) * 1.1


@pytest.mark.parametrize("shape,status", [
    (dict(T=8, d=12, E=4, top_k=2, ffn=16), 1),       # d not a multiple of 8
    (dict(T=8, d=16, E=4, top_k=2, ffn=20), 1),       # ffn not a multiple of 8
    (dict(T=8, d=16, E=2, top_k=3, ffn=16), 1),       # k > E
    (dict(T=9, d=16, E=4, top_k=2, ffn=16, num_segments=2), 1),  # T % S != 0
    (dict(T=8, d=16, E=257, top_k=2, ffn=16), 2),     # too many experts
    (dict(T=8, d=16, E=16, top_k=9, ffn=16), 2),      # k > 8
    (dict(T=-1, d=16, E=4, top_k=2, ffn=16), 1),
    (dict(T=130, d=16, E=4, top_k=2, ffn=16, num_segments=65), 2),
])
def test_invalid_shapes_are_rejected_on_the_host(lib, shape, status):
    s = moe.Shape(**shape)
    assert moe.workspace_bytes(s) == 0
    st = lib.moe_route(ctypes.byref(s.c()), None, None, None, None, None, None)
    assert st == status


def test_null_pointers_and_small_workspace_are_rejected_on_the_host(lib):
    s = moe.Shape(T=64, d=64, E=4, top_k=2, ffn=64)
    c = ctypes.byref(s.c())
    assert lib.moe_route(c, None, None, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(c, None, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check fails first
    nb = moe.workspace_bytes(s)
    assert lib.moe_expert_ffn(c, fake, fake, fake, fake, fake, fake, fake, nb - 1, None) == \
        moe.MOE_ERR_WORKSPACE
    assert lib.moe_layer_forward(c, fake, fake, None, fake, fake, fake, None, fake, nb - 1, None) == \
        moe.MOE_ERR_WORKSPACE
    # misaligned pointer
    mis = ctypes.c_void_p((1 << 20) + 8)
    assert lib.moe_expert_ffn(c, mis, fake, fake, fake, fake, fake, fake, nb, None) == \
        moe.MOE_ERR_INVALID_ARG
    bad_tune = moe.Tuning(schedule=7)
    assert lib.moe_expert_ffn_tuned(c, ctypes.byref(bad_tune.c()), fake, fake, fake, fake, fake, fake,
                                    fake, nb, None) == moe.MOE_ERR_INVALID_ARG
    for bad in (dict(orientation=3), dict(orientation=-1)):
        bad_tune = moe.Tuning(**bad)  # no such orientation
        assert lib.moe_expert_ffn_tuned(c, ctypes.byref(bad_tune.c()), fake, fake, fake, fake, fake, fake,
                                        fake, nb, None) == moe.MOE_ERR_INVALID_ARG
    bad_tune = moe.Tuning(l2_block_n=48)
    assert lib.moe_expert_ffn_tuned(c, ctypes.byref(bad_tune.c()), fake, fake, fake, fake, fake, fake,
                                    fake, nb, None) == moe.MOE_ERR_INVALID_ARG


def test_index_and_gate_arrays_must_be_4_byte_aligned(lib):
    # the checks run before any launch: every other pointer is a fake, aligned address
    s = moe.Shape(T=64, d=64, E=4, top_k=2, ffn=64)
    c = ctypes.byref(s.c())
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 2)
    segs = (ctypes.c_void_p * 1)(1 << 21)
    assert lib.moe_combine(c, fake, odd, fake, segs, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(c, fake, fake, odd, segs, None) == moe.MOE_ERR_INVALID_ARG
    nb = moe.workspace_bytes(s)
    for i in range(3):  # topk_idx, row_of_slot, slot_of_row
        args = [fake, odd if i == 0 else fake, fake, fake, odd if i == 1 else fake,
                odd if i == 2 else fake, fake, fake]
        assert lib.moe_dispatch(c, *args, nb, None) == moe.MOE_ERR_INVALID_ARG
        assert lib.moe_dispatch_noalloc(c, *args[:7], None) == moe.MOE_ERR_INVALID_ARG


def test_empty_call_enqueues_nothing(lib):
    s = moe.Shape(T=0, d=64, E=4, top_k=2, ffn=64)
    assert moe.workspace_bytes(s) > 0
    c = ctypes.byref(s.c())
    assert lib.moe_route(c, None, None, None, None, None, None) == moe.MOE_OK
    assert lib.moe_combine(c, None, None, None, None, None) == moe.MOE_OK
    fake = ctypes.c_void_p(1 << 20)
    nb = moe.workspace_bytes(s)
    assert lib.moe_expert_ffn(c, None, None, None, None, None, None, fake, nb, None) == moe.MOE_OK
    assert lib.moe_layer_forward(c, None, None, None, None, None, None, None, fake, nb, None) == moe.MOE_OK


def test_binding_rejects_wrong_tensors_before_the_library():
    import torch
    s = moe.Shape(T=4, d=8, E=2, top_k=1, ffn=8)
    with pytest.raises(TypeError):
        moe.route(s, torch.zeros(4, 8), torch.zeros(2, 8, dtype=torch.bfloat16), None,
                  torch.zeros(4, dtype=torch.int32), torch.zeros(4))
    with pytest.raises(ValueError):  # CPU tensors are refused: no host fallback exists
        moe.route(s, torch.zeros(4, 8, dtype=torch.bfloat16), torch.zeros(2, 8, dtype=torch.bfloat16),
                  None, torch.zeros(4, dtype=torch.int32), torch.zeros(4))


def test_h_ring_workspace_layout_and_checks(lib):
    """An h ring shrinks only the h region, which is the last one: every other
    region keeps its offset, so moe_dispatch accepts either workspace. A ring
    needs the interleaved schedule."""
    s = moe.Shape(T=4096, d=2048, E=64, top_k=6, ffn=1408)
    ring = moe.Tuning(h_ring_rows=40)
    full_nb, ring_nb = moe.workspace_bytes(s), moe.workspace_bytes(s, ring)
    assert ring_nb < full_nb
    for r in range(13):
        off_f, nb_f = moe.workspace_region(s, r)
        off_r, nb_r = moe.workspace_region(s, r, ring)
        assert off_f == off_r
        if r == moe.WS.H:
            assert nb_r == 40 * 256 * 1408 * 2 and off_r + nb_r <= ring_nb
        else:
            assert nb_f == nb_r and off_r + nb_r <= moe.workspace_region(s, moe.WS.H)[0]
    c = ctypes.byref(s.c())
    for bad in (moe.Tuning(h_ring_rows=40, schedule=moe.SCHEDULE_EXPERT_WAVE), moe.Tuning(h_ring_rows=-1)):
        assert lib.moe_workspace_bytes_tuned(c, ctypes.byref(bad.c())) == 0
    fake = ctypes.c_void_p(1 << 20)
    bad = moe.Tuning(h_ring_rows=40, schedule=moe.SCHEDULE_EXPERT_WAVE)
    assert lib.moe_expert_ffn_tuned(c, ctypes.byref(bad.c()), fake, fake, fake, fake, fake, fake,
                                    fake, full_nb, None) == moe.MOE_ERR_INVALID_ARG
    # the untuned FFN needs the full workspace; a ring-sized one is refused
    assert lib.moe_expert_ffn(c, fake, fake, fake, fake, fake, fake, fake, ring_nb, None) == \
        moe.MOE_ERR_WORKSPACE


def test_fused_combine_belongs_to_the_layer_call(lib):
    s = moe.Shape(T=64, d=64, E=4, top_k=2, ffn=64)
    c = ctypes.byref(s.c())
    fake = ctypes.c_void_p(1 << 20)
    nb = moe.workspace_bytes(s)
    for bad in (moe.Tuning(fused_combine=1), moe.Tuning(fused_combine=2)):
        assert lib.moe_expert_ffn_tuned(c, ctypes.byref(bad.c()), fake, fake, fake, fake, fake, fake,
                                        fake, nb, None) == moe.MOE_ERR_INVALID_ARG


def test_row_order_values_are_checked(lib):
    s = moe.Shape(T=64, d=64, E=4, top_k=2, ffn=64)
    c = ctypes.byref(s.c())
    fake = ctypes.c_void_p(1 << 20)
    nb = moe.workspace_bytes(s)
    for bad in (moe.Tuning(row_order=3), moe.Tuning(row_order=-1)):
        assert lib.moe_expert_ffn_tuned(c, ctypes.byref(bad.c()), fake, fake, fake, fake, fake, fake,
                                        fake, nb, None) == moe.MOE_ERR_INVALID_ARG



def test_layer_kernel_launches(lib):
    """Host-side count of the layer's launches: route (one kernel, or four when
    it filters then verifies: the default above 128 experts), four dispatch
    kernels, the grouped GEMM and the combine (none when the combine is fused
    into the GEMM)."""
    fine = moe.Shape(T=16384, d=4096, E=256, top_k=8, ffn=2048)
    assert moe.layer_kernel_launches(fine) == 10
    assert moe.layer_kernel_launches(fine, moe.Tuning(fused_combine=1)) == 9
    assert moe.layer_kernel_launches(fine, moe.Tuning(router=moe.ROUTER_DIRECT)) == 7
    mid = moe.Shape(T=16384, d=2048, E=64, top_k=8, ffn=1024)
    assert moe.layer_kernel_launches(mid) == 7
    assert moe.layer_kernel_launches(mid, moe.Tuning(router=moe.ROUTER_FILTER_VERIFY)) == 10
    at_128 = moe.Shape(T=1024, d=512, E=128, top_k=8, ffn=64)
    assert moe.layer_kernel_launches(at_128) == 7
    bad = moe.Shape(T=10, d=12, E=4, top_k=2, ffn=16)  # d not a multiple of 8
    assert moe.layer_kernel_launches(bad) == 0
    assert moe.layer_kernel_launches(fine, moe.Tuning(router=3)) == 0


def test_route_filtered_host_checks(lib):
    """moe_route_filtered rejects bad arguments before enqueuing anything."""
    s = moe.Shape(T=64, d=64, E=4, top_k=2, ffn=64)
    c = ctypes.byref(s.c())
    nb = moe.route_scratch_bytes(s)
    assert nb >= 256 + 64 * 64 + 64
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: a host check fails first
    assert lib.moe_route_filtered(c, None, None, None, None, None, None, 0, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_route_filtered(c, fake, fake, None, fake, fake, fake, nb - 1, None) == moe.MOE_ERR_WORKSPACE
    odd = ctypes.c_void_p((1 << 20) + 16)  # 16-byte but not 256-byte aligned scratch
    assert lib.moe_route_filtered(c, fake, fake, None, fake, fake, odd, nb, None) == moe.MOE_ERR_INVALID_ARG
    empty = moe.Shape(T=0, d=64, E=4, top_k=2, ffn=64)
    assert lib.moe_route_filtered(ctypes.byref(empty.c()), None, None, None, None, None, None, 0, None) == \
        moe.MOE_OK
    bad = moe.Shape(T=8, d=12, E=4, top_k=2, ffn=16)
    assert moe.route_scratch_bytes(bad) == 0
    assert lib.moe_route_filtered(ctypes.byref(bad.c()), fake, fake, None, fake, fake, fake, nb, None) == \
        moe.MOE_ERR_INVALID_ARG


def test_layer_routes_directly_when_x_perm_cannot_hold_the_scratch(lib):
    """The filter-then-verify router keeps its scratch in the X_PERM region
    (T*k*d*2 bytes); with k*d*2 below its ~69 bytes per token the layer
    routes directly instead."""
    roomy = moe.Shape(T=1000, d=64, E=200, top_k=1, ffn=16)
    tight = moe.Shape(T=1000, d=8, E=200, top_k=1, ffn=16)
    assert moe.layer_kernel_launches(roomy) == 10
    assert moe.layer_kernel_launches(tight) == 7
    assert moe.layer_kernel_launches(tight, moe.Tuning(router=moe.ROUTER_FILTER_VERIFY)) == 7


def test_route_filtered_rejects_a_huge_feature_dimension(lib):
    s = moe.Shape(T=1, d=1 << 20, E=4, top_k=2, ffn=8)
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the shape check fails first
    nb = moe.route_scratch_bytes(s)
    assert nb > 0
    assert lib.moe_route_filtered(ctypes.byref(s.c()), fake, fake, None, fake, fake, fake, nb, None) == \
        moe.MOE_ERR_UNSUPPORTED
