"""GPU grouped SwiGLU GEMM (moe_expert_ffn) against the oracle's per-row expert
FFN: h and y_perm within the bf16 tolerances, on ragged expert sizes (empty
experts, one-row experts, tiles that straddle experts, K and N tails) in both
operand orientations (tokens as the MMA's M rows or as its N columns), every
tile schedule bit-identical within an orientation, and every Linear-2 tile's
ready flag published."""
import numpy as np
import pytest
import torch

import grouped_gemm_softmax_gb300 as moe
import oracle
import synth
from gpu_helpers import assert_close, bits, need_gpu, to_f64

pytestmark = pytest.mark.gpu


def make_case(counts, d, F, seed=0):
    counts = np.asarray(counts, np.int64)
    E = len(counts)
    R = int(counts.sum())
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = synth.gaussian_bf16((R, d), 1.0, seed, synth.TID_ROWS, "cuda")
    w1 = synth.gaussian_bf16((E, F, d), d ** -0.5, seed, synth.TID_W1, "cuda")
    w3 = synth.gaussian_bf16((E, F, d), d ** -0.5, seed, synth.TID_W3, "cuda")
    w2 = synth.gaussian_bf16((E, d, F), F ** -0.5, seed, synth.TID_W2, "cuda")
    return dict(counts=counts, offsets=offsets, x=x, w1=w1, w3=w3, w2=w2, E=E, R=R, d=d, F=F)


def run_ffn(c, tuning=None, ws=None):
    # the shape's T*k must equal R: use k = 1 and T = R
    s = moe.Shape(T=c["R"], d=c["d"], E=c["E"], top_k=1, ffn=c["F"])
    if ws is None:
        ws = moe.alloc_workspace(s)
    y = torch.full((c["R"], c["d"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    off = torch.from_numpy(c["offsets"]).cuda()
    moe.expert_ffn(s, c["x"], off, c["w1"], c["w3"], c["w2"], y, ws, tuning=tuning)
    st = moe.last_device_status(ws)
    assert st == moe.MOE_OK, (st, moe.last_device_detail())
    ring = tuning is not None and tuning.h_ring_rows > 0  # then h holds only the last rows
    h = None if ring else moe.ws_view(ws, s, moe.WS.H, torch.bfloat16, (c["R"], c["F"])).clone()
    return s, ws, h, y


def oracle_rows(c, rows):
    er = np.repeat(np.arange(c["E"]), c["counts"]).astype(np.int32)[rows]
    return oracle.ffn_rows(bits(c["x"])[rows], er, bits(c["w1"]), bits(c["w3"]), bits(c["w2"]), c["E"],
                           keep_h=True)


CASES = {
    "single_expert_one_tile": ([128], 256, 256),
    "single_expert_ragged": ([300], 256, 512),
    "tiny_like": ([70, 0, 129, 1, 255, 57, 0, 0], 256, 512),
    "k_and_n_tails": ([200, 33, 140], 136, 200),
    "wide_d_tail": ([260, 70], 1160, 128),
    "dit_like_d": ([130, 5, 400], 1152, 384),
    "many_small_experts": ([3, 1, 0, 7, 130, 2, 0, 64] * 8, 128, 256),
    "one_row": ([1], 64, 64),
    # the smallest widths the shape rules allow: feature and ffn widths of 8
    # and 24/40, far below one 64-wide k-block (zero-filled past the end)
    "min_widths": ([20, 5], 8, 8),
    "small_widths": ([33, 0, 17], 24, 40),
}


# (CTAs per tile, operand orientation): single CTAs and pairs with tokens as M
# rows, pairs with tokens as N columns
MODES = {"m1": dict(cta_group=1, orientation=moe.ORIENT_TOKENS_M),
         "m2": dict(cta_group=2, orientation=moe.ORIENT_TOKENS_M),
         "n1": dict(cta_group=1, orientation=moe.ORIENT_TOKENS_N),
         "n2": dict(cta_group=2, orientation=moe.ORIENT_TOKENS_N)}
TILE_ROWS = {"m1": 128, "m2": 256, "n1": 256, "n2": 256}  # token rows of a scheduler row
L1_COLS = {"m1": 128, "m2": 128, "n1": 64, "n2": 128}     # h columns of a Linear-1 tile
L2_COLS = {"m1": 256, "m2": 256, "n1": 128, "n2": 256}    # y columns of a Linear-2 tile (d = 256)


@pytest.mark.parametrize("mode", ["m1", "n1", "n2"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_ffn_parity(name, mode):
    need_gpu()
    counts, d, F = CASES[name]
    c = make_case(counts, d, F, seed=len(name))
    _, _, h, y = run_ffn(c, tuning=moe.Tuning(**MODES[mode]))
    rows = np.arange(c["R"])
    href, yref = oracle_rows(c, rows)
    assert_close(to_f64(h), href, f"{name} {mode} h")
    assert_close(to_f64(y), yref, f"{name} {mode} y")


@pytest.mark.parametrize("mode", sorted(MODES))
def test_ffn_schedules_and_grids_are_bit_identical(mode):
    """The tile order never changes a result: every schedule, lead, raster group
    and grid size gives the same bits (within one tile shape)."""
    need_gpu()
    c = make_case([70, 0, 129, 1, 255, 57, 300, 12] * 4, 256, 384, seed=9)
    _, _, h0, y0 = run_ffn(c, tuning=moe.Tuning(**MODES[mode]))
    variants = [dict(schedule=moe.SCHEDULE_EXPERT_WAVE), dict(lead_rows=1), dict(lead_rows=50),
                dict(num_ctas=2), dict(num_ctas=7), dict(group_rows=1), dict(group_rows=4),
                dict(schedule=moe.SCHEDULE_EXPERT_WAVE, num_ctas=6, group_rows=2),
                dict(row_order=1), dict(row_order=2), dict(row_order=2, num_ctas=6, group_rows=2),
                dict(row_order=2, lead_rows=1)]
    for v in variants:
        t = moe.Tuning(**MODES[mode], **v)
        _, _, h, y = run_ffn(c, tuning=t)
        assert torch.equal(h.view(torch.int16), h0.view(torch.int16)), t
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16)), t


def test_cta_pairs_match_single_ctas():
    need_gpu()
    c = make_case([70, 0, 129, 1, 255, 57, 300, 12], 256, 384, seed=10)
    _, _, h1, y1 = run_ffn(c, tuning=moe.Tuning(**MODES["m1"]))
    _, _, h2, y2 = run_ffn(c, tuning=moe.Tuning(**MODES["m2"]))
    href, yref = oracle_rows(c, np.arange(c["R"]))
    assert_close(to_f64(h2), href, "pairs h")
    assert_close(to_f64(y2), yref, "pairs y")
    # the same MMA arithmetic per element: expected bit-identical
    assert torch.equal(h1.view(torch.int16), h2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_tokens_as_n_columns_match_tokens_as_m_rows():
    """Swapping the MMA operands changes only the fp32 accumulation order: both
    orientations meet the oracle, and agree with each other to a few bf16 ulps."""
    need_gpu()
    c = make_case([70, 0, 129, 1, 255, 57, 300, 12, 16, 17, 15], 512, 640, seed=11)
    _, _, hm, ym = run_ffn(c, tuning=moe.Tuning(**MODES["m2"]))
    _, _, hn, yn = run_ffn(c, tuning=moe.Tuning(**MODES["n2"]))
    href, yref = oracle_rows(c, np.arange(c["R"]))
    assert_close(to_f64(hn), href, "tokens-as-N h")
    assert_close(to_f64(yn), yref, "tokens-as-N y")
    # each result is the bf16 rounding of nearly the same fp32 value
    for a, b in ((hm, hn), (ym, yn)):
        da, db = to_f64(a), to_f64(b)
        assert np.all(np.abs(da - db) <= 2.0 ** -6 * np.abs(da) + 1e-6)


def test_default_orientation_puts_tokens_on_n_for_small_experts():
    """The default for 300-row experts is tokens as N columns: bit-identical to
    asking for it."""
    need_gpu()
    c = make_case([300, 200, 280], 256, 256, seed=12)
    _, _, hd, yd = run_ffn(c)
    _, _, hn, yn = run_ffn(c, tuning=moe.Tuning(orientation=moe.ORIENT_TOKENS_N))
    assert torch.equal(yd.view(torch.int16), yn.view(torch.int16))


@pytest.mark.parametrize("mode", sorted(MODES))
def test_h_ring_is_bit_identical_to_full_h(mode):
    """h as a ring of Q scheduler rows (Linear-1 of row p waits for the
    Linear-2 tiles of row p - Q): the same bits as with every row in place,
    for the smallest ring the raster group allows and a larger one, with many
    wrap-arounds."""
    need_gpu()
    c = make_case([70, 0, 129, 1, 255, 57, 300, 12] * 8, 256, 384, seed=13)
    base = dict(MODES[mode], group_rows=4)
    _, _, h0, y0 = run_ffn(c, tuning=moe.Tuning(**base))
    # the reference output itself against the oracle (every row)
    href, yref = oracle_rows(c, np.arange(c["R"]))
    assert_close(to_f64(h0), href, f"{mode} h")
    assert_close(to_f64(y0), yref, f"{mode} y")
    group = 4 // MODES[mode]["cta_group"]  # raster group in scheduler rows
    for ring, order in ((3 * group, 0), (13, 0), (3 * group, 2)):
        t = moe.Tuning(**base, h_ring_rows=ring, row_order=order)
        s = moe.Shape(T=c["R"], d=c["d"], E=c["E"], top_k=1, ffn=c["F"])
        ws = moe.alloc_workspace(s, tuning=t)
        assert ws.numel() < moe.workspace_bytes(s)
        _, _, _, y = run_ffn(c, tuning=t, ws=ws)
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16)), ring


def test_h_ring_below_the_deadlock_free_size_is_refused():
    need_gpu()
    c = make_case([300, 200], 256, 256, seed=14)
    s = moe.Shape(T=c["R"], d=c["d"], E=c["E"], top_k=1, ffn=c["F"])
    t = moe.Tuning(h_ring_rows=8)  # default raster group here: 8 pair rows -> needs >= 24
    ws = moe.alloc_workspace(s, tuning=t)
    y = torch.zeros(c["R"], c["d"], dtype=torch.bfloat16, device="cuda")
    off = torch.from_numpy(c["offsets"]).cuda()
    with pytest.raises(moe.MoEError) as e:
        moe.expert_ffn(s, c["x"], off, c["w1"], c["w3"], c["w2"], y, ws, tuning=t)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    assert torch.all(y == 0)


@pytest.mark.parametrize("n2", [64, 128, 192, 256])
def test_ffn_l2_tile_widths(n2):
    need_gpu()
    c = make_case([150, 90], 384, 256, seed=n2)
    _, _, h, y = run_ffn(c, tuning=moe.Tuning(l2_block_n=n2, orientation=moe.ORIENT_TOKENS_M))
    href, yref = oracle_rows(c, np.arange(c["R"]))
    assert_close(to_f64(y), yref, f"N2={n2} y")


@pytest.mark.parametrize("mode", sorted(MODES))
def test_ready_flags_carry_the_call_epoch(mode):
    need_gpu()
    counts = [70, 0, 129, 1, 255]
    c = make_case(counts, 256, 256, seed=4)
    t = moe.Tuning(**MODES[mode])
    cg = MODES[mode]["cta_group"]
    s, ws, _, _ = run_ffn(c, tuning=t)
    tr = TILE_ROWS[mode]
    rows = int(sum((n + tr - 1) // tr for n in counts))  # scheduler rows
    p2 = 256 // L2_COLS[mode]  # d = 256
    nflags = rows * p2 * cg  # one flag per CTA of each Linear-2 tile
    flags = moe.ws_view(ws, s, moe.WS.L2_FLAGS, torch.int32, (nflags,)).cpu().numpy()
    assert flags[0] != 0 and np.all(flags == flags[0])
    done = moe.ws_view(ws, s, moe.WS.L1_DONE, torch.int32, (rows,)).cpu().numpy()
    assert np.all(done == (256 // L1_COLS[mode]) * cg)  # F = 256: Linear-1 tiles per row, one count per CTA
    run_ffn(c, tuning=t, ws=ws)
    flags2 = moe.ws_view(ws, s, moe.WS.L2_FLAGS, torch.int32, (nflags,)).cpu().numpy()
    assert np.all(flags2 == flags2[0]) and flags2[0] != flags[0]


def test_bad_expert_offsets_are_reported_not_computed():
    need_gpu()
    c = make_case([100, 50], 64, 64, seed=5)
    c["offsets"] = np.array([0, 120, 100], np.int32)  # decreasing: invalid
    s = moe.Shape(T=c["R"], d=c["d"], E=c["E"], top_k=1, ffn=c["F"])
    ws = moe.alloc_workspace(s)
    y = torch.full((c["R"], c["d"]), 7.0, dtype=torch.bfloat16, device="cuda")
    moe.expert_ffn(s, c["x"], torch.from_numpy(c["offsets"]).cuda(), c["w1"], c["w3"], c["w2"], y, ws)
    assert moe.last_device_status(ws) == moe.MOE_ERR_INVALID_ARG
    assert torch.all(y == 7.0)  # nothing was written
