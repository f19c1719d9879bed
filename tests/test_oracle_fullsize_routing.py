"""The routing decision of every full-size workload, on the CPU: how many tokens
would be routed differently by fp64 logits than by the fp32 logits the selection
is decided on, and that each such difference lies within the fp32 rounding
bound of the logits (Cui et al., "Fine-grained Computation-Communication
Overlap ...", section 2.1 step 1: the router selects the top-k experts from a
probability distribution)."""
import pytest

import oracle
import synth
from routing_checks import check_fp64_selection


@pytest.mark.parametrize("name", ["tiny", "mid", "dit", "fine", "coarse"])
def test_fp_sensitive_tokens_are_within_the_fp32_bound(name):
    cfg = synth.CONFIGS[name]
    inp = synth.make_inputs(cfg, seed=0, device="cpu", weights=False)
    b = synth.bf16_bits
    xb, wb = b(inp.x), b(inp.wr)
    bias = None if inp.bias is None else inp.bias.numpy()
    r = oracle.route(xb, wb, bias, cfg.k, keep_logits=True)
    sens = check_fp64_selection(r.idx, xb, wb, r)
    print(f"{name}: {len(sens)} of {cfg.T} tokens fp-sensitive {list(sens[:8])}")
    assert len(sens) <= max(1, cfg.T // 1000)


def test_the_bound_check_rejects_a_wrong_order():
    """A selection that puts a clearly smaller logit first is caught."""
    import numpy as np
    from conftest import f32_to_bf16_bits
    rng = np.random.default_rng(9)
    T, d, E, k = 8, 64, 6, 2
    xb = f32_to_bf16_bits(rng.standard_normal((T, d)))
    wb = f32_to_bf16_bits(rng.standard_normal((E, d)) / 8.0)
    r = oracle.route(xb, wb, None, k, keep_logits=True)
    wrong = r.idx.copy()
    wrong[3] = wrong[3][::-1]           # second choice first
    r.fp_sensitive[:] = True           # look at every token
    check_fp64_selection(r.idx, xb, wb, r)
    with pytest.raises(AssertionError):
        check_fp64_selection(wrong, xb, wb, r)
