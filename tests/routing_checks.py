"""Checks on the routing decision shared by the CPU and GPU tests.

The selection is decided on fp32 logits summed in ascending feature order (the
kernel's precision). A token whose top-k would come out differently from fp64
logits is "fp-sensitive"; on such a token the fp32 choice must still be a valid
descending selection of the fp64 logits once the fp32 rounding is allowed for:
|z32 - z64| <= gamma_d * sum_i |x_i w_i| + 2u |z| (forward error bound of
recursive summation, u = 2^-24, gamma_d = d u / (1 - d u), plus the bias add)."""
import numpy as np

from conftest import bf16_bits_to_f64


def fp32_error_bound(x_row_bits, wr_bits, z64_row):
    u = 2.0 ** -24
    d = x_row_bits.shape[0]
    gam = d * u / (1 - d * u)
    x = np.abs(bf16_bits_to_f64(x_row_bits))
    w = np.abs(bf16_bits_to_f64(wr_bits))
    return gam * (w @ x) + 2 * u * (np.abs(z64_row) + 1e-30)


def check_fp64_selection(idx, x_bits, wr_bits, route):
    """idx: [T,k] selection to check (the GPU's, or the oracle's own); route: an
    oracle.Route with fp64 logits (keep_logits=True). Returns the fp-sensitive
    token ids after asserting that on each of them every step of the selection
    picks an expert whose fp64 logit is within the combined fp32 error bounds of
    the largest one still available."""
    sens = np.nonzero(route.fp_sensitive)[0]
    E = wr_bits.shape[0]
    for t in sens:
        z = route.z64[t]
        bound = fp32_error_bound(x_bits[t], wr_bits, z)
        avail = np.ones(E, bool)
        for a in idx[t]:
            others = np.nonzero(avail)[0]
            worst = np.max(z[others] - z[a] - bound[a] - bound[others])
            assert worst <= 0.0, f"token {t}: choice {a} trails an available expert by more than the fp32 bound"
            avail[a] = False
    return sens
