"""The argument behind filter-then-verify routing, checked on the CPU.

The layer's router for more than 128 experts computes every logit approximately
on tensor cores, bounds the error of both that sum and the exact sequential fp32
sum by gamma * |x| |w| (gamma = gamma_d(2^-24) + gamma_d(2^-21), Cauchy-Schwarz
for sum |x w|), and sums exactly only the experts whose upper end reaches the
k-th largest lower end. Here the tensor-core sum is modelled pessimistically:
each K = 16 step adds its 16 exact products to the accumulator after truncating
every term toward zero to 24 bits below the largest magnitude among them, then
rounds the result toward zero to fp32. The tests check, on random, tied,
near-tied and wide-range inputs, that the interval holds the exact sequential
sum and that the candidate set holds the exact top k (ties to the lower expert).
"""
import numpy as np
import pytest


def bf16(a):
    """Round float32 values to the nearest bf16 (ties to even), kept as float32."""
    b = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16 << 16
    return b.astype(np.uint32).view(np.float32)


def sequential_sum(x, w):
    """z[t, e] = fp32 sum over i in ascending order of x[t, i] * w[e, i] (each
    bf16 product is exact in fp32, so one rounding per step)."""
    acc = np.zeros((x.shape[0], w.shape[0]), dtype=np.float32)
    for i in range(x.shape[1]):
        acc = (acc + np.outer(x[:, i], w[:, i]).astype(np.float32)).astype(np.float32)
    return acc


def truncate_to(v, ulp):
    return np.trunc(v / ulp) * ulp


def tensor_core_model(x, w, kstep=16):
    """Pessimistic K-step accumulation: per step, every product and the
    accumulator truncated to 24 bits of the step's largest magnitude, summed,
    and the sum truncated to fp32."""
    acc = np.zeros((x.shape[0], w.shape[0]), dtype=np.float64)
    for k0 in range(0, x.shape[1], kstep):
        p = x[:, None, k0:k0 + kstep].astype(np.float64) * w[None, :, k0:k0 + kstep].astype(np.float64)
        big = np.maximum(np.abs(p).max(axis=2), np.abs(acc))
        e = np.floor(np.log2(np.where(big > 0, big, 1.0)))
        ulp = np.ldexp(1.0, (e - 23).astype(np.int64))[..., None]
        s = truncate_to(p, ulp).sum(axis=2) + truncate_to(acc[..., None], ulp)[..., 0]
        # toward zero to fp32
        f = s.astype(np.float32).astype(np.float64)
        over = np.abs(f) > np.abs(s)
        f[over] = np.nextafter(f[over].astype(np.float32), np.float32(0)).astype(np.float64)
        acc = f
    return acc


def gamma(n, u):
    return n * u / (1.0 - n * u)


def candidates(z_tc, xn, wn, d, k):
    b = (gamma(d, 2.0 ** -24) + gamma(d, 2.0 ** -21)) * np.outer(xn, wn)
    lo, hi = z_tc - b, z_tc + b
    tau = -np.sort(-lo, axis=1)[:, k - 1]
    return hi >= tau[:, None], b


def exact_topk(z, k):
    # descending, ties to the lower expert: a stable sort of -z
    return np.argsort(-z.astype(np.float64), axis=1, kind="stable")[:, :k]


def check(x, w, k):
    d = x.shape[1]
    z = sequential_sum(x, w).astype(np.float64)
    z_tc = tensor_core_model(x, w)
    xn = np.sqrt((x.astype(np.float64) ** 2).sum(1))
    wn = np.sqrt((w.astype(np.float64) ** 2).sum(1))
    cand, b = candidates(z_tc, xn, wn, d, k)
    assert np.all(np.abs(z_tc - z) <= b), "the interval misses an exact sum"
    top = exact_topk(z, k)
    assert np.all(np.take_along_axis(cand, top, axis=1)), "a selected expert was filtered out"
    return cand.sum(1)


@pytest.mark.parametrize("T,d,E,k,seed", [(64, 1024, 64, 8, 0), (96, 512, 40, 4, 1), (32, 2048, 128, 2, 2)])
def test_random_rows(T, d, E, k, seed):
    rng = np.random.default_rng(seed)
    x = bf16(rng.standard_normal((T, d)))
    w = bf16(rng.standard_normal((E, d)) / np.sqrt(d))
    n = check(x, w, k)
    assert n.min() >= k and n.mean() < E / 2  # the filter keeps the top k and drops most experts


def test_ties_near_ties_and_wide_range():
    rng = np.random.default_rng(3)
    T, d, E, k = 48, 512, 32, 4
    x = bf16(rng.standard_normal((T, d)))
    w = bf16(rng.standard_normal((E, d)) / np.sqrt(d))
    w[5] = w[3]                                          # an exact tie on every token
    near = w[1].copy().view(np.uint32)
    near[d // 2] += 1 << 16                              # one bf16 ulp in one feature
    w[2] = near.view(np.float32)
    x[:8] = bf16(np.tile(w[1] * 8.0 * np.sqrt(d), (8, 1)))  # tokens that prefer experts 1 and 2
    x[8:12, : d // 4] = bf16(x[8:12, : d // 4] * 2.0 ** 40)  # a wide dynamic range within the row
    x[12:16] = 0.0                                       # every logit zero: all experts tie
    n = check(x, w, k)
    assert np.all(n[12:16] == E)


def test_coherent_truncation_stays_inside_the_interval():
    """All-positive inputs make every truncation of the model fall the same
    way, so its error adds up instead of cancelling: it is then far above the
    sequential sum's own error, and still inside the interval."""
    rng = np.random.default_rng(4)
    d = 2048
    x = bf16(1.0 + rng.random((16, d)))
    w = bf16((1.0 + rng.random((24, d))) / d)
    real = x.astype(np.float64) @ w.astype(np.float64).T
    z = sequential_sum(x, w).astype(np.float64)
    z_tc = tensor_core_model(x, w)
    e_tc = (np.abs(z_tc - real) / real).max()
    e_seq = (np.abs(z - real) / real).max()
    assert e_tc > 5 * e_seq
    assert (np.abs(z_tc - z) / real).max() <= gamma(d, 2.0 ** -24) + gamma(d, 2.0 ** -21)
    check(x, w, 4)
