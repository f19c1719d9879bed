"""The grouped GEMM's tile order (Xian et al., "X-Stage ...", section 4.2,
Algorithm 1, taken as one sequence whose tiles the CTAs claim by ticket), on
the CPU: the closed-form ticket decode the kernel uses reproduces the
step-by-step merge of the Linear-1 and Linear-2 tile streams, and every wait a
tile can make (Linear-2 on its row's Linear-1 tiles; with an h ring of
Q >= D + 2 * group rows, Linear-1 of row p on the Linear-2 tiles of row p - Q)
is on a tile with a smaller ticket, which is what makes the waits
deadlock-free. A restatement of the kernel's formulas (TileSource,
stream_tile, group_of_row in grouped_gemm.cu), checked against brute force."""
import random


def layout(rows_per_expert, GM, mixed):
    row_start = [0]
    for n in rows_per_expert:
        row_start.append(row_start[-1] + n)
    return dict(E=len(rows_per_expert), row_start=row_start, P=row_start[-1], GM=GM, mixed=mixed)


def group_of_row(c, m):
    GM = c["GM"]
    if c["mixed"]:  # raster groups over the global row sequence
        g0 = m - m % GM
        return g0, min(GM, c["P"] - g0)
    rs = c["row_start"]
    e = max(i for i in range(c["E"]) if rs[i] <= m)  # experts without rows share row_start
    g0 = m - (m - rs[e]) % GM
    return g0, min(GM, rs[e + 1] - g0)


def stream_tile(c, k, Pn):
    g0, gs = group_of_row(c, k // Pn)
    i = k - g0 * Pn
    return g0 + i % gs, i // gs  # (row, n)


def stream_in_order(c, Pn):
    """Brute force: per expert (or over all rows), groups of GM rows, N-tile-major."""
    out = []
    rs, GM = c["row_start"], c["GM"]
    spans = [(0, c["P"])] if c["mixed"] else [(rs[e], rs[e + 1]) for e in range(c["E"])]
    for r0, r1 in spans:
        g = r0
        while g < r1:
            gs = min(GM, r1 - g)
            out += [(r, n) for n in range(Pn) for r in range(g, g + gs)]
            g += gs
    return out


def merge(c, P1, P2, D):
    """Brute force: one cursor pair walking both streams with step 1; the
    Linear-2 tile goes out once the largest row seen so far in its stream plus
    D is at most the Linear-1 cursor's row."""
    s1, s2 = stream_in_order(c, P1), stream_in_order(c, P2)
    k1 = k2 = 0
    out, maxrow = [], -1
    while k1 < len(s1) or k2 < len(s2):
        p1 = k1 // P1 if k1 < len(s1) else 1 << 30
        if k2 < len(s2) and max(maxrow, s2[k2][0]) + D <= p1:
            maxrow = max(maxrow, s2[k2][0])
            out.append((1,) + s2[k2])
            k2 += 1
        else:
            out.append((0,) + s1[k1])
            k1 += 1
    return out


def decode(c, P1, P2, D, q):
    """The kernel's decode: segment b holds the Linear-2 tiles with key b, then
    the P1 Linear-1 tiles of row block b; S(b) = b*P1 + C(b - D - 1)."""
    P = c["P"]
    tot1, tot2 = P * P1, P * P2

    def C(m):  # Linear-2 positions whose largest row so far is <= m
        if m < 0:
            return 0
        if m >= P - 1:
            return tot2
        g0, gs = group_of_row(c, m)
        return g0 * P2 + (m - g0 + 1) if m < g0 + gs - 1 else (g0 + gs) * P2

    if q >= tot1 + tot2:
        return None
    lo, hi = 0, P
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if mid * P1 + C(mid - D - 1) <= q:
            lo = mid
        else:
            hi = mid - 1
    b = lo
    c0 = C(b - D - 1)
    n2 = (C(b - D) if b < P else tot2) - c0
    off = q - (b * P1 + c0)
    if off < n2:
        return (1,) + stream_tile(c, c0 + off, P2)
    return (0,) + stream_tile(c, b * P1 + (off - n2), P1)


def random_case(rng):
    E = rng.randint(1, 12)
    rpe = [rng.choice([0, 1, 1, 2, 3, 5, 9, 17]) for _ in range(E)]
    if sum(rpe) == 0:
        rpe[0] = 1
    GM = rng.choice([1, 2, 3, 4, 8])
    return layout(rpe, GM, rng.random() < 0.3), rng.randint(1, 5), rng.randint(1, 5), GM + rng.randint(0, 6)


def test_decode_reproduces_the_merge():
    rng = random.Random(1)
    for _ in range(400):
        c, P1, P2, D = random_case(rng)
        ref = merge(c, P1, P2, D)
        assert [decode(c, P1, P2, D, q) for q in range(len(ref))] == ref
        assert decode(c, P1, P2, D, len(ref)) is None
        assert all(stream_tile(c, k, P1) == t for k, t in enumerate(stream_in_order(c, P1)))


def test_every_wait_is_on_a_smaller_ticket():
    rng = random.Random(2)
    for _ in range(400):
        c, P1, P2, D = random_case(rng)
        order = merge(c, P1, P2, D)
        pos = {t: i for i, t in enumerate(order)}
        Q = D + 2 * c["GM"]  # the smallest ring the kernel accepts for this lead
        for t, i in pos.items():
            if t[0] == 1:  # Linear-2 tile: every Linear-1 tile of its row
                assert all(pos[(0, t[1], n)] < i for n in range(P1))
            elif t[1] >= Q:  # ring: the slot's previous row fully read
                assert all(pos[(1, t[1] - Q, n)] < i for n in range(P2))


def test_a_smaller_ring_can_wait_on_a_later_tile():
    """Q = D + group + 1 (the rule of an earlier build) is not enough once a
    raster group's later passes wait for its last row."""
    rng = random.Random(3)
    violated = 0
    for _ in range(200):
        c, P1, P2, D = random_case(rng)
        if c["GM"] < 2 or P2 < 2:
            continue
        order = merge(c, P1, P2, c["GM"])
        pos = {t: i for i, t in enumerate(order)}
        Q = 2 * c["GM"] + 1
        violated += any(t[0] == 0 and t[1] >= Q and not all(pos[(1, t[1] - Q, n)] < i for n in range(P2))
                        for t, i in pos.items())
    assert violated > 0
