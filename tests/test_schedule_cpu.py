"""The persistent GEMM kernel's work split, restated on the host: whole tiles
round-robin over the grid, then the remaining tiles' K-tiles split evenly
over min(grid, units) CTAs (with splitting turned off, over as many CTAs as
there are remaining tiles, one tile each).  Checks that every (tile, k-tile) unit is owned by
exactly one CTA, that the CTAs sharing a split tile are exactly the
contiguous range the kernel's reducer sums over, and that the partial-tile
slots (two per CTA) never collide."""

import itertools

import pytest


def schedule(T, KT, G, whole=False, cap=0):
    W = T // G
    if whole:
        cap = 1
    if cap == 0 and W > 0 and T % G:
        W -= 1          # stream-K over the last two waves
    U = (T - W * G) * KT
    Gs = U if U < G else G
    if cap and U:
        r = U // KT
        Gs = min(Gs, r * min(cap, G // r))

    def sk_begin(c):
        return (c * U) // Gs

    def cta_of_unit(u):
        return ((u + 1) * Gs - 1) // U

    owner, slots, items_of = {}, set(), {}
    for c in range(G):
        items = [(c + it * G, 0, KT) for it in range(W)]
        if c < Gs and U > 0:
            u, ue = sk_begin(c), sk_begin(c + 1)
            assert ue > u, "a CTA of the split owns no unit"
            while u < ue:
                tl, k0 = divmod(u, KT)
                se = min((tl + 1) * KT, ue)
                items.append((W * G + tl, k0, k0 + se - u))
                u = se
        items_of[c] = items
        for t, k0, k1 in items:
            for k in range(k0, k1):
                assert (t, k) not in owner
                owner[(t, k)] = c
            if not (k0 == 0 and k1 == KT):
                us = (t - W * G) * KT
                which = 0 if sk_begin(c) >= us else 1
                assert (c, which) not in slots
                slots.add((c, which))
    return W, cta_of_unit, owner, items_of


@pytest.mark.parametrize("T,KT,G", list(itertools.product(
    [1, 2, 3, 8, 32, 149, 150, 256, 300, 4096], [1, 2, 3, 32, 64], [1, 7, 37, 148])))
def test_schedule_partition(T, KT, G):
    W, cta_of_unit, owner, _ = schedule(T, KT, G)
    assert len(owner) == T * KT
    for t in range(W * G, T):
        us = (t - W * G) * KT
        owners = {owner[(t, k)] for k in range(KT)}
        if len(owners) > 1:
            assert owners == set(range(cta_of_unit(us), cta_of_unit(us + KT - 1) + 1))


@pytest.mark.parametrize("T,KT,G", list(itertools.product(
    [1, 3, 149, 150, 300, 4096], [1, 3, 32], [1, 7, 148])))
def test_two_wave_stream_k_has_two_contributors_per_split_tile(T, KT, G):
    """With at least one whole wave and tiles left over, the stream-K region
    spans more than G tiles, so every split tile has exactly two contributors
    and the later one meets it as its first item."""
    W, cta_of_unit, owner, items_of = schedule(T, KT, G)
    if T // G == 0 or T % G == 0 or KT == 1:
        return
    for t in range(W * G, T):
        owners = sorted({owner[(t, k)] for k in range(KT)})
        assert len(owners) <= 2
        if len(owners) == 2:
            later = owners[1]
            first_split = next(it for it in items_of[later] if not (it[1] == 0 and it[2] == KT))
            assert first_split[0] == t


@pytest.mark.parametrize("T,KT,G", list(itertools.product(
    [1, 3, 149, 150, 300, 4096], [1, 3, 32], [1, 7, 148])))
def test_schedule_whole_tiles_never_split(T, KT, G):
    _, _, owner, items_of = schedule(T, KT, G, whole=True)
    assert len(owner) == T * KT
    items = [it for its in items_of.values() for it in its]
    assert all(k0 == 0 and k1 == KT for _, k0, k1 in items)
    assert sorted(t for t, _, _ in items) == list(range(T))


@pytest.mark.parametrize("T,KT,G,cap", list(itertools.product(
    [1, 3, 64, 149, 256, 300], [1, 3, 32, 64], [7, 148], [2, 3, 4, 64])))
def test_schedule_split_cap(T, KT, G, cap):
    """With a cap, every leftover tile is shared by exactly min(cap, G/r, KT)
    CTAs (r leftover tiles)."""
    W, _, owner, _ = schedule(T, KT, G, cap=cap)
    assert len(owner) == T * KT
    r = T - W * G
    for t in range(W * G, T):
        owners = {owner[(t, k)] for k in range(KT)}
        assert len(owners) == min(cap, G // r, KT)


def _fastdiv(d):
    """Divider constants for division by an invariant d (Granlund and
    Montgomery 1994): s = ceil(log2 d), m = floor(2^32 (2^s - d) / d) + 1."""
    s = 0
    while (1 << s) < d:
        s += 1
    return ((1 << 32) * ((1 << s) - d)) // d + 1, s


def test_fastdiv_constants_fit_and_divide_exactly():
    """The multiply-high division the kernel's schedule uses equals integer
    division for every dividend below 2^31 (checked at the edges, at
    multiples of the divisor and on random dividends)."""
    import random
    rnd = random.Random(5)
    divisors = list(range(1, 300)) + [2 ** k for k in range(1, 31)] + \
        [2 ** k + 1 for k in range(1, 30)] + [2 ** k - 1 for k in range(2, 31)] + \
        [rnd.randrange(1, 2 ** 31) for _ in range(200)]
    for d in divisors:
        m, s = _fastdiv(d)
        assert 0 <= m < 2 ** 32
        ns = {0, 1, d - 1, d, d + 1, 2 ** 31 - 1, 2 ** 31 - 2}
        ns |= {q * d + r for q in (1, 2, 7, (2 ** 31 - 1) // d) for r in (0, d - 1) if q * d + r < 2 ** 31}
        ns |= {rnd.randrange(0, 2 ** 31) for _ in range(50)}
        for n in ns:
            if 0 <= n < 2 ** 31:
                hi = (n * m) >> 32
                assert hi + n < 2 ** 32
                assert (hi + n) >> s == n // d, (d, n)
