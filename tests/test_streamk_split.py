"""The narrow grouped GEMMs' stream-K split, checked on the host.

The kernel gives CTA b of G the stages [U b / G, U (b + 1) / G) of the
U = tiles x stages-per-tile sequence and finishes a tile split between CTAs
with the last of its parts. These are the same integer formulas, restated,
with the properties the kernel relies on: every stage is taken exactly once,
each CTA's pieces are one contiguous run of tiles, a tile's parts are the
non-empty ranges between the CTA holding its first stage and the one holding
its last, and no CTA needs more than its two partial-sum slots (first tile,
last tile) with no two parts of a tile sharing a slot.
"""
import pytest


def cta_of(U, G, u):
    return ((u + 1) * G + U - 1) // U - 1


def pieces(U, G, NST, b):
    """CTA b's pieces in stage order."""
    u, end = U * b // G, U * (b + 1) // G
    out = []
    while u < end:
        tile = u // NST
        s0 = u - tile * NST
        s1 = min(NST, s0 + (end - u))
        out.append((tile, s0, s1))
        u += s1 - s0
    return out


def kernel_order(U, G, NST, b):
    """The order the kernel visits them: partial first tile, partial last
    tile, then the whole tiles (the same closed forms as the kernel)."""
    ub, ue = U * b // G, U * (b + 1) // G
    f_tile, l_tile = ub // NST, (ue - 1) // NST if ue > 0 else 0
    f_s0, l_s1 = ub - f_tile * NST, ue - l_tile * NST
    f_s1 = l_s1 if l_tile == f_tile else NST
    f_part = ue > ub and (f_s0 != 0 or f_s1 != NST)
    l_part = ue > ub and l_tile != f_tile and l_s1 != NST
    w_first = f_tile + 1 if f_part else f_tile
    w_last = (l_tile - 1 if l_part else l_tile) if ue > ub else -1
    out = []
    if f_part:
        out.append((f_tile, f_s0, f_s1))
    if l_part:
        out.append((l_tile, 0, l_s1))
    out += [(t, 0, NST) for t in range(w_first, w_last + 1)]
    return out


@pytest.mark.parametrize("tiles,NST,G", [(384, 28, 152), (896, 6, 152), (24, 28, 152),
                                         (3, 1, 8), (1, 3, 8), (1, 1, 152), (5472, 28, 152),
                                         (7, 5, 3), (100, 1, 152), (2, 7, 152)])
def test_split_covers_every_stage_once_and_parts_agree(tiles, NST, G):
    U = tiles * NST
    seen = {}
    slot_use = {}
    for b in range(G):
        ps = pieces(U, G, NST, b)
        ko = kernel_order(U, G, NST, b)
        assert sorted(ko) == sorted(ps)
        whole = [p for p in ko if p[1:] == (0, NST)]
        assert ko[len(ko) - len(whole):] == whole   # partial pieces come first
        t_first = (U * b // G) // NST
        for i, (tile, s0, s1) in enumerate(ps):
            assert 0 <= s0 < s1 <= NST
            if 0 < i < len(ps) - 1:
                assert (s0, s1) == (0, NST)        # middle pieces are whole tiles
            for s in range(s0, s1):
                key = (tile, s)
                assert key not in seen
                seen[key] = b
            if i:
                assert tile == ps[i - 1][0] + 1    # a contiguous run of tiles
            whole = s0 == 0 and s1 == NST
            c_first = cta_of(U, G, tile * NST)
            c_last = cta_of(U, G, tile * NST + NST - 1)
            assert whole == (c_first == c_last)
            if not whole:
                slot = 0 if tile == t_first else 1
                assert (b, slot) not in slot_use
                slot_use[(b, slot)] = tile
    assert len(seen) == U
    # each split tile: its parts are exactly the non-empty CTAs in [c_first, c_last],
    # and each reads back from the slot it wrote
    for tile in range(tiles):
        c_first = cta_of(U, G, tile * NST)
        c_last = cta_of(U, G, tile * NST + NST - 1)
        owners = sorted({seen[(tile, s)] for s in range(NST)})
        has_part = [c for c in range(c_first, c_last + 1) if U * (c + 1) // G > U * c // G]
        assert owners == has_part
        if len(owners) > 1:
            for c in owners:
                slot = 0 if tile == (U * c // G) // NST else 1
                assert slot_use[(c, slot)] == tile
