"""The plane-aligned windows of the tiled kernel's odd-row NCHW form (2 or 3
channels, binary16 and binary32), checked on the CPU: the index arithmetic of
odd_nchw_window / odd_nchw_chunks / odd_nchw_band in
image_preprocessing_gb300/csrc/fused_norm.cu, restated here, must produce
every element of every plane of a band exactly once, at the tile offset the
band's bulk store expects, from the source byte the operation's definition
names (the pixel itself, or its mirror in the same row when flipped:
FusedNormalization article §五), must zero exactly the elements inside the
erase rectangle in output coordinates (article §十二), and must read shared
memory only inside the stage (or the header or previous stage before it) and
write only inside the plane's tile.

The GPU parity tests then check the bytes themselves against the oracle, and
the checked build (test_bounds_checked.py) guards the same reads and stores
on the device."""
import random

import pytest


def _ru(v, a):
    return (v + a - 1) // a * a


def _band(W, C, R, rows, D, phi0, off_in, flip, y_begin=0, rect=None, header=384, OB=2):
    EPC = 16 // OB                               # elements per 16-byte chunk
    WP = EPC + (C - 1) * D
    GEW = WP * C
    NWW = (GEW + 3) // 4
    WC = W * C
    in_stage = _ru(R * WC + 64, 128)             # the planner's odd-row stage: 64 bytes of slack
    plane = _ru(R * W * OB + 16, 16)             # a plane's tile: the band's elements + 16
    E = rows * W
    wc_inv = ((1 << 32) + WC - 1) // WC
    sh = [OB * ((phi0 + c * D) % EPC) for c in range(C)]   # each plane tile's alignment shift
    kadj = [(phi0 + c * D) // EPC for c in range(C)]
    erow_lo, erow_hi, ecol_lo, ecol_hi = rect if rect else (0, 0, 0, 0)
    band_erased = erow_lo < erow_hi and erow_lo < y_begin + rows and erow_hi > y_begin
    produced = [[0] * E for _ in range(C)]
    ng = (E - 1 + phi0 + (C - 1) * D) // EPC + 1
    for g in range(ng):
        pw = EPC * g - phi0 - (C - 1) * D
        e0 = pw * C
        assert e0 + GEW - 1 > 0
        r1 = split_px = 0
        if flip or band_erased:
            r1 = ((e0 + GEW - 1) * wc_inv) >> 32
            assert r1 == (e0 + GEW - 1) // WC    # the one-multiply division is exact here
            r1 = min(r1, rows - 1)
            split = r1 * WC - e0
            split_px = split // C if split > 0 else 0
        reads = []
        if not flip:
            q = off_in + e0
            reads.append(q - q % 4)
            window = {sb: q + sb for sb in range(GEW)}
        else:
            assert (e0 - r1 * WC) % C == 0       # so C's truncating division is exact
            x0b = (e0 - r1 * WC) // C
            qb = off_in + r1 * WC + C * (W - x0b - WP)
            reads.append(qb - qb % 4)
            window = {sb: qb + sb for sb in range(GEW)}
            if split_px > 0 and r1 > 0:
                qa = qb - WC - C * W
                reads.append(qa - qa % 4)
                for sb in range(C * (WP - split_px), GEW):
                    window[sb] = qa + sb
        for a in reads:   # NWW + 1 aligned words from a
            assert -header <= a and a + 4 * (NWW + 1) <= in_stage, (W, C, R, g, a)
        lo_a = hi_a = lo_b = hi_b = 0
        if band_erased:
            ya, yb = y_begin + r1 - 1, y_begin + r1
            xa = pw - (r1 - 1) * W
            xb = pw - r1 * W
            if split_px > 0 and erow_lo <= ya < erow_hi:
                lo_a, hi_a = max(ecol_lo - xa, 0), min(ecol_hi - xa, split_px)
            if erow_lo <= yb < erow_hi:
                lo_b, hi_b = max(ecol_lo - xb, split_px), min(ecol_hi - xb, WP)
        for c in range(C):
            sc = pw + (C - 1 - c) * D
            if sc + EPC <= 0 or sc >= E:
                continue
            at = 16 * (g - kadj[c])
            assert g >= kadj[c] and 0 <= at and at + 16 <= plane, (W, C, g, c, at)
            assert at == sh[c] + OB * sc           # the chunk starts on the tile's 16-byte frame
            for i in range(EPC):
                j = (C - 1 - c) * D + i
                sb = C * (WP - 1 - j) + c if flip else C * j + c
                e = sc + i
                if 0 <= e < E:
                    r, x = divmod(e, W)
                    xs = W - 1 - x if flip else x
                    assert window[sb] == off_in + r * WC + xs * C + c, (W, C, g, c, i, flip)
                    erased = (lo_a <= j < hi_a) or (lo_b <= j < hi_b)
                    want = erow_lo <= y_begin + r < erow_hi and ecol_lo <= x < ecol_hi
                    assert erased == want, (W, C, g, c, i, rect)
                    produced[c][e] += 1
    assert all(pr == [1] * E for pr in produced)


@pytest.mark.parametrize("OB", [2, 4])
@pytest.mark.parametrize("W,C,D", [(299, 3, 1), (227, 3, 1), (13, 3, 1), (10, 3, 1), (301, 2, 1), (9, 2, 1),
                                   (299, 3, 0), (28, 3, 0), (12, 2, 0), (8, 3, 0), (5, 3, 1), (6, 2, 0)])
def test_plane_windows_cover_every_plane_once_within_bounds(W, C, D, OB):
    EPC = 16 // OB
    if W < EPC + (C - 1) * D:
        pytest.skip("rows shorter than a window take the plane-run stores")
    shapes = ((1, 1), (10, 10), (10, 7)) if W > 100 else ((1, 1), (10, 10), (10, 7), (23, 23))
    for R, rows in shapes:
        for phi0 in range(EPC):
            for off_in in (0, 15) if W > 100 else (0, 5, 15):
                for flip in (False, True):
                    _band(W, C, R, rows, D, phi0, off_in, flip, OB=OB)


@pytest.mark.parametrize("OB", [2, 4])
@pytest.mark.parametrize("W,C,D", [(299, 3, 1), (13, 3, 1), (9, 2, 1), (28, 3, 0)])
def test_plane_windows_zero_the_erased_elements(W, C, D, OB):
    rng = random.Random(20 + W + C + D + OB)
    for _ in range(60):
        R = rng.choice((1, 3, 10))
        rows = rng.randint(1, R)
        y_begin = rng.randint(0, 40)
        y0 = rng.randint(y_begin - 3, y_begin + rows + 2)
        x0 = rng.randint(-2, W)
        rect = (y0, y0 + rng.randint(0, rows + 3), x0, x0 + rng.randint(0, W + 2))
        _band(W, C, R, rows, D, rng.randrange(16 // OB), rng.choice((0, 7, 15)), rng.random() < 0.5, y_begin, rect,
              OB=OB)
