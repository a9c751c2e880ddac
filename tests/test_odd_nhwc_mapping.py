"""The tile-aligned groups of the tiled kernel's odd-row NHWC form (1 or 3
channels), checked on the CPU: the index arithmetic of odd_nhwc_group /
odd_nhwc_band in image_preprocessing_gb300/csrc/fused_norm.cu, restated here,
must produce every output element of a band exactly once, at the tile offset
the band's bulk store expects, from the source byte the operation's definition
names (the pixel itself, or its mirror in the same row when flipped:
FusedNormalization article §五), and must read shared memory only inside the
stage (or the bytes before it: the header or the previous stage) and write
only inside the output tile.

This is the emulation the kernel's index arithmetic was checked with before
and after its GPU runs; the GPU parity tests then check the bytes themselves
against the oracle, and the checked build (test_bounds_checked.py) guards the
same reads and stores on the device."""
import pytest


def _ru(v, a):
    return (v + a - 1) // a * a


def _band(W, C, R, rows, OB, sh, off_in, flip, header=384):
    P = 8 if C == 3 else 16 // C
    GE, EPC, WC, NW = P * C, 16 // OB, W * C, (P * C) // 4
    in_stage = _ru(R * WC + 64, 128)              # the planner's odd-row stage: 64 bytes of slack
    out_stage = _ru(R * WC * OB + 32, 128)        # and 32 bytes of tile slack
    E = rows * WC
    phi = (sh // OB) % EPC
    psi = phi
    while psi % C:
        psi += EPC
    assert psi < GE and psi % C == 0 and psi % EPC == phi
    tile0 = sh - psi * OB
    wc_inv = ((1 << 32) + WC - 1) // WC
    produced = [0] * E
    for g in range((E + psi + GE - 1) // GE):
        e0 = g * GE - psi
        r1 = ((e0 + GE - 1) * wc_inv) >> 32
        assert r1 == (e0 + GE - 1) // WC          # the one-multiply division is exact here
        r1 = min(r1, rows - 1)
        split = r1 * WC - e0
        split_px = split // C if split > 0 else 0
        window = {}
        reads = []
        if not flip:
            q = off_in + e0
            reads.append(q - q % 4)
            window = {sb: q + sb for sb in range(GE)}
        else:
            x0b = (e0 - r1 * WC) // C
            qb = off_in + r1 * WC + C * (W - x0b - P)
            reads.append(qb - qb % 4)
            window = {sb: qb + sb for sb in range(GE)}
            if split_px > 0 and r1 > 0:
                qa = qb - WC - C * W
                reads.append(qa - qa % 4)
                for sb in range(C * (P - split_px), GE):
                    window[sb] = qa + sb
        for a in reads:   # NW + 1 aligned words from a
            assert -header <= a and a + 4 * (NW + 1) <= in_stage, (W, C, R, g, a)
        for k in range(GE):
            i, c = divmod(k, C)
            sb = C * (P - 1 - i) + c if flip else k
            e = e0 + k
            if 0 <= e < E:
                r, w = divmod(e, WC)
                x = w // C
                xs = W - 1 - x if flip else x
                assert window[sb] == off_in + r * WC + xs * C + c, (W, C, g, k, flip)
                assert tile0 + (g * GE + k) * OB == sh + e * OB
                produced[e] += 1
        for qc in range(GE * OB // 16):
            if e0 + qc * EPC >= E:
                break
            if e0 + (qc + 1) * EPC <= 0:
                continue
            t = tile0 + g * GE * OB + 16 * qc
            assert t % 16 == 0 and 0 <= t and t + 16 <= out_stage, (W, C, g, qc, t)
    assert produced == [1] * E


@pytest.mark.parametrize("W,C", [(299, 3), (227, 3), (28, 3), (13, 3), (299, 1), (28, 1), (17, 1)])
@pytest.mark.parametrize("OB", [2, 4])
def test_tile_aligned_groups_cover_the_band_once_within_bounds(W, C, OB):
    for R, rows in ((1, 1), (10, 10), (10, 7), (28, 28)):
        for sh in range(0, 16, OB):
            for off_in in (0, 3, 9, 15):
                for flip in (False, True):
                    _band(W, C, R, rows, OB, sh, off_in, flip)
