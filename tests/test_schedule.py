"""The tc GEMM's schedule (host arithmetic, no GPU): the tile width, the cut of
the last partial wave and its split along K.  The work each CTA does is
rebuilt here from the schedule's description (the uncut tiles round robin; a
cut piece p in two parts, stages [0, split_kh) first on CTA p, the rest last
on CTA split_p + p) and checked to cover every (weight-row tile, token) pair
and every K stage exactly once, with each piece's second part after its
first."""
import numpy as np
import pytest

SHAPES = [(512, 5120, 5120), (512, 34816, 5120), (512, 5120, 17408), (1024, 5120, 5120),
          (1024, 34816, 5120), (1024, 5120, 17408), (64, 20480, 256), (48, 20480, 384),
          (64, 256, 512), (8192, 5120, 5120), (1, 16, 128), (300, 1024, 1024), (513, 5120, 5120)]


@pytest.fixture(scope="module")
def h32():
    import hadamard_rotated_bit_gb300 as m
    try:
        m.lib()
    except ImportError as e:
        pytest.skip(str(e))
    return m


def _pieces(M, N, sch):
    """(token start, token count, weight-row tile) of each work unit."""
    bn, k, tf, total = sch["bn"], sch["tail_k"], sch["tail_first"], sch["total"]
    chunks = (M + bn - 1) // bn

    def tile(t):
        wt, ch = divmod(t, chunks)
        g0 = ch * bn
        return g0, min(bn, M - g0), wt

    units = []
    for t in range(total):
        if t < tf:
            units.append(tile(t))
        else:
            p = t - tf
            g0, chi, wt = tile(tf + p // k)
            sub = p % k
            pw = ((chi + k - 1) // k + 15) // 16 * 16
            w = max(0, min(pw, chi - sub * pw))
            units.append((g0 + sub * pw, w, wt))
    return units


def _cover(M, N, K, sms, sch):
    nst = K // 128
    units = _pieces(M, N, sch)
    tf, grid, P, kh = sch["tail_first"], sch["grid"], sch["split_p"], sch["split_kh"]
    seen = {}   # (wt, token) -> list of (stage range, cta, position)
    for c in range(grid):
        items = []
        if P and c < P:
            items.append((tf + c, 0, kh))
        for t in range(c, tf if P else sch["total"], grid):
            items.append((t, 0, nst))
        if P and P <= c < 2 * P:
            items.append((tf + c - P, kh, nst))
        for pos, (u, s0, s1) in enumerate(items):
            g0, w, wt = units[u]
            for tok in range(g0, g0 + w):
                seen.setdefault((wt, tok), []).append((s0, s1, c, pos, len(items)))
    nt = (N + 127) // 128
    assert set(seen) == {(wt, tok) for wt in range(nt) for tok in range(M)}
    for key, parts in seen.items():
        parts.sort()
        assert parts[0][0] == 0 and parts[-1][1] == nst, key
        for a, b in zip(parts, parts[1:]):
            assert a[1] == b[0], key              # K stages continue, none twice
        if len(parts) == 2:                       # a split piece: first part first on
            (_, _, c1, pos1, _), (_, _, c2, pos2, n2) = parts   # its CTA, second last
            assert c1 != c2 and pos1 == 0 and pos2 == n2 - 1 and pos2 >= 1, key
        else:
            assert len(parts) == 1, key


@pytest.mark.parametrize("sms", [152, 148, 132, 160, 8])
def test_schedule_covers_every_output_once(h32, sms):
    for M, N, K in SHAPES:
        for ws in (False, True):
            sch = h32.h32_gemm_tc_schedule(M, N, K, sms, ws)
            assert sch["grid"] <= sms and sch["grid"] <= sch["total"]
            if not ws:
                assert sch["split_p"] == 0 and sch["ws_bytes"] == 0
            if sch["split_p"]:
                P = sch["split_p"]
                assert 2 * P <= sch["grid"] <= sch["tail_first"]
                assert P == sch["total"] - sch["tail_first"] and 1 <= sch["split_kh"] < K // 128
                assert sch["ws_bytes"] == 256 + 128 * 16 * 8 + P * 128 * sch["ws_ld"] * 4
            _cover(M, N, K, sms, sch)


def test_chain_projections_split_on_152_sms(h32):
    """The pp512 projections: attention and FFN down (160 tiles: 8 over a full
    wave) split 64 pieces of 16 tokens at half of K; gate/up (1088 tiles: 24
    over seven waves) keeps the cut without the split, whose simulated gain (3%)
    is below the 5% the split must show.  At 1024 tokens attention and FFN down
    split 64 pieces of 32 tokens."""
    att = h32.h32_gemm_tc_schedule(512, 5120, 5120, 152, True)
    down = h32.h32_gemm_tc_schedule(512, 5120, 17408, 152, True)
    gu = h32.h32_gemm_tc_schedule(512, 34816, 5120, 152, True)
    assert (att["split_p"], att["ws_ld"], att["split_kh"]) == (64, 16, 20)
    assert (down["split_p"], down["ws_ld"], down["split_kh"]) == (64, 16, 68)
    assert (gu["split_p"], gu["tail_k"]) == (0, 4)
    for K in (5120, 17408):
        long = h32.h32_gemm_tc_schedule(1024, 5120, K, 152, True)
        assert (long["split_p"], long["ws_ld"]) == (64, 32)
    # tiny shapes never fill a wave: nothing to split
    assert h32.h32_gemm_tc_schedule(64, 256, 512, 152, True)["split_p"] == 0


def test_schedule_rejects_bad_shapes(h32):
    for M, N, K, sms in [(0, 16, 128, 152), (4, 15, 128, 152), (4, 16, 100, 152),
                         (4, 16, 128, 0)]:
        with pytest.raises(h32.H32Error):
            h32.h32_gemm_tc_schedule(M, N, K, sms, True)
