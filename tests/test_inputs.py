"""The seeded input module shared by the tests and the benchmark (CPU only):
the same seed gives the same inputs, and the large-shape tile sample holds
every ragged edge tile."""
import numpy as np

import qk_inputs as qi


def test_generators_are_deterministic():
    a = qi.int8_problem(37, 24, 64, seed=3, bias=True)
    b = qi.int8_problem(37, 24, 64, seed=3, bias=True)
    for x, y in ((a.A, b.A), (a.B, b.B), (a.sa, b.sa), (a.sb, b.sb), (a.bias, b.bias)):
        assert np.array_equal(x, y)
    c = qi.mx_problem(qi.FMT_MXFP8_E4M3, 9, 32, 96, seed=1)
    d = qi.mx_problem(qi.FMT_MXFP8_E4M3, 9, 32, 96, seed=1)
    assert np.array_equal(c.A, d.A) and np.array_equal(c.sB, d.sB)
    e = qi.int8_problem(37, 24, 64, seed=4)
    assert not np.array_equal(a.A, e.A)


def _check_tiles(M, N, tiles, tile=128):
    assert tiles == sorted(set(tiles))                       # sorted, no duplicates
    for (m0, m1, n0, n1) in tiles:
        assert m0 % tile == 0 and n0 % tile == 0
        assert 0 <= m0 < m1 <= M and 0 <= n0 < n1 <= N
        assert m1 - m0 == min(tile, M - m0) and n1 - n0 == min(tile, N - n0)


def test_sample_tiles_hold_every_ragged_edge_tile():
    for M, N in ((30000, 21504), (64, 21504), (129, 264), (300, 520), (1, 8), (16384, 7168)):
        tiles = qi.sample_tiles(M, N, 12, 5)
        _check_tiles(M, N, tiles)
        assert tiles == qi.sample_tiles(M, N, 12, 5)         # seeded
        mt, nt = -(-M // 128), -(-N // 128)
        got = {(m0 // 128, n0 // 128) for (m0, _, n0, _) in tiles}
        assert (0, 0) in got and (mt - 1, nt - 1) in got
        if M % 128:
            assert all((mt - 1, bn) in got for bn in range(nt))
        else:
            assert any(bm == mt - 1 for bm, _ in got)
        if N % 128:
            assert all((bm, nt - 1) in got for bm in range(mt))
        else:
            assert any(bn == nt - 1 for _, bn in got)
