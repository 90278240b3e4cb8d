"""The CTA-pair kernels' work schedule and automatic tile choice, run on the
host through the library's test hooks (the same code the kernels compile,
built for the host; no GPU needed).

The stream-K tail must hand every K block of every tile to exactly one pair,
cut each tile at most once, pair each "init" unit with the previous pair's
"publish" unit at the same cut, put the publish first and the init last in a
pair's stream-K work, and never give a pair more K blocks than dealing whole
tiles round-robin would.  The automatic choice is pinned on the shapes whose
four schedules were timed on a GB300."""
import ctypes

import pytest

SK_AUTO, SK_OFF, SK_ON = 0, 1, 2
PAIR, WIDE = 1, 5
F16, TF32 = 0, 1


@pytest.fixture(scope="module")
def L():
    import dense_gemm_09_gb300 as dg
    dg.build()
    return dg.lib()


def units(L, tiles, pairs, kb, sk, pair):
    n = L.dgemm_test_pair_units(tiles, pairs, kb, sk, pair, None, 0)
    assert n >= 0
    buf = (ctypes.c_int64 * (5 * max(n, 1)))()
    assert L.dgemm_test_pair_units(tiles, pairs, kb, sk, pair, ctypes.addressof(buf), n) == n
    return [tuple(buf[5 * i:5 * i + 5]) for i in range(n)]


def check_schedule(L, tiles, pairs, kb, sk):
    owner = {}
    published = {}
    per_pair = []
    for c in range(pairs):
        us = units(L, tiles, pairs, kb, sk, c)
        cut = [u for u in us if u[0] < sk]
        for i, (t, k0, k1, init, pub) in enumerate(us):
            assert 0 <= t < tiles and 0 <= k0 < k1 <= kb
            assert init == (k0 > 0) and pub == (k1 < kb)
            if init:
                assert t < sk and i == len(cut) - 1, "init is the last stream-K unit"
                assert published.get(c - 1) == (t, k0), "the previous pair published this cut"
            if pub:
                assert t < sk and i == 0, "publish is the first unit"
                published[c] = (t, k1)
            for k in range(k0, k1):
                assert (t, k) not in owner, "K block handed out twice"
                owner[(t, k)] = c
        per_pair.append(sum(u[2] - u[1] for u in us))
    assert len(owner) == tiles * kb, "every K block of every tile is handed out"
    return max(per_pair)


@pytest.mark.parametrize("pairs", [2, 3, 38, 76])
@pytest.mark.parametrize("kb", [1, 2, 7, 64])
def test_schedule_covers_and_pairs(L, pairs, kb):
    for tiles in list(range(1, 3 * pairs + 3)) + [5 * pairs + 1, 7 * pairs - 1]:
        rr = check_schedule(L, tiles, pairs, kb, 0)
        assert rr == -(-tiles // pairs) * kb  # round-robin: ceil(T / P) whole tiles
        sk = L.dgemm_test_stream_k_tiles(tiles, pairs, kb, 1, SK_ON)
        if tiles <= pairs:
            assert sk == 0
            continue
        assert sk == pairs + tiles % pairs
        worst = check_schedule(L, tiles, pairs, kb, sk)
        assert worst <= rr
        # the busiest pair carries its share of the cut tiles, rounded up
        assert worst <= (tiles // pairs - 1) * kb + -(-sk * kb // pairs)


def test_headline_schedule(L):
    """8192 x 8192 x 4096 FP16 on 76 pairs: 1024 tiles of 256 x 256, 64 K blocks."""
    sk = L.dgemm_test_stream_k_tiles(1024, 76, 64, 1, SK_AUTO)
    assert sk == 76 + 1024 % 76
    assert check_schedule(L, 1024, 76, 64, sk) < 14 * 64  # round-robin needs 14 whole tiles


def test_stream_k_rule(L):
    # automatic: only when the last round's idle share is worth ~8 us
    assert L.dgemm_test_stream_k_tiles(152, 76, 64, 1, SK_AUTO) == 0     # divides evenly
    assert L.dgemm_test_stream_k_tiles(77, 76, 4, 1, SK_AUTO) == 0       # too little to save
    assert L.dgemm_test_stream_k_tiles(128, 76, 64, 2, SK_AUTO) == 128   # 4096^3, wide tiles
    assert L.dgemm_test_stream_k_tiles(76, 76, 64, 1, SK_ON) == 0        # no more tiles than pairs
    assert L.dgemm_test_stream_k_tiles(100, 76, 64, 1, SK_OFF) == 0
    assert L.dgemm_test_stream_k_tiles(100, 76, 64, 3, SK_ON) == -1
    assert L.dgemm_test_pair_units(100, 76, 64, 50, 0, None, 0) == -1   # region smaller than the pairs
    assert L.dgemm_test_pair_units(100, 76, 64, 0, 76, None, 0) == -1   # no such pair


# (kind, M, N, K) -> (variant, stream-K mode): the fastest of the four pair
# schedules in the GB300 timings of the tuning tool
CHOICES = [
    (F16, 8192, 8192, 4096, PAIR, SK_ON),
    (F16, 4096, 4096, 4096, PAIR, SK_ON),
    (F16, 12288, 12288, 12288, WIDE, SK_ON),
    (F16, 16384, 16384, 16384, WIDE, SK_OFF),
    (F16, 8192, 8448, 4096, PAIR, SK_OFF),
    (F16, 2048, 2048, 2048, PAIR, SK_OFF),
    (TF32, 8192, 8192, 4096, WIDE, SK_OFF),
    (TF32, 4096, 4096, 4096, PAIR, SK_ON),
    (TF32, 12288, 12288, 4096, WIDE, SK_ON),
]


@pytest.mark.parametrize("kind,M,N,K,variant,mode", CHOICES)
def test_automatic_choice(L, kind, M, N, K, variant, mode):
    v, bn, sp = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    assert L.dgemm_test_choose_config(kind, M, N, K, 152, ctypes.byref(v), ctypes.byref(bn), ctypes.byref(sp)) == 0
    assert (v.value, bn.value, sp.value) == (variant, 256, mode)


def test_choose_config_validates(L):
    v = ctypes.c_int()
    assert L.dgemm_test_choose_config(7, 256, 256, 256, 152, ctypes.byref(v), ctypes.byref(v), ctypes.byref(v)) == 1
    assert L.dgemm_test_choose_config(0, 0, 256, 256, 152, ctypes.byref(v), ctypes.byref(v), ctypes.byref(v)) == 1
    assert L.dgemm_test_choose_config(0, 256, 256, 256, 152, None, ctypes.byref(v), ctypes.byref(v)) == 1
