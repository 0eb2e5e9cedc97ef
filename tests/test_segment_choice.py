"""The automatic segment length of the split prefill (kda_auto_segment_tokens,
host only): no split when the (sequence, head) chains fill the GPU, the
wave-filling lengths on the long-context shapes (uniform and packed batches),
and the documented limits."""
import pytest

from gated_delta_rule_48_gb300 import binding as kb

SMS = 152


@pytest.fixture(scope="module")
def choose():
    kb.build()
    return lambda T, N, H, sms, uniform=True: kb.kda_auto_segment_tokens(T, N, H, sms, uniform)


def test_enough_chains_means_no_split(choose):
    assert choose(4 * 4096, 4, 32, SMS) == -1          # 128 chains, 64 chunks each
    assert choose(152 * 65536, 152, 1, SMS) == -1      # one chain per SM
    assert choose(1 << 20, 1, 200, SMS) == -1          # more chains than SMs


def test_long_context_shapes(choose):
    # uniform 1 x 65,536 tokens, H16: 10 segments, 144 units in each pass (16
    # replays of segment 0 + 128 summaries, then 144 replays), one wave each;
    # 105 chunks leave a 79-chunk last segment, about as long as a 105-chunk
    # replay that loads its T records (0.77 x 105 = 80.9)
    assert choose(65536, 1, 16, SMS) == 105 * 64
    # uniform 8 x 131,072 tokens, H8: 3 segments, one wave per pass; 739
    # chunks leave a last segment of 570 (0.77 x 739 = 569.0)
    assert choose(8 * 131072, 8, 8, SMS) == 739 * 64
    # packed, the same totals: the second pass counted as 8 H s units, so 7
    # segments of 293 chunks (three waves per pass)
    assert choose(8 * 131072, 8, 8, SMS, False) == 293 * 64


def test_lengths_are_whole_chunks_and_at_least_four(choose):
    for T, N, H in ((65536, 1, 16), (8 * 131072, 8, 8), (3 * 50000 + 1, 3, 4),
                    (1 << 22, 2, 2), (4096, 1, 1)):
        L = choose(T, N, H, SMS)
        if L != -1:
            assert L % 64 == 0 and L >= 4 * 64
            assert L < (T + N - 1) // N  # a split cuts every sequence


def test_short_sequences_are_not_split(choose):
    assert choose(256, 1, 1, SMS) == -1   # 4 chunks: no two segments of 4
    assert choose(0, 1, 1, SMS) == -1


def test_huge_sequences_choose_quickly(choose):
    import time
    t = time.perf_counter()
    L = choose(1 << 40, 1, 1, SMS)  # 2^34 chunks: the candidate count is bounded
    assert time.perf_counter() - t < 0.1
    assert L % 64 == 0 and -(-(1 << 40) // L) <= 8 * SMS


def test_invalid_sizes(choose):
    for args in ((-1, 1, 1, SMS), (4096, 0, 1, SMS), (4096, 1, 0, SMS), (4096, 1, 1, 0)):
        assert choose(*args) == -1


def modelled(T, N, H, sms, L, uniform):
    """Chunk-times x 100 of the split passes as kda.h documents them (L in
    chunks, None = no split)."""
    chains, n = N * H, -(-(-(-T // N)) // 64)
    waves = lambda u: -(-u // sms)
    if L is None:
        return waves(chains) * (n + 2) * 100
    segs = -(-n // L)
    last = n - (segs - 1) * L
    w1 = waves(chains * (segs - 1))
    first = w1 * (L + 2) * 100
    if uniform:  # segments 1 .. segs-2 load their T records (0.77 of a chunk-time each)
        second = w1 * (max(77 * L if segs > 2 else 0, 100 * last) + 200)
    else:
        second = waves(chains * segs) * (L + 2) * 100
    return first + second + segs * 100


@pytest.mark.parametrize("uniform", [True, False])
@pytest.mark.parametrize("T,N,H,sms", [(65536, 1, 16, 152), (8 * 131072, 8, 8, 152),
                                       (65536, 1, 16, 76), (3 * 40000, 3, 5, 152),
                                       (1 << 21, 1, 1, 152), (1 << 20, 2, 24, 152)])
def test_choice_minimises_the_documented_model(choose, T, N, H, sms, uniform):
    L = choose(T, N, H, sms, uniform)
    got = modelled(T, N, H, sms, None if L == -1 else L // 64, uniform)
    n = -(-(-(-T // N)) // 64)
    cap = max(2, 8 * sms // (N * H))  # at most 8 waves of replay units
    others = [modelled(T, N, H, sms, c, uniform) for c in range(4, n) if 2 <= -(-n // c) <= cap]
    assert got <= min(others + [modelled(T, N, H, sms, None, uniform)])
