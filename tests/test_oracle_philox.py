"""Pins for the oracle's Philox: a library routine and published known answers."""
import os

import numpy as np

from oracle.philox import philox4, philox4x32_10, to_uniform, uniforms

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def test_known_answers_4x32():
    rows = [ln.split() for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        w = [int(x, 16) for x in r]
        assert philox4x32_10(w[0:4], w[4:6]) == tuple(w[6:10])


def test_same_round_code_at_width64_matches_numpy_philox():
    # numpy.random.Philox is Philox4x64-10; it increments the counter before each
    # block. The oracle's round function, instantiated at W=64, must agree.
    rng = np.random.default_rng(1234)
    for _ in range(5):
        key = [int(x) for x in rng.integers(0, 2**63, size=2, dtype=np.int64)]
        ctr = [int(x) for x in rng.integers(0, 2**62, size=4, dtype=np.int64)]
        bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                              counter=np.array(ctr, dtype=np.uint64))
        raw = [int(x) for x in bg.random_raw(8)]
        c1 = [ctr[0] + 1] + ctr[1:]
        c2 = [ctr[0] + 2] + ctr[1:]
        assert list(philox4(c1, key, 64)) == raw[:4]
        assert list(philox4(c2, key, 64)) == raw[4:]


def test_uniform_conversion_is_exact_24bit_grid():
    assert to_uniform(0) == 0.0
    assert to_uniform(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert to_uniform(0x00000100) == 2.0 ** -24
    assert to_uniform(0x000000FF) == 0.0
    for w in (0x12345678, 0x80000000, 0xDEADBEEF):
        u = to_uniform(w)
        assert float(np.float32(u)) == u and u * 2**24 == (w >> 8)


def test_stream_layout_is_a_pure_function_of_seed_offset_sequence_position():
    a = uniforms(7, 3, 1, 2)
    assert a == uniforms(7, 3, 1, 2)
    key = (7, 0)
    w = philox4x32_10((2, 1, 3, 0), key)
    assert a == (to_uniform(w[0]), to_uniform(w[1]))
    # the high halves of seed and offset land in key[1] and counter[3]
    s, o = (5 << 32) | 9, (11 << 32) | 4
    w = philox4x32_10((0, 0, 4, 11), (9, 5))
    assert uniforms(s, o, 0, 0) == (to_uniform(w[0]), to_uniform(w[1]))
    assert len({uniforms(7, 3, b, i) for b in range(4) for i in range(4)}) == 16
