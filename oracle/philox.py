"""Philox-4xW-10 counter-based generator, written from its published definition.

TEST INFRASTRUCTURE: part of the CPU oracle. Only tests/, the smoke check and
bench.py's CPU-baseline leg may import this module; the product path never does.

Source: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random
numbers: as easy as 1, 2, 3", SC'11, section 3.3 (the Philox S-box: one
multiply-high/low per pair of words, a fixed word permutation and a key XOR),
with the multipliers and Weyl key increments the paper gives for N=4, W=32 and
W=64. Ten rounds; the key is bumped by the Weyl constants before every round
but the first.

The speculative-decoding pages ask only that the randomness be a pure function
of (seed, sequence, position); they name no generator. The layout used by the
whole library (both the oracle and the CUDA path) is:

    key     = (seed & 0xffffffff, seed >> 32)
    counter = (position i, sequence b, offset & 0xffffffff, offset >> 32)
    word 0 -> acceptance uniform u, word 1 -> sampling uniform v
    uniform = (word >> 8) * 2**-24            (exact in fp32 and float64)

Pure-Python integers; slow and obviously correct.
"""
from __future__ import annotations

_CONST = {
    32: dict(M0=0xD2511F53, M1=0xCD9E8D57, W0=0x9E3779B9, W1=0xBB67AE85),
    64: dict(M0=0xD2E7470EE14C6C93, M1=0xCA5A826395121157,
             W0=0x9E3779B97F4A7C15, W1=0xBB67AE8584CAA73B),
}


def _mulhilo(a: int, b: int, width: int) -> tuple[int, int]:
    prod = a * b
    mask = (1 << width) - 1
    return prod >> width, prod & mask


def philox4(counter, key, width: int = 32, rounds: int = 10) -> tuple[int, int, int, int]:
    """One Philox-4xW block: four W-bit words from a 4-word counter and 2-word key."""
    c = _CONST[width]
    mask = (1 << width) - 1
    c0, c1, c2, c3 = (int(x) & mask for x in counter)
    k0, k1 = (int(x) & mask for x in key)
    for r in range(rounds):
        if r > 0:
            k0 = (k0 + c["W0"]) & mask
            k1 = (k1 + c["W1"]) & mask
        hi0, lo0 = _mulhilo(c["M0"], c0, width)
        hi1, lo1 = _mulhilo(c["M1"], c2, width)
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def philox4x32_10(counter, key) -> tuple[int, int, int, int]:
    return philox4(counter, key, width=32, rounds=10)


def to_uniform(word: int) -> float:
    """Top 24 bits of a 32-bit word as a float in [0, 1): exact in fp32 and float64."""
    return (int(word) >> 8) * (2.0 ** -24)


def uniforms(seed: int, offset: int, b: int, i: int) -> tuple[float, float]:
    """(u, v) for sequence b, position i: u decides acceptance, v drives sampling."""
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    ctr = (i, b, offset & 0xFFFFFFFF, (offset >> 32) & 0xFFFFFFFF)
    w = philox4x32_10(ctr, key)
    return to_uniform(w[0]), to_uniform(w[1])
