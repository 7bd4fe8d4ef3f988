"""GPU: seeded random verify calls against the float64 oracle.

Random batch sizes, depths, vocabularies (16-byte aligned rows and not), dtypes,
temperatures (0 included), top-k, top-p, draft quality, masked and quantised
rows. The mix reaches every kernel route: key-histogram (bf16, aligned, at least
16 units), cluster kernel (fp32, unaligned or small batches, hand-backs) and
greedy. Tokens and n_accepted must match the oracle except on boundary draws."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_30_gb300 as sv
from tests.parity_util import ParityReport, compare, oracle_verify

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed):
    g = torch.Generator().manual_seed(seed)
    rng = np.random.default_rng(seed)
    B = int(rng.choice([1, 3, 4, 8, 17]))
    K = int(rng.choice([1, 2, 4, 7]))
    V = int(rng.choice([8, 64, 1000, 1024, 2048, 4097, 8192]))
    dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
    s = float(rng.uniform(0.5, 1.5))
    ranks = torch.argsort(torch.rand(B * (2 * K + 1), V, generator=g), dim=1).float() + 1
    z = (-s * torch.log(ranks) + 0.5 * torch.randn(B * (2 * K + 1), V, generator=g)).view(B, 2 * K + 1, V)
    a = float(rng.uniform(0.0, 1.0))
    tgt = z[:, : K + 1].clone()
    drf = a * tgt[:, :K] + (1 - a) * z[:, K + 1:]
    if rng.random() < 0.3:                                   # quantised logits: ties
        q = float(rng.choice([0.125, 0.5, 1.0]))
        tgt, drf = torch.round(tgt / q) * q, torch.round(drf / q) * q
    if rng.random() < 0.3:                                   # masked tokens
        m = torch.rand(V, generator=g) < 0.5
        tgt[:, :, m] = -float("inf")
        drf[:, :, m] = -float("inf")
        tgt[:, :, int(torch.nonzero(~m)[0]) if (~m).any() else 0] = 1.0
    T = torch.tensor(rng.choice([0.0, 0.3, 0.7, 1.0, 1.6], size=B), dtype=torch.float32)
    k = torch.tensor(rng.choice([0, 1, 5, 20, V], size=B), dtype=torch.int32)
    P = torch.tensor(rng.choice([1.0, 0.95, 0.8, 0.5], size=B), dtype=torch.float32)
    top = torch.topk(drf, min(4, V), dim=-1).indices
    dtok = top.gather(-1, torch.randint(0, min(4, V), (B, K, 1), generator=g)).squeeze(-1).to(torch.int32)
    return tgt.to(dtype), drf.to(dtype), dtok, T, k, P


@pytest.mark.parametrize("block", range(6))
def test_random_calls_match_the_oracle(block):
    total = ParityReport()
    for seed in range(block * 12, block * 12 + 12):
        tgt, drf, dtok, T, k, P = _case(seed)
        out, n = sv.spec_verify(tgt.to(DEV), drf.to(DEV), dtok.to(DEV), T.to(DEV), k.to(DEV),
                                P.to(DEV), seed=seed, offset=3 * seed)
        torch.cuda.synchronize()
        res = oracle_verify(tgt, drf, dtok, T, k, P, seed, 3 * seed, parallel=False)
        rep = compare(out.cpu(), n.cpu(), res, T)
        assert not rep.bad_mismatches, (seed, tuple(tgt.shape), tgt.dtype, rep.bad_mismatches[:2])
        total.add(rep)
    print("fuzz block", block, total)
