"""GPU: acceptance telemetry (spec_accept_histogram) is bit-exact against a host
count, accumulates across calls, and feeds the depth tuner's sweep."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_30_gb300 as sv
from speculative_decoding_verification_30_gb300 import tuner
from speculative_decoding_verification_30_gb300.workloads import (WORKLOADS, draft_tokens_by_rank,
                                                                   make_batch)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _host_hist(n, K):
    n = np.asarray(n)
    h = np.bincount(np.where((n >= 0) & (n <= K), n, K + 1), minlength=K + 2)
    return h.astype(np.int64)


@pytest.mark.parametrize("B,K", [(1, 1), (1000, 4), (70_000, 16), (513, 7)])
def test_histogram_equals_a_host_count(B, K):
    g = torch.Generator().manual_seed(B + K)
    n = torch.randint(-1, K + 1, (B,), generator=g, dtype=torch.int32)
    n[::97] = K + 5                                   # out-of-range values land in the error bin
    h = sv.spec_accept_histogram(n.to(DEV), K)
    torch.cuda.synchronize()
    assert h.cpu().numpy().tolist() == _host_hist(n.numpy(), K).tolist()


def test_histogram_accumulates_across_calls():
    K = 4
    a = torch.tensor([0, 1, 4, 4, -1], dtype=torch.int32)
    b = torch.tensor([2, 2, 3], dtype=torch.int32)
    h = sv.spec_accept_histogram(a.to(DEV), K)
    sv.spec_accept_histogram(b.to(DEV), K, h)
    torch.cuda.synchronize()
    assert h.cpu().tolist() == [1, 1, 2, 1, 2, 1]


def test_histogram_of_a_verify_call():
    w = WORKLOADS["nucleus_batch"]
    b = make_batch(w, 5, B=16, device=DEV)
    d = draft_tokens_by_rank(b.draft, 5, w.cid).to(DEV)
    _, n = sv.spec_verify(b.target, b.draft, d, b.temperature.to(DEV), b.top_k.to(DEV),
                          b.top_p.to(DEV), seed=3, offset=1)
    h = sv.spec_accept_histogram(n, w.K)
    torch.cuda.synchronize()
    assert h.cpu().tolist() == _host_hist(n.cpu().numpy(), w.K).tolist()


def test_sweep_measures_more_tokens_per_step_with_a_better_draft():
    lo = tuner.sweep(0.3, [1, 4], B=32, V=32_768, steps=2)
    hi = tuner.sweep(0.97, [1, 4], B=32, V=32_768, steps=2)
    for res in (lo, hi):
        for K, r in res.items():
            # the expected-token formula on the measured rates reproduces the measured mean
            assert r["predicted"] == pytest.approx(r["tokens_per_step"], rel=1e-9)
            assert sum(r["hist"]) == 2 * 32 and r["hist"][K + 1] == 0
    assert hi[4]["tokens_per_step"] > lo[4]["tokens_per_step"]
    assert hi[4]["tokens_per_step"] > hi[1]["tokens_per_step"]
    assert hi[4]["rates"][0] > lo[4]["rates"][0]
