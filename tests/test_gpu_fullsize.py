"""GPU parity at the full sizes of the benchmark workloads, in the launch
configuration the bench times (one spec_verify call per batch).

Every sequence of the nucleus serving batch (B=64) and of the greedy batch
(B=256) is checked against the float64 oracle, and so is every sequence of the
mixed fp32 batch at its full size (B=512, K=5); the
tiny verify runs all of its 1000 steps and the MTP-decode shape a stretch of
its steps. Tokens and n_accepted must be identical except on sequences whose
oracle draws include a boundary draw (an acceptance or sampling uniform within
1e-6 of its decision boundary); temperature-0 sequences have no exceptions. The
boundary counts are printed with the draw counts.
"""
import pytest
import torch

import speculative_decoding_verification_30_gb300 as sv
from speculative_decoding_verification_30_gb300.workloads import (WORKLOADS, draft_tokens_by_rank,
                                                                   make_batch)
from tests.parity_util import ParityReport, compare, oracle_verify

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _verify(batch, dtok, seed, offset, greedy=False):
    out, n = sv.spec_verify(batch.target, None if greedy else batch.draft, dtok.to(DEV),
                            batch.temperature.to(DEV), batch.top_k.to(DEV), batch.top_p.to(DEV),
                            seed=seed, offset=offset)
    torch.cuda.synchronize()
    return out.cpu(), n.cpu()


@pytest.mark.parametrize("name,step", [("nucleus_batch", 0), ("nucleus_batch", 1)])
def test_full_nucleus_batch_every_sequence(name, step):
    w = WORKLOADS[name]
    b = make_batch(w, step, device=DEV)
    dtok = sv.spec_sample(b.draft, b.temperature.to(DEV), b.top_k.to(DEV), b.top_p.to(DEV),
                          seed=4242, offset=10_000 + step)
    out, n = _verify(b, dtok, 1234, step)
    res = oracle_verify(b.target, b.draft, dtok, b.temperature, b.top_k, b.top_p, 1234, step)
    rep = compare(out, n, res, b.temperature)
    print(name, "full B=64:", rep)
    assert rep.sequences == w.B
    assert not rep.bad_mismatches, rep.bad_mismatches[:3]


def test_full_greedy_batch_is_bit_exact():
    w = WORKLOADS["greedy"]
    b = make_batch(w, 0, device=DEV)
    dtok = draft_tokens_by_rank(b.draft, 0, w.cid)
    out, n = _verify(b, dtok, 1, 0, greedy=True)
    res = oracle_verify(b.target, None, dtok, b.temperature, b.top_k, b.top_p, 1, 0)
    rep = compare(out, n, res, b.temperature)
    print("greedy full B=256:", rep)
    assert rep.greedy == w.B and rep.mismatches == 0, rep.bad_mismatches[:3]
    # sequences whose draft equals the target (every 5th) accept every drafted argmax
    dt = dtok.cpu()
    assert all(int(n[s]) == w.K for s in range(0, w.B, 5) if bool((dt[s] == out[s, : w.K]).all()))


def test_full_greedy_batch_with_draft_logits_matches_without():
    w = WORKLOADS["greedy"]
    b = make_batch(w, 1, device=DEV)
    dtok = draft_tokens_by_rank(b.draft, 1, w.cid)
    a = _verify(b, dtok, 1, 0, greedy=True)
    c = _verify(b, dtok, 1, 0, greedy=False)
    assert torch.equal(a[0], c[0]) and torch.equal(a[1], c[1])


def test_full_mixed_batch_every_sequence():
    w = WORKLOADS["mixed"]
    b = make_batch(w, 0, device=DEV)
    dtok = draft_tokens_by_rank(b.draft, 0, w.cid)
    out, n = _verify(b, dtok, 77, 3)
    res = oracle_verify(b.target, b.draft, dtok, b.temperature, b.top_k, b.top_p, 77, 3)
    rep = compare(out, n, res, b.temperature)
    print("mixed full B=512 K=5 fp32, every sequence:", rep)
    assert rep.sequences == w.B
    assert not rep.bad_mismatches, rep.bad_mismatches[:3]
    # every sequence produced a well-formed row: n in [0, K], tokens after n+1 are -1
    nn = n.numpy()
    assert ((nn >= 0) & (nn <= w.K)).all()
    for s in range(w.B):
        assert (out[s, nn[s] + 1:] == -1).all() and (out[s, : nn[s] + 1] >= 0).all()


def test_tiny_all_steps():
    w = WORKLOADS["tiny"]
    total = ParityReport()
    batches = [make_batch(w, step, device=DEV) for step in range(w.steps)]
    dts = [draft_tokens_by_rank(bb.draft, step, w.cid) for step, bb in enumerate(batches)]
    outs = [_verify(bb, dts[step], 0, step) for step, bb in enumerate(batches)]
    for step, bb in enumerate(batches):
        res = oracle_verify(bb.target, bb.draft, dts[step], bb.temperature, bb.top_k, bb.top_p,
                            0, step, parallel=False)
        total.add(compare(outs[step][0], outs[step][1], res, bb.temperature))
    print("tiny, all", w.steps, "steps:", total)
    assert total.sequences == w.steps and not total.bad_mismatches, total.bad_mismatches[:3]


def test_mtp_decode_steps():
    w = WORKLOADS["mtp_decode"]
    steps = 300
    total = ParityReport()
    for s0 in range(0, steps, 50):
        chunk = []
        for step in range(s0, s0 + 50):
            bb = make_batch(w, step, device=DEV)
            dt = draft_tokens_by_rank(bb.draft, step, w.cid)
            chunk.append((step, bb, dt, _verify(bb, dt, 0, step)))
        for step, bb, dt, (out, n) in chunk:
            res = oracle_verify(bb.target, bb.draft, dt, bb.temperature, bb.top_k, bb.top_p, 0, step,
                                parallel=False)
            total.add(compare(out, n, res, bb.temperature))
    print("mtp_decode,", steps, "steps:", total)
    assert not total.bad_mismatches, total.bad_mismatches[:3]
