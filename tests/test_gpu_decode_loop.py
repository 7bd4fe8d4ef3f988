"""GPU: the device-resident decode-loop step (spec_verify_step).

The step keeps its Philox offset in device memory and hands each sequence's
last emitted token to the next step. Eager calls and a CUDA graph captured once
and replayed must give bit-identical results to spec_verify called with
offsets base, base + 1, ... on the same inputs, and agree with the float64 oracle
at those offsets (tokens and n exact except on boundary draws)."""
import pytest
import torch

import speculative_decoding_verification_30_gb300 as sv
from speculative_decoding_verification_30_gb300.workloads import (WORKLOADS, draft_tokens_by_rank,
                                                                   make_batch)
from tests.parity_util import compare, oracle_verify

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(name, step, B):
    w = WORKLOADS[name]
    b = make_batch(w, step, B=B, device=DEV)
    d = draft_tokens_by_rank(b.draft, step, w.cid).to(DEV)
    return (b.target, b.draft, d, b.temperature.to(DEV), b.top_k.to(DEV), b.top_p.to(DEV))


@pytest.mark.parametrize("name,B", [("nucleus_batch", 16), ("greedy", 8), ("mixed", 6)])
def test_eager_steps_match_spec_verify_and_hand_off(name, B):
    K = WORKLOADS[name].K
    base = 40
    off = torch.tensor([base], dtype=torch.int64, device=DEV)
    ws = sv.Workspace(B, K)
    out = torch.empty(B, K + 1, dtype=torch.int32, device=DEV)
    n = torch.empty(B, dtype=torch.int32, device=DEV)
    nxt = torch.empty(B, dtype=torch.int32, device=DEV)
    slen = torch.full((B,), 100, dtype=torch.int32, device=DEV)
    expect_len = torch.full((B,), 100, dtype=torch.int32)
    for step in range(3):
        tg, dr, d, T, k, P = _inputs(name, step, B)
        ref_tok, ref_n = sv.spec_verify(tg, dr, d, T, k, P, seed=5, offset=base + step)
        sv.spec_verify_step(tg, dr, d, T, k, P, 5, off, out, n, ws, nxt, slen)
        torch.cuda.synchronize()
        assert torch.equal(out.cpu(), ref_tok.cpu()) and torch.equal(n.cpu(), ref_n.cpu())
        # and against the float64 oracle at the offset the step read from device memory
        res = oracle_verify(tg, None if name == "greedy" else dr, d, T, k, P, 5, base + step)
        rep = compare(out.cpu(), n.cpu(), res, T)
        assert not rep.bad_mismatches, (step, rep.bad_mismatches[:3])
        rn = ref_n.cpu()
        last = torch.tensor([int(ref_tok[b, rn[b]]) if rn[b] >= 0 else -1 for b in range(B)],
                            dtype=torch.int32)
        assert torch.equal(nxt.cpu(), last)
        expect_len += torch.where(rn >= 0, rn + 1, torch.zeros_like(rn))
        assert torch.equal(slen.cpu(), expect_len)
    assert int(off.item()) == base + 3
    assert int(ws.buf.count_nonzero()) == 0


@pytest.mark.parametrize("name,B", [("nucleus_batch", 16), ("greedy", 8), ("mixed", 6)])
def test_a_captured_step_replays_bit_exactly(name, B):
    K = WORKLOADS[name].K
    base = 7
    static = [t.clone() for t in _inputs(name, 0, B)]
    off = torch.tensor([base], dtype=torch.int64, device=DEV)
    ws = sv.Workspace(B, K)
    out = torch.empty(B, K + 1, dtype=torch.int32, device=DEV)
    n = torch.empty(B, dtype=torch.int32, device=DEV)
    nxt = torch.empty(B, dtype=torch.int32, device=DEV)
    slen = torch.zeros(B, dtype=torch.int32, device=DEV)
    # warm-up outside capture (kernel attributes are set on the first call), then reset
    sv.spec_verify_step(*static, 3, off, out, n, ws, nxt, slen)
    torch.cuda.synchronize()
    off.fill_(base)
    slen.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sv.spec_verify_step(*static, 3, off, out, n, ws, nxt, slen)
    torch.cuda.synchronize()
    off.fill_(base)                 # capture does not run the kernels; start the loop here
    slen.zero_()
    total = torch.zeros(B, dtype=torch.int32)
    for step in range(4):
        fresh = _inputs(name, 10 + step, B)
        for dst, src in zip(static, fresh):
            dst.copy_(src)
        g.replay()
        ref_tok, ref_n = sv.spec_verify(*fresh, seed=3, offset=base + step)
        torch.cuda.synchronize()
        assert torch.equal(out.cpu(), ref_tok.cpu()), step
        assert torch.equal(n.cpu(), ref_n.cpu()), step
        tg, dr, d, T, k, P = fresh
        res = oracle_verify(tg, None if name == "greedy" else dr, d, T, k, P, 3, base + step)
        rep = compare(out.cpu(), n.cpu(), res, T)
        assert not rep.bad_mismatches, (step, rep.bad_mismatches[:3])
        rn = ref_n.cpu()
        total += torch.where(rn >= 0, rn + 1, torch.zeros_like(rn))
    assert int(off.item()) == base + 4
    assert torch.equal(slen.cpu(), total)
    assert int(ws.buf.count_nonzero()) == 0
