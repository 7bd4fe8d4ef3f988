"""GPU: the rate of forgiven mismatches stays under 1e-5 of draws.

Parity allows a token or n_accepted to differ from the float64 oracle only on a
boundary draw (an acceptance or sampling uniform within 1e-6 of its decision
boundary; "MTPLX: native MTP speculative decoding on Apple Silicon", section 3.3:
the verifier is exact, so nothing else may differ). The allowance is read as a
budget on forgiven mismatches: the mismatches that do occur, all of which must be
on boundary draws, must number fewer than 1e-5 of all draws (acceptance tests plus
the one sample per sequence). Boundary draws themselves are counted and reported;
their rate is a property of the input (about 2e-6 per acceptance draw, and far more
for samples from a wide nucleus, where tokens carry ~1e-5 of mass each).

More than 1e5 draws per dtype: vocabulary 1024 (so the oracle finishes in seconds),
mixed per-sequence temperature / top-k / top-p, fp32 rows (row-streaming kernel)
and bf16 rows (key-histogram kernel), 45,000 sequences each in calls of 2,500.
"""
import pytest
import torch

import speculative_decoding_verification_30_gb300 as sv
from speculative_decoding_verification_30_gb300.workloads import (Workload, draft_tokens_by_rank,
                                                                   make_batch)
from tests.parity_util import ParityReport, compare, oracle_verify

pytestmark = pytest.mark.gpu
DEV = "cuda"
B, K, V = 45_000, 2, 1024
CHUNK = 2_500


@pytest.fixture(scope="module")
def report():
    return {}


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_forgiven_mismatches_stay_under_1e5_of_draws(dtype, report):
    # the mixed workload's parameter recipe at a small vocabulary
    w = Workload("mixed", B, K, V, dtype, 1, cid=5)
    total = ParityReport()
    for c0 in range(0, B, CHUNK):
        b = make_batch(w, 100 + c0 // CHUNK, B=CHUNK)
        dtok = draft_tokens_by_rank(b.draft, c0, w.cid)
        out, n = sv.spec_verify(b.target.to(DEV), b.draft.to(DEV), dtok.to(DEV),
                                b.temperature.to(DEV), b.top_k.to(DEV), b.top_p.to(DEV),
                                seed=2024, offset=c0)
        torch.cuda.synchronize()
        res = oracle_verify(b.target, b.draft, dtok, b.temperature, b.top_k, b.top_p, 2024, c0)
        total.add(compare(out.cpu(), n.cpu(), res, b.temperature))
    report[str(dtype)] = total
    rate = total.excused / total.draws
    print(f"{dtype}: {total}; forgiven-mismatch rate {rate:.2e}; "
          f"boundary-draw sequences {total.boundary / total.sequences:.2e} of sequences")
    assert total.draws >= 100_000
    assert not total.bad_mismatches, total.bad_mismatches[:3]
    assert total.excused < 1e-5 * total.draws, (total.excused, total.draws)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_row_kernel_results_are_identical_across_calls(dtype):
    # the row kernels take rows from a work counter, so which CTA serves which row
    # changes from call to call; the outputs must not (a stale or racing read would
    # show here before it shows against the oracle)
    w = Workload("mixed", CHUNK, K, V, dtype, 1, cid=5)
    b = make_batch(w, 100, B=CHUNK)
    dtok = draft_tokens_by_rank(b.draft, 0, w.cid)
    args = [x.to(DEV) for x in (b.target, b.draft, dtok, b.temperature, b.top_k, b.top_p)]
    first = None
    for _ in range(8):
        out, n = sv.spec_verify(*args, seed=2024, offset=0)
        torch.cuda.synchronize()
        if first is None:
            first = (out.clone(), n.clone())
        else:
            assert torch.equal(out, first[0]) and torch.equal(n, first[1])
