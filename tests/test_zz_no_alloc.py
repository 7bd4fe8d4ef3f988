"""GPU: spec_verify_noalloc (fixed library scratch, no workspace argument) gives the
same results as spec_verify with a caller workspace, on two consecutive calls.

The file name sorts last so that the run also covers the case where other tests
have used the library before; the test does not depend on that order."""
import pytest
import torch

import speculative_decoding_verification_30_gb300 as sv
from speculative_decoding_verification_30_gb300.workloads import (WORKLOADS, draft_tokens_by_rank,
                                                                   make_batch)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(name, step, B):
    w = WORKLOADS[name]
    b = make_batch(w, step, B=B)
    dtok = draft_tokens_by_rank(b.draft, step, w.cid)
    return (b.target.to(DEV), b.draft.to(DEV), dtok.to(DEV), b.temperature.to(DEV),
            b.top_k.to(DEV), b.top_p.to(DEV))


@pytest.mark.parametrize("name,B", [("mixed", 12), ("nucleus_batch", 6), ("greedy", 8)])
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(name, B):
    ws = sv.Workspace(B, WORKLOADS[name].K, DEV)
    for call, step in enumerate((3, 4)):
        tgt, drf, dtok, T, k, P = _inputs(name, step, B)
        seed, offset = 77 + call, 1000 * step + call
        ref_tok, ref_n = sv.spec_verify(tgt, drf, dtok, T, k, P, seed=seed, offset=offset,
                                        workspace=ws)
        got_tok, got_n = sv.spec_verify_noalloc(tgt, drf, dtok, T, k, P, seed=seed,
                                                offset=offset)
        torch.cuda.synchronize()
        # same kernels on the same inputs and uniforms: token ids are integers, the
        # tolerance is exact equality
        assert torch.equal(ref_n.cpu(), got_n.cpu()), (name, call)
        assert torch.equal(ref_tok.cpu(), got_tok.cpu()), (name, call)


def test_noalloc_rejects_batches_beyond_the_scratch():
    B, K, V = 65535, 16, 8
    assert sv.spec_verify_workspace_bytes(B, K) > sv.NOALLOC_SCRATCH_BYTES
    tgt = torch.zeros(B, K + 1, V, device=DEV)
    dtok = torch.zeros(B, K, dtype=torch.int32, device=DEV)
    T, k, P = (torch.zeros(B, device=DEV), torch.zeros(B, dtype=torch.int32, device=DEV),
               torch.ones(B, device=DEV))
    with pytest.raises(sv.SpecVerifyError, match="status 7"):
        sv.spec_verify_noalloc(tgt, None, dtok, T, k, P, seed=0, offset=0)


def test_noalloc_after_a_rejected_call_still_matches():
    # a call rejected before launching (here an unaligned pointer, status 6) must
    # leave the shared scratch usable: the next call equals the workspace entry point
    name, B = "nucleus_batch", 6
    tgt, drf, dtok, T, k, P = _inputs(name, 5, B)
    lib = sv.load()
    K, V = WORKLOADS[name].K, WORKLOADS[name].V
    out = torch.empty(B, K + 1, dtype=torch.int32, device=DEV)
    n = torch.empty(B, dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.spec_verify_noalloc(tgt.data_ptr(), drf.data_ptr(), sv.SV_BF16, dtok.data_ptr(),
                                 T.data_ptr() + 1, k.data_ptr(), P.data_ptr(), 3, 4, B, K, V,
                                 out.data_ptr(), n.data_ptr(), stream)
    assert st == 6
    ref_tok, ref_n = sv.spec_verify(tgt, drf, dtok, T, k, P, seed=3, offset=4)
    got_tok, got_n = sv.spec_verify_noalloc(tgt, drf, dtok, T, k, P, seed=3, offset=4)
    torch.cuda.synchronize()
    assert torch.equal(ref_n.cpu(), got_n.cpu()) and torch.equal(ref_tok.cpu(), got_tok.cpu())
