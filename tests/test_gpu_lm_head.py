"""GPU: the LM-head logits GEMM (tcgen05 tensor cores, TMA, TMEM accumulator)
against the float64 oracle, and the verify step fed from hidden states.

Logits z = h . W^T ("Apple Silikon İçin Cihaz Üstü Çıkarımı Optimize Etme",
decode section: the output projection ends every decode step). The kernel
accumulates bf16 products in fp32, so every logit must lie within the oracle's
fp32 accumulation bound (oracle.lm_head.logit_error_bound) of the exact value;
shapes include M and N that are not multiples of the 128 x 128 tile and more
than one 64-wide K slice."""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_30_gb300 as sv
from oracle import lm_head
from tests.parity_util import compare, f64, oracle_verify

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(M, N, d, seed, rows=None):
    g = torch.Generator().manual_seed(seed)
    h = (torch.randn(M, d, generator=g) * 0.5).to(torch.bfloat16)
    W = (torch.randn(N, d, generator=g) * 0.05).to(torch.bfloat16)
    z, flag = sv.spec_lm_head_logits(h.to(DEV), W.to(DEV))
    torch.cuda.synchronize()
    assert int(flag.item()) == 0, "a bounded wait of the GEMM timed out"
    got = z.cpu().double().numpy()
    sel = np.arange(M) if rows is None else rows
    ref = lm_head.lm_head_logits(f64(h)[sel], f64(W))
    bound = lm_head.logit_error_bound(f64(h)[sel], f64(W))
    err = np.abs(got[sel] - ref)
    assert np.all(err <= bound + 1e-30), (float(err.max()), float(bound.max()))
    return float((err / np.maximum(bound, 1e-30)).max())


@pytest.mark.parametrize("M,N,d", [(128, 128, 64), (130, 300, 128), (320, 1000, 512), (7, 129, 192)])
def test_lm_head_logits_within_fp32_bound(M, N, d):
    worst = _case(M, N, d, seed=M * 7 + N + d)
    print(f"M={M} N={N} d={d}: worst error / bound = {worst:.3f}")


def test_lm_head_logits_full_vocabulary_sampled_rows():
    # the nucleus batch's 320 target rows against a 151,936-token head, d = 1024;
    # every column of 24 sampled rows is checked
    rows = np.array(sorted(set(range(0, 320, 14)) | {319}))
    worst = _case(320, 151_936, 1024, seed=3, rows=rows)
    print(f"full vocabulary: worst error / bound = {worst:.3f}")


def test_verify_from_hidden_matches_oracle():
    # logits from hidden states (target and draft heads), then the verify step;
    # tokens may differ from the oracle's float64 logits only where a decision
    # margin lies within the fp32 perturbation (here: boundary draws)
    B, K, V, d = 8, 2, 2048, 256
    g = torch.Generator().manual_seed(11)
    ht = (torch.randn(B, K + 1, d, generator=g) * 0.5).to(torch.bfloat16)
    Wt = (torch.randn(V, d, generator=g) * 0.1).to(torch.bfloat16)
    hd = (0.6 * ht[:, :K].float() + 0.4 * torch.randn(B, K, d, generator=g) * 0.5).to(torch.bfloat16)
    dtok = torch.randint(0, V, (B, K), generator=g, dtype=torch.int32)
    T = torch.tensor([1.0, 0.7, 0.0, 1.2, 0.9, 1.0, 0.5, 0.0])
    k = torch.tensor([0, 20, 0, 50, 0, 5, 0, 0], dtype=torch.int32)
    P = torch.tensor([0.95, 1.0, 1.0, 0.9, 0.8, 1.0, 0.95, 1.0])
    out, n, flag = sv.spec_verify_from_hidden(ht.to(DEV), Wt.to(DEV), hd.to(DEV), Wt.to(DEV),
                                              dtok.to(DEV), T.to(DEV), k.to(DEV), P.to(DEV), seed=5,
                                              offset=9)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    zt = lm_head.lm_head_logits(f64(ht), f64(Wt))
    zd = lm_head.lm_head_logits(f64(hd), f64(Wt))
    res = oracle_verify(torch.from_numpy(zt), torch.from_numpy(zd), dtok, T, k, P, 5, 9,
                        parallel=False)
    rep = compare(out.cpu(), n.cpu(), res, T)
    print("verify from hidden:", rep)
    assert not rep.bad_mismatches, rep.bad_mismatches[:3]
