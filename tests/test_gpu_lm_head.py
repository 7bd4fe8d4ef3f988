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


# --- greedy verify fused with the LM head (no logit row written) -------------

def _greedy_inputs(B, K, V, d, seed, rows_for=None, corrupt=0.25):
    """Hidden states, head, and drafted tokens: the exact (float64) argmax of each
    drafted position, replaced by a random id with probability `corrupt`, for the
    sequences in rows_for (all by default); random ids elsewhere."""
    g = torch.Generator().manual_seed(seed)
    h = (torch.randn(B, K + 1, d, generator=g) * 0.5).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g) * 0.1).to(torch.bfloat16)
    seqs = np.arange(B) if rows_for is None else np.asarray(rows_for)
    zt = lm_head.lm_head_logits(f64(h)[seqs], f64(W))              # [S, K+1, V]
    bound = lm_head.logit_error_bound(f64(h)[seqs], f64(W))
    dt = torch.randint(0, V, (B, K), generator=g).numpy()
    keep = torch.rand(B, K, generator=g).numpy() >= corrupt
    ex = zt[:, :K].argmax(-1)
    dt[seqs] = np.where(keep[seqs], ex, dt[seqs])
    return h, W, torch.from_numpy(dt.astype(np.int32)), seqs, zt, bound


def _check_greedy(out, n, dt, seqs, zt, bound):
    """Exact agreement with the oracle for every sequence whose rows all have a
    maximum clear of the runner-up by more than the two logits' fp32 bounds;
    elsewhere every kept drafted token and the emitted token must be maxima of
    their rows within those bounds. Returns the number of unclear sequences."""
    from oracle import sampler
    K1 = zt.shape[1]
    K = K1 - 1
    unclear = 0
    for s, b in enumerate(seqs):
        r = sampler.verify_sequence(zt[s], None, dt[b].tolist(), 0.0, 0, 1.0, 0, 0, int(b))
        clear = True
        for i in range(K1):
            t2 = np.argsort(-zt[s, i])[:2]
            if zt[s, i, t2[0]] - zt[s, i, t2[1]] <= bound[s, i, t2[0]] + bound[s, i, t2[1]]:
                clear = False
        if clear:
            assert list(out[b]) == list(r.tokens) and int(n[b]) == r.n_accepted, (b, out[b], r.tokens)
            continue
        unclear += 1
        nb = int(n[b])
        assert 0 <= nb <= K

        def is_max(i, v):
            top = int(zt[s, i].argmax())
            return zt[s, i, v] >= zt[s, i, top] - (bound[s, i, v] + bound[s, i, top])
        for q in range(nb):
            assert out[b][q] == dt[b][q] and is_max(q, int(dt[b][q])), (b, q)
        assert is_max(nb, int(out[b][nb])), (b, nb)
        assert nb == K or out[b][nb] != dt[b][nb]
        assert all(x == -1 for x in out[b][nb + 1:])
    return unclear


def test_greedy_from_hidden_matches_oracle():
    # M = 160 rows (ragged against the 128-row tile), V = 5000 (ragged against the
    # 256-column tile), four 64-wide K slices
    B, K, V, d = 40, 3, 5000, 256
    h, W, dt, seqs, zt, bound = _greedy_inputs(B, K, V, d, seed=21)
    ws = sv.Workspace(B, K, DEV)
    out, n, flag = sv.spec_verify_greedy_from_hidden(h.to(DEV), W.to(DEV), dt.to(DEV), workspace=ws)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    o, nn = out.cpu().numpy(), n.cpu().numpy()
    unclear = _check_greedy(o, nn, dt.numpy(), seqs, zt, bound)
    assert unclear <= B // 10, unclear
    assert sorted(set(nn.tolist())) != [0], "the drafts should be accepted at some positions"
    # the row keys live in the workspace and are left zeroed; a second call agrees
    assert int(ws.buf[: B * (K + 1) * 8].count_nonzero()) == 0
    out2, n2, _ = sv.spec_verify_greedy_from_hidden(h.to(DEV), W.to(DEV), dt.to(DEV), workspace=ws)
    assert torch.equal(out2, out) and torch.equal(n2, n)


def test_greedy_from_hidden_data_errors():
    # a hidden state holding +inf gives a row with infinite logits; drafted ids
    # outside [0, V) are data errors; the other sequences are unaffected
    B, K, V, d = 6, 2, 1000, 128
    h, W, dt, seqs, _, _ = _greedy_inputs(B, K, V, d, seed=5)
    h[1, 2, 7] = float("inf")
    dt[2, 0] = V
    dt[3, 1] = -1
    zt = lm_head.lm_head_logits(f64(h), f64(W))
    bound = lm_head.logit_error_bound(f64(h), f64(W))
    out, n, flag = sv.spec_verify_greedy_from_hidden(h.to(DEV), W.to(DEV), dt.to(DEV))
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    o, nn = out.cpu().numpy(), n.cpu().numpy()
    from oracle import sampler
    for b in (1, 2, 3):
        assert sampler.verify_sequence(zt[b], None, dt[b].tolist(), 0.0, 0, 1.0, 0, 0, b).error
        assert nn[b] == -1 and (o[b] == -1).all()
    ok = np.array([0, 4, 5])
    assert _check_greedy(o, nn, dt.numpy(), ok, zt[ok], bound[ok]) <= 1


def test_greedy_from_hidden_full_vocabulary_and_unfused_path():
    # the greedy batch's shape from hidden states (B = 256, K = 3, V = 151,936,
    # d = 1,024): 16 sampled sequences against the oracle, and every sequence
    # against the unfused path (GEMM to fp32 rows, then spec_verify on them), which
    # reduces the same accumulator values and must agree exactly
    B, K, V, d = 256, 3, 151_936, 1024
    sample = np.arange(0, B, 16)
    h, W, dt, seqs, zt, bound = _greedy_inputs(B, K, V, d, seed=8, rows_for=sample)
    hd, Wd, dtd = h.to(DEV), W.to(DEV), dt.to(DEV)
    out, n, flag = sv.spec_verify_greedy_from_hidden(hd, Wd, dtd)
    T = torch.zeros(B, device=DEV)
    kk = torch.zeros(B, dtype=torch.int32, device=DEV)
    P = torch.ones(B, device=DEV)
    out_u, n_u, flag_u = sv.spec_verify_from_hidden(hd, Wd, None, None, dtd, T, kk, P)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0 and int(flag_u.item()) == 0
    assert torch.equal(out, out_u) and torch.equal(n, n_u)
    o, nn = out.cpu().numpy(), n.cpu().numpy()
    unclear = _check_greedy(o, nn, dt.numpy(), seqs, zt, bound)
    assert unclear <= 4, unclear


def test_greedy_from_hidden_exact_ties_take_the_lowest_id():
    # W[v] = e_(v mod 4) with d = 64: the logits are exact integers repeating with
    # period 4 across three 256-column tiles, so each row's maximum appears about 150
    # times; the merged key must name the lowest id (the oracle's closed form)
    B, K, V, d = 3, 2, 600, 64
    W = torch.zeros(V, d)
    W[torch.arange(V), torch.arange(V) % 4] = 1.0
    h = torch.zeros(B, K + 1, d)
    h[:, :, :4] = torch.tensor([[1.0, 5.0, 2.0, 0.0], [3.0, 0.0, 3.0, 1.0], [0.0, 0.0, 0.0, 4.0]])
    dtok = torch.tensor([[1, 0], [5, 0], [1, 2]], dtype=torch.int32)
    out, n, flag = sv.spec_verify_greedy_from_hidden(h.to(torch.bfloat16).to(DEV), W.to(torch.bfloat16).to(DEV),
                                                     dtok.to(DEV))
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    assert out.cpu().tolist() == [[1, 0, 3], [1, -1, -1], [1, 0, -1]]
    assert n.cpu().tolist() == [2, 0, 1]
