"""Seeded synthetic logit workloads for the verify-and-sample step.

This module only draws inputs. It contains none of the method's arithmetic (no
softmax, truncation, acceptance or sampling), so both the CUDA path and the CPU
oracle can be fed from it.

The pages measure live decodes of real models (Qwen3.5/3.6 with an MTP head,
LLaMA-3-70B with an 8B draft); no weights exist here, so rows are synthetic
with the shape of such logits:

* target row: a random permutation gives every token a rank r in 1..V, and
  z = -s * ln(r) + 0.5 * N(0, 1)   (Zipf-like head, noisy tail);
* draft row: alpha * z + (1 - alpha) * z', with z' an independent copy made by
  the same recipe (its own permutation and noise);
* every (sequence, position) row is independent; rows are cast to the
  workload's dtype (bf16 round-to-nearest-even) and both sides read those bytes.

Vocabulary V = 151,936 (Qwen's padded vocabulary).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

QWEN_VOCAB = 151_936


@dataclass
class Workload:
    name: str
    B: int
    K: int
    V: int
    dtype: torch.dtype
    steps: int                      # steps the configuration is quoted on
    description: str = ""
    cid: int = 0

    def rows_per_step(self) -> int:
        """Logit rows one verify call consumes: B*(K+1) target + B*K draft."""
        return self.B * (2 * self.K + 1)

    def bytes_per_step(self, needed_only: bool = False, greedy: bool = False) -> int:
        es = torch.finfo(self.dtype).bits // 8
        rows = self.B * (self.K + 1) if (needed_only and greedy) else self.rows_per_step()
        return rows * self.V * es


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 1024, torch.float32, 1000,
                     "B=1 K=1 V=1024 fp32, T=1 top_k=20 top_p=0.95, alpha=0.7", cid=1),
    "mtp_decode": Workload("mtp_decode", 1, 1, QWEN_VOCAB, torch.bfloat16, 10_000,
                           "B=1 K=1 V=151936 bf16, T=1 top_k=20 top_p=0.95, alpha=0.7", cid=2),
    "nucleus_batch": Workload("nucleus_batch", 64, 4, QWEN_VOCAB, torch.bfloat16, 200,
                              "B=64 K=4 V=151936 bf16, T=0.6 top_p=0.95 no top_k, "
                              "alpha~U(0.4,0.95)", cid=3),
    "greedy": Workload("greedy", 256, 3, QWEN_VOCAB, torch.bfloat16, 200,
                       "B=256 K=3 V=151936 bf16, T=0; every 5th sequence has draft == target, "
                       "others alpha=0.7", cid=4),
    "mixed": Workload("mixed", 512, 5, QWEN_VOCAB, torch.float32, 50,
                      "B=512 K=5 V=151936 fp32, s~U(0.8,1.5), alpha~U(0.2,0.95), "
                      "T~U(0.3,1.2), top_k in {0,20,50}, top_p in {0.8,0.95,1.0}", cid=5),
}


def _generator(device, *seed_parts) -> torch.Generator:
    seed = 0
    for p in seed_parts:
        seed = (seed * 1_000_003 + int(p) + 1) % (2**62)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def zipf_rows(R: int, V: int, s: torch.Tensor, g: torch.Generator, device) -> torch.Tensor:
    """R independent rows z = -s*ln(rank) + 0.5*N(0,1) (float32), s: [R]."""
    u = torch.rand(R, V, generator=g, device=device)
    perm = torch.argsort(u, dim=1)                     # token placed at each rank
    base = -torch.log(torch.arange(1, V + 1, device=device, dtype=torch.float32))
    z = torch.empty(R, V, device=device, dtype=torch.float32)
    z.scatter_(1, perm, base.expand(R, V) * s.view(R, 1).to(torch.float32))
    z += 0.5 * torch.randn(R, V, generator=g, device=device)
    return z


@dataclass
class Batch:
    target: torch.Tensor            # [B, K+1, V]
    draft: torch.Tensor             # [B, K, V]
    temperature: torch.Tensor       # [B] float32
    top_k: torch.Tensor             # [B] int32
    top_p: torch.Tensor             # [B] float32
    meta: dict = field(default_factory=dict)


def make_batch(w: Workload, step: int = 0, device="cpu", B: int | None = None,
               chunk_rows: int = 512) -> Batch:
    """The seeded batch for workload `w` at `step` (B may be reduced for tests)."""
    B = w.B if B is None else B
    K, V = w.K, w.V
    g = _generator(device, 0, w.cid, step)
    gp = _generator("cpu", 0, w.cid, step, 7)         # per-sequence parameters, on the host

    if w.name in ("tiny", "mtp_decode"):
        s = torch.full((B,), 1.1)
        alpha = torch.full((B,), 0.7)
        T = torch.full((B,), 1.0)
        k = torch.full((B,), 20, dtype=torch.int32)
        P = torch.full((B,), 0.95)
    elif w.name == "nucleus_batch":
        s = torch.full((B,), 1.1)
        alpha = 0.4 + 0.55 * torch.rand(B, generator=gp)
        T = torch.full((B,), 0.6)
        k = torch.zeros(B, dtype=torch.int32)
        P = torch.full((B,), 0.95)
    elif w.name == "greedy":
        s = torch.full((B,), 1.1)
        alpha = torch.full((B,), 0.7)
        T = torch.zeros(B)
        k = torch.zeros(B, dtype=torch.int32)
        P = torch.ones(B)
    elif w.name == "mixed":
        s = 0.8 + 0.7 * torch.rand(B, generator=gp)
        alpha = 0.2 + 0.75 * torch.rand(B, generator=gp)
        T = 0.3 + 0.9 * torch.rand(B, generator=gp)
        k = torch.tensor([0, 20, 50], dtype=torch.int32)[torch.randint(0, 3, (B,), generator=gp)]
        P = torch.tensor([0.8, 0.95, 1.0])[torch.randint(0, 3, (B,), generator=gp)]
    else:
        raise KeyError(w.name)

    target = torch.empty(B, K + 1, V, dtype=w.dtype, device=device)
    draft = torch.empty(B, K, V, dtype=w.dtype, device=device)
    # rows are generated sequence by sequence in chunks to bound temporary memory
    per_seq = 2 * K + 1
    seqs_per_chunk = max(1, chunk_rows // per_seq)
    for b0 in range(0, B, seqs_per_chunk):
        b1 = min(B, b0 + seqs_per_chunk)
        nb = b1 - b0
        s_rows = s[b0:b1].repeat_interleave(per_seq).to(device)
        z = zipf_rows(nb * per_seq, V, s_rows, g, device).view(nb, per_seq, V)
        tgt = z[:, :K + 1]
        z_own = z[:, K + 1:]                            # independent copies for the drafts
        a = alpha[b0:b1].to(device).view(nb, 1, 1)
        drf = a * tgt[:, :K] + (1 - a) * z_own
        target[b0:b1] = tgt.to(w.dtype)
        draft[b0:b1] = drf.to(w.dtype)
        if w.name == "greedy":
            same = [b - b0 for b in range(b0, b1) if b % 5 == 0]
            if same:
                idx = torch.tensor(same, device=device)
                draft[b0:b1][idx] = target[b0:b1][idx, :K]
    return Batch(target, draft, T.to(torch.float32), k, P.to(torch.float32),
                 meta=dict(alpha=alpha, s=s, workload=w.name, step=step))


def draft_tokens_by_rank(draft: torch.Tensor, step: int = 0, cid: int = 0,
                         max_rank: int = 8) -> torch.Tensor:
    """Synthetic drafted tokens [B, K] int32: for each draft row, the token at a
    random rank r of that row (r = 1 with probability 1/2, 2 with 1/4, ...,
    capped at max_rank). A stand-in for the drafter's own draw that needs no
    sampler; the verifier accepts any token id in [0, V)."""
    B, K, V = draft.shape
    g = _generator("cpu", 0, cid, step, 11)
    u = torch.rand(B, K, generator=g)
    r = torch.clamp((-torch.log2(1.0 - u)).floor().long(), max=max_rank - 1)   # geometric
    top = torch.topk(draft.float(), max_rank, dim=-1).indices                    # [B, K, max_rank]
    return torch.gather(top, -1, r.to(top.device).unsqueeze(-1)).squeeze(-1).to(torch.int32)


def hidden_batch(B: int, K1: int, d: int, V: int, seed: int = 0, device="cpu"):
    """Seeded final hidden states [B, K1, d] and an LM-head weight [V, d], bf16:
    h ~ 0.5 N(0, 1) and W ~ 0.1 N(0, 1) elementwise, so that a logit h . W_v has a
    standard deviation of 0.05 sqrt(d). No trained weights exist here; these stand
    in for a model's last hidden states and its output projection."""
    g = _generator(device, 0, 6, seed)
    h = (0.5 * torch.randn(B, K1, d, generator=g, device=device)).to(torch.bfloat16)
    W = torch.empty(V, d, dtype=torch.bfloat16, device=device)
    for v0 in range(0, V, 16384):                       # bounded fp32 temporaries
        v1 = min(V, v0 + 16384)
        W[v0:v1] = (0.1 * torch.randn(v1 - v0, d, generator=g, device=device)).to(torch.bfloat16)
    return h, W
