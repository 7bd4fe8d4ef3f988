"""GB300-native speculative-decoding verify-and-sample.

Thin Python binding over the C ABI in include/spec_verify.h (libspec_verify.so,
built in-tree by `_build.build()`). The binding only marshals arguments:
every step of the computation runs in the library's CUDA kernels. PyTorch is
used for device memory and streams. There is no CPU fallback: the calls raise
if the library is missing or a tensor is not on a CUDA device.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB, build

__all__ = ["load", "spec_verify", "spec_verify_noalloc", "spec_verify_workspace_bytes",
           "spec_truncated_probs", "NOALLOC_SCRATCH_BYTES",
           "spec_sample", "spec_philox_uniforms", "spec_lm_head_logits", "spec_verify_from_hidden",
           "spec_verify_greedy_from_hidden", "sv_version", "Workspace", "SV_BF16", "SV_F32", "SpecVerifyError"]

SV_BF16, SV_F32 = 0, 1
_STATUS = {0: "ok", 1: "null pointer", 2: "shape", 3: "dtype", 4: "workspace", 5: "cuda",
           6: "alignment", 7: "scratch"}
NOALLOC_SCRATCH_BYTES = 1 << 20     # SV_NOALLOC_SCRATCH_BYTES in include/spec_verify.h
_lib = None


class SpecVerifyError(RuntimeError):
    pass


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the in-tree CUDA library."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB
    if not os.path.exists(path):
        build()
    lib = ctypes.CDLL(path)
    vp, i32, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
    lib.spec_verify_workspace_bytes.argtypes = [i32, i32]
    lib.spec_verify_workspace_bytes.restype = sz
    lib.spec_verify.argtypes = [vp, vp, i32, vp, vp, vp, vp, u64, u64, i32, i32, i32, vp, vp,
                                vp, sz, vp]
    lib.spec_verify.restype = i32
    lib.spec_verify_noalloc.argtypes = [vp, vp, i32, vp, vp, vp, vp, u64, u64, i32, i32, i32, vp,
                                        vp, vp]
    lib.spec_verify_noalloc.restype = i32
    lib.spec_truncated_probs.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp]
    lib.spec_truncated_probs.restype = i32
    lib.spec_sample.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, u64, u64, vp, vp]
    lib.spec_sample.restype = i32
    lib.spec_philox_uniforms.argtypes = [u64, u64, i32, i32, vp, vp]
    lib.spec_philox_uniforms.restype = i32
    lib.spec_verify_step.argtypes = [vp, vp, i32, vp, vp, vp, vp, u64, vp, i32, i32, i32, vp, vp,
                                     vp, vp, vp, sz, vp]
    lib.spec_verify_step.restype = i32
    lib.spec_accept_histogram.argtypes = [vp, i32, i32, vp, vp]
    lib.spec_accept_histogram.restype = i32
    lib.spec_lm_head_logits.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
    lib.spec_lm_head_logits.restype = i32
    lib.spec_verify_from_hidden.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp, vp, vp, u64, u64, i32,
                                            i32, i32, vp, vp, vp, vp, vp, sz, vp]
    lib.spec_verify_from_hidden.restype = i32
    lib.spec_verify_greedy_from_hidden.argtypes = [vp, vp, i32, vp, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    lib.spec_verify_greedy_from_hidden.restype = i32
    lib.sv_status_string.argtypes = [i32]
    lib.sv_status_string.restype = ctypes.c_char_p
    lib.sv_version.argtypes = []
    lib.sv_version.restype = i32
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        msg = load().sv_status_string(status).decode()
        raise SpecVerifyError(f"{what}: {msg} (status {status})")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    raise SpecVerifyError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise SpecVerifyError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise SpecVerifyError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise SpecVerifyError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def sv_version() -> int:
    return int(load().sv_version())


def spec_verify_workspace_bytes(B: int, K: int) -> int:
    return int(load().spec_verify_workspace_bytes(B, K))


class Workspace:
    """Zero-initialised device workspace for spec_verify (reused across calls on one stream)."""

    def __init__(self, B: int, K: int, device=None):
        self.B, self.K = B, K
        self.nbytes = spec_verify_workspace_bytes(B, K)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device or "cuda")

    def fits(self, B: int, K: int) -> bool:
        return spec_verify_workspace_bytes(B, K) <= self.nbytes


def spec_verify(target: torch.Tensor, draft: torch.Tensor | None, draft_tokens: torch.Tensor,
                temperature: torch.Tensor, top_k: torch.Tensor, top_p: torch.Tensor,
                seed: int, offset: int, out_tokens: torch.Tensor | None = None,
                out_n: torch.Tensor | None = None, workspace: Workspace | None = None,
                stream=None):
    """Verify-and-sample for a batch; returns (out_tokens [B, K+1] int32, n_accepted [B] int32)."""
    B, K1, V = target.shape
    K = K1 - 1
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty(B, K + 1, dtype=torch.int32, device=dev)
    if out_n is None:
        out_n = torch.empty(B, dtype=torch.int32, device=dev)
    if workspace is None or not workspace.fits(B, K):
        workspace = Workspace(B, K, dev)
    if draft is not None and (draft.shape != (B, K, V) or draft.dtype != target.dtype):
        raise SpecVerifyError("draft must be [B, K, V] with the target's dtype")
    st = load().spec_verify(
        _dev(target, "target"), None if draft is None else _dev(draft, "draft"),
        _dtype_code(target), _dev(draft_tokens, "draft_tokens", torch.int32),
        _dev(temperature, "temperature", torch.float32), _dev(top_k, "top_k", torch.int32),
        _dev(top_p, "top_p", torch.float32), seed & (2**64 - 1), offset & (2**64 - 1), B, K, V,
        _dev(out_tokens, "out_tokens", torch.int32), _dev(out_n, "out_n", torch.int32),
        workspace.buf.data_ptr(), workspace.nbytes, _stream(stream))
    _check(st, "spec_verify")
    return out_tokens, out_n


def spec_verify_noalloc(target: torch.Tensor, draft: torch.Tensor | None,
                        draft_tokens: torch.Tensor, temperature: torch.Tensor,
                        top_k: torch.Tensor, top_p: torch.Tensor, seed: int, offset: int,
                        out_tokens: torch.Tensor | None = None, out_n: torch.Tensor | None = None,
                        stream=None):
    """spec_verify with the library's fixed device scratch instead of a workspace.

    Calls on one device must not overlap (they share the scratch); batches whose
    workspace would exceed NOALLOC_SCRATCH_BYTES raise (status 7)."""
    B, K1, V = target.shape
    K = K1 - 1
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty(B, K + 1, dtype=torch.int32, device=dev)
    if out_n is None:
        out_n = torch.empty(B, dtype=torch.int32, device=dev)
    if draft is not None and (draft.shape != (B, K, V) or draft.dtype != target.dtype):
        raise SpecVerifyError("draft must be [B, K, V] with the target's dtype")
    st = load().spec_verify_noalloc(
        _dev(target, "target"), None if draft is None else _dev(draft, "draft"),
        _dtype_code(target), _dev(draft_tokens, "draft_tokens", torch.int32),
        _dev(temperature, "temperature", torch.float32), _dev(top_k, "top_k", torch.int32),
        _dev(top_p, "top_p", torch.float32), seed & (2**64 - 1), offset & (2**64 - 1), B, K, V,
        _dev(out_tokens, "out_tokens", torch.int32), _dev(out_n, "out_n", torch.int32),
        _stream(stream))
    _check(st, "spec_verify_noalloc")
    return out_tokens, out_n


def spec_truncated_probs(logits: torch.Tensor, temperature: torch.Tensor, top_k: torch.Tensor,
                         top_p: torch.Tensor, out: torch.Tensor | None = None, stream=None):
    """Truncated, renormalised fp32 distributions of R rows [R, V] (per-row parameters)."""
    R, V = logits.shape
    if out is None:
        out = torch.empty(R, V, dtype=torch.float32, device=logits.device)
    st = load().spec_truncated_probs(
        _dev(logits, "logits"), _dtype_code(logits), R, V,
        _dev(temperature, "temperature", torch.float32), _dev(top_k, "top_k", torch.int32),
        _dev(top_p, "top_p", torch.float32), _dev(out, "out", torch.float32), _stream(stream))
    _check(st, "spec_truncated_probs")
    return out


def spec_sample(logits: torch.Tensor, temperature: torch.Tensor, top_k: torch.Tensor,
                top_p: torch.Tensor, seed: int, offset: int, out: torch.Tensor | None = None,
                stream=None):
    """Draft-side sampler over [B, K, V] rows with per-sequence parameters -> [B, K] int32."""
    B, K, V = logits.shape
    if out is None:
        out = torch.empty(B, K, dtype=torch.int32, device=logits.device)
    st = load().spec_sample(
        _dev(logits, "logits"), _dtype_code(logits), B, K, V,
        _dev(temperature, "temperature", torch.float32), _dev(top_k, "top_k", torch.int32),
        _dev(top_p, "top_p", torch.float32), seed & (2**64 - 1), offset & (2**64 - 1),
        _dev(out, "out", torch.int32), _stream(stream))
    _check(st, "spec_sample")
    return out


def spec_philox_uniforms(seed: int, offset: int, B: int, K1: int, device="cuda", stream=None):
    """The library's Philox grid indices [B, K1, 2] (acceptance, sampling) as int64."""
    out = torch.empty(B * K1 * 2, dtype=torch.int32, device=device)
    st = load().spec_philox_uniforms(seed & (2**64 - 1), offset & (2**64 - 1), B, K1,
                                     out.data_ptr(), _stream(stream))
    _check(st, "spec_philox_uniforms")
    return (out.to(torch.int64) & 0xFFFFFFFF).view(B, K1, 2)


def spec_accept_histogram(n_accepted: torch.Tensor, K: int, hist: torch.Tensor | None = None,
                          stream=None) -> torch.Tensor:
    """Adds out_n_accepted of one verify call to an acceptance histogram [K+2] (int64 on
    the device; bins 0..K count accepted-prefix lengths, bin K+1 data errors)."""
    B = n_accepted.numel()
    if hist is None:
        hist = torch.zeros(K + 2, dtype=torch.int64, device=n_accepted.device)
    if hist.numel() != K + 2 or hist.dtype != torch.int64 or not hist.is_contiguous():
        raise ValueError("hist must be a contiguous int64 tensor of K+2 counters")
    st = load().spec_accept_histogram(_dev(n_accepted, "n_accepted", torch.int32), B, K,
                                      _dev(hist, "hist"), _stream(stream))
    _check(st, "spec_accept_histogram")
    return hist


def spec_verify_step(target: torch.Tensor, draft: torch.Tensor | None, draft_tokens: torch.Tensor,
                     temperature: torch.Tensor, top_k: torch.Tensor, top_p: torch.Tensor,
                     seed: int, offset: torch.Tensor, out_tokens: torch.Tensor,
                     out_n: torch.Tensor, workspace: Workspace,
                     next_token: torch.Tensor | None = None, seq_len: torch.Tensor | None = None,
                     stream=None):
    """A graph-capturable verify step: the Philox offset lives in `offset` (a one-element
    int64 device tensor, advanced by one per step); `next_token` [B] receives each
    sequence's last emitted token and `seq_len` [B] grows by the tokens emitted."""
    B, K1, V = target.shape
    K = K1 - 1
    if offset.numel() != 1 or offset.dtype != torch.int64:
        raise SpecVerifyError("offset must be a one-element int64 device tensor")
    if not workspace.fits(B, K):
        raise SpecVerifyError("workspace too small for this batch")
    if draft is not None and (draft.shape != (B, K, V) or draft.dtype != target.dtype):
        raise SpecVerifyError("draft must be [B, K, V] with the target's dtype")
    st = load().spec_verify_step(
        _dev(target, "target"), None if draft is None else _dev(draft, "draft"),
        _dtype_code(target), _dev(draft_tokens, "draft_tokens", torch.int32),
        _dev(temperature, "temperature", torch.float32), _dev(top_k, "top_k", torch.int32),
        _dev(top_p, "top_p", torch.float32), seed & (2**64 - 1), _dev(offset, "offset"), B, K, V,
        _dev(out_tokens, "out_tokens", torch.int32), _dev(out_n, "out_n", torch.int32),
        None if next_token is None else _dev(next_token, "next_token", torch.int32),
        None if seq_len is None else _dev(seq_len, "seq_len", torch.int32),
        workspace.buf.data_ptr(), workspace.nbytes, _stream(stream))
    _check(st, "spec_verify_step")


def spec_lm_head_logits(hidden: torch.Tensor, weight: torch.Tensor, out: torch.Tensor | None = None,
                        flag: torch.Tensor | None = None, stream=None):
    """logits [..., V] fp32 = hidden [..., d] . weight [V, d]^T on the tensor cores
    (bf16 operands). Returns (logits, flag); flag [1] int32 becomes 1 if a wait of
    the kernel timed out."""
    d = hidden.shape[-1]
    V = weight.shape[0]
    if weight.dim() != 2 or weight.shape[1] != d:
        raise SpecVerifyError("weight must be [V, d] with the hidden states' d")
    M = hidden.numel() // d
    dev = hidden.device
    if out is None:
        out = torch.empty(*hidden.shape[:-1], V, dtype=torch.float32, device=dev)
    if flag is None:
        flag = torch.zeros(1, dtype=torch.int32, device=dev)
    st = load().spec_lm_head_logits(_dev(hidden, "hidden", torch.bfloat16), _dev(weight, "weight", torch.bfloat16),
                                    M, V, d, _dev(out, "out", torch.float32), _dev(flag, "flag", torch.int32),
                                    _stream(stream))
    _check(st, "spec_lm_head_logits")
    return out, flag


def spec_verify_from_hidden(hidden_target: torch.Tensor, weight_target: torch.Tensor,
                            hidden_draft: torch.Tensor | None, weight_draft: torch.Tensor | None,
                            draft_tokens: torch.Tensor, temperature: torch.Tensor,
                            top_k: torch.Tensor, top_p: torch.Tensor, seed: int = 0, offset: int = 0,
                            logits_scratch: torch.Tensor | None = None,
                            flag: torch.Tensor | None = None, out_tokens: torch.Tensor | None = None,
                            out_n: torch.Tensor | None = None, workspace: "Workspace | None" = None,
                            stream=None):
    """spec_verify on logit rows computed from hidden states on the tensor cores:
    hidden_target [B, K+1, d] and weight_target [V, d] (bf16) give the target rows,
    hidden_draft [B, K, d'] and weight_draft [V, d'] the draft rows (None for a
    greedy batch). Returns (out_tokens, out_n, flag); the results are valid only
    when flag stays 0 (a timed-out wait of a GEMM sets it)."""
    B, K1, d = hidden_target.shape
    K = K1 - 1
    V = weight_target.shape[0]
    dev = hidden_target.device
    if logits_scratch is None:
        logits_scratch = torch.empty(B * (2 * K + 1) * V, dtype=torch.float32, device=dev)
    if flag is None:
        flag = torch.zeros(1, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(B, K + 1, dtype=torch.int32, device=dev)
    if out_n is None:
        out_n = torch.empty(B, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = Workspace(B, K, dev)
    hd = _dev(hidden_draft, "hidden_draft", torch.bfloat16) if hidden_draft is not None else None
    wd = _dev(weight_draft, "weight_draft", torch.bfloat16) if weight_draft is not None else None
    dd = hidden_draft.shape[-1] if hidden_draft is not None else 64
    st = load().spec_verify_from_hidden(
        _dev(hidden_target, "hidden_target", torch.bfloat16),
        _dev(weight_target, "weight_target", torch.bfloat16), d, hd, wd, dd,
        _dev(draft_tokens, "draft_tokens", torch.int32), _dev(temperature, "temperature", torch.float32),
        _dev(top_k, "top_k", torch.int32), _dev(top_p, "top_p", torch.float32), seed, offset, B, K, V,
        _dev(logits_scratch, "logits_scratch", torch.float32), _dev(flag, "flag", torch.int32),
        _dev(out_tokens, "out_tokens", torch.int32), _dev(out_n, "out_n", torch.int32),
        workspace.buf.data_ptr(), workspace.nbytes, _stream(stream))
    _check(st, "spec_verify_from_hidden")
    return out_tokens, out_n, flag


def spec_verify_greedy_from_hidden(hidden_target: torch.Tensor, weight: torch.Tensor,
                                   draft_tokens: torch.Tensor, flag: torch.Tensor | None = None,
                                   out_tokens: torch.Tensor | None = None, out_n: torch.Tensor | None = None,
                                   workspace: "Workspace | None" = None, stream=None):
    """Greedy (temperature 0) verify fused with the LM head: hidden_target
    [B, K+1, d] and weight [V, d] (bf16) give the target rows, whose argmax the
    GEMM epilogue keeps without writing the logits. Returns (out_tokens, out_n,
    flag); the results are valid only when flag stays 0."""
    B, K1, d = hidden_target.shape
    K = K1 - 1
    V = weight.shape[0]
    if weight.dim() != 2 or weight.shape[1] != d:
        raise SpecVerifyError("weight must be [V, d] with the hidden states' d")
    dev = hidden_target.device
    if flag is None:
        flag = torch.zeros(1, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty(B, K + 1, dtype=torch.int32, device=dev)
    if out_n is None:
        out_n = torch.empty(B, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = Workspace(B, K, dev)
    st = load().spec_verify_greedy_from_hidden(
        _dev(hidden_target, "hidden_target", torch.bfloat16), _dev(weight, "weight", torch.bfloat16), d,
        _dev(draft_tokens, "draft_tokens", torch.int32), B, K, V, _dev(flag, "flag", torch.int32),
        _dev(out_tokens, "out_tokens", torch.int32), _dev(out_n, "out_n", torch.int32),
        workspace.buf.data_ptr(), workspace.nbytes, _stream(stream))
    _check(st, "spec_verify_greedy_from_hidden")
    return out_tokens, out_n, flag
