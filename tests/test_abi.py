"""Host-side checks of the C ABI (no GPU needed): the library builds, loads,
exports every function include/*.h declares, and rejects bad arguments before
launching anything."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_30_gb300 as sv
from speculative_decoding_verification_30_gb300 import _build

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include")


def declared_functions():
    names = set()
    for h in sorted(os.listdir(INCLUDE)):
        if not h.endswith(".h"):
            continue
        src = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:sv_status|size_t|int|const char\*)\s+(\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_library_builds_and_exports_every_declared_symbol():
    path = _build.build()
    lib = ctypes.CDLL(path)
    names = declared_functions()
    assert {"spec_verify", "spec_verify_workspace_bytes", "spec_truncated_probs",
            "spec_sample", "sv_status_string", "spec_lm_head_logits", "spec_verify_from_hidden",
            "spec_verify_greedy_from_hidden"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_version_and_status_strings():
    lib = sv.load()
    assert sv.sv_version() >= 100
    for s in range(8):
        assert lib.sv_status_string(s)


def test_workspace_size():
    assert sv.spec_verify_workspace_bytes(64, 4) >= 64 * 5 * 8 + 64 * 4
    assert sv.spec_verify_workspace_bytes(0, 4) == 0


def _verify(**kw):
    lib = sv.load()
    a = dict(t=1 << 12, d=1 << 12, dt=0, tok=1 << 12, T=1 << 12, k=1 << 12, P=1 << 12,
             B=2, K=2, V=1024, ot=1 << 12, on=1 << 12, ws=1 << 12, wsb=1 << 20)
    a.update(kw)
    return lib.spec_verify(a["t"], a["d"], a["dt"], a["tok"], a["T"], a["k"], a["P"], 0, 0,
                           a["B"], a["K"], a["V"], a["ot"], a["on"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(t=None), 1), (dict(tok=None), 1), (dict(ws=None), 1), (dict(ot=None), 1),
    (dict(B=0), 2), (dict(K=0), 2), (dict(K=17), 2), (dict(V=1), 2), (dict(V=262145), 2),
    (dict(dt=7), 3), (dict(wsb=8), 4), (dict(ws=(1 << 12) + 8), 4), (dict(t=(1 << 12) + 1), 6),
])
def test_argument_errors_are_reported_without_launching(kw, status):
    assert _verify(**kw) == status


def test_other_entry_points_validate_arguments():
    lib = sv.load()
    assert lib.spec_truncated_probs(None, 0, 1, 10, 1 << 12, 1 << 12, 1 << 12, 1 << 12, None) == 1
    assert lib.spec_truncated_probs(1 << 12, 0, 0, 10, 1 << 12, 1 << 12, 1 << 12, 1 << 12, None) == 2
    assert lib.spec_sample(1 << 12, 1, 1, 1, 1, 1 << 12, 1 << 12, 1 << 12, 0, 0, 1 << 12, None) == 2
    assert lib.spec_philox_uniforms(0, 0, 0, 1, 1 << 12, None) == 2
    assert lib.spec_philox_uniforms(0, 0, 1, 1, None, None) == 1


def test_noalloc_entry_point_rejects_oversized_batches_before_any_cuda_call():
    lib = sv.load()
    args = lambda B, K: (1 << 12, 1 << 12, 0, 1 << 12, 1 << 12, 1 << 12, 1 << 12, 0, 0, B, K,
                         1024, 1 << 12, 1 << 12, None)
    need = sv.spec_verify_workspace_bytes(65535, 16)
    assert need > sv.NOALLOC_SCRATCH_BYTES
    assert lib.spec_verify_noalloc(*args(65535, 16)) == 7
    assert lib.spec_verify_noalloc(*args(0, 4)) == 2
    assert lib.spec_verify_noalloc(*args(4, 17)) == 2


def test_lm_head_entry_points_validate_before_launching():
    lib = sv.load()
    A = 1 << 12

    def lm(h=A, w=A, M=128, N=256, d=128, z=A, f=A):
        return lib.spec_lm_head_logits(h, w, M, N, d, z, f, None)
    assert lm(h=None) == 1 and lm(z=None) == 1 and lm(f=None) == 1
    assert lm(M=0) == 2 and lm(N=0) == 2 and lm(d=0) == 2 and lm(d=96) == 2 and lm(d=65600) == 2
    assert lm(N=65535 * 256 + 1) == 2 and lm(M=2**31 - 128) == 2
    assert lm(h=A + 8) == 6 and lm(w=A + 4) == 6 and lm(z=A + 2) == 6

    wsb = sv.spec_verify_workspace_bytes(2, 2)

    def vh(ht=A, wt=A, d=128, hd=A, wd=A, dd=64, B=2, K=2, V=1024, z=A, ws=A, wsb=wsb):
        return lib.spec_verify_from_hidden(ht, wt, d, hd, wd, dd, A, A, A, A, 0, 0, B, K, V, z, A, A, A,
                                           ws, wsb, None)
    assert vh(ht=None) == 1 and vh(z=None) == 1 and vh(ws=None) == 1
    assert vh(hd=None) == 1                    # draft hidden states without their weight
    assert vh(B=0) == 2 and vh(K=17) == 2 and vh(V=1) == 2 and vh(V=262145) == 2
    assert vh(d=65) == 2 and vh(dd=100) == 2
    assert vh(z=A + 4) == 6 and vh(ht=A + 8) == 6
    assert vh(wsb=8) == 4

    def gh(ht=A, w=A, d=128, dt=A, B=2, K=2, V=1024, f=A, ot=A, on=A, ws=A, wsb=wsb):
        return lib.spec_verify_greedy_from_hidden(ht, w, d, dt, B, K, V, f, ot, on, ws, wsb, None)
    assert gh(ht=None) == 1 and gh(w=None) == 1 and gh(dt=None) == 1 and gh(f=None) == 1
    assert gh(ot=None) == 1 and gh(on=None) == 1 and gh(ws=None) == 1
    assert gh(B=0) == 2 and gh(B=65536) == 2 and gh(K=0) == 2 and gh(K=17) == 2
    assert gh(V=1) == 2 and gh(V=262145) == 2 and gh(d=0) == 2 and gh(d=96) == 2 and gh(d=65600) == 2
    assert gh(ht=A + 8) == 6 and gh(w=A + 4) == 6 and gh(dt=A + 2) == 6 and gh(on=A + 1) == 6
    assert gh(ws=A + 8) == 4 and gh(wsb=wsb - 1) == 4


def test_launch_cache_is_per_device_and_thread_safe():
    # Grid sizes and kernel attributes are cached per (device, kernel, shared memory):
    # a process driving two GPUs must not reuse the first GPU's SM count on the
    # second. The hook runs the library's cache with two fake devices (152 and 132
    # SMs, two CTAs per SM) from eight host threads, without a GPU.
    lib = sv.load()
    lib.sv_test_launch_cache.argtypes = [ctypes.c_void_p]
    lib.sv_test_launch_cache.restype = ctypes.c_int
    out = (ctypes.c_int * 6)()
    assert lib.sv_test_launch_cache(ctypes.cast(out, ctypes.c_void_p)) == 0
    assert list(out[:4]) == [152 * 2, 132 * 2, 152 * 2 + 1, 132 * 2 + 1]
    assert out[4] == 4            # one entry per (device, kernel)
    assert out[5] == 1            # every thread saw the same values


def test_binding_rejects_bad_tensors_before_calling_the_library():
    # argument marshalling only: shape and device errors surface as SpecVerifyError
    # before anything reaches the C ABI (no GPU needed)
    import torch
    h = torch.zeros(2, 3, 64, dtype=torch.bfloat16)
    W = torch.zeros(100, 128, dtype=torch.bfloat16)
    dt = torch.zeros(2, 2, dtype=torch.int32)
    with pytest.raises(sv.SpecVerifyError, match="weight must be"):
        sv.spec_verify_greedy_from_hidden(h, W, dt)
    with pytest.raises(sv.SpecVerifyError, match="weight must be"):
        sv.spec_lm_head_logits(h, W)
    W64 = torch.zeros(100, 64, dtype=torch.bfloat16)
    flag = torch.zeros(1, dtype=torch.int32)
    out, n = torch.zeros(2, 3, dtype=torch.int32), torch.zeros(2, dtype=torch.int32)
    ws = type("W", (), {"buf": torch.zeros(16, dtype=torch.uint8), "nbytes": 16})()
    with pytest.raises(sv.SpecVerifyError, match="CUDA tensor"):
        sv.spec_verify_greedy_from_hidden(h, W64, dt, flag=flag, out_tokens=out, out_n=n, workspace=ws)
