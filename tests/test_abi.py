"""Host-side checks of the C ABI (no GPU needed): the library builds, loads,
exports every function include/spec_verify.h declares, and rejects bad
arguments before launching anything."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_30_gb300 as sv
from speculative_decoding_verification_30_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "spec_verify.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:sv_status|size_t|int|const char\*)\s+(\w+)\s*\(",
                                 src, flags=re.M)))


def test_library_builds_and_exports_every_declared_symbol():
    path = _build.build()
    lib = ctypes.CDLL(path)
    names = declared_functions()
    assert {"spec_verify", "spec_verify_workspace_bytes", "spec_truncated_probs",
            "spec_sample", "sv_status_string"} <= set(names)
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
