"""Host-side checks of the C ABI (no GPU needed): the library builds and
exports every entry point that include/moe.h declares, the ctypes structs
match the C layout, and host-detectable errors are returned before any
CUDA work is enqueued."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from ragged_grouped_gemm_gb300 import _lib, build
from ragged_grouped_gemm_gb300.inputs import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_route", "moe_route_from_logits", "moe_permute", "moe_grouped_ffn", "moe_combine",
                     "moe_backward", "moe_update_bias", "moe_workspace_size", "moe_get_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\sT\s(moe_\w+)", out.stdout))
    for name in declared_functions():
        assert name in exported, name
        assert name in _lib.SIGNATURES, name
        assert getattr(lib, name) is not None


def test_ctypes_structs_match_c_layout():
    structs = {"moe_desc_t": _lib.MoeDesc, "moe_expert_weights_t": _lib.MoeExpertWeights,
               "moe_ffn_saved_t": _lib.MoeFfnSaved, "moe_fwd_state_t": _lib.MoeFwdState,
               "moe_grads_t": _lib.MoeGrads, "moe_expert_weights_mx_t": _lib.MoeExpertWeightsMx}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'  printf("{cname} %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'  printf("{cname}.{fname} %zu\\n", offsetof({cname}, {fname}));')
    lines.append("  return 0; }")
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "probe.c")
        exe = os.path.join(tmp, "probe")
        open(src, "w").write("\n".join(lines))
        subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    got = dict(line.rsplit(" ", 1) for line in out.strip().splitlines())
    for cname, py in structs.items():
        assert int(got[cname]) == ctypes.sizeof(py), cname
        for fname, _ in py._fields_:
            assert int(got[f"{cname}.{fname}"]) == getattr(py, fname).offset, (cname, fname)


def _desc(**kw):
    from ragged_grouped_gemm_gb300.api import make_desc
    d = make_desc(CONFIGS["tiny"])
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_workspace_sizes(lib):
    from ragged_grouped_gemm_gb300.api import make_desc
    prev = 0
    for name in ("tiny", "small_softmax", "small_sigmoid", "mixtral", "dsv3"):
        d = make_desc(CONFIGS[name])
        f, b = ctypes.c_size_t(), ctypes.c_size_t()
        assert lib.moe_workspace_size(ctypes.byref(d), ctypes.byref(f), ctypes.byref(b)) == 0
        assert 0 < f.value <= b.value
    d = _desc()
    for n in (1, 100, 1000, 10000):
        d.n_tok = n
        b = ctypes.c_size_t()
        assert lib.moe_workspace_size(ctypes.byref(d), None, ctypes.byref(b)) == 0
        assert b.value >= prev
        prev = b.value


@pytest.mark.parametrize("field,value,code", [
    ("top_k", 0, 1), ("top_k", 9, 1), ("d_model", 96, 1), ("d_ff", 100, 1), ("gate", 2, 1),
    ("n_exp", 2000, 1), ("precision", 3, 2), ("n_shared", 2, 2), ("n_tok", -1, 1), ("top_k", 33, 1),
])
def test_invalid_descriptions_rejected(lib, field, value, code):
    d = _desc(**{field: value})
    b = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(d), None, ctypes.byref(b)) == code
    assert lib.moe_update_bias(ctypes.byref(d), None, None, 1e-3, 0, None) == code


def test_null_and_misaligned_arguments_rejected_on_host(lib):
    d = _desc()
    # no workspace
    assert lib.moe_route(ctypes.byref(d), None, None, None, None, None, None, None, None, None, 0, None) == 3
    # workspace too small
    assert lib.moe_route(ctypes.byref(d), None, None, None, None, None, None, None, None, 256, 16, None) == 3
    f = ctypes.c_size_t()
    lib.moe_workspace_size(ctypes.byref(d), ctypes.byref(f), None)
    big = f.value + 1024
    # null inputs with an adequate (fake, never dereferenced) workspace address
    assert lib.moe_route(ctypes.byref(d), None, None, None, None, None, None, None, None, 4096, big, None) == 1
    assert lib.moe_permute(ctypes.byref(d), None, None, None, None, None, None, 4096, big, None) == 1
    # misaligned
    assert lib.moe_combine(ctypes.byref(d), 4097, 8, 8, None, 8192, None) == 1
    assert lib.moe_update_bias(ctypes.byref(d), 64, 64, 1e-3, 7, None) == 1
    assert lib.moe_get_device_status(None, None, None) == 1


def test_status_strings(lib):
    for code in range(6):
        assert lib.moe_status_string(code)
    assert lib.moe_abi_version() == 1


def test_timing_entry_points_validate_on_host(lib):
    import ctypes as ct
    ms, n, u = ct.c_double(), ct.c_int64(), ct.c_int64()
    assert lib.moe_timing_enable(0) == 1                  # capacity out of range
    assert lib.moe_timing_enable((1 << 20) + 1) == 1
    assert lib.moe_timing_read(4, ct.byref(ms), ct.byref(n), None) == 1     # unknown kind
    assert lib.moe_timing_read(-1, ct.byref(ms), ct.byref(n), None) == 1
    assert lib.moe_timing_read(3, None, ct.byref(n), None) == 1
    assert lib.moe_timing_disable() == 0
    # nothing recorded: zero time, zero launches
    assert lib.moe_timing_read(3, ct.byref(ms), ct.byref(n), ct.byref(u)) == 0
    assert (ms.value, n.value, u.value) == (0.0, 0, 0)


def test_selftest_wait_timeout_validates_on_host(lib):
    # no or misaligned workspace, limit of zero or above one second: rejected before any launch
    assert lib.moe_selftest_wait_timeout(None, 4096, 50000, 1, None) == 3
    assert lib.moe_selftest_wait_timeout(4097, 4096, 50000, 1, None) == 3
    assert lib.moe_selftest_wait_timeout(4096, 4, 50000, 1, None) == 3
    assert lib.moe_selftest_wait_timeout(4096, 4096, 0, 1, None) == 1
    assert lib.moe_selftest_wait_timeout(4096, 4096, 2_000_000_000, 1, None) == 1
