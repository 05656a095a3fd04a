"""The C ABI library: it builds, loads, exports every declared symbol, and
its host-side checks reject bad arguments before touching a device.  No GPU
compute here."""
import ctypes
import os
import re
import subprocess

import pytest

import speculative_decoding_verification_23_gb300 as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    return sv.load_library()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "spec_verify.h")).read()
    return sorted(set(re.findall(r"^\s*(?:size_t|int64_t|int|const char \*)\s*\**(spec_\w+)\(", text, re.M)))


def test_header_declares_the_python_names():
    assert sorted(sv.EXPORTED) == _declared_symbols()


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", sv.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (spec_\w+)", out))
    for name in _declared_symbols():
        assert name in exported, name
        assert hasattr(lib, name)


def test_struct_layout_matches_header(tmp_path):
    """Field offsets of the ctypes mirror equal the C compiler's."""
    fields = [f[0] for f in sv.SpecArgs._fields_]
    c = tmp_path / "layout.c"
    body = "\n".join(f'  printf("{f} %zu\\n", offsetof(spec_args, {f}));' for f in fields)
    c.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "spec_verify.h"\n'
                 'int main(void) {\n' + body + '\n  printf("size %zu\\n", sizeof(spec_args));\n  return 0;\n}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(c), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                        check=True).stdout.splitlines())
    for f in fields:
        assert int(got[f]) == getattr(sv.SpecArgs, f).offset, f
    assert int(got["size"]) == ctypes.sizeof(sv.SpecArgs)


def test_status_strings(lib):
    assert sv.status_string(0) == "ok"
    for code in range(-8, 0):
        assert sv.status_string(code) != "unknown status"


def test_workspace_size_grows_with_batch(lib):
    a = sv.spec_workspace_bytes(1, 4, 1024)
    b = sv.spec_workspace_bytes(64, 512, 152064)
    assert 0 < a < b and b % 256 == 0


@pytest.mark.parametrize("B,total", [(1, 0), (3, 7), (256, 1152), (4096, 32768)])
def test_workspace_covers_the_top_p_records(lib, B, total):
    """The top-p path keeps a 32-byte record per logical row (2 total + B),
    one word, and kept-token lists of 1024 int32 entries per row on average
    (2^23 at most): spec_workspace_bytes covers them for any V."""
    nr = 2 * total + B
    need = nr * 32 + 4 * min(nr * 1024, 1 << 23)
    for V in (16, 152064):
        assert sv.spec_workspace_bytes(B, total, V) >= need


def _args(**kw):
    a = sv.SpecArgs()
    a.B, a.V, a.total_drafts, a.max_k, a.dtype = 1, 16, 1, 1, sv.SPEC_F32
    a.cu_draft, a.target_logits, a.ld_target = 256, 512, 16
    a.draft_logits, a.ld_draft, a.draft_tokens = 1024, 16, 2048
    a.temperature = a.tv_budget = a.uniforms = 4096
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _call(lib, a, ws_bytes=None, ws=1 << 20):
    n = sv.spec_workspace_bytes(a.B, a.total_drafts, a.V) if ws_bytes is None else ws_bytes
    return lib.spec_verify_sample(ctypes.byref(a), 8192, 8192, None, ws, n, None)


def test_host_checks_reject_bad_arguments(lib):
    assert lib.spec_verify_sample(None, None, None, None, None, 0, None) == sv.SPEC_ERR_NULL
    assert _call(lib, _args(dtype=7)) == sv.SPEC_ERR_DTYPE
    assert _call(lib, _args(max_k=33)) == sv.SPEC_ERR_K_TOO_LARGE
    assert _call(lib, _args(B=0)) == sv.SPEC_ERR_SHAPE
    assert _call(lib, _args(ld_target=8)) == sv.SPEC_ERR_SHAPE
    assert _call(lib, _args(target_logits=520)) == sv.SPEC_ERR_ALIGN
    assert _call(lib, _args(ld_target=17)) == sv.SPEC_ERR_ALIGN
    assert _call(lib, _args(dtype=sv.SPEC_BF16, ld_target=20, ld_draft=24)) == sv.SPEC_ERR_ALIGN
    assert _call(lib, _args(uniforms=0)) == sv.SPEC_ERR_NULL
    assert _call(lib, _args(), ws_bytes=16) == sv.SPEC_ERR_WORKSPACE
    assert _call(lib, _args(), ws=(1 << 20) + 64) == sv.SPEC_ERR_WORKSPACE
    assert _call(lib, _args(total_drafts=5)) == sv.SPEC_ERR_SHAPE   # more drafts than B*max_k


def test_no_device_is_an_error_not_a_fallback(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _call(lib, _args()) == sv.SPEC_ERR_DEVICE
    a = _args()
    n = sv.spec_workspace_bytes(1, 1, 16)
    assert lib.spec_verify_greedy(ctypes.byref(a), 8192, 8192, None, 1 << 20, n, None) == sv.SPEC_ERR_DEVICE
