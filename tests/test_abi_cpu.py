"""Host-side checks of the C ABI that need no GPU: the library loads, exports every symbol the
header declares, and its pure host queries answer (no kernel is launched here)."""

import os
import re
import subprocess

import pytest

import diffusion_transformer_gb300 as D

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libdit():
    from diffusion_transformer_gb300 import build
    build.build()
    return D.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "dit.h")).read()
    return sorted(set(re.findall(r"DIT_API\s+[\w\s\*]+?\b(dit_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["dit_block_forward", "dit_block_forward_int8", "dit_euler_step", "dit_denoise",
              "dit_workspace_bytes", "dit_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(libdit):
    out = subprocess.run(["nm", "-D", "--defined-only", D.library_path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (dit_\w+)", out))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    for n in _declared():
        getattr(libdit, n)  # resolvable through ctypes too


def test_binding_covers_every_declared_symbol():
    for n in _declared():
        assert hasattr(D, n), n


def test_status_strings_and_version(libdit):
    assert D.dit_version() >= 100
    for s in (0, -1, -2, -3, -4, -5):
        assert D.dit_status_string(s) and D.dit_status_string(s) != "unknown status"


def test_workspace_sizes_host_only(libdit):
    d = D.DitDims(3072, 24, 128, 12288)
    ws = D.dit_workspace_bytes(d, 128, 4096, 0)
    R = 4224
    expect = 2 * R * 3072 + 3 * 24 * R * 128 * 2 + R * 3072 * 2 + R * 12288 * 2
    assert abs(ws - expect) < 8 * 256
    assert D.dit_workspace_bytes(D.DitDims(3072, 24, 96, 12288), 128, 4096, 0) == 0   # unsupported head dim
    assert D.dit_workspace_bytes(d, 128, 0, 0) == 0                                  # no image rows
    assert D.dit_vt_stride(4224) == 4224 and D.dit_vt_stride(4225) == 4232
    assert D.dit_block_noalloc_max_bytes() == 64 << 20
    assert D.dit_workspace_bytes(D.DitDims(3072, 24, 128, 12288), 64, 1024, 0) <= D.dit_block_noalloc_max_bytes()


def test_invalid_arguments_rejected_before_any_cuda_call(libdit):
    import ctypes
    L = libdit
    # null dims / null pointers: validation returns before touching CUDA
    assert L.dit_block_forward(None, None, None, 0, None, 1, None, None, None, None, None, None, 0, None) == -1
    assert L.dit_euler_step(None, None, 5, ctypes.c_float(1.0), ctypes.c_float(0.5), None) == -1
    assert L.dit_rope_tables(4, 2, 2, 96, ctypes.c_float(1e4), ctypes.c_void_p(16), ctypes.c_void_p(16), None) == -2
    assert L.dit_dequant_int8(ctypes.c_void_p(16), ctypes.c_void_p(16), 4, 33, ctypes.c_void_p(16), None) == -2
