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


def _ru(n, a=256):
    return (n + a - 1) // a * a


@pytest.mark.parametrize("H,nh,hd,F,L,N", [(3072, 24, 128, 12288, 128, 4096), (256, 4, 64, 768, 8, 64),
                                           (3072, 24, 128, 12288, 0, 1), (512, 8, 64, 1536, 13, 90)])
def test_workspace_variants_host_only(libdit, H, nh, hd, F, L, N):
    # block workspace: h, q, k, vt (rows padded to 8), o, a, each 256-byte aligned; variants add
    # the int8lin slots (two of the largest dequantised linear), the W8A8 slots and per-row scales,
    # the parallel block's [Wqkv ; Wup] and [Wout | Wdown] slots, the double-stream block's two
    # text + image slots
    d = D.DitDims(H, nh, hd, F)
    R = L + N
    block = (_ru(R * H * 2) + 2 * _ru(nh * R * hd * 2) + _ru(nh * hd * _ru(R, 8) * 2) + _ru(R * H * 2) +
             _ru(R * F * 2))
    slot = _ru(max(3 * H * H, H * H, 2 * F * H, H * F) * 2)
    par = _ru((3 * H + 2 * F) * H * 2) + _ru(H * (H + F) * 2)
    expect = {0: block, 1: block + 2 * slot, 2: block, 3: block, 4: block + 2 * slot + _ru(R * 4),
              5: block + par, 6: block + 4 * slot, 7: block + par + 2 * _ru(R, 64) * 4, 8: block + 4 * slot + _ru(R * 4)}
    for variant, want in expect.items():
        assert D.dit_workspace_bytes(d, L, N, variant) == want, variant
    assert D.dit_workspace_bytes(d, L, N, 9) == 0 and D.dit_workspace_bytes(d, L, N, -1) == 0


def test_new_entries_reject_invalid_arguments_before_any_cuda_call(libdit):
    import ctypes
    L = libdit
    p = ctypes.c_void_p(256)
    # LoRA merge: null pointers, empty sizes
    assert L.dit_lora_merge(None, 4, 4, p, p, 8, p, None) == -1
    assert L.dit_lora_merge(p, 0, 4, p, p, 8, p, None) == -1
    assert L.dit_lora_merge(p, 4, 4, p, p, 0, p, None) == -1
    # int8lin parallel / double-stream blocks: null dims or weights
    args = (None, 0, None, 1, None, None, None, None, None, None, 0, None)
    assert L.dit_parallel_block_forward_int8(None, None, *args) == -1
    assert L.dit_double_block_forward_int8(None, None, None, *args) == -1
    assert L.dit_parallel_block_forward_w8a8(None, None, *args) == -1
    assert L.dit_double_block_forward_w8a8(None, None, None, *args) == -1
    # no-allocation block: every argument is checked before the scratch address is looked up (that
    # lookup is the call's first CUDA call), so on this GPU-less host the errors are the argument
    # errors, never DIT_ECUDA
    na = (None, 0, None, 1, None, None, None, None, None, None)
    assert L.dit_block_forward_noalloc(None, None, *na) == -1
    dims = D.dit_dims(3072, 24, 128, 12288, 1e-6, 1e-6, 0)
    assert L.dit_block_forward_noalloc(ctypes.byref(dims), None, *na) == -1                # no weights, no rows
    bad = D.dit_dims(3072, 24, 96, 12288, 1e-6, 1e-6, 0)
    mod = D.dit_mod(256, None, 1)
    assert L.dit_block_forward_noalloc(ctypes.byref(bad), None, None, 0, p, 1, None, None, p, p,
                                       ctypes.byref(mod), None) == -2                     # head_dim 96
    w = D.dit_block_w(256, 256, 256, 256, None, None, None, None)
    assert L.dit_block_forward_noalloc(ctypes.byref(dims), ctypes.byref(w), None, 0, p, 0, None, None, p, p,
                                       ctypes.byref(mod), None) == -1                     # N = 0
    wmis = D.dit_block_w(256, 258, 256, 256, None, None, None, None)
    assert L.dit_block_forward_noalloc(ctypes.byref(dims), ctypes.byref(wmis), None, 0, p, 8, None, None, p, p,
                                       ctypes.byref(mod), None) == -1                     # misaligned weight
    # the 1024sq shape exceeds the static array: rejected with DIT_EWORKSPACE, still before CUDA
    assert L.dit_block_forward_noalloc(ctypes.byref(dims), ctypes.byref(w), p, 128, p, 4096, p, p, p, p,
                                       ctypes.byref(mod), None) == -3


def test_header_is_plain_c_and_links(libdit, tmp_path):
    # a C11 client (no C++) includes the header, takes every declared entry point's address, links
    # against libdit.so and calls the host-only queries
    import shutil
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    names = _declared()
    src = tmp_path / "client.c"
    src.write_text(
        '#include "dit.h"\n#include <stdio.h>\n'
        "typedef void (*fn_t)(void);\n"
        "static const fn_t fns[] = {\n" + ",\n".join(f"  (fn_t){n}" for n in names) + "\n};\n"
        "int main(void) {\n"
        "  dit_dims d = {3072, 24, 128, 12288, 1e-6f, 1e-6f, 0};\n"
        '  printf("%d %zu %zu %s\\n", dit_version(), sizeof(fns) / sizeof(fns[0]),\n'
        "         dit_workspace_bytes(&d, 128, 4096, 0), dit_status_string(DIT_EWORKSPACE));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "client"
    libdir = os.path.dirname(D.library_path)
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-L", libdir, "-ldit", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert int(out[0]) == D.dit_version() and int(out[1]) == len(names)
    assert int(out[2]) == D.dit_workspace_bytes(D.DitDims(3072, 24, 128, 12288), 128, 4096, 0)
    assert " ".join(out[3:]) == D.dit_status_string(-3)


def test_missing_library_fails_loudly():
    # no fallback: with the library absent every call raises instead of computing anything elsewhere
    import sys
    code = ("import diffusion_transformer_gb300 as D\n"
            "D.library_path = '/nonexistent/libdit.so'\nD._lib = None\n"
            "try:\n    D.dit_version()\nexcept RuntimeError as e:\n    print('raised', e)\n")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT).stdout
    assert out.startswith("raised") and "not built" in out
