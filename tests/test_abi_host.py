"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point the header declares, and rejects bad arguments before
launching anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsc.h")


@pytest.fixture(scope="module")
def L():
    from dynamic_short_convolution_gb300 import build, _abi

    build.build()
    return _abi.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsc_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_abi():
    names = _declared()
    for n in ("dsc_fwd", "dsc_bwd", "dsc_lowrank_fwd", "dsc_lowrank_bwd", "dsc_lowrank_bwd_workspace_bytes",
              "dsc_static_fwd", "dsc_static_bwd", "dsc_decode_step", "dsc_status_string", "dsc_sync_status"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    from dynamic_short_convolution_gb300 import _abi

    for n in _declared():
        assert hasattr(L, n), f"libdsc.so does not export {n}"
        assert n in _abi.SIGNATURES, f"binding has no signature for {n}"


def test_header_compiles_as_c_and_links(L, tmp_path):
    """A plain C99 program includes the header, links libdsc.so and gets an argument error back (no GPU call)."""
    import shutil
    import subprocess

    from dynamic_short_convolution_gb300 import build

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(build.nvcc()))), "include")
    src = tmp_path / "use_dsc.c"
    src.write_text(
        "#include <stdio.h>\n#include \"dsc.h\"\n"
        "int main(void) {\n"
        "    dsc_status s = dsc_fwd(0, 0, 0, 0, 8, 64, 4, 1, DSC_BF16, 0, 0, 0);\n"
        "    printf(\"%d %s\\n\", dsc_version(), dsc_status_string(s));\n"
        "    return s == DSC_ERR_INVALID_ARG ? 0 : 1;\n"
        "}\n")
    exe = tmp_path / "use_dsc"
    libdir = os.path.dirname(build.LIB)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror=implicit-function-declaration", "-I",
                        os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe), "-L", libdir,
                        "-ldsc", f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and "DSC_ERR_INVALID_ARG" in r.stdout, r.stdout + r.stderr


def test_binding_refuses_host_tensors():
    """The Python entry points take CUDA tensors only; host tensors are refused before the library is used."""
    import torch

    import dynamic_short_convolution_gb300 as dsc

    x = torch.zeros(1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        dsc.dsc_fwd(x, torch.zeros(1, 8, 4, 4, dtype=torch.bfloat16))
    with pytest.raises(TypeError):
        dsc.dsc_static_fwd(x, torch.zeros(64, 4, dtype=torch.bfloat16))
    with pytest.raises(TypeError):
        dsc.dsc_decode_step(x[0], torch.zeros(8, 4, 4, dtype=torch.bfloat16), None, None)


def test_status_strings(L):
    assert L.dsc_status_string(0) == b"DSC_OK"
    assert L.dsc_status_string(4) == b"DSC_ERR_TIMEOUT"
    assert L.dsc_version() >= 10000


def test_rejects_bad_arguments_before_any_launch(L):
    p = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    bf16, f32 = 1, 0
    # non-positive sizes, W out of range, D % H != 0, bad dtype, n_docs < 1 with offsets
    assert L.dsc_fwd(p, p, p, 0, 8, 64, 4, 1, bf16, None, 0, None) == 1
    assert L.dsc_fwd(p, p, p, 1, 8, 64, 9, 1, bf16, None, 0, None) == 1
    assert L.dsc_fwd(p, p, p, 1, 8, 64, 0, 1, bf16, None, 0, None) == 1
    assert L.dsc_fwd(p, p, p, 1, 8, 64, 4, 3, bf16, None, 0, None) == 1
    assert L.dsc_fwd(p, p, p, 1, 8, 64, 4, 1, 7, None, 0, None) == 1
    assert L.dsc_fwd(p, p, p, 1, 8, 64, 4, 1, bf16, p, 0, None) == 1
    assert L.dsc_fwd(None, p, p, 1, 8, 64, 4, 1, bf16, None, 0, None) == 1
    assert L.dsc_fwd(ctypes.c_void_p(0x10001), p, p, 1, 8, 64, 4, 1, bf16, None, 0, None) == 1  # not element-aligned
    assert L.dsc_bwd(p, p, p, p, None, 1, 8, 64, 4, 1, bf16, None, 0, None) == 1
    assert L.dsc_fwd(p, p, p, 1 << 16, 1 << 16, 8, 4, 1, bf16, None, 0, None) == 1  # int32 size limit
    # low-rank: fp32 unsupported, R out of range unsupported
    assert L.dsc_lowrank_fwd(p, p, p, p, p, 1, 8, 64, 4, 16, f32, None, 0, None) == 2
    # (every call below is rejected before any launch: the pointers are not device memory)
    for r in (12, 264, 512):  # R a multiple of 8, at most 256
        assert L.dsc_lowrank_fwd(p, p, p, p, p, 1, 8, 64, 4, r, bf16, None, 0, None) == 2
        assert L.dsc_lowrank_bwd(p, p, p, p, p, p, p, p, p, None, 1, 8, 64, 4, r, bf16, None, 0, None) == 2
        assert L.dsc_lowrank_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 8, 64, 4, r, bf16, None, 0, None) == 2
    assert L.dsc_lowrank_fwd(p, p, p, p, p, 1, 8, 64, 4, 0, bf16, None, 0, None) == 1
    assert L.dsc_lowrank_bwd(p, p, p, p, p, p, p, p, p, None, 1, 8, 64, 4, 0, bf16, None, 0, None) == 1
    assert L.dsc_lowrank_bwd(p, p, p, p, None, p, p, p, p, None, 1, 8, 64, 4, 16, bf16, None, 0, None) == 1  # no dy
    # the backward's workspace: 16 bytes per filter column (the bias rows) and 256 rows of padding, rounded up
    # to 1 KB, then the reordered copy of U (2 bytes per element), whatever B and T; a null workspace is refused
    for b, t, r in ((8, 2048, 8), (1, 5, 64), (8, 2048, 256)):
        rows = (16 * (2048 * 4 + 256) + 1023) // 1024 * 1024
        assert L.dsc_lowrank_bwd_workspace_bytes(b, t, 2048, 4, r) == rows + (2 * r * 2048 * 4 + 255) // 256 * 256
    assert L.dsc_lowrank_bwd(p, p, p, p, p, p, p, p, p, None, 1, 8, 64, 4, 16, bf16, None, 0, None) == 1
    # the allocation-free entry point's array holds 8 MiB of workspace: D = 16384, W = 4, R = 64 needs 9 MiB
    assert L.dsc_lowrank_bwd_workspace_bytes(1, 8, 16384, 4, 64) > 8 << 20
    assert L.dsc_lowrank_bwd_noalloc(p, p, p, p, p, p, p, p, p, 1, 8, 16384, 4, 64, bf16, None, 0, None) == 1
    # the low-rank forward with z from the layer input: its own limits (R <= 128, Dm % 8 == 0) and pointers
    def zp(x, h, W1, b1, U, bias, y, *rest):
        return L.dsc_lowrank_zproj_fwd(x, h, W1, b1, U, bias, y, *rest)
    assert zp(p, p, p, None, p, p, p, 1, 8, 64, 64, 4, 64, f32, None, 0, None) == 2
    assert zp(p, p, p, None, p, p, p, 1, 8, 64, 64, 4, 136, bf16, None, 0, None) == 2
    assert zp(p, p, p, p, p, p, p, 1, 8, 64, 60, 4, 64, bf16, None, 0, None) == 2
    assert zp(p, p, p, None, p, p, p, 1, 8, 64, 0, 4, 64, bf16, None, 0, None) == 1
    assert zp(p, None, p, None, p, p, p, 1, 8, 64, 64, 4, 64, bf16, None, 0, None) == 1
    assert zp(p, p, None, None, p, p, p, 1, 8, 64, 64, 4, 64, bf16, None, 0, None) == 1
    assert zp(p, p, p, None, p, p, None, 1, 8, 64, 64, 4, 64, bf16, None, 0, None) == 1
    assert zp(p, p, p, None, p, p, p, 1, 8, 64, 64, 9, 64, bf16, None, 0, None) == 1
    assert zp(p, p, ctypes.c_void_p(0x10008), None, p, p, p, 1, 8, 64, 64, 4, 64, bf16, None, 0, None) == 2  # W1
    assert zp(p, p, p, ctypes.c_void_p(0x10002), p, p, p, 1, 8, 64, 64, 4, 64, bf16, None, 0, None) == 1  # b1 unaligned
    assert zp(p, p, p, None, p, p, p, 1 << 16, 1 << 10, 64, 64, 4, 64, bf16, None, 0, None) == 1  # B*T*Dm >= 2^31
    # the projection: H must divide D and be 1, 2, 4 or a multiple of 8; Dm % 8
    assert L.dsc_proj_fwd(p, p, p, None, p, 1, 8, 64, 64, 4, 12, bf16, None, 0, None) == 1
    assert L.dsc_proj_fwd(p, p, p, None, p, 1, 8, 64, 48, 4, 12, bf16, None, 0, None) == 2
    assert L.dsc_proj_fwd(p, p, p, None, p, 1, 8, 60, 64, 4, 16, bf16, None, 0, None) == 2
    assert L.dsc_proj_fwd(p, p, p, None, p, 1, 8, 64, 64, 4, 16, f32, None, 0, None) == 2
    assert L.dsc_validate_cu_seqlens(None, 3, 1, 8, None) == 1
    # static convolution: the same size, W, dtype and alignment rules; dw must be fp32-aligned
    assert L.dsc_static_fwd(p, p, p, 0, 8, 64, 4, bf16, None, 0, None) == 1
    assert L.dsc_static_fwd(p, p, p, 1, 8, 64, 9, bf16, None, 0, None) == 1
    assert L.dsc_static_fwd(p, p, p, 1, 8, 64, 4, 7, None, 0, None) == 1
    assert L.dsc_static_fwd(p, p, p, 1, 8, 64, 4, bf16, p, 0, None) == 1
    assert L.dsc_static_bwd(p, p, p, p, ctypes.c_void_p(0x10002), 1, 8, 64, 4, bf16, None, 0, None) == 1
    assert L.dsc_static_bwd(p, p, p, None, p, 1, 8, 64, 4, bf16, None, 0, None) == 1
    # decode step: D % H, W range, missing history for W > 1, missing positions
    assert L.dsc_decode_step(p, p, p, p, p, 4, 64, 4, 3, bf16, None) == 1
    assert L.dsc_decode_step(p, p, p, p, p, 4, 64, 9, 1, bf16, None) == 1
    assert L.dsc_decode_step(p, p, None, p, p, 4, 64, 4, 1, bf16, None) == 1
    assert L.dsc_decode_step(p, p, p, None, p, 4, 64, 4, 1, bf16, None) == 1
    assert L.dsc_decode_step(p, p, p, p, p, 0, 64, 4, 1, bf16, None) == 1


def test_loading_without_gpu_reports_cuda_error_not_crash(L):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    p = ctypes.c_void_p(0x10000)
    assert L.dsc_fwd(p, p, p, 1, 8, 64, 4, 1, 1, None, 0, None) == 3
