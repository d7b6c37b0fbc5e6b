"""Host-side checks of the C ABI (no GPU needed).

The library must build for sm_103a, load, export exactly the entry points
include/lora_punica.h declares, and reject bad arguments on the host with
the documented negative status codes before anything is launched.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lora_punica.h")


@pytest.fixture(scope="module")
def lib():
    from expand_gemm_gb300 import build as pkg_build
    from expand_gemm_gb300 import _lib
    pkg_build()
    return _lib.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \t\*]*?\b(lora_\w+)\s*\(", text, flags=re.M)))


def _exported(path):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True,
                         text=True, check=True).stdout
    return sorted(l.split()[-1] for l in out.splitlines() if " T " in l)


def test_header_declares_the_three_steps():
    names = _declared()
    for fn in ("lora_meta_prepare", "lora_shrink", "lora_expand"):
        assert fn in names


def test_library_exports_every_declared_symbol_and_nothing_else(lib):
    from expand_gemm_gb300 import _lib
    exported = _exported(_lib.LIB_PATH)
    declared = _declared()
    assert exported == declared, (exported, declared)
    assert sorted(_lib.EXPORTS) == declared
    for name in declared:
        assert hasattr(lib, name)


def test_version_and_status_strings(lib):
    assert lib.lora_version() == 1
    assert lib.lora_status_string(0) == b"ok"
    for code in range(-1, -10, -1):
        s = lib.lora_status_string(code)
        assert s and s != b"unknown status"
    assert lib.lora_status_string(-99) == b"unknown status"


def _meta(max_loras=4, max_tokens=16, null_field=None):
    from expand_gemm_gb300 import _lib
    vals = {f: 0x1000 * (i + 1) for i, (f, _) in enumerate(_lib.LoraMetaC._fields_[:7])}
    if null_field:
        vals[null_field] = 0
    return _lib.LoraMetaC(*[vals[f] for f, _ in _lib.LoraMetaC._fields_[:7]],
                          max_loras, max_tokens)


def test_meta_prepare_rejects_bad_arguments(lib):
    m = _meta()
    assert lib.lora_meta_prepare(0x1000, 4, None, None) == -1
    assert lib.lora_meta_prepare(0x1000, 4, ctypes.byref(_meta(null_field="error_word")), None) == -1
    assert lib.lora_meta_prepare(0x1000, 17, ctypes.byref(m), None) == -6
    assert lib.lora_meta_prepare(0x1000, -1, ctypes.byref(m), None) == -2
    assert lib.lora_meta_prepare(None, 3, ctypes.byref(m), None) == -1
    assert lib.lora_meta_prepare(0x1000, 1, ctypes.byref(_meta(max_loras=0)), None) == -2
    assert lib.lora_meta_prepare(0x1000, 1, ctypes.byref(_meta(max_loras=1025)), None) == -2


def test_read_no_lora_rejects_null_arguments(lib):
    out = ctypes.c_int32(7)
    assert lib.lora_meta_read_no_lora(None, None, ctypes.byref(out)) == -1
    assert lib.lora_meta_read_no_lora(ctypes.byref(_meta()), None, None) == -1
    assert lib.lora_meta_read_no_lora(ctypes.byref(_meta(null_field="no_lora_flag")), None,
                                      ctypes.byref(out)) == -1
    assert out.value == 7


def test_shrink_rejects_bad_arguments(lib):
    m = _meta()
    A = (ctypes.c_void_p * 2)(0x2000, 0x3000)
    ok = dict(x=0x4000, T=8, H=64, ld=64, A=A, S=2, r=16, y=0x5000)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.lora_shrink(a["x"], a["T"], a["H"], a["ld"], a["A"], a["S"], a["r"],
                               a["y"], ctypes.byref(m), 1.0, None)
    assert call(S=0) == -5
    assert call(S=9) == -5
    assert call(r=12) == -4
    assert call(r=136) == -4
    assert call(T=17) == -6
    assert call(ld=32) == -2
    assert call(H=60, ld=64) == -3
    assert call(x=0x4002) == -3
    assert call(A=(ctypes.c_void_p * 2)(0x2000, 0)) == -1
    assert call(A=(ctypes.c_void_p * 2)(0x2000, 0x3008)) == -3
    assert lib.lora_shrink(0x4000, 8, 64, 64, A, 2, 16, 0x5000, None, 1.0, None) == -1
    assert call(T=0) == 0        # nothing to do: returns before any launch


def test_expand_rejects_bad_arguments(lib):
    m = _meta()
    B = (ctypes.c_void_p * 2)(0x2000, 0x3000)
    sizes = (ctypes.c_int32 * 2)(64, 32)
    ok = dict(x=0x4000, B=B, sizes=sizes, S=2, r=16, y=0x5000, ld=96, T=8, off=0)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.lora_expand(a["x"], a["B"], None, a["sizes"], a["S"], a["r"], a["y"],
                               a["ld"], a["T"], a["off"], 1, ctypes.byref(m), None)
    assert call(S=0) == -5
    assert call(r=20) == -4
    assert call(ld=95) == -7
    assert call(off=8) == -7
    assert call(off=-1) == -2
    assert call(T=17) == -6
    assert call(sizes=(ctypes.c_int32 * 2)(64, -1)) == -2
    assert call(B=(ctypes.c_void_p * 2)(0, 0x3000)) == -1
    assert call(x=0x4004) == -3
    assert call(T=0) == 0


def test_linear_noalloc_rejects_sizes_above_its_buffer(lib):
    """Checked on the host before any CUDA call: slices, rank, and
    num_slices * num_tokens * rank against the fixed buffer."""
    from expand_gemm_gb300 import _lib
    m = _meta(max_tokens=1 << 20)
    A = (ctypes.c_void_p * 2)(0x2000, 0x3000)
    B = (ctypes.c_void_p * 2)(0x6000, 0x7000)
    sizes = (ctypes.c_int32 * 2)(64, 64)

    def call(T, S=2, r=16):
        return lib.lora_linear_noalloc(0x1000, T, 0x4000, 64, 64, A, B, None, sizes, S, r, 1.0,
                                       0x5000, 128, ctypes.byref(m), None)
    cap = _lib.LORA_NOALLOC_MAX_FLOATS
    assert call(cap // 32 + 1) == -9
    assert call(cap // 16 + 1, S=1) == -9
    assert call(1 << 20, S=2, r=128) == -9
    assert call(8, S=0) == -5
    assert call(8, S=2, r=12) == -4
    assert call(-1) == -2


def test_expand_bf16_rejects_bad_arguments(lib):
    """Same host checks as lora_expand, on a bf16 input."""
    m = _meta()
    B = (ctypes.c_void_p * 2)(0x2000, 0x3000)
    sizes = (ctypes.c_int32 * 2)(64, 32)
    ok = dict(x=0x4000, B=B, sizes=sizes, S=2, r=16, y=0x5000, ld=96, T=8, off=0)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.lora_expand_bf16(a["x"], a["B"], None, a["sizes"], a["S"], a["r"], a["y"],
                                    a["ld"], a["T"], a["off"], 1, ctypes.byref(m), None)
    assert call(S=0) == -5
    assert call(S=9) == -5
    assert call(r=20) == -4
    assert call(ld=95) == -7
    assert call(off=-1) == -2
    assert call(T=17) == -6
    assert call(sizes=(ctypes.c_int32 * 2)(64, -1)) == -2
    assert call(B=(ctypes.c_void_p * 2)(0, 0x3000)) == -1
    assert call(x=0x4002) == -3
    assert call(T=0) == 0


def test_linear_rejects_bad_arguments(lib):
    """lora_linear's own checks, all on the host before any CUDA call."""
    m = _meta()
    A = (ctypes.c_void_p * 2)(0x2000, 0x3000)
    B = (ctypes.c_void_p * 2)(0x6000, 0x7000)
    sizes = (ctypes.c_int32 * 2)(64, 64)
    ok = dict(meta=ctypes.byref(m), A=A, B=B, sizes=sizes, S=2, r=16, T=8, H=64, x_ld=64)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.lora_linear(0x1000, a["T"], 0x4000, a["H"], a["x_ld"], a["A"], a["B"], None,
                               a["sizes"], a["S"], a["r"], 1.0, 0x8000, 0x5000, 128, a["meta"],
                               None)
    assert call(meta=None) == -1
    assert call(A=None) == -1
    assert call(B=None) == -1
    assert call(sizes=None) == -1
    assert call(S=0) == -5
    assert call(S=9) == -5
    assert call(r=12) == -4
    assert call(r=136) == -4
    assert call(T=-1) == -2
    assert call(x_ld=32) == -2
    assert call(T=17) == -6


def test_header_is_plain_c_and_links(lib, tmp_path):
    """A C99 program (no C++, no CUDA headers) includes the header, links
    the library and calls entry points that need no GPU."""
    import shutil
    import subprocess
    from expand_gemm_gb300 import _lib
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    src = tmp_path / "consumer.c"
    src.write_text(
        '#include <stdio.h>\n'
        '#include "lora_punica.h"\n'
        'int main(void)\n'
        '{\n'
        '    lora_meta_t m = {0};\n'
        '    int32_t out = 7;\n'
        '    printf("%d %s %d %d\\n", lora_version(), lora_status_string(LORA_ERR_RANK),\n'
        '           lora_meta_read_no_lora(&m, NULL, &out), out);\n'
        '    return 0;\n'
        '}\n')
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(_lib.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), str(src), "-L", libdir, "-llora_punica",
                    "-Wl,-rpath," + libdir, "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert out[0] == "1" and out[-2:] == ["-1", "7"]
    assert " ".join(out[1:-2]) == lib.lora_status_string(-4).decode()
