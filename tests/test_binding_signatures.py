"""The Python binding's ctypes signatures against the C header: every function the binding
declares has the header's parameter count, integer widths and pointer positions, and the two
option / plan structs have the header's size and field offsets (compiled with the host C
compiler). A mismatch would pass garbage through the ABI without any error."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxfp4_gb300.h")

_SCALAR = {"int": ctypes.c_int, "unsigned": ctypes.c_uint, "int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t,
           "void": None}


def _prototypes():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    out = {}
    for m in re.finditer(r"([A-Za-z_][\w\s]*?)(\*?)\s*(mxfp4_\w+)\s*\(([^)]*)\)\s*;", text):
        ret = (m.group(1).split()[-1], bool(m.group(2)))
        params = [] if m.group(4).strip() in ("", "void") else [p.strip() for p in m.group(4).split(",")]
        out[m.group(3)] = (ret, [("*" in p, p.replace("const", "").replace("*", " ").split()[0]) for p in params])
    return out


def _kind(ct):
    """'ptr' for any pointer-like ctypes type, else the ctypes scalar class itself."""
    if ct in (ctypes.c_void_p, ctypes.c_char_p) or (isinstance(ct, type) and issubclass(ct, ctypes._Pointer)):
        return "ptr"
    return ct


@pytest.fixture(scope="module")
def lib():
    import block_scaled_mxfp4_bf16_gb300 as mx
    return mx.load_library()


def test_header_parses_every_entry_point():
    protos = _prototypes()
    for name in ("mxfp4_quantize", "mxfp4_prepack_b", "mxfp4_gemm", "mxfp4_gemm_host", "mxfp4_gemm_noalloc",
                 "mxfp4_gemm_plan_model", "mxfp4_version"):
        assert name in protos, name
    assert protos["mxfp4_gemm"][1][0] == (True, "void")
    assert len(protos["mxfp4_gemm_host"][1]) == 13


def test_binding_signatures_match_the_header(lib):
    checked = 0
    protos = _prototypes()
    for name, ((ret, ret_ptr), params) in protos.items():
        fn = getattr(lib, name)
        argtypes = fn.argtypes
        if argtypes is None:           # configured without arguments: must take none
            assert params == [], name
        else:
            assert len(argtypes) == len(params), name
            for i, ((is_ptr, ctype), ct) in enumerate(zip(params, argtypes)):
                want = "ptr" if is_ptr else _SCALAR[ctype]
                assert _kind(ct) == want, f"{name} argument {i}: {ct} for {ctype}{'*' if is_ptr else ''}"
        want_ret = "ptr" if ret_ptr else _SCALAR[ret]
        assert _kind(fn.restype) == want_ret, f"{name} returns {fn.restype}, header {ret}"
        checked += 1
    assert checked == len(protos) >= 18


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs the host C compiler")
def test_option_and_plan_structs_match_the_header(tmp_path):
    import block_scaled_mxfp4_bf16_gb300 as mx
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "mxfp4_gb300.h"\n'
        "int main(void) {\n"
        '  printf("%zu %zu %zu %zu\\n", sizeof(mxfp4_gemm_options), offsetof(mxfp4_gemm_options, path),\n'
        "         offsetof(mxfp4_gemm_options, splits), offsetof(mxfp4_gemm_options, m_tile));\n"
        '  printf("%zu %zu %zu %zu\\n", sizeof(mxfp4_plan_info), offsetof(mxfp4_plan_info, reduction),\n'
        "         offsetof(mxfp4_plan_info, tmem_cols), offsetof(mxfp4_plan_info, reserved));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    opt, plan = [list(map(int, line.split())) for line in subprocess.run(
        [str(exe)], check=True, capture_output=True, text=True).stdout.splitlines()]
    O, P = mx._Options, mx._PlanInfo
    assert opt == [ctypes.sizeof(O), O.path.offset, O.splits.offset, O.m_tile.offset]
    assert plan == [ctypes.sizeof(P), P.reduction.offset, P.tmem_cols.offset, P.reserved.offset]


def test_noalloc_scratch_size_matches_the_header():
    # the no-allocation GEMM's tests size their shapes against the library's fixed scratch
    m = re.search(r"#define\s+MXFP4_NOALLOC_SCRATCH_BYTES\s+\(([\du\s*]+)\)", open(HEADER).read())
    value = 1
    for factor in m.group(1).replace("u", "").split("*"):
        value *= int(factor)
    import test_zz_no_alloc
    assert test_zz_no_alloc.NOALLOC_BYTES == value == 32 << 20


@pytest.mark.skipif(shutil.which("gcc") is None or shutil.which("g++") is None, reason="needs gcc and g++")
@pytest.mark.parametrize("compiler,std", [("gcc", "c99"), ("gcc", "c11"), ("g++", "c++17")])
def test_header_is_strict_c_and_cpp(tmp_path, compiler, std):
    # the boundary is a plain C header: C callers include it as well as C++ ones
    src = tmp_path / "use.c"
    src.write_text('#include "mxfp4_gb300.h"\nint main(void) { return MXFP4_OK; }\n')
    lang = ["-x", "c++"] if compiler == "g++" else []
    subprocess.run([compiler, f"-std={std}", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I",
                    os.path.join(ROOT, "include"), *lang, "-c", str(src), "-o", str(tmp_path / "use.o")], check=True)
