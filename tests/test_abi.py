"""Host-side checks of the C-ABI library: it loads, exports every declared
symbol, and rejects bad arguments before any device work."""

import ctypes

import pytest

from precision_mx_quantize_gb300 import mxq
from tests.libutil import ensure_built, header_prototypes, header_symbols


@pytest.fixture(scope="module")
def lib():
    return ensure_built()


def test_exports_every_declared_symbol(lib):
    names = header_symbols()
    assert "mxq_quantize" in names and "mxq_gemm" in names
    for n in names:
        assert hasattr(lib, n), n
    bound = {n for n, _, _ in mxq.SIGNATURES}
    assert set(names) <= bound


def test_bounds_checked_build_exports_the_same_symbols(lib):
    # the bounds-checked variant is built from the same sources beside the
    # library and loads on its own
    from precision_mx_quantize_gb300 import build as _build
    dbg = ctypes.CDLL(_build.LIB_DEBUG)
    for n in header_symbols():
        assert hasattr(dbg, n), n
    dbg.mxq_status_str.restype = ctypes.c_char_p
    assert dbg.mxq_status_str(7) == b"index out of bounds (bounds-checked build)"


def test_version_and_status_strings(lib):
    assert lib.mxq_version() >= 1
    assert lib.mxq_status_str(0) == b"ok"
    assert lib.mxq_status_str(5) == b"device-side wait timed out"
    assert lib.mxq_status_str(99) == b"unknown status"


def test_argument_errors_return_before_device_work(lib):
    p = ctypes.c_void_p(16 * 1024)  # never dereferenced: every call below fails its checks
    E4, E2, ROW, COL = mxq.E4M3, mxq.E2M1, mxq.ROWWISE, mxq.COLWISE_T
    # empty tensors are a no-op
    assert mxq.mxq_quantize(p, 0, 64, ROW, E4, p, p, None) == 0
    # row-wise needs cols % 32 == 0
    assert mxq.mxq_quantize(p, 64, 48, ROW, E4, p, p, None) == 1
    # col-wise needs rows % 32 == 0
    assert mxq.mxq_quantize(p, 40, 64, COL, E2, p, p, None) == 1
    # bad enums and null pointers
    assert mxq.mxq_quantize(p, 64, 64, 7, E4, p, p, None) == 1
    assert mxq.mxq_quantize(p, 64, 64, ROW, 9, p, p, None) == 1
    assert mxq.mxq_quantize(None, 64, 64, ROW, E4, p, p, None) == 1
    # misaligned input pointer
    assert mxq.mxq_quantize(ctypes.c_void_p(16 * 1024 + 2), 64, 64, ROW, E4, p, p, None) == 2
    # dual needs both dims % 32
    assert mxq.mxq_quantize_dual(p, 64, 40, E4, 0, p, p, E2, 1, p, p, None) == 1
    # negative sizes
    assert mxq.mxq_hadamard_quantize(p, -32, 64, ROW, E2, p, p, None) == 1
    assert mxq.mxq_dequantize(p, p, 64, 48, ROW, E4, p, 0, None) == 1
    assert mxq.mxq_dequantize(p, p, 64, 64, ROW, E4, p, 3, None) == 1
    # the dual pass takes E5M2 on either side, with the same shape rules
    assert mxq.mxq_quantize_dual(p, 64, 40, mxq.E5M2, 0, p, p, E2, 1, p, p, None) == 1
    assert mxq.mxq_quantize_dual(p, 64, 64, mxq.E5M2, 0, p, p, 9, 1, p, p, None) == 1
    assert mxq.mxq_quantize(p, 64, 64, ROW, 3, p, p, None) == 1
    # ablation: a sign mask needs the rotation; the usual shape rules apply
    A = mxq.mxq_quantize_ablation
    assert A(p, 64, 64, ROW, E2, 0, 0x5, 1, 7, p, p, None) == 1
    assert A(p, 64, 48, ROW, E4, 1, 0x5, 1, 7, p, p, None) == 1
    assert A(p, 40, 64, COL, E2, 0, 0, 1, 7, p, p, None) == 1
    assert A(p, 64, 64, 5, E4, 1, 0, 1, 7, p, p, None) == 1
    assert A(p, 64, 64, ROW, 9, 1, 0, 1, 7, p, p, None) == 1
    assert A(ctypes.c_void_p(16 * 1024 + 2), 64, 64, ROW, E4, 0, 0, 1, 7, p, p, None) == 2
    assert A(p, 0, 64, ROW, E4, 1, 0xFFFFFFFF, 1, 2 ** 64 - 1, p, p, None) == 0


def test_tc_scale_buffer_sizes(lib):
    assert mxq.mxq_scales_tc_bytes(128, 128) == 512
    assert mxq.mxq_scales_tc_bytes(129, 256) == 2 * 2 * 512
    assert mxq.mxq_scales_tc_bytes(8192, 4096) == 64 * 32 * 512 == 8192 * 4096 // 32
    assert mxq.mxq_scales_tc_bytes(64, 96) == 0
    assert mxq.mxq_scales_tc_bytes(0, 128) == 0


def _ctype_of(decl):
    """The ctypes type a C parameter declaration needs (pointers as void*)."""
    if "*" in decl:
        return "ptr"
    t = decl.replace("const ", "").split()[0]
    return {"int64_t": ctypes.c_int64, "int": ctypes.c_int, "size_t": ctypes.c_size_t,
            "uint64_t": ctypes.c_uint64, "uint32_t": ctypes.c_uint32}[t]


def test_binding_signatures_match_the_header():
    # a ctypes signature with a missing or mistyped parameter would hand the
    # library shifted arguments (and the GPU a wrong pointer): every bound
    # function takes exactly the header's parameters, in order
    protos = header_prototypes()
    sigs = {n: args for n, _, args in mxq.SIGNATURES}
    assert set(protos) == set(sigs)
    for name, decls in protos.items():
        args = sigs[name]
        assert len(args) == len(decls), name
        for i, (decl, arg) in enumerate(zip(decls, args)):
            want = _ctype_of(decl)
            if want == "ptr":
                assert arg in (ctypes.c_void_p, ctypes.c_char_p), (name, i, decl)
            else:
                assert arg is want, (name, i, decl, arg)


def test_gemm_problem_struct_matches_the_header(tmp_path):
    # the binding's ctypes mirror of mxq_gemm_problem has the C layout: a C
    # program compiled against the header prints sizeof and every offset
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    import os
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    src = tmp_path / "layout.c"
    fields = [f for f, _ in mxq.GemmProblem._fields_]
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"mxq.h\"\nint main(void) {\n"
                   "  printf(\"%zu\", sizeof(mxq_gemm_problem));\n" +
                   "".join(f"  printf(\" %zu\", offsetof(mxq_gemm_problem, {f}));\n" for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "layout"
    cuda_inc = "/usr/local/cuda/include"
    subprocess.run([cc, "-I", inc, "-I", cuda_inc, str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [ctypes.sizeof(mxq.GemmProblem)] + [getattr(mxq.GemmProblem, f).offset for f in fields]
    assert got == want


def test_gemm_grouped_argument_errors(lib):
    p = ctypes.c_void_p(16 * 1024)
    arr = (mxq.GemmProblem * 9)()
    for i in range(9):
        arr[i] = mxq.GemmProblem(p.value, p.value, p.value, p.value, p.value, 256, 256, 256, 0)
    addr = ctypes.addressof(arr)
    assert mxq.mxq_gemm_grouped(None, 1, mxq.E4M3, None) == 1
    assert mxq.mxq_gemm_grouped(addr, 0, mxq.E4M3, None) == 1
    assert mxq.mxq_gemm_grouped(addr, 9, mxq.E4M3, None) == 1
    arr[1].K = 96                      # K % 32 == 0 but not % 128 (chunk-layout scales)
    assert mxq.mxq_gemm_grouped(addr, 2, mxq.E4M3, None) == 1
    arr[1].K = 256
    arr[1].out_dtype = 5
    assert mxq.mxq_gemm_grouped(addr, 2, mxq.E4M3, None) == 1
    arr[1].out_dtype = 0
    arr[1].N = 258                     # fp32 rows must stay 16-byte aligned
    assert mxq.mxq_gemm_grouped(addr, 2, mxq.E4M3, None) == 2
