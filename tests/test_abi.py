"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

* include/fp8q.h and libfp8q.so agree: every function the header declares is
  exported, and the binding's list matches the header;
* a C program that includes the header and calls every entry point links
  against the library;
* argument validation returns the documented status before touching a
  device (bad enums, inner dimensions not multiples of 16, misaligned
  pointers, a missing workspace).
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8q.h")


@pytest.fixture(scope="module")
def lib():
    from scaled_quantize_fp8_warp_gb300 import build_lib
    import scaled_quantize_fp8_warp_gb300 as fq
    build_lib.build()
    return fq.load_library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_layer_entry_points():
    fns = header_functions()
    for name in ("fp8_amax", "fp8_quantize_tensor", "fp8_quantize_tile1x128",
                 "fp8_quantize_delayed", "fp8_gemm_fprop", "fp8_gemm_dgrad", "fp8_gemm_wgrad",
                 "fp8_linear_autocast"):
        assert name in fns


def test_library_exports_every_declared_symbol(lib):
    import scaled_quantize_fp8_warp_gb300 as fq
    fns = header_functions()
    assert sorted(fq.EXPORTS) == fns
    out = subprocess.run(["nm", "-D", "--defined-only", fq.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [f for f in fns if f not in exported]
    assert not missing, missing


def test_c_program_links_against_header(tmp_path, lib):
    import scaled_quantize_fp8_warp_gb300 as fq
    src = tmp_path / "use.c"
    calls = "\n".join(f"  (void)&{f};" for f in header_functions())
    src.write_text('#include "fp8q.h"\nint main(void) {\n' + calls + "\n  return 0;\n}\n")
    exe = tmp_path / "use"
    cuda_inc = "/usr/local/cuda/include"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", cuda_inc, str(src), "-o", str(exe), fq.LIB_PATH,
                    "-Wl,-rpath," + os.path.dirname(fq.LIB_PATH)], check=True)


def test_struct_sizes_match_header(tmp_path, lib):
    import scaled_quantize_fp8_warp_gb300 as fq
    src = tmp_path / "sz.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "fp8q.h"\n'
                   'int main(void){printf("%zu %zu %zu %zu\\n", sizeof(fp8q_amax_history),'
                   ' sizeof(fp8q_operand), offsetof(fp8q_amax_history, next),'
                   ' offsetof(fp8q_operand, scale_stride_row));return 0;}\n')
    exe = tmp_path / "sz"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", "/usr/local/cuda/include",
                    str(src), "-o", str(exe)], check=True)
    hist, op, nxt, srow = map(int, subprocess.run([str(exe)], capture_output=True, text=True,
                                                  check=True).stdout.split())
    assert hist == fq.HISTORY_BYTES and nxt == 4 * fq.HISTORY_LEN
    assert op == ctypes.sizeof(fq.Operand)
    assert srow == fq.Operand.scale_stride_row.offset


def test_status_strings(lib):
    for code in range(8):
        assert lib.fp8q_status_string(code)
    assert b"unknown" in lib.fp8q_status_string(99)


def test_validation_before_device(lib):
    import scaled_quantize_fp8_warp_gb300 as fq
    P = ctypes.c_void_p
    aligned, odd = P(0x10000), P(0x10008)
    # quantize: cols % 16 != 0, bad format, misaligned output
    assert lib.fp8_quantize_tensor(aligned, fq.DT_BF16, 16, 24, fq.E4M3, aligned, None, aligned,
                                   None, 0, None) == 1
    assert lib.fp8_quantize_tensor(aligned, fq.DT_BF16, 16, 32, 7, aligned, None, aligned, None,
                                   0, None) == 1
    assert lib.fp8_quantize_tensor(aligned, fq.DT_BF16, 16, 32, fq.E4M3, aligned, None, odd,
                                   None, 0, None) == 2
    # transposed output needs rows % 16 == 0
    assert lib.fp8_quantize_tensor(aligned, fq.DT_BF16, 20, 32, fq.E4M3, aligned, None, None,
                                   aligned, 0, None) == 1
    # tile: pairs must be complete
    assert lib.fp8_quantize_tile1x128(aligned, fq.DT_BF16, 16, 32, fq.E4M3, aligned, None, None,
                                      None, 0, None) == 1
    assert lib.fp8_amax(odd, fq.DT_BF16, 64, aligned, None) == 2
    assert lib.fp8_amax(aligned, 5, 64, aligned, None) == 1
    # gemm: N and K multiples of 16
    op = fq.Operand(0x10000, fq.E4M3, fq.SCALE_TENSOR, 0x20000, 0, 0)
    assert lib.fp8_gemm(ctypes.byref(op), ctypes.byref(op), aligned, fq.DT_BF16, 32, 24, 32,
                        None) == 1
    assert lib.fp8_gemm(ctypes.byref(op), ctypes.byref(op), aligned, fq.DT_BF16, 32, 32, 40,
                        None) == 1
    bad = fq.Operand(0x10008, fq.E4M3, fq.SCALE_TENSOR, 0x20000, 0, 0)
    assert lib.fp8_gemm(ctypes.byref(bad), ctypes.byref(op), aligned, fq.DT_BF16, 32, 32, 32,
                        None) == 2
    bad = fq.Operand(0x10000, fq.E4M3, 9, 0x20000, 0, 0)
    assert lib.fp8_gemm(ctypes.byref(bad), ctypes.byref(op), aligned, fq.DT_BF16, 32, 32, 32,
                        None) == 1
    # quantize with its own amax: the amax output is required and 4-byte aligned
    assert lib.fp8_quantize_tensor_current(aligned, fq.DT_BF16, 16, 32, fq.E4M3, None, None,
                                           aligned, None, 0, None) == 1
    assert lib.fp8_quantize_tensor_current(aligned, fq.DT_BF16, 16, 32, fq.E4M3, P(0x10002),
                                           None, aligned, None, 0, None) == 2
    assert lib.fp8_quantize_tensor_current(aligned, fq.DT_BF16, 16, 24, fq.E4M3, aligned, None,
                                           aligned, None, 0, None) == 1
    # gemm with fused amax: needs a 4-byte aligned amax, then validates as fp8_gemm
    assert lib.fp8_gemm_amax(ctypes.byref(op), ctypes.byref(op), aligned, fq.DT_BF16, 32, 32,
                             32, None, None) == 1
    assert lib.fp8_gemm_amax(ctypes.byref(op), ctypes.byref(op), aligned, fq.DT_BF16, 32, 32,
                             32, P(0x10002), None) == 2
    assert lib.fp8_gemm_amax(ctypes.byref(op), ctypes.byref(op), aligned, fq.DT_BF16, 32, 24,
                             32, aligned, None) == 1
    # autocast: workspace too small
    assert lib.fp8_linear_autocast(aligned, aligned, fq.DT_BF16, 32, 32, 32, 0, None, None,
                                   aligned, fq.DT_BF16, aligned, 16, None) == 4
    # delayed recipe needs histories
    assert lib.fp8_linear_autocast(aligned, aligned, fq.DT_BF16, 32, 32, 32, 1, None, None,
                                   aligned, fq.DT_BF16, aligned, 1 << 30, None) == 1


def test_workspace_size_formula(lib):
    import scaled_quantize_fp8_warp_gb300 as fq
    M, N, K = 15872, 4096, 4096
    got = lib.fp8q_linear_workspace_size(fq.RECIPE_BLOCK, M, N, K)
    r = lambda b: (b + 255) // 256 * 256
    assert got == r(M * K) + r(N * K) + 4 * 256 + r(4 * (K // 128) * M) + r(4 * (N // 128) * (K // 128))


def test_product_package_has_no_oracle_dependency():
    """The product package never imports the oracle or falls back to torch math."""
    pkg = os.path.join(ROOT, "scaled_quantize_fp8_warp_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "fp8_oracle" not in text, f
