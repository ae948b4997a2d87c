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
                   'int main(void){printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(fp8q_amax_history),'
                   ' sizeof(fp8q_operand), offsetof(fp8q_amax_history, next),'
                   ' offsetof(fp8q_operand, scale_stride_row), sizeof(fp8q_gemm_desc),'
                   ' offsetof(fp8q_gemm_desc, K));return 0;}\n')
    exe = tmp_path / "sz"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", "/usr/local/cuda/include",
                    str(src), "-o", str(exe)], check=True)
    hist, op, nxt, srow, gd, gdk = map(int, subprocess.run([str(exe)], capture_output=True,
                                                           text=True, check=True).stdout.split())
    assert gd == ctypes.sizeof(fq.GemmDesc) and gdk == fq.GemmDesc.K.offset
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
    # sizes whose byte counts overflow int64 are rejected before any arithmetic on them
    big = 1 << 40
    assert lib.fp8_quantize_tensor(aligned, fq.DT_BF16, big, big, fq.E4M3, aligned, None,
                                   aligned, None, 0, None) == 1
    assert lib.fp8_quantize_tile1x128(aligned, fq.DT_F32, big, big, fq.E4M3, aligned, aligned,
                                      None, None, 0, None) == 1
    assert lib.fp8_amax(aligned, fq.DT_F32, 1 << 62, aligned, None) == 1
    assert lib.fp8_gemm(ctypes.byref(op), ctypes.byref(op), aligned, fq.DT_BF16, big, big, 32,
                        None) == 1
    assert lib.fp8_gemm(ctypes.byref(op), ctypes.byref(op), aligned, fq.DT_BF16, 32, 32,
                        1 << 60, None) == 1
    # autocast: workspace too small
    assert lib.fp8_linear_autocast(aligned, aligned, fq.DT_BF16, 32, 32, 32, 0, None, None,
                                   aligned, fq.DT_BF16, aligned, 16, None) == 4
    # delayed recipe needs histories
    assert lib.fp8_linear_autocast(aligned, aligned, fq.DT_BF16, 32, 32, 32, 1, None, None,
                                   aligned, fq.DT_BF16, aligned, 1 << 30, None) == 1


def _has_cuda_device():
    import torch
    return torch.cuda.is_available()


@pytest.mark.skipif(_has_cuda_device(),
                    reason="valid layouts would reach a kernel launch on placeholder pointers")
def test_role_wrappers_reject_undocumented_scale_layouts(lib):
    """fp8_gemm_fprop/_dgrad/_wgrad know each operand's [rows, K] and accept
    only the scale strides the quantize calls write; anything else would index
    past the scale array on the device, so it is refused before any device
    work (INVALID_ARG, 1).  A documented layout passes validation and then
    fails only at the device check (CUDA, 6: there is no GPU here)."""
    import scaled_quantize_fp8_warp_gb300 as fq
    P = ctypes.c_void_p
    y = P(0x40000)
    M, N, K = 256, 384, 512
    ten = fq.Operand(0x10000, fq.E4M3, fq.SCALE_TENSOR, 0x20000, 0, 0)

    def fprop(a, b):
        return lib.fp8_gemm_fprop(ctypes.byref(a), ctypes.byref(b), y, fq.DT_BF16, M, N, K, None)

    def tile(rows, sr, sk):
        return fq.Operand(0x10000, fq.E4M3, fq.SCALE_TILE_1x128, 0x20000, sr, sk)

    def block(sr, sk):
        return fq.Operand(0x10000, fq.E4M3, fq.SCALE_BLOCK_128x128, 0x20000, sr, sk)

    # x [M, K] with 1x128 tiles: stride_row 1, stride_k M
    assert fprop(tile(M, 1, M), ten) == 6
    assert fprop(tile(M, 1, M - 16), ten) == 1
    assert fprop(tile(M, M, 1), ten) == 1
    # w [N, K] with 128x128 blocks: (ceil(K/128), 1) or, read transposed, (1, ceil(N/128))
    xt = tile(M, 1, M)
    assert fprop(xt, block(K // 128, 1)) == 6
    assert fprop(xt, block(1, 3)) == 6
    assert fprop(xt, block(1, 4)) == 1
    assert fprop(xt, block(K // 128 + 1, 1)) == 1
    # row scales: stride_row 1
    rowop = fq.Operand(0x10000, fq.E4M3, fq.SCALE_ROW, 0x20000, 1, 0)
    assert fprop(rowop, rowop) == 6
    rowbad = fq.Operand(0x10000, fq.E4M3, fq.SCALE_ROW, 0x20000, 2, 0)
    assert fprop(rowbad, rowop) == 1
    # dgrad: g [M, N] tiles need stride_k M; w_t [K, N] blocks of w read transposed
    g = tile(M, 1, M)
    wt = block(1, K // 128)
    assert lib.fp8_gemm_dgrad(ctypes.byref(g), ctypes.byref(wt), y, fq.DT_BF16, M, N, K,
                              None) == 6
    assert lib.fp8_gemm_dgrad(ctypes.byref(g), ctypes.byref(block(1, N // 128)), y,
                              fq.DT_BF16, M, N, K, None) == 1
    # wgrad: g_t [N, M] and x_t [K, M] column tiles: stride_k = N and K respectively
    gt, xt2 = tile(N, 1, N), tile(K, 1, K)
    assert lib.fp8_gemm_wgrad(ctypes.byref(gt), ctypes.byref(xt2), y, fq.DT_BF16, M, N, K,
                              None) == 6
    assert lib.fp8_gemm_wgrad(ctypes.byref(xt2), ctypes.byref(gt), y, fq.DT_BF16, M, N, K,
                              None) == 1


def test_grouped_gemm_validation_before_device(lib):
    """fp8_gemm_grouped: a count outside [0, 3] or null descriptors are
    INVALID_ARG (1); count 0 does nothing (OK, 0); every descriptor is checked
    like the role wrappers check theirs (an undocumented scale stride is 1)
    before any device work.  These cases never reach a launch."""
    import scaled_quantize_fp8_warp_gb300 as fq
    P = ctypes.c_void_p
    assert lib.fp8_gemm_grouped(None, 0, fq.DT_BF16, None) == 0
    assert lib.fp8_gemm_grouped(None, 1, fq.DT_BF16, None) == 1
    M, N, K = 256, 384, 512
    ten = fq.Operand(0x10000, fq.E4M3, fq.SCALE_TENSOR, 0x20000, 0, 0)
    badtile = fq.Operand(0x10000, fq.E4M3, fq.SCALE_TILE_1x128, 0x20000, 1, M - 16)
    arr = (fq.GemmDesc * 4)()
    for i in range(4):
        arr[i] = fq.GemmDesc(ten, ten, 0x40000, M, N, K)
    assert lib.fp8_gemm_grouped(ctypes.cast(arr, P), 4, fq.DT_BF16, None) == 1
    assert lib.fp8_gemm_grouped(ctypes.cast(arr, P), -1, fq.DT_BF16, None) == 1
    arr[1] = fq.GemmDesc(badtile, ten, 0x40000, M, N, K)
    assert lib.fp8_gemm_grouped(ctypes.cast(arr, P), 3, fq.DT_BF16, None) == 1
    arr[1] = fq.GemmDesc(ten, ten, 0x40000, M, N + 8, K)      # N % 16 != 0
    assert lib.fp8_gemm_grouped(ctypes.cast(arr, P), 3, fq.DT_BF16, None) == 1
    arr[1] = fq.GemmDesc(ten, ten, 0x40008, M, N, K)          # C not 16-byte aligned
    assert lib.fp8_gemm_grouped(ctypes.cast(arr, P), 3, fq.DT_BF16, None) == 2


@pytest.mark.skipif(_has_cuda_device(),
                    reason="valid descriptors would reach a kernel launch on placeholder pointers")
def test_grouped_gemm_valid_descriptors_reach_the_device_check(lib):
    import scaled_quantize_fp8_warp_gb300 as fq
    M, N, K = 256, 384, 512
    ten = fq.Operand(0x10000, fq.E4M3, fq.SCALE_TENSOR, 0x20000, 0, 0)
    arr = (fq.GemmDesc * 3)()
    for i in range(3):
        arr[i] = fq.GemmDesc(ten, ten, 0x40000, M, N, K)
    assert lib.fp8_gemm_grouped(ctypes.cast(arr, ctypes.c_void_p), 3, fq.DT_BF16, None) == 6


def test_linear_sizes_that_overflow_are_rejected(lib):
    """M*K or N*K past int64 must not wrap into a small workspace size: the
    size query returns 0 and both forwards return INVALID_ARG (1) before any
    device work -- in particular the workspace-free forward, whose scratch
    limit check would otherwise pass on a wrapped size."""
    import scaled_quantize_fp8_warp_gb300 as fq
    P = ctypes.c_void_p
    big, K = 1 << 40, 1 << 30
    for recipe in (fq.RECIPE_TENSOR_CURRENT, fq.RECIPE_BLOCK):
        assert lib.fp8q_linear_workspace_size(recipe, big, 16, K) == 0
        assert lib.fp8q_linear_workspace_size(recipe, 16, big, K) == 0
        assert lib.fp8_linear_autocast(P(0x10000), P(0x10000), fq.DT_BF16, big, 16, K, recipe,
                                       None, None, P(0x10000), fq.DT_BF16, P(0x10000), 1 << 62,
                                       None) == 1
        assert lib.fp8_linear_autocast_noalloc(P(0x10000), P(0x10000), fq.DT_BF16, 16, big, K,
                                               recipe, None, None, P(0x10000), fq.DT_BF16,
                                               None) == 1
    # products that wrap to exactly 2^64 (0 mod 2^64) are caught too
    assert lib.fp8q_linear_workspace_size(fq.RECIPE_TENSOR_CURRENT, 1 << 34, 16, 1 << 30) == 0
    # a size that fits is still computed
    assert lib.fp8q_linear_workspace_size(fq.RECIPE_TENSOR_CURRENT, 1 << 20, 16, 1 << 20) > 0


def test_linear_train_validation_before_device(lib):
    """fp8_linear_train(_host): M, N, K multiples of 16, a valid recipe, the
    three histories for delayed scaling, a large enough 256-byte aligned
    workspace -- all checked before any device work."""
    import scaled_quantize_fp8_warp_gb300 as fq
    P = ctypes.c_void_p
    a = P(0x10000)
    need = lib.fp8q_linear_train_workspace_size(fq.RECIPE_BLOCK, 256, 128, 64)
    assert need > 0
    assert lib.fp8q_linear_train_workspace_size(9, 256, 128, 64) == 0
    assert lib.fp8q_linear_train_workspace_size(fq.RECIPE_BLOCK, -1, 128, 64) == 0
    hneed = lib.fp8q_linear_train_host_workspace_size(fq.RECIPE_BLOCK, fq.DT_BF16, fq.DT_BF16,
                                                      256, 128, 64)
    assert hneed == need + 2 * (256 * 64 + 128 * 64 + 256 * 128) * 2
    args = lambda M, N, K, rec, ws, wsz: (a, a, a, fq.DT_BF16, M, N, K, rec, None, None, None,
                                          a, a, a, fq.DT_BF16, ws, wsz, None)
    for fn in (lib.fp8_linear_train, lib.fp8_linear_train_host):
        assert fn(*args(256, 128, 72, fq.RECIPE_BLOCK, a, 1 << 30)) == 1       # K % 16
        assert fn(*args(200, 128, 64, fq.RECIPE_BLOCK, a, 1 << 30)) == 1       # M % 16
        assert fn(*args(256, 128, 64, 7, a, 1 << 30)) == 1                     # recipe
        assert fn(*args(256, 128, 64, fq.RECIPE_TENSOR_DELAYED, a, 1 << 30)) == 1   # histories
        assert fn(*args(256, 128, 64, fq.RECIPE_BLOCK, a, 64)) == 4            # workspace
        assert fn(*args(256, 128, 64, fq.RECIPE_BLOCK, P(0x10010), 1 << 30)) == 2   # alignment


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


def header_prototypes():
    """{name: (return type, [parameter types])} of every function include/fp8q.h
    declares, parameter names dropped."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for ret, name, args in re.findall(
            r"^\s*((?:const\s+)?[A-Za-z_0-9]+\s*\*?)\s*([a-z_0-9]+)\s*\(([^;{]*?)\)\s*;",
            text, flags=re.M | re.S):
        params = []
        for a in args.replace("\n", " ").split(","):
            a = re.sub(r"\s+", " ", a).strip()
            if a and a != "void":
                params.append(re.sub(r"\s*[A-Za-z_0-9]+$", "", a).strip())   # drop the name
        out[name] = (re.sub(r"\s+", " ", ret).strip(), params)
    return out


def _ctype_class(t: str) -> str:
    """The ctypes class a C parameter or return type needs."""
    t = t.replace("const ", "")
    if t == "char *":
        return "char_p"
    if t.endswith("*") or t == "cudaStream_t":
        return "pointer"
    return {"int": "i32", "int32_t": "i32", "int64_t": "i64", "size_t": "size"}[t]


def _ctypes_class(ct) -> str:
    import scaled_quantize_fp8_warp_gb300 as fq
    if ct is ctypes.c_char_p:
        return "char_p"
    if ct is ctypes.c_void_p or ct is ctypes.POINTER(fq.Operand):
        return "pointer"
    return {ctypes.c_int: "i32", ctypes.c_int64: "i64", ctypes.c_size_t: "size"}[ct]


def test_binding_signatures_match_the_header():
    """Every argument the binding marshals has the width and kind the header
    declares (a missing or mis-sized argument would be undefined behaviour)."""
    import scaled_quantize_fp8_warp_gb300 as fq
    protos = header_prototypes()
    sigs = fq.signatures()
    assert sorted(protos) == sorted(sigs)
    for name, (ret, params) in protos.items():
        res, args = sigs[name]
        assert _ctype_class(ret) == _ctypes_class(res), name
        assert [_ctype_class(p) for p in params] == [_ctypes_class(a) for a in args], name


@pytest.mark.skipif(_has_cuda_device(),
                    reason="valid combinations would reach a kernel launch on placeholder pointers")
def test_random_arguments_get_a_status_not_a_crash(lib):
    """Seeded random arguments (sizes negative, zero, odd, huge; bad enums;
    null, aligned or misaligned placeholder pointers) to the quantize, amax
    and GEMM entry points: every call returns a documented status and none
    touches memory before its checks.  Here no device exists, so arguments
    that pass validation stop at the device check (ARCH 3 or CUDA 6)."""
    import random
    import scaled_quantize_fp8_warp_gb300 as fq
    rng = random.Random(1234)
    P = ctypes.c_void_p
    sizes = [-1, 0, 1, 15, 16, 17, 128, 130, 4096, 1 << 31, 1 << 40, (1 << 62) + 16]
    ptrs = [None, P(0x10000), P(0x10008), P(0x10004)]
    dts = [fq.DT_F32, fq.DT_BF16, 2, -1]
    fmts = [fq.E4M3, fq.E5M2, 2, -1]
    scalings = [fq.SCALE_TENSOR, fq.SCALE_TILE_1x128, fq.SCALE_BLOCK_128x128, fq.SCALE_ROW,
                fq.SCALE_MX_1x32, 5, -1]
    documented = {1, 2, 3, 6, 7}
    pick = rng.choice
    for _ in range(3000):
        kind = rng.randrange(6)
        if kind == 0:
            rc = lib.fp8_amax(pick(ptrs), pick(dts), pick(sizes), pick(ptrs), None)
        elif kind == 1:
            rc = lib.fp8_quantize_tensor(pick(ptrs), pick(dts), pick(sizes), pick(sizes),
                                         pick(fmts), pick(ptrs), pick(ptrs), pick(ptrs),
                                         pick(ptrs), rng.randrange(2), None)
        elif kind == 2:
            rc = lib.fp8_quantize_tile1x128(pick(ptrs), pick(dts), pick(sizes), pick(sizes),
                                            pick(fmts), pick(ptrs), pick(ptrs), pick(ptrs),
                                            pick(ptrs), rng.randrange(2), None)
        elif kind == 3:
            rc = lib.fp8_quantize_block128x128(pick(ptrs), pick(dts), pick(sizes), pick(sizes),
                                               pick(fmts), pick(ptrs), pick(ptrs), pick(ptrs),
                                               rng.randrange(2), None)
        elif kind == 4:
            rc = lib.fp8_quantize_mxfp8(pick(ptrs), pick(dts), pick(sizes), pick(sizes),
                                        pick(fmts), pick(ptrs), pick(ptrs), pick(ptrs),
                                        pick(ptrs), None)
        else:
            def operand():
                d, s = pick(ptrs), pick(ptrs)
                return fq.Operand(d.value if d is not None else None, pick(fmts), pick(scalings),
                                  s.value if s is not None else None, pick(sizes[:6]),
                                  pick(sizes[:6]))
            a, b = operand(), operand()
            fn = pick([lib.fp8_gemm, lib.fp8_gemm_fprop, lib.fp8_gemm_dgrad, lib.fp8_gemm_wgrad])
            rc = fn(ctypes.byref(a), ctypes.byref(b), pick(ptrs), pick(dts), pick(sizes),
                    pick(sizes), pick(sizes), None)
        assert rc in documented, (kind, rc)
