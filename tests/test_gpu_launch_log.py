"""No silent fallback: with FP8Q_LOG=1 every call names the kernel that
served it.  A child process (the switch is read once per process) runs one
call of each kind and the test checks the kernel named for each, so a
dispatch change that routes a scaling to another kernel fails here."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import torch
import scaled_quantize_fp8_warp_gb300 as fq
fq.load_library()
x = torch.randn(512, 256, device="cuda", dtype=torch.bfloat16)
w = torch.randn(384, 256, device="cuda", dtype=torch.bfloat16)
w64 = torch.randn(64, 256, device="cuda", dtype=torch.bfloat16)
T = fq.GemmOperand.tensor
def mark(name):
    import sys
    print("=== " + name, file=sys.stderr, flush=True)
mark("amax")
ax = fq.fp8_amax(x)
mark("tensor cast")
qx, qxt, sx = fq.fp8_quantize_tensor(x, fq.E4M3, ax, want_qt=True)
aw = fq.fp8_amax(w)
qw, _, sw = fq.fp8_quantize_tensor(w, fq.E4M3, aw)
a64 = fq.fp8_amax(w64)
q64, _, s64 = fq.fp8_quantize_tensor(w64, fq.E4M3, a64)
mark("pair gemm")
fq.fp8_gemm_fprop(T(qx, 0, sx), T(qw, 0, sw))
mark("one-SM gemm")
fq.fp8_gemm_fprop(T(qx, 0, sx), T(q64, 0, s64))
mark("tile cast")
qa, sa, _, _ = fq.fp8_quantize_tile1x128(x, fq.E4M3, rows=True)
mark("block cast")
qb, _, sb = fq.fp8_quantize_block128x128(w, fq.E4M3)
mark("block gemm")
fq.fp8_gemm_fprop(fq.GemmOperand.tile(qa, 0, sa), fq.GemmOperand.block(qb, 0, sb))
mark("mx cast")
mxa = fq.fp8_quantize_mxfp8(x, fq.E4M3, rows=True)
mxb = fq.fp8_quantize_mxfp8(w, fq.E4M3, rows=True)
mark("mx gemm")
fq.fp8_gemm_fprop(fq.GemmOperand.mx(mxa[0], 0, mxa[1]), fq.GemmOperand.mx(mxb[0], 0, mxb[1]))
mark("one-call tensor")
fq.fp8_quantize_tensor_current(x, fq.E4M3)
mark("end")
torch.cuda.synchronize()
assert fq.device_status() == 0
"""

EXPECT = {
    "amax": ["launch amax_kernel bf16 input, 131072 elements"],
    "tensor cast": ["launch quant2d_kernel mode tensor bf16 input"],
    "pair gemm": ["launch gemm_tensor_pair_kernel unit 256x256", "scales tensor out bf16"],
    "one-SM gemm": ["launch gemm_tensor_kernel unit 128x64"],
    "tile cast": ["launch quant2d_kernel mode tile_rows"],
    "block cast": ["launch quant2d_kernel mode block"],
    "block gemm": ["launch gemm_blockscaled_kernel unit 128x256", "promoted per K block"],
    "mx cast": ["launch quant2d_kernel mode mx"],
    "mx gemm": ["launch gemm_mx_kernel unit 128x256", "scales mx"],
    "one-call tensor": ["launch quant2d_kernel mode tensor_fused", "cooperative"],
}


def test_every_call_names_its_kernel():
    env = dict(os.environ, FP8Q_LOG="1")
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    sections, cur = {}, None
    for line in r.stderr.splitlines():
        if line.startswith("=== "):
            cur = line[4:]
            sections[cur] = []
        elif cur is not None and line.startswith("[fp8q]"):
            sections[cur].append(line)
    for name, needles in EXPECT.items():
        text = "\n".join(sections.get(name, []))
        for n in needles:
            assert n in text, f"{name}: '{n}' not in:\n{text}"
