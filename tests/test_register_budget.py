"""Build-time guard of the decode kernel's register budget (no GPU needed): the bf16 decode at
head_dim 128 must keep three CTAs per SM (192 threads each), which its HBM throughput depends on
(at two CTAs per SM the 64x4096 call measured 183 instead of 168 us). ptxas's own report."""

import os
import re
import subprocess
import tempfile

import pytest

from paged_kv_attention_gb300 import build

SRC = os.path.join(os.path.dirname(build.__file__), "csrc", "decode.cu")


def have_nvcc():
    try:
        return bool(build.nvcc())
    except RuntimeError:
        return False


def ptxas_registers(src):
    with tempfile.TemporaryDirectory() as d:
        r = subprocess.run([build.nvcc(), *build._flags(False), "-Xptxas", "-v", "-c", src,
                            "-o", os.path.join(d, "x.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    regs, current = {}, None
    for line in r.stderr.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            current = m.group(1)
        m = re.search(r"Used (\d+) registers", line)
        if m and current:
            regs[current] = int(m.group(1))
            current = None
    return regs


@pytest.mark.skipif(not have_nvcc(), reason="no nvcc")
def test_bf16_decode_keeps_three_ctas_per_sm():
    regs = ptxas_registers(SRC)
    name = next(k for k in regs if "decode_tc_kernelILi128ELi1ELi0E" in k)
    # registers are allocated in steps of 8 per thread: 3 CTAs x 6 warps x 32 threads x 112 <= 65536
    assert regs[name] <= 112, f"{regs[name]} registers: fewer than 3 CTAs per SM"
