"""CPU-only guard on the expert GEMMs' register use (no GPU needed: nvcc
cross-compiles for sm_103a).  The GEMM CTA has ten warps, so two of the four
sub-partitions hold three of them and each thread gets at most 168 registers;
anything above spills to local memory, which the small L1 beside the GEMM's
shared memory mostly misses.  The store epilogue (expert wgrads, down and
gate/up dgrads) must not spill at all, and the SwiGLU-backward epilogue stays
within the 84 bytes of spill stores of its 32-column stash form (it spilled
208 before), so a change that brings the spills back fails here first."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GEMM = os.path.join(ROOT, "mixture_experts_layer_device_gb300", "csrc", "gemm.cu")


def _ptxas_report(tmp_path):
    nvcc = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
    if not os.path.exists(nvcc) and not shutil.which("nvcc"):
        pytest.skip("nvcc not available")
    cmd = [nvcc if os.path.exists(nvcc) else "nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
           "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"), "-Xptxas", "-v", "-c", GEMM,
           "-o", str(tmp_path / "gemm.o")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stderr


def _kernels(report):
    """{mangled gemm_kernel name: (registers, spill store bytes, spill load bytes)}"""
    out, name, spills = {}, None, None
    for line in report.splitlines():
        m = re.search(r"Compiling entry function '(\S*gemm_kernel\S*)'", line)
        if m:
            name, spills = m.group(1), None
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and name:
            spills = (int(m.group(1)), int(m.group(2)))
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and name and spills is not None:
            out[name] = (int(m.group(1)), spills[0], spills[1])
            name = None
    return out


def _find(kernels, fmt, bn, epi, ring=0, dump=0):
    key = "gemm_kernelILi%dELi%dELi%dELb%dELb%d" % (fmt, bn, epi, ring, dump)
    hits = [v for k, v in kernels.items() if key in k and "gemm_pair" not in k]
    assert len(hits) == 1, (key, sorted(kernels))
    return hits[0]


@pytest.fixture(scope="module")
def kernels(tmp_path_factory):
    return _kernels(_ptxas_report(tmp_path_factory.mktemp("ptxas")))


def test_store_epilogue_gemms_do_not_spill(kernels):
    regs, st, ld = _find(kernels, fmt=1, bn=256, epi=0)   # MXFP8, 256-wide tiles, bf16 store
    assert regs <= 168
    assert st == 0 and ld == 0


def test_swiglu_backward_epilogue_spills_stay_small(kernels):
    regs, st, ld = _find(kernels, fmt=1, bn=256, epi=2)   # MXFP8 down dgrad + SwiGLU backward
    assert regs <= 168
    assert st <= 96 and ld <= 160, (st, ld)
