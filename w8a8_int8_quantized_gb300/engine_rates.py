"""Build and run the tensor-engine probe (engine_probe.cu) and print its JSON.

    python -m w8a8_int8_quantized_gb300.engine_rates

It measures the dense rate of the GPU's only INT8 tensor instruction (mma.sync s8), the
tcgen05 kind::f16 rates the GEMM runs at, the issue cost of the MMA-issuing thread, and the
exactness of fp32 TMEM accumulation for int8-valued operands.  Needs nvcc and a GB300.
"""

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "engine_probe.cu")
EXE = os.path.join(HERE, "_build", "engine_probe")


def build():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    os.makedirs(os.path.dirname(EXE), exist_ok=True)
    if os.path.exists(EXE) and os.path.getmtime(EXE) >= os.path.getmtime(SRC):
        return EXE
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", SRC, "-o", EXE]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed:\n{r.stdout}\n{r.stderr}")
    return EXE


def main():
    exe = build()
    r = subprocess.run([exe], capture_output=True, text=True)
    sys.stdout.write(r.stdout)
    sys.stderr.write(r.stderr)
    return r.returncode


if __name__ == "__main__":
    sys.exit(main())
