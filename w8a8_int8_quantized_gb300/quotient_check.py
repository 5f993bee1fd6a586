"""Build and run quotient_check.cu: the row rules' division-free codes against the IEEE float32
quotient -- the symmetric rule exhaustively over bf16 rows, the affine rule over every bf16 value
of 65536 hashed row ranges.  Prints JSON; needs nvcc and a GB300.

    python -m w8a8_int8_quantized_gb300.quotient_check
"""

import json
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "quotient_check.cu")
EXE = os.path.join(HERE, "_build", "quotient_check")


def build():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    os.makedirs(os.path.dirname(EXE), exist_ok=True)
    deps = [SRC, os.path.join(HERE, "csrc", "common.cuh")]
    if os.path.exists(EXE) and all(os.path.getmtime(EXE) >= os.path.getmtime(d) for d in deps):
        return EXE
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
           "-I", os.path.join(HERE, "csrc"), "-I", os.path.join(os.path.dirname(HERE), "include"), SRC, "-o", EXE]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed:\n{r.stdout}\n{r.stderr}")
    return EXE


def run():
    """Returns the parsed JSON result."""
    r = subprocess.run([build()], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"quotient_check failed:\n{r.stdout}\n{r.stderr}")
    return json.loads(r.stdout)


if __name__ == "__main__":
    print(json.dumps(run()))
    sys.exit(0)
