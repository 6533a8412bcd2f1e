"""Write page4_pattern.txt: oracle checksums for the day-74 program's own inputs.

Calls only the oracle package and the seeded input module.  The fixture lets
any machine (x86 here, Arm on the GPU host) confirm that its oracle build gives
bit-for-bit the same FP32 chain result, and gives the GPU tests an expected
value that never came from the CUDA path.

Inputs: "pipelined_gemm.cu", main(): a[i] = (i % 97) * 0.01f,
b[i] = (i % 53) * 0.02f - 0.5f, square sizes 512 (the program's first size).
Run: python tests/golden/make_golden.py
"""
import hashlib
import math
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from async_copy_pipelined_gb300 import inputs  # noqa: E402

SIZE = 512
SAMPLES = [(0, 0), (0, 511), (511, 0), (511, 511), (97, 53), (255, 256), (300, 17)]


def main():
    a = inputs.matrix_f32("page4a", SIZE, SIZE, 0, 0)
    b = inputs.matrix_f32("page4b", SIZE, SIZE, 0, 0)
    c32 = oracle.gemm_fmaf_chain(a, b, SIZE, SIZE, SIZE)
    c64 = oracle.gemm_f64(a, b, SIZE, SIZE, SIZE)
    lines = [
        "# Oracle checksums for the day-74 program's input pattern at N=512",
        "# (\"pipelined_gemm.cu\", main: a[i]=(i%97)*0.01f, b[i]=(i%53)*0.02f-0.5f).",
        "# Written by tests/golden/make_golden.py, which calls only oracle/.",
        f"N {SIZE}",
        "a_sha256 " + hashlib.sha256(a.tobytes()).hexdigest(),
        "b_sha256 " + hashlib.sha256(b.tobytes()).hexdigest(),
        "fmaf_sha256 " + hashlib.sha256(c32.tobytes()).hexdigest(),
        "f64_fsum " + repr(math.fsum(c64.ravel().tolist())),
    ]
    for (i, j) in SAMPLES:
        lines.append(f"sample {i} {j} fmaf_bits 0x{int(c32[i, j].view(np.uint32)):08x} f64 {float(c64[i, j])!r}")
    with open(os.path.join(HERE, "page4_pattern.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
