"""Write the stored oracle fixtures under tests/golden/.

Every expected value comes from the oracle (oracle/vbq_oracle.py), and every
input comes from the seeded generators. The CUDA path plays no part here. The
pages print no worked example, so these fixtures pin the oracle against
regressions. They also give the GPU tests small, fixed inputs.

Run: python tests/golden/make_golden.py
"""

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

from oracle import vbq_oracle as O  # noqa: E402
from synth import CONFIG0_PROBS, gen_matrix, gen_x, stress_bits, gen_matrix_with_bits  # noqa: E402
from tests.oracle_pins import tiny_case  # noqa: E402


def write(name, what, codes, bits, scales, X):
    X = np.atleast_2d(X)
    fx = {
        "name": name,
        "what": what,
        "grid": "w = s_g * (q - (2^b_g - 1)/2), groups of 64 along K (VBQ abstract; grid fixed by this project)",
        "codes": codes.tolist(),
        "bits": bits.tolist(),
        "scales_f16_bits": scales.tolist(),
        "x_bf16_bits": X.tolist(),
        "w_f32_bits": O.dequant(codes, bits, scales).view(np.uint32).tolist(),
        "y": O.gemm(codes, bits, scales, X).tolist(),
    }
    with open(os.path.join(HERE, name + ".json"), "w") as f:
        json.dump(fx, f, separators=(",", ":"))


def main():
    c, b, s, x = tiny_case(0)
    write("tiny_all_widths", "4x128, every 1- and 2-bit code, all four widths, batch 1", c, b, s, x)
    m = gen_matrix(16, 256, CONFIG0_PROBS, seed=21)
    write("mix16x256_b2", "16x256 iid mixed widths (1/2/4/8 at .69/.15/.11/.05), batch 2", m.codes, m.bits,
          m.scales, gen_x(256, seed=21, batch=2))
    bits = stress_bits("e", 8, 512)
    m = gen_matrix_with_bits(bits, 22, (9, 9))
    write("banded8x512", "8x512, first quarter of groups 8-bit, rest 1-bit, batch 1", m.codes, m.bits,
          m.scales, gen_x(512, seed=22))


if __name__ == "__main__":
    main()
