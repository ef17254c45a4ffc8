"""Writes tests/golden/*.txt from the float64 oracle and the seeded generator.

The pages print no worked numeric example for the FFN block, so the stored
values here are regression anchors written by this script, which calls only
``oracle`` and ``synth``.  Re-run it only when the oracle's arithmetic changes
for a reason that cites the passage it follows.
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth   # noqa: E402


def main():
    o = oracle.get()
    inp = synth.make_block_inputs(synth.C1_TINY_F32, seed=0, rows=4, d=32, ffn=48)
    y = o.block_from_inputs(inp, nthreads=1)
    with open(os.path.join(HERE, "block_tiny_f32_seed0_4x32x48.txt"), "w") as f:
        f.write("# oracle y for synth.make_block_inputs(C1_TINY_F32, seed=0, rows=4, d=32, ffn=48)\n")
        f.write("# recipe: x~N(0,1), g=1+0.1N(0,1), W~N(0,1/fan_in), eps=1e-6, fp32 storage\n")
        for row in y:
            f.write(" ".join(f"{v:.17g}" for v in row) + "\n")
    inp = synth.make_q4_inputs(synth.C5_DECODE_Q4, seed=0, rows=2, d=128, ffn=256)
    y = o.q4_block_from_inputs(inp, nthreads=1)
    with open(os.path.join(HERE, "block_q4_seed0_2x128x256.txt"), "w") as f:
        f.write("# oracle y for synth.make_q4_inputs(C5_DECODE_Q4, seed=0, rows=2, d=128, ffn=256)\n")
        f.write("# recipe: q~U{-8..7}, s=|N(0,1)|/(8 sqrt(fan_in)) fp16, x~N(0,1) bf16, eps=1e-6\n")
        for row in y:
            f.write(" ".join(f"{v:.17g}" for v in row) + "\n")


if __name__ == "__main__":
    main()
