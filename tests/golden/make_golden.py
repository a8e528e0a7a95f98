"""Write tests/golden/tiny_mqa_decode.txt from the fp64 oracle.

The workload is the pages' tiny MQA decode ("Run Gemma4 head_dim 512 attention on
Triton", Test Coverage: partial and exact-multiple last pages): batch 2, 8 query heads on
1 kv head, head_dim 512, page_size 16, kv_len 37 and 64, seeded random page order.
The stored values are the oracle's lse per (sequence, head) and, per row, the first 8
output elements and the row sum of the output.  This script calls only oracle/ and synth.
"""

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402


def main():
    c = synth.workload("tiny_mqa_decode")
    out, lse = oracle.full(c, threads=1)
    path = os.path.join(HERE, "tiny_mqa_decode.txt")
    with open(path, "w") as f:
        f.write("# oracle output for the tiny MQA decode workload (see make_golden.py)\n")
        f.write("# b h lse sum(out) out[0..7]\n")
        for b in range(c.batch):
            for h in range(c.Hq):
                row = out[b, h]
                vals = " ".join(repr(float(x)) for x in row[:8])
                f.write(f"{b} {h} {float(lse[b, h])!r} {float(row.sum())!r} {vals}\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
