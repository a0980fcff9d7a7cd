"""Write the stored expected values under tests/golden/.

Calls only the seeded generators (synth) and the CPU oracle (oracle); nothing
here touches the CUDA library.  Run from the repository root:

    python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402


def main():
    case = synth.full_tile_case()
    fr, tc, fs, ts = oracle.full_tile_sum(case["values"], case["count"], case["initial"],
                                          case["tile_size"])
    with open(os.path.join(HERE, "full_tile_case.txt"), "w") as f:
        f.write("# One 63x32 f32 segment, uniform on the 2**-23 grid from the seeded generator\n")
        f.write("# (workload seed 1), count 61, initial 0.5, tile 8; expected outputs from the\n")
        f.write("# fp64 oracle (exact for grid values).  Written by make_golden.py.\n")
        f.write(f"final_row {fr}\ntail_count {tc}\nfull_sum {fs.hex()}\ntail_sum {ts.hex()}\n")


if __name__ == "__main__":
    main()
