"""Write tiny_oracle_digest.txt: the oracle's routing and a sample of its
output on the tiny workload (T=8, H=256, E=288, I=64, seed 0).

Calls only the oracle (and the seeded input generator).  Rerun after a change
to the oracle's arithmetic that a passage of the pages justifies:
    python tests/golden/make_tiny_digest.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synthetic  # noqa: E402
from moe_inputs import make_inputs  # noqa: E402


def main():
    wl = synthetic.WORKLOADS["tiny"]
    inp = make_inputs(wl)
    out, idx, w = oracle.moe_forward(inp.x, inp.w_router, inp.b_router, inp.experts, inp.shared,
                                     "bf16")
    lines = ["# Oracle digest of the tiny workload (T=8, H=256, E=288, I=64, seed 0).",
             "# Written by tests/golden/make_tiny_digest.py, which calls only the oracle.",
             f"# tokens redrawn for the top-8 boundary gap: {inp.redraws}",
             "# idx t e_0..e_7   |   out t h value"]
    for t in range(wl.T):
        lines.append("idx %d %s" % (t, " ".join(str(int(e)) for e in idx[t])))
    rng = np.random.default_rng(0)
    for t in range(wl.T):
        for h in sorted(rng.choice(wl.H, 6, replace=False)):
            lines.append("out %d %d %.17g" % (t, h, out[t, h]))
    with open(os.path.join(HERE, "tiny_oracle_digest.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
