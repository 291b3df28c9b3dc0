"""Write the stored expected values under tests/golden/.

Every stored value comes from the fp64 oracle (``oracle``) on inputs from
``attn_inputs``; nothing here touches the CUDA path.  Run from the repository
root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import attn_inputs  # noqa: E402
import oracle  # noqa: E402

ROWS = [0, 1, 63, 127, 128, 200, 255]


def tiny_fixture():
    w = attn_inputs.WORKLOADS["tiny"]
    x = w.inputs()
    o, lse = oracle.attn_fwd(x.q, x.k, x.v, False, w.scale)
    flat_o = o.reshape(-1, w.D)
    return {
        "source": "fp64 oracle (oracle.attn_fwd) on attn_inputs.WORKLOADS['tiny']",
        "workload": {"B": w.B, "H": w.H, "S": w.S, "D": w.D, "dtype": w.dtype,
                     "causal": False, "seed": w.seed, "scale": w.scale},
        "lse": [float(t) for t in lse.reshape(-1)],
        "o_rows": {str(r): [float(t) for t in flat_o[r]] for r in ROWS},
    }


def main():
    path = os.path.join(HERE, "tiny_fp16_noncausal_oracle.json")
    with open(path, "w") as f:
        json.dump(tiny_fixture(), f, indent=0)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
