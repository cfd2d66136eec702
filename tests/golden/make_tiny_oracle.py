"""Writes tests/golden/tiny_oracle.txt: the oracle's routing and output on the
tiny workload (T=4, H=256, E=8, k=2, I=512, seed 0, inputs drawn on the CPU).
Calls only oracle/ and the seeded input generators."""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle as O  # noqa: E402


def compute(inp):
    res = O.moe_ffn_forward(inp["x"].double().numpy(), inp["norm_w"].double().numpy(), inp["eps"],
                            inp["k"], inp["w13"].double().numpy(), inp["w2"].double().numpy(),
                            router_w=inp["router_w"].double().numpy())
    return res


def parse(path):
    d = {}
    with open(path) as f:
        for ln in f:
            if ln.startswith("#") or not ln.strip():
                continue
            key, shape, vals = ln.split(":", 2)
            shp = tuple(int(s) for s in shape.split("x"))
            d[key] = np.array([float(v) for v in vals.split()]).reshape(shp)
    return d


def main():
    import workloads
    res = compute(workloads.make_inputs("c1_tiny", "cpu"))
    with open(os.path.join(HERE, "tiny_oracle.txt"), "w") as f:
        f.write("# oracle output for the tiny workload (seed 0, CPU generator); "
                "written by make_tiny_oracle.py\n")
        for key in ("ids", "topk_w", "out"):
            a = np.asarray(res[key], dtype=np.float64)
            f.write(f"{key}:{'x'.join(str(s) for s in a.shape)}:"
                    + " ".join(repr(float(v)) for v in a.reshape(-1)) + "\n")


if __name__ == "__main__":
    main()
