"""Writes oracle_regression.json: tiny oracle results frozen as a regression
fixture.  Calls only the oracle (and numpy for the seeded inputs)."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402


def cases():
    rng = np.random.default_rng(20261202)
    out = []
    for name, Hqk, HV, per_channel in (("kda_d4", 1, 1, True), ("gdn_d4_grouped", 1, 2, False)):
        lengths = [3, 0, 2]
        T, D = sum(lengths), 4
        q = rng.standard_normal((T, Hqk, D))
        k = rng.standard_normal((T, Hqk, D)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
        v = rng.standard_normal((T, HV, D))
        g = rng.uniform(-2, 0, (T, HV, D) if per_channel else (T, HV))
        b = rng.uniform(0, 1, (T, HV))
        h0 = rng.standard_normal((3, HV, D, D))
        do = rng.standard_normal((T, HV, D))
        cu = [0, 3, 3, 5]
        inputs = dict(q=q, k=k, v=v, g=g, beta=b, h0=h0, dout=do)
        out.append((name, cu, inputs))
    return out


def main():
    data = {}
    for name, cu, x in cases():
        r = oracle.run(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, 0.5, h0=x["h0"], dout=x["dout"])
        data[name] = {
            "cu_seqlens": cu,
            "scale": 0.5,
            "inputs": {k: v.tolist() for k, v in x.items()},
            "outputs": {k: v.tolist() for k, v in r.items()},
        }
    with open(os.path.join(HERE, "oracle_regression.json"), "w") as f:
        json.dump(data, f)


if __name__ == "__main__":
    main()
