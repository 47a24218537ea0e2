"""Write tests/golden/oracle_linear_small.json: stored inputs and the oracle's
binary64 outputs for a few small linears.

Calls only ``oracle`` and ``synthetic_inputs``.  The stored values pin the
oracle's results across machines (x86 build host, Arm GPU host): the test
re-runs the oracle on the stored inputs and demands identical bits.  Shapes
cover several groups, a ragged zeros word (G = 3) and M = 1..3.

Usage: python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synthetic_inputs as si  # noqa: E402

CASES = [(1, 5, 384), (3, 7, 256), (2, 4, 1152)]


def main():
    out = {"what": "W4A16 linear, group 128: y = x @ ((q - z) * s)^T in binary64 "
                   "(forum thread 'vLLM on Hygon Z100', section 四).",
           "writer": "tests/golden/make_golden.py (oracle only)",
           "cases": []}
    for i, (M, N, K) in enumerate(CASES):
        seed = si.config_seed(60, 0, i)
        qw, s, zw = si.layer(seed, N, K)
        x = si.x(seed, M, K)
        qn, sn, zn, xn = si.as_u32(qw), si.as_u16(s), si.as_u32(zw), si.as_u16(x)
        y = oracle.linear(xn, qn, sn, zn, nthreads=1)
        out["cases"].append({
            "M": M, "N": N, "K": K, "group": 128,
            "x_f16_bits": xn.reshape(-1).tolist(),
            "qweight_u32": qn.reshape(-1).tolist(),
            "scales_f16_bits": sn.reshape(-1).tolist(),
            "zeros_u32": zn.reshape(-1).tolist(),
            "y_f64_hex": [float(v).hex() for v in y.reshape(-1)],
        })
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_linear_small.json")
    with open(path, "w") as f:
        json.dump(out, f, separators=(",", ":"))
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
