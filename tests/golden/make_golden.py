"""Writes the oracle's regression fixtures under tests/golden/.

Calls only the fp64 oracle (and the seeded input generator).  The pages print
no worked numeric example for attention, so these fixtures are the oracle's
own outputs on seeded inputs, kept to catch unintended changes to the oracle;
they are checked by tests/test_oracle_golden.py and used as expected values
by the GPU parity tests of the fp32 workload.

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

from oracle import attention_fp64 as A  # noqa: E402
from exact_io_aware_36_gb300 import inputs as I  # noqa: E402

ROWS = [0, 1, 17, 63, 64, 100, 127]


def c1_fixture():
    w = I.workload("c1_fp32_fwd")
    x = I.make_inputs(w, seed=0)
    O, lse = A.attention_forward(x.q, x.k, x.v, w.scale, w.causal, x.cu_seqlens)
    return {
        "workload": w.name, "seed": 0, "scale": w.scale,
        "source": "oracle.attention_fp64.attention_forward on exact_io_aware_36_gb300.inputs",
        "rows": ROWS,
        "O": [[float(v) for v in O[t, 0]] for t in ROWS],
        "LSE": [float(lse[0, t]) for t in ROWS],
        "O_sum": float(O.sum()), "LSE_sum": float(lse.sum()),
    }


def small_bwd_fixture():
    w = I.small_case("bf16", causal=True, Hq=4, Hkv=2, d=64, alibi=True,
                     seqlens=(37, 130, 1), name="golden_small_bwd")
    x = I.make_inputs(w, seed=7)
    dq, dk, dv, O, lse, D = A.attention_backward(x.q, x.k, x.v, x.do, w.scale, True,
                                                 x.cu_seqlens, x.alibi_slopes)
    return {
        "workload": "small bf16 causal ALiBi GQA 4/2 d=64, seqlens (37,130,1)", "seed": 7,
        "source": "oracle.attention_fp64.attention_backward on exact_io_aware_36_gb300.inputs",
        "sums": {n: float(a.sum()) for n, a in
                 (("O", O), ("LSE", lse), ("D", D), ("dQ", dq), ("dK", dk), ("dV", dv))},
        "absmax": {n: float(np.abs(a).max()) for n, a in
                   (("O", O), ("dQ", dq), ("dK", dk), ("dV", dv))},
    }


if __name__ == "__main__":
    for name, fn in (("c1_fp32_rows.json", c1_fixture), ("small_bwd_sums.json", small_bwd_fixture)):
        with open(os.path.join(HERE, name), "w") as f:
            json.dump(fn(), f, indent=1)
        print("wrote", name)
