"""Writes tests/golden/kda_t5_d4.json: a small fixed case and the fp64 oracle's
output for it.  The pages print no numeric worked example of KDA, so this
fixture is a regression record of the oracle (it calls only ``oracle``); its
correctness rests on the pins in tests/test_oracle_pins.py.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def case():
    # small exact decimals so the inputs can be read by eye
    T, H, K = 5, 1, 4
    q = np.array([[1, 0, 2, -1], [0.5, 1, 0, 0], [0, 0, 1, 1], [2, -1, 0.5, 0], [1, 1, 1, 1]],
                 dtype=np.float64).reshape(T, H, K)
    k = np.array([[1, 1, 0, 0], [0, 1, -1, 0], [1, 0, 0, 2], [0.5, 0.5, 0.5, -0.5],
                  [0, 0, 3, 1]], dtype=np.float64).reshape(T, H, K)
    v = np.array([[1, 2, 3, 4], [-1, 0, 1, 0], [0.25, 0.5, -0.5, 2], [3, -2, 1, 0],
                  [0, 1, 0, -1]], dtype=np.float64).reshape(T, H, K)
    g = np.array([[0, 1, -1, 2], [0.5, 0.5, 0.5, 0.5], [-2, 0, 2, 0], [1, -1, 1, -1],
                  [0, 0, 0, 0]], dtype=np.float64).reshape(T, H, K)
    b = np.array([[0.0], [1.0], [-1.0], [2.0], [0.5]])
    return dict(q_raw=q, k_raw=k, v=v, g_raw=g, beta_raw=b, scale=0.5, lower_bound=-5.0,
                eps=1e-6)


if __name__ == "__main__":
    c = case()
    o, S = oracle.fwd_raw(c["q_raw"], c["k_raw"], c["v"], c["g_raw"], c["beta_raw"], c["scale"],
                          c["lower_bound"], eps=c["eps"])
    rec = {
        "about": "KDA forward, 5 tokens, 1 head, d_k = d_v = 4, zero initial state; "
                 "regression record of the fp64 oracle (the pages print no numeric example)",
        "inputs": {k_: (v_.tolist() if isinstance(v_, np.ndarray) else v_) for k_, v_ in c.items()},
        "out": o.tolist(), "final_state": S.tolist(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "kda_t5_d4.json")
    with open(path, "w") as f:
        json.dump(rec, f, indent=1)
    print("wrote", path)
