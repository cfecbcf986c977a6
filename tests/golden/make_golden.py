"""Writes tests/golden/exact_k4.json: a tiny worked example of the recurrence in
exact rational arithmetic.  Calls only oracle/ (oracle.exact).

The pages print no worked example, so the fixture is built from the
recurrence's definition ("gated_delta_recurrence_fwd_gpu" summary; the gated
delta rule step of "core.ssm.ops.gdp.fused_recurrent") on inputs chosen so
that nothing needs rounding: dyadic values (exact in float32) and q/k vectors
whose norms are integers, with eps = 0 and K = 4 (scale 1/2).

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import exact  # noqa: E402


def dyadic_case():
    K = V = 4
    nk, nv = 1, 2
    # integer norms: (1,2,2,4)->5 (2,-3,6,0)->7 (4,4,-7,0)->9 (2,4,5,-6)->9 (-1,2,-2,4)->5
    qs = [[1, 2, 2, 4], [2, -3, 6, 0], [4, 4, -7, 0], [2, 4, 5, -6], [-1, 2, -2, 4]]
    ks = [[2, 4, 5, 6], [1, -2, 2, 4], [2, 3, 6, 0], [-4, 4, 7, 0], [2, -4, 5, 6]]
    vs = [[0.5, -1.25, 2.0, 0.75, -0.5, 1.0, 0.25, -2.0],
          [1.5, 0.0, -0.75, 1.25, 2.0, -1.5, 0.5, 0.25],
          [-1.0, 0.5, 0.25, -0.25, 1.75, 0.75, -1.25, 1.0],
          [0.25, 1.75, -2.0, 0.5, -0.75, 0.0, 1.5, -0.5],
          [2.0, -0.5, 1.0, -1.75, 0.25, 1.25, -1.0, 0.75]]
    qkv = [[float(x) for x in qs[t] + ks[t]] + vs[t] for t in range(5)]
    decay = [[0.875, 0.5], [1.0, 0.75], [0.9375, 0.625], [0.5, 1.0], [0.75, 0.875]]
    beta = [[0.5, 0.25], [1.0, 0.75], [0.125, 0.0], [0.375, 0.5], [0.625, 1.0]]
    state = [[[[((3 * s + 5 * h + 7 * i + 11 * j) % 9 - 4) / 8.0 for j in range(V)]
               for i in range(K)] for h in range(nv)] for s in range(3)]
    return dict(K=K, V=V, nk=nk, nv=nv, qkv=qkv, decay=decay, beta=beta, state=state,
                slot_idx=[2, 0], offsets=[0, 3, 5])


def main():
    c = dyadic_case()
    S0 = {s: c["state"][s] for s in range(3)}
    out, fin = exact.fwd_exact(c["qkv"], c["decay"], c["beta"], S0, c["slot_idx"],
                               c["offsets"], nk=c["nk"], nv=c["nv"], K=c["K"], V=c["V"],
                               use_l2norm=True, eps=0)
    T, cols = 5, c["nv"] * c["V"]
    doc = {
        "about": "exact rational outputs of the gated delta rule on a dyadic K=V=4 case "
                 "(l2norm on, eps=0, scale=K^-0.5=1/2); written by make_golden.py",
        "inputs": c,
        "out_exact": [[str(out[(t, j)]) for j in range(cols)] for t in range(T)],
        "final_state_exact": {f"{s},{h}": [[str(x) for x in row] for row in S]
                              for (s, h), S in fin.items()},
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "exact_k4.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
