"""Write tests/golden/ns_small_cases.json from the fp64 oracle (and nothing else).

The inputs are small hand-chosen matrices whose normalized singular values are
rational (Pythagorean triples), so that tests can also check every stored value
against the exact rational closed form U diag(p^k(s/||s||)) V^T at run time.
The stored values are regression pins of the oracle: a later change to its arithmetic
shows up as a mismatch here.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import muon_ref  # noqa: E402

CASES = [
    # name, matrix, ns_steps
    ("diag_3_4", [[3.0, 0.0], [0.0, 4.0]], 5),
    ("wide_2x3", [[0.0, 3.0, 0.0], [4.0, 0.0, 0.0]], 5),
    ("tall_3x2", [[0.0, 0.0], [-3.0, 0.0], [0.0, 4.0]], 5),
    ("scalar_neg7", [[-7.0]], 5),
    ("diag_5_12_one_step", [[5.0, 0.0], [0.0, 12.0]], 1),
    ("diag_5_12_zero_steps", [[5.0, 0.0], [0.0, 12.0]], 0),
    ("rank1_2x2", [[3.0, 4.0], [6.0, 8.0]], 5),
]


def main():
    out = {
        "source": "oracle/muon_ref.py newton_schulz (fp64); see make_golden.py",
        "coeffs": [muon_ref.NS_A, muon_ref.NS_B, muon_ref.NS_C],
        "cases": [],
    }
    for name, X, steps in CASES:
        O = muon_ref.newton_schulz(X, steps)
        out["cases"].append({"name": name, "input": X, "ns_steps": steps,
                             "output": O.tolist()})
    path = os.path.join(HERE, "ns_small_cases.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
