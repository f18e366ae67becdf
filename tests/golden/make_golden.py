"""Writes tests/golden/brute_tiny.json from the exact rational brute force
(oracle.brute) only.  Run from the repository root:  python -m tests.golden.make_golden"""
import json
import os

from oracle import brute
from tests.oracle_pins import brute_case

SEED, T, D = 7, 5, 4


def main():
    case = brute_case(SEED, T=T, d=D)
    o, S = brute.brute_recurrence(*case)
    out = {"about": "exact KDA recurrence on a tiny rational case (tests.oracle_pins.brute_case)",
           "seed": SEED, "T": T, "d": D,
           "o": [[str(x) for x in r] for r in o], "S": [[str(x) for x in r] for r in S]}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "brute_tiny.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
