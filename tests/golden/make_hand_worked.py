"""Writes the 'expected' values of hand_worked_n1.json from its closed-form expressions.

Uses only the math module (never the oracle or the CUDA library).
Run: python tests/golden/make_hand_worked.py
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))
PATH = os.path.join(HERE, "hand_worked_n1.json")
ENV = {"log": math.log, "exp": math.exp, "__builtins__": {}}


def ev(expr, **kw):
    return float(eval(expr, dict(ENV), kw))


def main():
    with open(PATH) as f:
        g = json.load(f)
    for c in g["scan_cases"]:
        c["expected"] = [ev(c["expected_expr"], t=t) for t in range(len(c["u"]))]
        c["final"] = ev(c["final_expr"])
    for c in g["update_cases"]:
        c["state_expected"] = ev(c["state_expr"])
        c["out_expected"] = ev(c["out_expr"])
    with open(PATH, "w") as f:
        json.dump(g, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
