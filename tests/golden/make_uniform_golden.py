"""Write uniform_logits.json: closed-form RNN-T losses for constant logits.

With every logit equal, each node's output distribution is uniform (p = 1/V),
every alignment emits exactly T blanks and U labels, and there are
C(T-1+U, U) alignments (the (t, u) lattice walks of the ESPnet GPURNNT docs /
warp-transducer blog section 1.1).  Hence

    loss = (T + U) * log V - log C(T-1+U, U).

This script uses only that formula (math.lgamma); it does not call the
oracle.  Shapes: the rnnt-loss-ascend README call example ("调用说明": T=[4, 6],
target_lengths=[2, 1], V=8, 24 rows) and a spread of larger lattices.
Run: python tests/golden/make_uniform_golden.py
"""
import json
import math
import os

CASES = [
    # (name, T list, U list, V, citation)
    ("readme_call_example", [4, 6], [2, 1], 8,
     "rnnt-loss-ascend README, section 调用说明 (24-row example)"),
    ("t1_u0", [1], [0], 5, "T=1, U=0 single node"),
    ("u0_long", [37], [0], 11, "U=0: blanks only"),
    ("t1_long_targets", [1], [9], 13, "T=1: all labels then the terminal blank"),
    ("mid", [120, 77, 5], [30, 12, 0], 40, "mixed lattice sizes"),
    ("bpe_like", [400], [75], 1024, "BPE-like lattice, V=1024"),
]


def log_binom(n, k):
    return math.lgamma(n + 1) - math.lgamma(k + 1) - math.lgamma(n - k + 1)


def main():
    out = []
    for name, T, U, V, cite in CASES:
        losses = [(t + u) * math.log(V) - log_binom(t - 1 + u, u) for t, u in zip(T, U)]
        out.append({"name": name, "T": T, "U": U, "V": V, "losses": losses, "source": cite})
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "uniform_logits.json")
    with open(path, "w") as f:
        json.dump({"formula": "(T+U)*log(V) - log(C(T-1+U, U))", "cases": out}, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
