"""Writes exact_rational_case.json: integer q, k, v with f~ = 0 and i~ = 0 (f = 1/2, i = 1),
d_qk = 4, and the exact h_t and final C of the mLSTM cell as fractions.

The values come from the unrolled sum of "xLSTM: How Exponential Gating and Matrix Memory
Scale Recurrent Neural Networks" (llms.blog), section 3 "The Parallel Dual Form"
(C_T = sum_t (prod_{tau=t+1..T} f_tau) i_t v_t k_t^T), with the normaliser of section 3
"Associative Matrix Cell State" (max(|n_t^T q_t|, 1)), evaluated in exact rational arithmetic.
Neither the oracle nor the CUDA library is called.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

from exact_case import exact_rational_case  # noqa: E402


def main():
    (q, k, v, ig, fg), h, C, _n = exact_rational_case()
    doc = {
        "citation": "llms.blog xLSTM page, section 3: unrolled C_T and retrieval "
                    "h = C q / max(|n^T q|, 1); f = sigmoid(0) = 1/2, i = exp(0) = 1, "
                    "k scaled by 1/sqrt(4)",
        "q": q.tolist(), "k": k.tolist(), "v": v.tolist(), "ig": ig.tolist(), "fg": fg.tolist(),
        "h": [[str(x) for x in row] for row in h],
        "C_last": [[str(x) for x in row] for row in C],
    }
    with open(os.path.join(HERE, "exact_rational_case.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()
