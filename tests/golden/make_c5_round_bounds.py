"""Write c5_round_bounds.json: the oracle's round bound for every row of config 5.

Config 5 is B=256, V=256000 (half Zipf(1.1) rows permuted, half near-flat softmax
rows, 5 % bad rows), joint top-k 128000 + top-p 0.99 + min-p 0.01.  For each row the
file holds ``oracle.filters.round_bound`` (the bound on the number of draws of the
dual-pivot sampler, from the FlashInfer blog's dual-pivot section: every failure
raises `low` past a token and at least halves high - low), 0 for a row whose allowed
set is empty or that is invalid, and the row's validity.  The benchmark reads these
stored values next to the kernels' round counts; it never runs the oracle itself.

    python tests/golden/make_c5_round_bounds.py
"""
from __future__ import annotations

import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

OUT = os.path.join(HERE, "c5_round_bounds.json")


def main() -> None:
    import numpy as np

    import workloads
    from oracle import filters

    w = workloads.config5()
    bounds, valid = [], []
    for i in range(w.batch_in):
        p = w.probs[i]
        ok = bool(filters.row_is_valid(p))
        args = (int(w.top_k[i]), float(w.top_p[i]), float(w.min_p[i]), "joint")
        b = filters.round_bound(p, *args) if ok else 0
        valid.append(ok and b > 0)
        bounds.append(int(b))
    digest = hashlib.sha256(np.ascontiguousarray(w.probs).tobytes()).hexdigest()[:16]
    with open(OUT, "w") as fh:
        json.dump({"workload": w.name, "probs_sha256_16": digest, "order": "joint",
                   "top_k": int(w.top_k[0]), "top_p": float(w.top_p[0]), "min_p": float(w.min_p[0]),
                   "bad_rows": [int(r) for r in w.bad_rows], "valid": valid, "round_bound": bounds}, fh)
        fh.write("\n")
    print(OUT, sum(valid), "valid rows, largest bound", max(bounds))


if __name__ == "__main__":
    main()
