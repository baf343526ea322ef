"""Writes tests/golden/hash_v1.txt: rows and sign words of hash_version 1 for a
fixed short token sequence under every table of the five workloads. Calls only
the CPU oracle (and the workload configs for the table shapes and hash seeds).

    python tests/golden/make_hash_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import oracle as orc  # noqa: E402
from hashed_head_gram_gb300 import workloads as W  # noqa: E402

TOKENS = np.array([[0, 1, 2, 1000, 2, 1000, 49999, 7],
                   [7, 7, 7, 7, 31, 0, 1, 2]], np.int32)


def main(path=os.path.join(os.path.dirname(os.path.abspath(__file__)), "hash_v1.txt")):
    lines = ["# hash_version 1 regression values, written by make_hash_golden.py (oracle only).",
             "# tokens: " + " ".join(map(str, TOKENS.reshape(-1))) + f" as [{TOKENS.shape[0]}, {TOKENS.shape[1]}]",
             "# columns: workload table flat_index order head row sign_word0_hex"]
    for cfg in range(1, 6):
        w = W.make_workload(cfg)
        for sp in w.tables:
            _, rows, signs, bad = orc.index(sp, TOKENS, None, 50304)
            assert bad == -1
            for i in range(rows.shape[0]):
                for o in range(rows.shape[1]):
                    for k in range(rows.shape[2]):
                        lines.append(f"{cfg} {sp.name} {i} {o} {k} {rows[i, o, k]} {signs[i, o, k, 0]:016x}")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
