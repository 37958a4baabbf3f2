"""Writes regression.txt: SHA-256 digests of the oracle's outputs on small
seeded inputs, so that any change to the oracle's arithmetic shows up as a
failing test (and has to be justified when the digests are rewritten).

Calls only the oracle and the input generator.  The inputs are the
`small_ints` stream (integers times 2^-4, no transcendental function), so the
digests are the same on every host.

    python tests/golden/make_regression.py
"""
import hashlib
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads  # noqa: E402

CASES = [(B, rows, hidden) for B in (64, 128, 256) for rows, hidden in [(8, 1024)]]


def digests():
    out = []
    for B, rows, hidden in CASES:
        xs = [workloads.generate("small_ints", rows, hidden, seed=s).reshape(-1) for s in range(3)]
        packed = [oracle.compress(x, B) for x in xs]
        dec = oracle.decompress(packed[0], xs[0].size, B)
        red = oracle.reduce_shards(packed, xs[0].size, B)
        for what, arr in (("compress", packed[0]), ("decompress", dec), ("reduce3", red)):
            out.append(f"B={B} rows={rows} hidden={hidden} {what} "
                       f"{hashlib.sha256(arr.tobytes()).hexdigest()}")
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "regression.txt"), "w") as f:
        f.write("\n".join(digests()) + "\n")
