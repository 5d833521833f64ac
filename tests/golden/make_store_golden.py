"""Writes tests/golden/store_tiny.txt: the compressed store of a tiny layer
(2 experts, d_model 64, d_ff 64, peaked codes, seed 13) as the oracle builds
it. Calls only oracle/ and the seeded generator; rerun it only when the
store's format itself is changed on purpose."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle.store as S  # noqa: E402
import synth  # noqa: E402

E, D, F, SEED = 2, 64, 64, 13


def build() -> dict:
    w = {nm: np.stack([synth.expert_weights(SEED, e, D, F, dist=synth.CODES_PEAKED)[nm].ravel()
                       for e in range(E)]) for nm in S.NAMES}
    return S.build_store(w, E, D, F)


def main():
    st = build()
    lines = ["# Compressed store of a tiny layer, written by make_store_golden.py from the",
             "# oracle (oracle/store_oracle.c): 2 experts, d_model 64, d_ff 64, peaked E2M1",
             "# codes, seed 13. Sections: records (8 words per tile), tables (256 entries",
             "# per expert and array, nonzero ones as byte:f), blob (hex, 32 bytes a line)."]
    lines.append("records")
    for r in st["records"].reshape(-1, 8):
        lines.append(" ".join(str(int(v)) for v in r))
    lines.append("tables")
    for t in st["tables"].reshape(-1, 256):
        lines.append(" ".join(f"{b}:{int(f)}" for b, f in enumerate(t) if f))
    lines.append("blob")
    b = st["blob"]
    for i in range(0, b.size, 32):
        lines.append(b[i:i + 32].tobytes().hex())
    with open(os.path.join(HERE, "store_tiny.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
