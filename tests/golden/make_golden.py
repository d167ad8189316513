"""Writes the stored oracle values in this folder.  Calls only ``oracle/`` and the seeded input generator.

The pages print no worked numeric example for this block, so nothing here is a page value: the files are
regression fixtures of the oracle on seeded inputs (they also catch a change of the seeded generator).
Run from the repository root:  python tests/golden/make_golden.py
"""

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402
import torch  # noqa: E402

from oracle import ref  # noqa: E402
from seeded_inputs import TINY, decode_inputs, fwd_inputs  # noqa: E402

FWD_ROWS = [(0, 0, 0), (0, 1, 3), (0, 127, 2), (0, 200, 1), (0, 255, 3)]
DEC_ROWS = [(0, 0), (1, 5), (2, 11)]


def main():
    w = TINY
    q, k, v = (t.to(torch.float64).numpy() for t in fwd_inputs(w.B, w.T, w.Hq, w.Hkv, w.D, seed=0))
    fwd = {}
    for W in w.windows:
        vals = ref.attn_fwd_rows(q, k, v, W, FWD_ROWS)
        fwd[str(W)] = [[float(x) for x in row[:16]] for row in vals]
    d = decode_inputs(3, 12, 4, 128, 64, 1, 63, seed=0, with_new=True)
    f = {n: (d[n].to(torch.float64).numpy() if d[n] is not None else None) for n in d}
    lens = d["cache_lens"].numpy()
    out, _ = ref.attn_decode(f["q"], f["kcache"], f["vcache"], lens, 16, f["k_new"], f["v_new"])
    doc = {
        "about": "oracle regression values (first 16 of 128 dims) on seeded inputs; written by make_golden.py",
        "fwd_workload": {"B": w.B, "T": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "seed": 0},
        "fwd_rows_b_i_h": FWD_ROWS,
        "fwd": fwd,
        "decode_workload": {"B": 3, "Hq": 12, "Hkv": 4, "D": 128, "Tcap": 64, "len_lo": 1, "len_hi": 63,
                            "seed": 0, "with_new": True, "window": 16, "cache_lens": lens.tolist()},
        "decode_rows_b_h": DEC_ROWS,
        "decode": [[float(x) for x in out[b, h, :16]] for (b, h) in DEC_ROWS],
    }
    with open(os.path.join(HERE, "oracle_tiny.json"), "w") as fh:
        json.dump(doc, fh, indent=1)
    print("wrote", os.path.join(HERE, "oracle_tiny.json"), np.asarray(fwd["128"]).shape)


if __name__ == "__main__":
    main()
