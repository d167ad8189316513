"""The oracle on seeded inputs still gives the stored regression values (CPU only).

``tests/golden/oracle_tiny.json`` was written by ``tests/golden/make_golden.py``, which calls only the oracle.
A failure here means the oracle's arithmetic or the seeded generator changed.
"""

import json
import os

import numpy as np
import torch

from oracle import ref
from seeded_inputs import decode_inputs, fwd_inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_regression_values():
    with open(os.path.join(HERE, "golden", "oracle_tiny.json")) as fh:
        doc = json.load(fh)
    w = doc["fwd_workload"]
    q, k, v = (t.to(torch.float64).numpy() for t in fwd_inputs(w["B"], w["T"], w["Hq"], w["Hkv"], w["D"], w["seed"]))
    rows = [tuple(r) for r in doc["fwd_rows_b_i_h"]]
    for W, exp in doc["fwd"].items():
        got = ref.attn_fwd_rows(q, k, v, int(W), rows)[:, :16]
        np.testing.assert_allclose(got, np.asarray(exp), rtol=1e-12, atol=1e-14)
    dw = doc["decode_workload"]
    d = decode_inputs(dw["B"], dw["Hq"], dw["Hkv"], dw["D"], dw["Tcap"], dw["len_lo"], dw["len_hi"],
                      seed=dw["seed"], with_new=dw["with_new"])
    assert d["cache_lens"].tolist() == dw["cache_lens"]
    f = {n: d[n].to(torch.float64).numpy() for n in ("q", "kcache", "vcache", "k_new", "v_new")}
    out, _ = ref.attn_decode(f["q"], f["kcache"], f["vcache"], d["cache_lens"].numpy(), dw["window"],
                             f["k_new"], f["v_new"])
    got = np.stack([out[b, h, :16] for (b, h) in doc["decode_rows_b_h"]])
    np.testing.assert_allclose(got, np.asarray(doc["decode"]), rtol=1e-12, atol=1e-14)
