"""Comparison helpers shared by the tests (no method arithmetic here)."""
from __future__ import annotations

import numpy as np


def rel_l2(a, b, floor=1e-6):
    """Per-vector relative L2 error ||a-b|| / max(||b||, floor) over the last axis."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    num = np.linalg.norm(a - b, axis=-1)
    den = np.maximum(np.linalg.norm(b, axis=-1), floor)
    return num / den


def near_tie(s, rel=1e-6, abs_=0.0):
    """True where s lies within rel*|s| (+abs_) of a rounding tie (a half-integer)."""
    s = np.asarray(s, np.float64)
    return np.abs(s - (np.floor(s) + 0.5)) <= rel * np.abs(s) + abs_


def code_mismatches(got, want, s_ref, rel=1e-6, abs_=0.0):
    """(n_mismatch, n_allowed_ok, ok) for int8 codes compared under the near-tie rule.

    A mismatch is allowed only at a near tie of the reference's pre-round value and
    only one code apart.
    """
    got = np.asarray(got, np.int32)
    want = np.asarray(want, np.int32)
    diff = got != want
    n = int(diff.sum())
    if n == 0:
        return 0, True
    tie = near_tie(np.asarray(s_ref)[diff], rel, abs_)
    one = np.abs(got[diff] - want[diff]) <= 1
    return n, bool(np.all(tie & one))


def read_golden(name):
    import os

    path = os.path.join(os.path.dirname(__file__), "golden", name)
    out = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (x.strip() for x in line.split("=", 1))
            out[k] = float(v) if "." in v else int(v)
    return out
