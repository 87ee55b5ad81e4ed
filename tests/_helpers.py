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


def tie_rows(qm):
    """Rows whose t * h values are exact half-integers (C = 0, smoothing off, so t = R and
    h = qm / max|row|) and the codes round-half-to-even gives them, typed out by hand.
    Row r is the base row times 2^(r - 1), so h = 2^(1 - r) exactly and every product
    stays a half-integer."""
    base = [qm, 0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, -3.5, qm - 0.5, -(qm - 0.5), 4.5, -4.5]
    if qm == 7:
        want = [7, 0, 2, 2, 4, 0, -2, -2, -4, 6, -6, 4, -4]
    elif qm == 31:
        want = [31, 0, 2, 2, 4, 0, -2, -2, -4, 30, -30, 4, -4]
    else:
        want = [127, 0, 2, 2, 4, 0, -2, -2, -4, 126, -126, 4, -4]
    S0 = np.zeros((1, 128, 128), np.float32)
    codes = np.zeros((1, 128, 128), np.int8)
    for r in range(3):
        S0[0, r, :len(base)] = np.float32(2.0 ** (r - 1)) * np.asarray(base, np.float32)
        codes[0, r, :len(want)] = want
    return S0, codes


def selection_ties():
    """States whose compensator selection (C = 4) meets exact score ties, with the ids
    the tie rule gives (reading R5: largest squared length, ties to the smallest id, rows
    0..127 before columns 128..255), worked out by hand:
    - a constant state: every line has the same length; taking row 0 shortens every
      column by one entry, so rows 1, 2, 3 follow;
    - row 5 and column 9 all ones: the row wins the tie; the column (127 ones left)
      beats the rows' single entries; then the residual is zero, every score ties at 0
      and id 0 wins twice (a zero line);
    - columns 20 and 10 all ones: the smaller column wins the tie, then the other;
      then zero lines at id 0."""
    cases = []
    S = np.full((1, 128, 128), 0.5, np.float32)
    cases.append((S, [0, 1, 2, 3]))
    S = np.zeros((1, 128, 128), np.float32)
    S[0, 5, :] = 1.0
    S[0, :, 9] = 1.0
    cases.append((S, [5, 128 + 9, 0, 0]))
    S = np.zeros((1, 128, 128), np.float32)
    S[0, :, 20] = 1.0
    S[0, :, 10] = 1.0
    cases.append((S, [128 + 10, 128 + 20, 0, 0]))
    return cases
