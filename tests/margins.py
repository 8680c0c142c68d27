"""Observed parity margins.

Every GPU-against-oracle comparison goes through `check`, which records the
largest error it saw beside its tolerance and then asserts. The session's
terminal summary (conftest.py) prints the table, so a run shows how close each
case came to its bound, not only that it passed.
"""
import os

OBSERVED = []


def check(err, tol, what=""):
    """Record `err` (a max abs error) against `tol` for the running test, then
    assert err <= tol."""
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    OBSERVED.append((test, what, float(err), float(tol)))
    assert err <= tol, f"{what or 'max abs error'}: {err:.4g} > {tol:.4g}"
