"""Planted mistakes in the channel-reader oracle: each mutant must make at least one pin of
tests/test_reader_pins.py fail (the pins would catch that kind of slip)."""
import numpy as np
import pytest

import oracle.reader as R
import test_reader_pins as pins

PINS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


def _fails(monkeypatch, name, fn):
    monkeypatch.setattr(R, name, fn)
    failed = 0
    for pin in PINS:
        try:
            pin()
        except Exception:  # an assertion, or a shape error the slip causes
            failed += 1
    return failed


_orig_rotate, _orig_ternary, _orig_scan = R.rotate, R.ternary_block, R.scan_mask
_orig_est = R.sketch_estimate


def _smallest_basis(wd, r):
    D = np.asarray(wd, np.float64).reshape(-1, np.asarray(wd).shape[-1])
    return np.linalg.eigh(D.T @ D)[1][:, :r]


MUTANTS = {
    "rotation without the signs": ("rotate", lambda x, s: _orig_rotate(x, np.ones_like(s))),
    "rotation not normalised": ("rotate", lambda x, s: _orig_rotate(x, s) * np.sqrt(2.0)),
    "ternary threshold 0.5": ("ternary_block", lambda r: (
        np.where(np.abs(r) > 0.5 * np.mean(np.abs(r)), np.sign(r), 0).astype(np.int8),
        _orig_ternary(r)[1])),
    "ternary scale over all coordinates": ("ternary_block", lambda r: (
        _orig_ternary(r)[0], float(np.mean(np.abs(r))))),
    "scan keeps the smallest": ("scan_mask", lambda xr, n: _orig_scan(-1.0 / (np.abs(xr) + 1e-9), n)),
    "scan one coordinate short": ("scan_mask", lambda xr, n: _orig_scan(xr, max(n - 1, 0))),
    "activation without the gate": ("silu", lambda z: np.asarray(z, np.float64)),
    "basis from the smallest eigenvalues": ("down_basis", lambda wd, r: _smallest_basis(wd, r)),
    "sketch ignores the scales": ("sketch_estimate", lambda c, s, xr, m: _orig_est(c, np.ones_like(s), xr, m)),
}


@pytest.mark.parametrize("label", sorted(MUTANTS))
def test_mutant_is_caught(monkeypatch, label):
    name, fn = MUTANTS[label]
    assert _fails(monkeypatch, name, fn) >= 1, label
