"""How the GPU tests compare a GPU result with the oracle's.  Holds none of
the method's arithmetic: norms of differences, counts and bookkeeping.

The bar (the same in every parity test):
  * output: relative L2 over the compared rows <= TOL; over every single row
    <= ROW_TOL, and at most MAX_ROWS_ABOVE_TOL of the rows (at least five)
    above TOL, so that neither a few corrupted rows nor many slightly wrong
    ones can hide in a large sample.  A single row may legitimately reach a
    few percent: where the FP32 scores of the GPU and the FP64 scores of the
    oracle round a block's largest weight code to different sides of a scale
    boundary, that block of P sits on a grid twice as fine or coarse, which
    moves each of its weights by up to half a step of the coarser grid (6 %
    for E4M3), and a row whose weight sits mostly in that block moves about
    as much.  Measured on GB300 over all the parity tests: the largest row
    error 4.9e-2 (rows dominated by one key); rows above TOL 0.26-1.05 % of
    a sample of 1526 rows (MXFP6, ten seeds of B=1 H=16 S=8192, mean 0.67 %;
    MXFP8 at most 0.4 %), so the count bound sits at twice the largest; a
    corrupted value gives errors of order one.  Rows
    whose gate decision legitimately differs -- a near-tie -- are left out
    of the per-row bounds, see below;
  * rollback decisions: identical per (row, tile) except near-ties, tiles
    whose gate margin |max s - m - theta| is below NEAR_TIE in score units,
    where the GPU's FP32 accumulation order may decide the other way.  The
    near-ties are counted; those decided differently -- the only decisions
    left out of the identity -- may be at most MAX_NEAR_TIE_FRAC of the gate
    decisions (tiles after the first of the compared rows).  (Near-ties
    themselves can be common: with four-bit operands and theta = 0 the
    scores sit on a coarse grid and a tile's maximum often equals the
    reference exactly; both sides then decide alike.)
Each comparison logs what it observed (one line; also appended to the file
named by FSA_PARITY_LOG when that is set), so the margin to the bar is on
record."""
from __future__ import annotations

import os

import numpy as np

TOL = 5e-3
ROW_TOL = 0.1
MAX_ROWS_ABOVE_TOL = 0.02
NEAR_TIE = 1e-4
MAX_NEAR_TIE_FRAC = 1e-3


def log(label: str, **vals) -> None:
    parts = []
    for k, v in vals.items():
        parts.append(f"{k}={v:.3e}" if isinstance(v, float) else f"{k}={v}")
    line = f"[parity] {label}: " + " ".join(parts)
    print(line)
    path = os.environ.get("FSA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")


def row_errors(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Relative L2 error of every row: |got_i - ref_i| / |ref_i|."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref, axis=1)
    num = np.linalg.norm(got - ref, axis=1)
    return num / np.where(den > 0, den, 1.0)


def check_out(label: str, got, ref, skip_rows=None, tol: float = TOL, row_tol: float = ROW_TOL):
    """Assert the output bar; returns (global relative L2, largest row error)."""
    got = np.asarray(got, np.float64).reshape(np.shape(ref))
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got)), f"{label}: non-finite output"
    g = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    re = row_errors(got, ref)
    keep = np.ones(len(re), bool)
    if skip_rows is not None:
        keep[np.asarray(skip_rows, np.int64)] = False
    worst = float(re[keep].max()) if keep.any() else 0.0
    above = int((re[keep] > tol).sum())
    log(label, rel_l2=g, max_row_rel_l2=worst, rows_above_tol=above, rows=int(len(re)),
        rows_skipped=int((~keep).sum()))
    assert g <= tol, f"{label}: relative L2 {g:.3e} > {tol:.0e}"
    assert worst <= row_tol, f"{label}: a row's relative L2 {worst:.3e} > {row_tol:.0e}"
    assert above <= max(5, MAX_ROWS_ABOVE_TOL * keep.sum()), \
        f"{label}: {above} of {int(keep.sum())} rows above {tol:.0e}"
    return g, worst


def check_bits(label: str, bits, ref_bits, margins):
    """Assert the rollback-decision bar.  bits / ref_bits / margins are
    [rows][tiles]; margins hold max s - m - theta (NaN where no decision
    exists: tile 0, tiles past the keys).  Returns the indices of the rows
    with a near-tie decided differently (to leave out of the per-row
    output bound) and the number of near-ties."""
    bits = np.asarray(bits)
    ref_bits = np.asarray(ref_bits)
    margins = np.asarray(margins, np.float64)
    assert set(np.unique(bits)) <= {0, 1}, f"{label}: rollback bytes other than 0/1"
    decided = ~np.isnan(margins)
    near = decided & (np.abs(np.nan_to_num(margins, nan=1.0)) < NEAR_TIE)
    n_dec, n_near = int(decided.sum()), int(near.sum())
    differ = bits != ref_bits
    bad = differ & ~near
    log(label, decisions=n_dec, firings=int(ref_bits.sum()), near_ties=n_near,
        near_ties_differing=int((differ & near).sum()), mismatches=int(bad.sum()))
    assert not bad.any(), f"{label}: {int(bad.sum())} rollback decisions differ outside near-ties"
    n_flip = int((differ & near).sum())
    assert n_flip <= max(1, MAX_NEAR_TIE_FRAC * n_dec), \
        f"{label}: {n_flip} near-ties of {n_dec} decisions decided differently"
    return np.nonzero((differ & near).any(axis=1))[0], n_near
