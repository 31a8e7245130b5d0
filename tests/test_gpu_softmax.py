"""fattn_softmax_rows (the online normaliser on its own) against the fp64 oracle.

Shapes: a single value; rows whose length is not a multiple of four (scalar
path); rows staged in shared memory; rows longer than the staging buffer (read
twice).  Values span large magnitudes and include -inf entries and an all -inf
row.  Bar: |y - y_ref| <= 1e-5 y_ref + 1e-9 and |lse - lse_ref| <= 1e-6 max(1,
|lse_ref|) + 1e-5 (fp32 arithmetic, exp2 with ~2^-22 relative error).
"""
import numpy as np
import pytest
import torch

import oracle
from online_softmax_08_gb300 import fattn

pytestmark = pytest.mark.gpu


def _rows(rows, cols, seed, scale=30.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((rows, cols), generator=g, dtype=torch.float32) * scale
    if cols > 3:
        x[0, ::3] = -float("inf")        # masked entries
    if rows > 2:
        x[2, :] = -float("inf")          # nothing visible in this row
    return x


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 7), (64, 4096), (9, 1000), (5, 50000),
                                       (2, 60001), (300, 257)])
def test_softmax_rows_matches_oracle(rows, cols):
    x = _rows(rows, cols, seed=rows * 7919 + cols)
    dev = torch.device("cuda:0")
    y, lse = fattn.softmax_rows(x.to(dev), with_lse=True)
    torch.cuda.synchronize()
    y_ref, lse_ref = oracle.softmax_rows(x.double().numpy())
    yg, lg = y.double().cpu().numpy(), lse.double().cpu().numpy()
    assert np.all(np.abs(yg - y_ref) <= 1e-5 * y_ref + 1e-9)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    assert np.all(np.abs(lg[fin] - lse_ref[fin]) <= 1e-6 * np.maximum(1.0, np.abs(lse_ref[fin])) + 1e-5)


def test_softmax_rows_in_place():
    x = _rows(4, 2048, seed=5)
    dev = torch.device("cuda:0")
    xd = x.to(dev)
    fattn.softmax_rows(xd, out=xd)
    torch.cuda.synchronize()
    y_ref, _ = oracle.softmax_rows(x.double().numpy())
    assert np.all(np.abs(xd.double().cpu().numpy() - y_ref) <= 1e-5 * y_ref + 1e-9)


def test_softmax_bench_workload_sampled():
    """The benchmark's workload (4096 rows of 32768 fp32 values), sampled rows
    against the oracle."""
    from online_softmax_08_gb300.inputs import SOFTMAX_WORKLOADS, make_softmax_input
    w = SOFTMAX_WORKLOADS["softmax_rows4096_cols32768_f32"]
    x = make_softmax_input(w["rows"], w["cols"], w["seed"])
    dev = torch.device("cuda:0")
    y, lse = fattn.softmax_rows(x.to(dev), with_lse=True)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, 1, 151, 152, w["rows"] - 1],
                                     np.random.default_rng(w["seed"]).integers(0, w["rows"], 11)]))
    y_ref, lse_ref = oracle.softmax_rows(x[rows].double().numpy())
    yg = y[rows].double().cpu().numpy()
    assert np.all(np.abs(yg - y_ref) <= 1e-5 * y_ref + 1e-9)
    assert np.all(np.abs(lse[rows].double().cpu().numpy() - lse_ref) <= 1e-6 * np.abs(lse_ref) + 1e-5)
