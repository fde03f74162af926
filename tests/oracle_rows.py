"""The oracle's mat-vec with its rows split over host threads, for full-size parity checks.

The oracle is C called through ctypes, which releases the interpreter lock, so row slices run in
parallel; each slice is an ordinary oracle call, so the result is the same as one call over all
rows."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle as O


def oracle_rows_threaded(ofmt, W, oqs, od, obs, order, threads=None):
    rows = W.shape[0]
    n = max(1, min(threads or os.cpu_count() or 1, rows // 64 or 1))
    cuts = [rows * i // n for i in range(n + 1)]
    with ThreadPoolExecutor(n) as ex:
        parts = list(ex.map(lambda i: O.qmatvec(ofmt, W[cuts[i]:cuts[i + 1]], oqs, od, obs, order), range(n)))
    return np.concatenate(parts, axis=1)
