"""Full-size parity helpers: the oracle over every channel (depthwise) or every
group (CCA) of a launch, run as independent channel blocks on all host cores.

Each depthwise channel, and each CCA group, is an independent computation, so
the oracle runs in place on disjoint blocks of the same full-size host arrays
(its C calls release the GIL), and the comparison of each block happens in
its worker, a few thousand rows at a time, to bound the temporaries.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from oracle.torch_io import np_to_f64

THREADS = max(1, os.cpu_count() or 1)


def pmap(fn, items):
    """fn over items on all host cores; returns the results in order."""
    with ThreadPoolExecutor(THREADS) as ex:
        return list(ex.map(fn, items))


def channel_blocks(C, unit=8, per_thread=2):
    """Contiguous channel slices (multiples of `unit`) covering [0, C)."""
    n = max(1, min(THREADS * per_thread, C // unit))
    edges = [(k * (C // unit) // n) * unit for k in range(n + 1)]
    edges[-1] = C
    return [slice(edges[k], edges[k + 1]) for k in range(n) if edges[k + 1] > edges[k]]


def count_out_of_tol(got, want, bf16, rows=4096):
    """Elements of got (storage bits or fp32) outside the tolerance of the parity
    tests against want: |err| <= 2e-2 + 2e-2*|ref| (bf16), max|err| <= 1e-5 (fp32).
    Returns (count, max |err|)."""
    bad, worst = 0, 0.0
    for r0 in range(0, got.shape[0], rows):
        g = np_to_f64(got[r0:r0 + rows])
        w = np_to_f64(want[r0:r0 + rows])
        err = np.abs(g - w)
        if err.size:
            worst = max(worst, float(err.max()))
        bad += int((err > (2e-2 + 2e-2 * np.abs(w)) if bf16 else err > 1e-5).sum())
    return bad, worst


def assert_blocks(results, what):
    """results: list of (block, bad count, max err, state mismatches) from workers."""
    bad = sum(r[1] for r in results)
    worst = max((r[2] for r in results), default=0.0)
    neq = sum(r[3] for r in results)
    assert bad == 0, f"{what}: {bad} elements out of tolerance (max |err| {worst:.3g})"
    assert neq == 0, f"{what}: {neq} state elements differ"
