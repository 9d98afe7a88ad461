"""bench.py's per-launch algorithmic bytes and flops (the roofline numerators),
counted from first principles on small CPU cases: every byte of x and out, the
weights, and per request the state columns read (S with history) and written
(S, or cap for a speculative step), at the pool's own element size."""
import pytest
import torch

import bench
from state_cached_causal_gb300 import synth

CPU = torch.device("cpu")


def _case(dtype, **kw):
    return synth.depthwise_case(77, CPU, C=64, width=4, dilation=3, act=1, dtype=dtype,
                                w_std=0.1, bias_std=0.02, **kw)


@pytest.mark.parametrize("pool_dtype", [None, torch.float32])
def test_varlen_and_update_bytes(pool_dtype):
    case = _case(torch.bfloat16, lens=[1, 5, 0, 20], spec_requests=3, n_spec=3,
                 padding_every=3)
    if pool_dtype is not None:
        case.pool = torch.zeros(case.pool.shape, dtype=pool_dtype)
    es = case.pool.element_size()
    fwd, upd = bench.depthwise_calls("t", case, None)
    S, C, cap = 9, 64, case.pool.shape[2]
    T = 26
    # sequences: slots of the varlen part (every 3rd is padding); history
    # columns are read only with has_init and a real slot
    reads = sum(1 for s in range(4) if int(case.state_idx[s]) >= 0 and int(case.has_init[s]))
    writes = sum(1 for s in range(4) if int(case.state_idx[s]) >= 0)
    weights = C * 4 * 2 + C * 2
    assert fwd.bytes == 2 * T * C * 2 + weights + C * es * S * (reads + writes)
    assert fwd.units == T * C
    R, q = 3, 4
    assert upd.bytes == 2 * R * q * C * 2 + weights + R * C * es * (S + cap)
    assert upd.units == R * q * C


def test_cca_bytes_and_flops():
    cc = synth.cca_case(78, CPU, lens=[1, 1, 9], decode_prefix=2, Hq=1, Hkv=1)
    (call,) = bench.cca_calls("z", cc, None)
    T, Cqk, Dv, n = 11, 256, 64, 2
    valid = sum(1 for s in cc.state_idx.tolist() if s >= 0)
    reads = sum(1 for s, h in zip(cc.state_idx.tolist(), cc.has_init.tolist()) if s >= 0 and h)
    weights = (Cqk * 2 + Cqk + Cqk * 128 * 2 + Cqk) * 2
    assert call.bytes == (2 * T * Cqk * 2 + 2 * T * Dv * 2 + weights + Dv * 2
                          + (reads + valid) * (n * Cqk * 2 + Dv * 2))
    # grouped stage: 2 flops per multiply-add, 128 inputs x 2 taps per output;
    # depthwise stage: 2 taps over T + 1 positions
    assert call.flops == 2.0 * T * Cqk * 128 * 2 + 2.0 * (T + 1) * Cqk * 2
