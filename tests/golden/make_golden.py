"""Writes the stored fixtures of this folder. Run from the repository root:

    python tests/golden/make_golden.py

The pages print no worked numeric example, so every stored value here is an
input drawn by the seeded generator (state_cached_causal_gb300.synth) or an
output of the oracle (oracle/) on it; nothing comes from the CUDA library.
Inputs are stored with the expected values, as raw bits in hex, so that the
fixtures do not depend on the random-number stream of a torch version.
"""
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle.torch_io import pool_np, to_np  # noqa: E402
from state_cached_causal_gb300 import synth  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def hexbits(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return {"dtype": "f32", "shape": list(a.shape), "hex": a.view(np.uint32).tobytes().hex()}
    if a.dtype == np.uint16:
        return {"dtype": "bf16", "shape": list(a.shape), "hex": a.tobytes().hex()}
    if a.dtype in (np.int32, np.uint8):
        return {"dtype": str(a.dtype), "shape": list(a.shape), "values": a.ravel().tolist()}
    raise TypeError(a.dtype)


def single_prefill():
    """1 sequence x 32 tokens x 64 channels, fp32, width 4, dilation 1, no bias, no
    activation, w ~ N(0, 0.25); its slot is zero. Run with has_init = 0 and with
    has_init = 1: the zero slot and the missing history must give the same bits."""
    fx = {"what": "one prefill on a zero slot, both has_init values",
          "passages": ["GDN page, _spec_aware_nonspec (prefill conv with has_initial_state)",
                       "Zaya page, _mix_with_state (history masked by has_history)"]}
    case = synth.single_prefill(torch.device("cpu"), has_init="none")
    x, w = to_np(case.x), to_np(case.w)
    pool0 = pool_np(case.pool).copy()
    fx["inputs"] = {"x": hexbits(x), "w": hexbits(w), "pool": hexbits(pool0),
                    "state_idx": hexbits(to_np(case.state_idx)),
                    "cu_seqlens": hexbits(to_np(case.cu_seqlens))}
    fx["width"], fx["dilation"], fx["act"] = case.width, case.dilation, case.act
    res = []
    for h in (0, 1):
        pool = pool0.copy()
        out = np.zeros_like(x)
        oracle.cconv_fwd_varlen(x, w, None, pool, to_np(case.state_idx),
                                to_np(case.cu_seqlens), np.array([h], np.uint8), case.width,
                                case.dilation, case.act, out)
        res.append((out, pool))
    assert all(np.array_equal(a.view(np.uint32), b.view(np.uint32)) for a, b in zip(*res))
    fx["expected"] = {"out": hexbits(res[0][0]), "pool": hexbits(res[0][1])}
    return fx


def spec_step():
    """2 speculative requests x (1+3) tokens x 16 channels, bf16, width 4,
    dilation 3 (S = 9, cap = 12), SiLU, num_accepted 1 and 4."""
    fx = {"what": "one speculative-decode step on a rolling buffer",
          "passages": ["GDN page, _spec_forward (prior at num_accepted - 1, kept columns, "
                       "new tokens)", "PLE page, _short_conv_dilated_dispatch (spec branch)"]}
    case = synth.depthwise_case(1100, torch.device("cpu"), lens=[], C=16, width=4, dilation=3,
                                act=1, dtype=torch.bfloat16, w_std=0.3, spec_requests=2,
                                n_spec=3, num_slots=3)
    na = np.array([1, 4], np.int32)
    x, w = to_np(case.x_spec), to_np(case.w)
    pool = pool_np(case.pool).copy()
    fx["inputs"] = {"x": hexbits(x), "w": hexbits(w), "pool": hexbits(pool),
                    "state_idx": hexbits(to_np(case.spec_state_idx)),
                    "num_accepted": hexbits(na)}
    fx["width"], fx["dilation"], fx["act"], fx["n_spec"] = 4, 3, 1, 3
    out = np.zeros_like(x)
    oracle.cconv_update(x, pool, w, None, to_np(case.spec_state_idx), 3, na, None, 4, 3, 1, out)
    fx["expected"] = {"out": hexbits(out), "pool": hexbits(pool)}
    return fx


if __name__ == "__main__":
    for name, fn in (("single_prefill", single_prefill), ("spec_step", spec_step)):
        with open(os.path.join(HERE, f"{name}.json"), "w") as f:
            json.dump(fn(), f, indent=0)
            f.write("\n")
        print("wrote", name)
