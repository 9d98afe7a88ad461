"""Stored fixtures (tests/golden/, written by tests/golden/make_golden.py from the
seeded generator and the oracle): the oracle must keep reproducing them bit for
bit, and -- on a GPU -- the library must match them (outputs within the
tolerance of their type, state bit for bit).

single_prefill: the zero slot read with has_init = 1 and the missing history of
has_init = 0 give identical outputs and state (GDN page, _spec_aware_nonspec;
Zaya page, _mix_with_state masks the history by has_history).
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    with open(os.path.join(HERE, f"{name}.json")) as f:
        return json.load(f)


def arr(d):
    if "values" in d:
        return np.array(d["values"], dtype=d["dtype"]).reshape(d["shape"])
    raw = bytes.fromhex(d["hex"])
    if d["dtype"] == "f32":
        return np.frombuffer(raw, dtype=np.uint32).view(np.float32).reshape(d["shape"]).copy()
    return np.frombuffer(raw, dtype=np.uint16).reshape(d["shape"]).copy()


def bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


def test_single_prefill_fixture_and_has_init_agreement():
    fx = load("single_prefill")
    i = {k: arr(v) for k, v in fx["inputs"].items()}
    assert not i["pool"].any(), "the slot of this fixture is zero"
    got = {}
    for h in (0, 1):
        pool = i["pool"].copy()
        out = np.zeros_like(i["x"])
        oracle.cconv_fwd_varlen(i["x"], i["w"], None, pool, i["state_idx"], i["cu_seqlens"],
                                np.array([h], np.uint8), fx["width"], fx["dilation"], fx["act"],
                                out)
        want = fx["expected"]           # one stored result for both has_init values
        assert np.array_equal(bits(out), bits(arr(want["out"])))
        assert np.array_equal(bits(pool), bits(arr(want["pool"])))
        got[h] = (out, pool)
    assert np.array_equal(bits(got[0][0]), bits(got[1][0]))
    assert np.array_equal(bits(got[0][1]), bits(got[1][1]))
    # the new state is the last S = 3 inputs
    assert np.array_equal(got[0][1][0].T, i["x"][-3:])


def test_spec_step_fixture():
    fx = load("spec_step")
    i = {k: arr(v) for k, v in fx["inputs"].items()}
    pool = i["pool"].copy()
    out = np.zeros_like(i["x"])
    oracle.cconv_update(i["x"], pool, i["w"], None, i["state_idx"], fx["n_spec"],
                        i["num_accepted"], None, fx["width"], fx["dilation"], fx["act"], out)
    assert np.array_equal(out, arr(fx["expected"]["out"]))
    assert np.array_equal(pool, arr(fx["expected"]["pool"]))
    # the last q = 4 columns of every rewritten slot are the new tokens
    for r, slot in enumerate(i["state_idx"]):
        assert np.array_equal(pool[slot, :, -4:].T, i["x"][4 * r:4 * r + 4])


def _dev(a, dev):
    t = torch.from_numpy(a.copy())
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.to(dev)


def _host(t):
    t = t.cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


@pytest.mark.gpu
def test_library_matches_the_fixtures():
    from state_cached_causal_gb300 import ops
    from tests.test_parity_depthwise import assert_out_close
    dev = torch.device("cuda")
    fx = load("single_prefill")
    i = {k: arr(v) for k, v in fx["inputs"].items()}
    for h in (0, 1):
        pool = _dev(i["pool"], dev)
        out = torch.zeros(i["x"].shape, device=dev)
        ops.cconv_fwd_varlen(_dev(i["x"], dev), _dev(i["w"], dev), None, pool,
                             _dev(i["state_idx"], dev), _dev(i["cu_seqlens"], dev),
                             torch.tensor([h], dtype=torch.uint8, device=dev), fx["width"],
                             fx["dilation"], fx["act"], out)
        torch.cuda.synchronize()
        want = fx["expected"]
        assert_out_close(_host(out), arr(want["out"]), torch.float32)
        assert np.array_equal(bits(_host(pool)), bits(arr(want["pool"])))
    fx = load("spec_step")
    i = {k: arr(v) for k, v in fx["inputs"].items()}
    pool = _dev(i["pool"], dev)
    x = _dev(i["x"], dev)
    out = torch.zeros_like(x)
    ops.cconv_update(x, pool, _dev(i["w"], dev), None, _dev(i["state_idx"], dev), fx["n_spec"],
                     _dev(i["num_accepted"], dev), None, fx["width"], fx["dilation"], fx["act"],
                     out)
    torch.cuda.synchronize()
    assert_out_close(_host(out), arr(fx["expected"]["out"]), torch.bfloat16)
    assert np.array_equal(_host(pool), arr(fx["expected"]["pool"]))
