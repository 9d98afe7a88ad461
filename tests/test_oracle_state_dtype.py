"""Pins for the oracle's state storage type (a conv-state pool whose dtype
differs from the activations', the mamba_cache_dtype of the
"Qwen4ExpPLELayer" get_state_dtype), against things other than the oracle's
own conversion code:

* The Zaya page's _mix_with_state fixes the rule: the history it reads is
  conv_state[slot].to(qk.dtype) and what it writes back is
  new_history.to(conv_state.dtype). So a call on a pool of the other type must
  equal the same call on a pool of the activations' type holding torch's
  conversion of it, with torch's conversion of the new state written back --
  on the columns the call rewrites, while every other element keeps its bits.
* fp32 activations with a bf16 pool: the widened pool is exact, so the whole
  pool after the call is torch's round-to-nearest-even of the same-type
  result.
* A wider pool holding values of the narrower type gives the same-type result
  exactly.

Conversions here are torch's (Tensor.to); the oracle's are its own C code.
No CUDA is involved.
"""
import numpy as np
import pytest
import torch

import oracle
from state_cached_causal_gb300 import synth
from tests._util import pool_np, to_np

CPU = torch.device("cpu")
OTHER = {torch.float32: torch.bfloat16, torch.bfloat16: torch.float32}


def _other_pool(pool, dtype, seed, representable=False):
    """A pool of `dtype` with pool's shape and layout: random values, or (for
    representable) pool's own values converted."""
    if representable or dtype == torch.bfloat16:
        return pool.to(dtype)           # keeps the strides of the view
    g = synth.generator(seed, CPU)
    new = torch.randn(pool.shape, generator=g).to(dtype)
    out = torch.empty_strided(pool.shape, pool.stride(), dtype=dtype)
    out.copy_(new)
    return out


def _bits(t):
    t = t.detach().cpu()
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _check_state(after, before, ref_after, written):
    """`after` (the other-type pool after the call) equals torch's conversion of
    the same-type result where `written`, and keeps its bits elsewhere."""
    want = torch.where(written, ref_after.to(after.dtype), before)
    assert torch.equal(_bits(after), _bits(want))


def _written(shape, slots, ncols):
    m = torch.zeros(shape, dtype=torch.bool)
    for s in slots:
        if s >= 0:
            m[s, :, :ncols] = True
    return m


LAYOUTS = ["DS", "SD"]


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("representable", [False, True])
def test_fwd_varlen_state_type(layout, act, representable):
    if representable and act == torch.float32:
        pytest.skip("a bf16 pool always holds values of fp32 activations")
    case = synth.depthwise_case(1201, CPU, lens=[5, 1, 0, 2, 9, 1], C=16, width=4, dilation=2,
                                act=1, dtype=act, w_std=0.5, bias_std=0.1, layout=layout,
                                padding_every=5, cap=9)
    sd = OTHER[act]
    pool_o = _other_pool(case.pool, sd, 7, representable)
    pool_ref = pool_o.to(act)                      # what the call reads, in torch
    before = pool_o.clone()
    x = to_np(case.x)
    out_m, out_r = np.zeros_like(x), np.zeros_like(x)
    pm, pr = pool_np(pool_o), pool_np(pool_ref)
    args = (to_np(case.state_idx), to_np(case.cu_seqlens), to_np(case.has_init), 4, 2, 1)
    oracle.cconv_fwd_varlen(x, to_np(case.w), to_np(case.bias), pm, *args, out_m)
    oracle.cconv_fwd_varlen(x, to_np(case.w), to_np(case.bias), pr, *args, out_r)
    assert np.array_equal(out_m, out_r)
    written = _written(pool_o.shape, case.state_idx.tolist(), 6)   # S = 6 of cap 9
    _check_state(pool_o, before, pool_ref, written)
    if representable:
        assert torch.equal(pool_o, pool_ref.to(sd))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("n_spec", [0, 3])
def test_update_state_type(layout, act, n_spec):
    case = synth.depthwise_case(1202, CPU, lens=[], C=16, width=4, dilation=3, act=1,
                                dtype=act, w_std=0.3, layout=layout, spec_requests=6,
                                n_spec=n_spec, cap=9 + n_spec + 1)
    sd = OTHER[act]
    pool_o = _other_pool(case.pool, sd, 8)
    pool_ref = pool_o.to(act)
    before = pool_o.clone()
    x = to_np(case.x_spec)
    out_m, out_r = np.zeros_like(x), np.zeros_like(x)
    sidx = case.spec_state_idx.clone()
    sidx[2] = -1                                   # a padding row
    hi = torch.tensor([1, 0, 1, 1, 0, 1], dtype=torch.uint8)
    na = to_np(case.num_accepted) if n_spec else None
    for pool, out in ((pool_o, out_m), (pool_ref, out_r)):
        oracle.cconv_update(x, pool_np(pool), to_np(case.w), None, to_np(sidx), n_spec, na,
                            to_np(hi), 4, 3, 1, out)
    assert np.array_equal(out_m, out_r)
    ncols = case.pool.shape[2] if n_spec else 9
    _check_state(pool_o, before, pool_ref, _written(pool_o.shape, sidx.tolist(), ncols))


@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
def test_fused_fwd_state_type(act):
    case = synth.depthwise_case(1203, CPU, lens=[4, 1, 7, 0, 2], C=16, width=3, dilation=2,
                                act=1, dtype=act, w_std=0.5, layout="DS")
    sd = OTHER[act]
    pool_o = _other_pool(case.pool, sd, 9)
    pool_ref = pool_o.to(act)
    before = pool_o.clone()
    x = to_np(case.x)
    g = torch.Generator().manual_seed(5)
    res0 = to_np(torch.randn(x.shape, generator=g).to(act))
    outer = to_np(torch.randn(x.shape, generator=g).to(act))
    perm = np.random.default_rng(1).permutation(x.shape[0]).astype(np.int32)
    res_m, res_r = res0.copy(), res0.copy()
    args = (to_np(case.state_idx), to_np(case.cu_seqlens), to_np(case.has_init), 3, 2, 1)
    oracle.cconv_fwd_varlen_fused(x, to_np(case.w), None, pool_np(pool_o), *args, res_m, outer,
                                  perm)
    oracle.cconv_fwd_varlen_fused(x, to_np(case.w), None, pool_np(pool_ref), *args, res_r, outer,
                                  perm)
    assert np.array_equal(res_m, res_r)
    _check_state(pool_o, before, pool_ref, _written(pool_o.shape, case.state_idx.tolist(), 4))


@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16])
def test_checkpoint_export_converts_to_the_pool_type(act):
    case = synth.depthwise_case(1204, CPU, lens=[12, 9], C=16, width=4, dilation=3, act=1,
                                dtype=act, w_std=0.5, cap=10, num_slots=6)
    sd = OTHER[act]
    pool_o = _other_pool(case.pool, sd, 10)
    before = pool_o.clone()
    x = to_np(case.x)
    oracle.cconv_checkpoint_export(x, pool_np(pool_o), np.array([0, 1], np.int32),
                                   np.array([12, 9], np.int32), np.array([4, 5], np.int32),
                                   to_np(case.cu_seqlens), 4, 3)
    want = before.clone()
    want[4, :, :9] = case.x[3:12].T.to(sd)         # offset 12 of request 0: rows 3..11
    want[5, :, :9] = case.x[12:21].T.to(sd)        # offset 9 of request 1: rows 12..20
    assert torch.equal(_bits(pool_o), _bits(want))


def test_cca_fp32_state():
    case = synth.cca_case(1205, CPU, lens=[1, 1, 3, 0, 0, 5], decode_prefix=2, Hq=2, Hkv=1,
                          head_dim=128, has_init="bernoulli")
    case.has_init[3], case.has_init[4] = 1, 0      # empty requests with and without history
    pool32 = _other_pool(case.pool, torch.float32, 11)
    g = torch.Generator().manual_seed(12)
    dst32 = torch.randn(case.delayed_state.shape, generator=g)
    pool_ref, dst_ref = pool32.to(torch.bfloat16), dst32.to(torch.bfloat16)
    before, dbefore = pool32.clone(), dst32.clone()
    T = case.qk.shape[0]
    outs = []
    for pool, dst in ((pool32, dst32), (pool_ref, dst_ref)):
        out_qk = np.zeros((T, case.Cqk), np.uint16)
        out_dp = np.zeros((T, case.Dv), np.uint16)
        oracle.cca_qk_conv(to_np(case.qk), to_np(case.w_dw), to_np(case.b_dw), to_np(case.w_gr),
                           to_np(case.b_gr), case.groups, case.t0, case.t1, to_np(case.delayed),
                           to_np(case.delayed_init), pool_np(pool), to_np(dst),
                           to_np(case.state_idx), to_np(case.cu_seqlens), to_np(case.has_init),
                           out_qk, out_dp)
        outs.append((out_qk, out_dp))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    sidx = case.state_idx.tolist()
    _check_state(pool32, before, pool_ref, _written(pool32.shape, sidx, case.meta["n"]))
    lens = case.meta["lens"]
    dwritten = torch.zeros(dst32.shape, dtype=torch.bool)
    for s, slot in enumerate(sidx):
        if slot >= 0 and (lens[s] > 0 or not case.has_init[s]):
            dwritten[slot] = True
    want = torch.where(dwritten, dst_ref.float(), dbefore)
    assert torch.equal(dst32, want)
    # the empty request with history keeps its fp32 delayed state bit for bit
    assert torch.equal(dst32[sidx[3]], dbefore[sidx[3]])
