"""GPU parity for conv-state pools of another storage type than the activations
(fp32 pools under bf16 activations, the usual mamba_cache_dtype, and bf16
pools under fp32 activations), every entry point through the C ABI vs the
oracle: outputs within the tolerance of the activations' type, the pool and
the delayed state bit for bit.

Pools hold random values of their own type (an fp32 pool is not limited to
bf16 values), so the conversions on both read and write are exercised.
"""
import numpy as np
import pytest
import torch

import oracle
from state_cached_causal_gb300 import ops, synth
from tests._util import pool_np, to_np
from tests.test_parity_cca import LENS, oracle_cca
from tests.test_parity_cca import check as check_cca
from tests.test_parity_depthwise import (assert_bits_equal, assert_out_close, check_fwd,
                                         check_upd, new_err)
from tests.test_parity_fused import oracle_fwd_fused, physical, rand_rows, run_fwd_fused

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
MIX = [(torch.bfloat16, torch.float32), (torch.float32, torch.bfloat16)]


def other_pool(shape, dtype, layout, seed):
    """A [slot, channel, column] pool view of `dtype` with random values:
    channel-first, column-first, or a slice of a wider channel-first buffer."""
    slots, C, cap = shape
    g = torch.Generator(device=DEV).manual_seed(seed)
    if layout == "DS":
        return torch.randn(slots, C, cap, generator=g, device=DEV).to(dtype)
    if layout == "SD":
        return torch.randn(slots, cap, C, generator=g, device=DEV).to(dtype).transpose(1, 2)
    return torch.randn(slots, C, cap + 3, generator=g, device=DEV).to(dtype)[:, :, 3:]


def _C(act):
    return 1040 if act == torch.bfloat16 else 520


@pytest.mark.parametrize("act,sd", MIX)
@pytest.mark.parametrize("layout", ["DS", "SD", "wide"])
@pytest.mark.parametrize("W,D", [(4, 1), (4, 3), (2, 2), (3, 4), (8, 8), (5, 3)])
def test_fwd_varlen_state_type(act, sd, layout, W, D):
    S = (W - 1) * D
    lens = [1, 1, 1, 0, 2, max(1, S - 1), S, S + 1, 63, 64, 65, 129, 200, 7]
    case = synth.depthwise_case(1300 + 10 * W + D, DEV, lens=lens, C=_C(act), width=W,
                                dilation=D, act=1, dtype=act, w_std=0.5, bias_std=0.1,
                                decode_prefix=3, padding_every=5, cap=S + 2)
    case.pool = other_pool(case.pool.shape, sd, layout, 1301 + W + D)
    check_fwd(case)


@pytest.mark.parametrize("act,sd", MIX)
@pytest.mark.parametrize("layout", ["DS", "SD", "wide"])
@pytest.mark.parametrize("n_spec", [0, 1, 3])
@pytest.mark.parametrize("W,D", [(4, 3), (6, 4)])
def test_update_state_type(act, sd, layout, n_spec, W, D):
    S = (W - 1) * D
    case = synth.depthwise_case(1320 + n_spec, DEV, lens=[], C=_C(act), width=W, dilation=D,
                                act=1, dtype=act, w_std=0.5, bias_std=0.1, spec_requests=67,
                                n_spec=n_spec, cap=S + n_spec + (1 if layout == "wide" else 0))
    g = torch.Generator(device=DEV).manual_seed(13)
    case.spec_has_init = (torch.rand(67, generator=g, device=DEV) < 0.8).to(torch.uint8)
    case.spec_state_idx[::9] = -1
    case.pool = other_pool(case.pool.shape, sd, layout, 1330 + n_spec)
    check_upd(case)


@pytest.mark.parametrize("act,sd", MIX)
def test_decode_on_a_widened_pool_keeps_the_other_columns(act, sd):
    # one-token decodes on a channel-first pool with spare columns: columns
    # >= S are not rewritten and keep their bits (an fp32 pool under bf16
    # activations goes through the bulk-copy pipeline with fp32 stages)
    W, D, S = 4, 1, 3
    case = synth.depthwise_case(1325, DEV, lens=[], C=_C(act), width=W, dilation=D, act=1,
                                dtype=act, w_std=0.5, bias_std=0.1, spec_requests=300,
                                n_spec=0, cap=S + 5)
    case.spec_has_init = torch.ones(300, dtype=torch.uint8, device=DEV)
    case.spec_has_init[::4] = 0
    case.pool = other_pool(case.pool.shape, sd, "DS", 1326)
    check_upd(case)


@pytest.mark.parametrize("act,sd", MIX)
def test_fused_fwd_state_type(act, sd):
    W, D = 4, 3
    lens = [1, 1, 0, 2, 9, 10, 64, 65, 129, 200, 7]
    case = synth.depthwise_case(1340, DEV, lens=lens, C=_C(act), width=W, dilation=D, act=1,
                                dtype=act, w_std=0.5, decode_prefix=2, padding_every=4)
    case.pool = other_pool(case.pool.shape, sd, "DS", 1341)
    T, C = case.num_tokens, case.C
    R = T + 21
    gc = torch.Generator(device="cpu").manual_seed(14)
    perm = torch.randperm(R, generator=gc)[:T].to(torch.int32).to(DEV)
    x_phys = physical(case.x, perm, R)
    res = rand_rows(R, C, 83, act)
    outer = rand_rows(R, C, 84, act)
    want_res, want_pool = oracle_fwd_fused(case, res, outer, perm, x_phys)
    err = new_err()
    got = res.clone()
    pool = run_fwd_fused(case, got, outer, perm, x_phys, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_out_close(to_np(got), want_res, act, "residual")
    assert_bits_equal(pool_np(pool), want_pool)


@pytest.mark.parametrize("act,sd", MIX)
@pytest.mark.parametrize("n_spec", [0, 3])
def test_fused_update_state_type(act, sd, n_spec):
    W, D = 4, 3
    case = synth.depthwise_case(1350 + n_spec, DEV, lens=[], C=_C(act), width=W, dilation=D,
                                act=1, dtype=act, w_std=0.5, spec_requests=29, n_spec=n_spec,
                                layout="SD")
    case.spec_has_init = torch.ones(29, dtype=torch.uint8, device=DEV)
    case.spec_state_idx[::7] = -1
    case.pool = other_pool(case.pool.shape, sd, "SD", 1351)
    q = 1 + n_spec
    Rl, C = 29 * q, case.C
    R = Rl + 11
    gc = torch.Generator(device="cpu").manual_seed(15)
    perm = torch.randperm(R, generator=gc)[:Rl].to(torch.int32).to(DEV)
    x_phys = physical(case.x_spec, perm, R)
    res = rand_rows(R, C, 85, act)
    outer = rand_rows(R, C, 86, act)
    na = case.num_accepted if n_spec else None
    want = to_np(res).copy()
    want_pool = pool_np(case.pool.clone())
    oracle.cconv_update_fused(to_np(x_phys), want_pool, to_np(case.w), None,
                              to_np(case.spec_state_idx), n_spec,
                              None if na is None else to_np(na), to_np(case.spec_has_init),
                              W, D, case.act, want, to_np(outer), to_np(perm))
    got = res.clone()
    pool = case.pool.clone()
    err = new_err()
    ops.cconv_update_fused(x_phys, pool, case.w, None, case.spec_state_idx, n_spec, na,
                           case.spec_has_init, W, D, case.act, got, outer, perm, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_out_close(to_np(got), want, act, "residual")
    assert_bits_equal(pool_np(pool), want_pool)


@pytest.mark.parametrize("act,sd", MIX)
@pytest.mark.parametrize("layout", ["DS", "SD"])
@pytest.mark.parametrize("spare", [0, 3])
def test_checkpoint_export_state_type(act, sd, layout, spare):
    W, D, S = 4, 3, 9
    lens = [3 * S + 5, S, 2 * S, 200]
    case = synth.depthwise_case(1360, DEV, lens=lens, C=_C(act), width=W, dilation=D, act=1,
                                dtype=act, w_std=0.5, num_slots=40, cap=S + spare)
    case.pool = other_pool(case.pool.shape, sd, layout, 1361)
    T = case.num_tokens
    ck_seq = torch.tensor([0, 0, 1, 2, 3, 3], dtype=torch.int32, device=DEV)
    ck_off = torch.tensor([S, 3 * S, S, 2 * S, 64, 200], dtype=torch.int32, device=DEV)
    ck_slot = torch.tensor([30, 31, 32, 33, 34, 35], dtype=torch.int32, device=DEV)
    want = pool_np(case.pool.clone())
    oracle.cconv_checkpoint_export(to_np(case.x), want, to_np(ck_seq), to_np(ck_off),
                                   to_np(ck_slot), to_np(case.cu_seqlens), W, D)
    pool = case.pool.clone()
    err = new_err()
    ops.cconv_checkpoint_export(case.x, pool, ck_seq, ck_off, ck_slot, case.cu_seqlens, W, D,
                                num_tokens=T, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_bits_equal(pool_np(pool), want)


def _fp32_state(case, layout, seed):
    case.pool = other_pool(case.pool.shape, torch.float32, layout, seed)
    g = torch.Generator(device=DEV).manual_seed(seed + 1)
    case.delayed_state = torch.randn(case.delayed_state.shape, generator=g, device=DEV)
    return case


@pytest.mark.parametrize("layout", ["DS", "SD", "wide"])
@pytest.mark.parametrize("t0,t1", [(2, 2), (3, 1), (4, 2)])
def test_cca_fp32_state(layout, t0, t1):
    case = synth.cca_case(1370 + t0 + t1, DEV, lens=LENS, decode_prefix=3, Hq=4, Hkv=2, t0=t0,
                          t1=t1, padding_every=6)
    check_cca(_fp32_state(case, layout, 1371))


def test_cca_fp32_state_empty_requests_keep_their_bits():
    case = synth.cca_case(1380, DEV, lens=[0, 0, 0, 3], decode_prefix=0, Hq=1, Hkv=1)
    case.has_init = torch.tensor([1, 0, 1, 1], dtype=torch.uint8, device=DEV)
    case.state_idx[2] = -1
    case = _fp32_state(case, "DS", 1381)
    before = case.delayed_state.clone()
    check_cca(case)
    # (check_cca runs on copies: run once more to look at the kept row itself)
    pool, dstate = case.pool.clone(), case.delayed_state.clone()
    T = int(case.qk.shape[0])
    out = torch.zeros_like(case.qk)
    dprev = torch.zeros_like(case.delayed)
    ops.cca_qk_conv(case.qk, case.w_dw, case.b_dw, case.w_gr, case.b_gr, case.groups, case.t0,
                    case.t1, case.delayed, case.delayed_init, pool, dstate, case.state_idx,
                    case.cu_seqlens, case.has_init, out, dprev, num_tokens=T)
    torch.cuda.synchronize()
    s0 = int(case.state_idx[0])
    assert torch.equal(dstate[s0].view(torch.int32), before[s0].view(torch.int32))


def test_cca_fused_fp32_state():
    Hq, Hkv = 4, 2
    case = synth.cca_case(1390, DEV, lens=LENS, decode_prefix=3, Hq=Hq, Hkv=Hkv,
                          padding_every=6)
    case = _fp32_state(case, "SD", 1391)
    T = int(case.qk.shape[0])
    g = torch.Generator(device=DEV).manual_seed(16)
    v_cur = torch.randn(T, case.Dv, generator=g, device=DEV).to(torch.bfloat16)
    out = torch.zeros((T, case.Cqk + 2 * case.Dv), device=DEV, dtype=torch.bfloat16)
    pool = case.pool.clone()
    dstate = case.delayed_state.clone()
    err = new_err()
    ops.cca_qk_conv_fused(case.qk, case.w_dw, case.b_dw, case.w_gr, case.b_gr, case.groups, Hq,
                          case.t0, case.t1, case.delayed, case.delayed_init, v_cur, pool, dstate,
                          case.state_idx, case.cu_seqlens, case.has_init, out, dev_err=err)
    chans, w_conv, w_dprev, w_pool, w_dstate = oracle_cca(case)
    want = np.zeros((T, case.Cqk + 2 * case.Dv), dtype=np.uint16)
    oracle.cca_project_epilogue(to_np(case.qk), w_conv, to_np(v_cur), w_dprev, Hq, Hkv, want)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = to_np(out)
    assert_out_close(got[:, :case.Cqk], want[:, :case.Cqk], torch.bfloat16, "query|key")
    assert_bits_equal(got[:, case.Cqk:], want[:, case.Cqk:], "value")
    assert_bits_equal(pool_np(pool), w_pool, "conv_state")
    assert_bits_equal(to_np(dstate), w_dstate, "delayed_state")


def test_cca_delayed_state_must_match_the_pool_type():
    case = synth.cca_case(1395, DEV, lens=[2], decode_prefix=0, Hq=1, Hkv=1)
    case.pool = other_pool(case.pool.shape, torch.float32, "DS", 1396)   # bf16 delayed state
    with pytest.raises(TypeError):
        check_cca(case)
