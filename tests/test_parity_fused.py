"""GPU parity: the fused entry points (residual epilogue and logical row order)
vs the oracle.

Residual rows within |err| <= 1e-5 (fp32) or 2e-2 + 2e-2*|ref| (bf16); the
state bit for bit; rows the call does not own untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from state_cached_causal_gb300 import ops, synth
from tests._util import pool_np, to_np
from tests.test_parity_depthwise import assert_bits_equal, assert_out_close, new_err

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def rand_rows(rows, C, seed, dtype):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return torch.randn(rows, C, generator=g, device=DEV).to(dtype)


def physical(x_log, perm, rows):
    """Physical tensor with logical row i at row perm[i] (other rows random)."""
    out = rand_rows(rows, x_log.shape[1], 77, x_log.dtype)
    out[perm.long()] = x_log
    return out


def run_fwd_fused(case, res, outer, perm, x_phys, err):
    pool = case.pool.clone()
    ops.cconv_fwd_varlen_fused(x_phys, case.w, case.bias, pool, case.state_idx, case.cu_seqlens,
                               case.has_init, case.width, case.dilation, case.act, res, outer,
                               perm, dev_err=err, num_tokens=case.num_tokens)
    return pool


def oracle_fwd_fused(case, res, outer, perm, x_phys):
    r = to_np(res).copy()
    pool = pool_np(case.pool.clone())
    oracle.cconv_fwd_varlen_fused(to_np(x_phys), to_np(case.w), to_np(case.bias), pool,
                                  to_np(case.state_idx), to_np(case.cu_seqlens),
                                  to_np(case.has_init), case.width, case.dilation, case.act, r,
                                  None if outer is None else to_np(outer),
                                  None if perm is None else to_np(perm))
    return r, pool


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("W,D", [(4, 1), (4, 3), (2, 2), (3, 4), (8, 8), (5, 2), (2, 7)])
@pytest.mark.parametrize("with_outer,with_perm", [(True, True), (False, False), (True, False)])
def test_fwd_fused(dtype, W, D, with_outer, with_perm):
    S = (W - 1) * D
    lens = [1, 1, 0, 2, S, S + 1, 64, 65, 129, 200, 7]
    case = synth.depthwise_case(600 + 10 * W + D, DEV, lens=lens, C=520 if dtype ==
                                torch.float32 else 1040, width=W, dilation=D, act=1,
                                dtype=dtype, w_std=0.5, bias_std=0.1, decode_prefix=2,
                                padding_every=4)
    T, C = case.num_tokens, case.C
    R = T + 37                                       # physical rows beyond the logical ones
    g = torch.Generator(device="cpu").manual_seed(5)
    perm = (torch.randperm(R, generator=g)[:T].to(torch.int32).to(DEV) if with_perm
            else None)
    x_phys = physical(case.x, perm, R) if with_perm else torch.cat(
        [case.x, rand_rows(R - T, C, 78, dtype)])
    res = rand_rows(R, C, 79, dtype)
    outer = rand_rows(R, C, 80, dtype) if with_outer else None
    want_res, want_pool = oracle_fwd_fused(case, res, outer, perm, x_phys)
    err = new_err()
    got = res.clone()
    pool = run_fwd_fused(case, got, outer, perm, x_phys, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_out_close(to_np(got), want_res, dtype, "residual")
    assert_bits_equal(pool_np(pool), want_pool)


@pytest.mark.parametrize("layout", ["DS", "SD"])
@pytest.mark.parametrize("n_spec", [0, 3])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("W,D", [(4, 3), (7, 6)])
def test_update_fused(layout, n_spec, dtype, W, D):
    case = synth.depthwise_case(700 + n_spec, DEV, lens=[], C=520 if dtype == torch.float32
                                else 1040, width=W, dilation=D, act=1, dtype=dtype, w_std=0.5,
                                bias_std=0.1, spec_requests=29, n_spec=n_spec, layout=layout)
    g = torch.Generator(device=DEV).manual_seed(6)
    case.spec_has_init = (torch.rand(29, generator=g, device=DEV) < 0.8).to(torch.uint8)
    case.spec_state_idx[::7] = -1
    q = 1 + n_spec
    Rl, C = 29 * q, case.C
    R = Rl + 11
    gc = torch.Generator(device="cpu").manual_seed(7)
    perm = torch.randperm(R, generator=gc)[:Rl].to(torch.int32).to(DEV)
    x_phys = physical(case.x_spec, perm, R)
    res = rand_rows(R, C, 81, dtype)
    outer = rand_rows(R, C, 82, dtype)
    na = case.num_accepted if n_spec else None
    want = to_np(res).copy()
    want_pool = pool_np(case.pool.clone())
    oracle.cconv_update_fused(to_np(x_phys), want_pool, to_np(case.w), to_np(case.bias),
                              to_np(case.spec_state_idx), n_spec,
                              None if na is None else to_np(na), to_np(case.spec_has_init),
                              W, D, case.act, want, to_np(outer), to_np(perm))
    got = res.clone()
    pool = case.pool.clone()
    err = new_err()
    ops.cconv_update_fused(x_phys, pool, case.w, case.bias, case.spec_state_idx, n_spec, na,
                           case.spec_has_init, W, D, case.act, got, outer, perm, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_out_close(to_np(got), want, dtype, "residual")
    assert_bits_equal(pool_np(pool), want_pool)


def test_mixed_batch_in_original_row_order():
    """The PLE dispatch on one mixed batch: spec requests and non-spec
    (decode + prefill) rows interleaved in physical order, each call reading
    and writing its own rows through token_indices, no reordering copies."""
    W, D, n_spec = 4, 3, 3
    q = 1 + n_spec
    C, dtype = 1024, torch.bfloat16
    base = synth.depthwise_case(801, DEV, lens=[1, 1, 1, 40, 130], C=C, width=W, dilation=D,
                                act=1, dtype=dtype, w_std=0.3, decode_prefix=3,
                                spec_requests=6, n_spec=n_spec, num_slots=32)
    T = base.num_tokens
    Rs = 6 * q
    R = T + Rs
    gc = torch.Generator(device="cpu").manual_seed(8)
    order = torch.randperm(R, generator=gc).to(torch.int32).to(DEV)
    nonspec_idx, spec_idx = order[:T].contiguous(), order[T:].contiguous()
    x = rand_rows(R, C, 83, dtype)
    x[nonspec_idx.long()] = base.x
    x[spec_idx.long()] = base.x_spec
    res = rand_rows(R, C, 84, dtype)
    outer = rand_rows(R, C, 85, dtype)
    # oracle: spec first, then the non-spec rows (the dispatch order)
    want = to_np(res).copy()
    want_pool = pool_np(base.pool.clone())
    oracle.cconv_update_fused(to_np(x), want_pool, to_np(base.w), None,
                              to_np(base.spec_state_idx), n_spec, to_np(base.num_accepted),
                              to_np(base.spec_has_init), W, D, 1, want, to_np(outer),
                              to_np(spec_idx))
    oracle.cconv_fwd_varlen_fused(to_np(x), to_np(base.w), None, want_pool,
                                  to_np(base.state_idx), to_np(base.cu_seqlens),
                                  to_np(base.has_init), W, D, 1, want, to_np(outer),
                                  to_np(nonspec_idx))
    got = res.clone()
    pool = base.pool.clone()
    err = new_err()
    ops.cconv_update_fused(x, pool, base.w, None, base.spec_state_idx, n_spec,
                           base.num_accepted, base.spec_has_init, W, D, 1, got, outer, spec_idx,
                           dev_err=err)
    ops.cconv_fwd_varlen_fused(x, base.w, None, pool, base.state_idx, base.cu_seqlens,
                               base.has_init, W, D, 1, got, outer, nonspec_idx, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_out_close(to_np(got), want, dtype, "residual")
    assert_bits_equal(pool_np(pool), want_pool)


def test_bad_row_index_sets_flag_and_skips():
    case = synth.depthwise_case(802, DEV, lens=[5, 70, 3], C=256, width=4, dilation=1, act=1,
                                dtype=torch.bfloat16, w_std=0.5, spec_requests=4, n_spec=1)
    T = case.num_tokens
    idx = torch.arange(T, dtype=torch.int32, device=DEV)
    cu = case.cu_seqlens.tolist()
    idx[cu[1] + 3] = T + 100                        # outside the physical rows
    res = rand_rows(T, case.C, 86, torch.bfloat16)
    got = res.clone()
    err = new_err()
    ops.cconv_fwd_varlen_fused(case.x, case.w, None, case.pool.clone(), case.state_idx,
                               case.cu_seqlens, case.has_init, 4, 1, 1, got, None, idx,
                               dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.DERR_ROW_INDEX
    # the chunk holding the bad row is skipped: its rows keep their values
    assert torch.equal(got[cu[1]:cu[1] + 64], res[cu[1]:cu[1] + 64])
    # update: the request with the bad row is skipped
    q = 2
    idx_u = torch.arange(4 * q, dtype=torch.int32, device=DEV)
    idx_u[q * 2] = -1
    res_u = rand_rows(4 * q, case.C, 87, torch.bfloat16)
    got_u = res_u.clone()
    err = new_err()
    ops.cconv_update_fused(case.x_spec, case.pool.clone(), case.w, None, case.spec_state_idx, 1,
                           case.num_accepted, None, 4, 1, 1, got_u, None, idx_u, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.DERR_ROW_INDEX
    assert torch.equal(got_u[2 * q:3 * q], res_u[2 * q:3 * q])


# ---- prefill checkpoint export ------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("layout", ["DS", "SD", "wide"])
@pytest.mark.parametrize("W,D", [(4, 3), (2, 1), (3, 4), (8, 8), (6, 5)])
def test_checkpoint_export(dtype, layout, W, D):
    S = (W - 1) * D
    lens = [3 * S + 5, S, 2 * S, 200]
    kw = dict(lens=lens, C=520 if dtype == torch.float32 else 1040, width=W, dilation=D, act=1,
              dtype=dtype, w_std=0.5, num_slots=40)
    if layout == "wide":
        case = synth.depthwise_case(900 + W * 10 + D, DEV, cap=S + 4, **kw)
        case.pool = case.pool[:, :, 2:]
    else:
        case = synth.depthwise_case(900 + W * 10 + D, DEV, layout=layout, **kw)
    T = case.num_tokens
    R = T + 9
    gc = torch.Generator(device="cpu").manual_seed(10)
    perm = torch.randperm(R, generator=gc)[:T].to(torch.int32).to(DEV)
    x_phys = physical(case.x, perm, R)
    ck_seq = torch.tensor([0, 0, 1, 2, 3, 3], dtype=torch.int32, device=DEV)
    ck_off = torch.tensor([S, 3 * S, S, 2 * S, 64, 200], dtype=torch.int32, device=DEV)
    ck_slot = torch.tensor([30, 31, 32, 33, 34, 35], dtype=torch.int32, device=DEV)
    want = pool_np(case.pool.clone())
    oracle.cconv_checkpoint_export(to_np(x_phys), want, to_np(ck_seq), to_np(ck_off),
                                   to_np(ck_slot), to_np(case.cu_seqlens), W, D, to_np(perm))
    pool = case.pool.clone()
    err = new_err()
    ops.cconv_checkpoint_export(x_phys, pool, ck_seq, ck_off, ck_slot, case.cu_seqlens, W, D,
                                perm, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_bits_equal(pool_np(pool), want)


def test_checkpoint_export_bad_entries_are_flagged_and_skipped():
    W, D, S = 4, 1, 3
    case = synth.depthwise_case(950, DEV, lens=[10, 5], C=256, width=W, dilation=D, act=1,
                                dtype=torch.bfloat16, w_std=0.5, num_slots=8)
    ck_seq = torch.tensor([0, 2, 1, 1], dtype=torch.int32, device=DEV)    # request 2: none
    ck_off = torch.tensor([4, 3, 2, 5], dtype=torch.int32, device=DEV)    # 2 < S
    ck_slot = torch.tensor([5, 6, 7, 8], dtype=torch.int32, device=DEV)   # slot 8 == num_slots
    pool = case.pool.clone()
    err = new_err()
    ops.cconv_checkpoint_export(case.x, pool, ck_seq, ck_off, ck_slot, case.cu_seqlens, W, D,
                                dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.DERR_CHECKPOINT
    want = pool_np(case.pool.clone())
    oracle.cconv_checkpoint_export(to_np(case.x), want, [0], [4], [5], to_np(case.cu_seqlens),
                                   W, D)
    assert_bits_equal(pool_np(pool), want)
