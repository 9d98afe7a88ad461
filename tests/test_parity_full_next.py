"""GPU parity at full size for the paths bench.py times beyond the hybrid step:
the fused PLE dispatch (spec + prefill rows in one physical tensor, random
request order), the fused Zaya tail, and fp32 conv-state pools under bf16
activations. The library runs the whole launch; the oracle checks sampled
channel slices (each channel is independent in the depthwise conv) or one kv
group (the fused CCA couples a kv group's query and key heads), whose values it
computes exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from state_cached_causal_gb300 import ops, synth
from tests._util import pool_np, to_np
from tests.test_parity_depthwise import (_slices, assert_bits_equal, assert_out_close, gpu_fwd,
                                         gpu_upd, new_err, oracle_fwd, oracle_upd)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda")


def _f32_pool(case, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    case.pool = torch.randn(case.pool.shape, generator=g, device=DEV)
    return case


def test_gdn_mixed_fp32_state_full_sampled():
    case = _f32_pool(synth.gdn_mixed(DEV), 3001)
    err = new_err()
    out, pool = gpu_fwd(case, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for sl in _slices(case.C):
        want_out, want_pool = oracle_fwd(case, chans=sl)
        assert_out_close(to_np(out)[:, sl], want_out, case.dtype)
        assert_bits_equal(pool_np(pool)[:, sl, :], want_pool)


def test_ple_spec_fp32_state_full_sampled():
    case = _f32_pool(synth.ple_spec(DEV), 3002)
    err = new_err()
    out, pool = gpu_fwd(case, err=err)
    out_s, pool = gpu_upd(case, pool=pool, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for sl in _slices(case.C):
        want_out, want_pool = oracle_fwd(case, chans=sl)
        want_s, want_pool = oracle_upd(case, pool_np_in=want_pool, chans=sl)
        assert_out_close(to_np(out)[:, sl], want_out, case.dtype)
        assert_out_close(to_np(out_s)[:, sl], want_s, case.dtype, "spec out")
        assert_bits_equal(pool_np(pool)[:, sl, :], want_pool)


def test_ple_fused_full_sampled():
    # the ple_spec batch with every request's rows at a random place of one
    # physical tensor: spec requests through cconv_update_fused, prefills
    # through cconv_fwd_varlen_fused, residual += conv + outer residual
    case = synth.ple_spec(DEV)
    q = 1 + case.n_spec
    T, C = case.num_tokens, case.C
    Rs = int(case.spec_state_idx.numel())
    R = T + Rs * q
    order = torch.randperm(R, generator=torch.Generator().manual_seed(3003)).to(torch.int32)
    idx_p, idx_s = order[:T].contiguous().to(DEV), order[T:].contiguous().to(DEV)
    x = torch.zeros(R, C, device=DEV, dtype=case.dtype)
    x[idx_p.long()] = case.x
    x[idx_s.long()] = case.x_spec
    g = torch.Generator(device=DEV).manual_seed(3004)
    res = torch.randn(R, C, generator=g, device=DEV).to(case.dtype)
    outer = torch.randn(R, C, generator=g, device=DEV).to(case.dtype)
    pool = case.pool.clone()
    got = res.clone()
    err = new_err()
    ops.cconv_update_fused(x, pool, case.w, case.bias, case.spec_state_idx, case.n_spec,
                           case.num_accepted, case.spec_has_init, case.width, case.dilation,
                           case.act, got, outer, idx_s, dev_err=err)
    ops.cconv_fwd_varlen_fused(x, case.w, case.bias, pool, case.state_idx, case.cu_seqlens,
                               case.has_init, case.width, case.dilation, case.act, got, outer,
                               idx_p, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for sl in _slices(C):
        sub = lambda t: np.ascontiguousarray(to_np(t)[:, sl])
        want = sub(res)
        want_pool = pool_np(case.pool)[:, sl, :].copy()
        w = np.ascontiguousarray(to_np(case.w)[sl])
        oracle.cconv_update_fused(sub(x), want_pool, w, None, to_np(case.spec_state_idx),
                                  case.n_spec, to_np(case.num_accepted), None, case.width,
                                  case.dilation, case.act, want, sub(outer), to_np(idx_s))
        oracle.cconv_fwd_varlen_fused(sub(x), w, None, want_pool, to_np(case.state_idx),
                                      to_np(case.cu_seqlens), to_np(case.has_init), case.width,
                                      case.dilation, case.act, want, sub(outer), to_np(idx_p))
        assert_out_close(to_np(got)[:, sl], want, case.dtype, "residual")
        assert_bits_equal(pool_np(pool)[:, sl, :], want_pool)


def test_zaya_fused_full_one_kv_group():
    # 16 query + 4 key heads; kv group j = 1 is query heads 4..7 and key head 1
    cc = synth.zaya_cca(DEV)
    Hq, Hkv, hd = 16, 4, 128
    T = int(cc.qk.shape[0])
    g = torch.Generator(device=DEV).manual_seed(3005)
    v_cur = torch.randn(T, cc.Dv, generator=g, device=DEV).to(torch.bfloat16)
    out = torch.zeros(T, cc.Cqk + 2 * cc.Dv, device=DEV, dtype=torch.bfloat16)
    pool, dstate = cc.pool.clone(), cc.delayed_state.clone()
    err = new_err()
    ops.cca_qk_conv_fused(cc.qk, cc.w_dw, cc.b_dw, cc.w_gr, cc.b_gr, cc.groups, Hq, cc.t0,
                          cc.t1, cc.delayed, cc.delayed_init, v_cur, pool, dstate, cc.state_idx,
                          cc.cu_seqlens, cc.has_init, out, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    heads = [4, 5, 6, 7, Hq + 1]
    chans = np.concatenate([np.arange(h * hd, (h + 1) * hd) for h in heads])
    sub = lambda a: None if a is None else np.ascontiguousarray(a[chans])
    qk = np.ascontiguousarray(to_np(cc.qk)[:, chans])
    p = pool_np(cc.pool)[:, chans, :].copy()
    ds = to_np(cc.delayed_state).copy()
    conv = np.zeros_like(qk)
    dprev = np.zeros_like(to_np(cc.delayed))
    oracle.cca_qk_conv(qk, sub(to_np(cc.w_dw)), sub(to_np(cc.b_dw)), sub(to_np(cc.w_gr)),
                       sub(to_np(cc.b_gr)), len(heads), cc.t0, cc.t1, to_np(cc.delayed),
                       to_np(cc.delayed_init), p, ds, to_np(cc.state_idx),
                       to_np(cc.cu_seqlens), to_np(cc.has_init), conv, dprev)
    want = np.zeros((T, len(heads) * hd + 2 * (hd // 2)), dtype=np.uint16)
    oracle.cca_project_epilogue(qk, conv, to_np(v_cur), dprev, 4, 1, want)
    got = to_np(out)
    assert_out_close(got[:, chans], want[:, :len(heads) * hd], torch.bfloat16, "query|key")
    assert_bits_equal(got[:, cc.Cqk:cc.Cqk + cc.Dv], to_np(v_cur), "v_current")
    assert_bits_equal(got[:, cc.Cqk + cc.Dv:], dprev, "delayed_prev")
    assert_bits_equal(pool_np(pool)[:, chans, :], p, "conv_state")
    assert_bits_equal(to_np(dstate), ds, "delayed_state")
