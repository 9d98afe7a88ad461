"""GPU parity at full size for the paths bench.py times beyond the hybrid step:
the fused PLE dispatch (spec + prefill rows in one physical tensor, random
request order), the fused Zaya tail, and fp32 conv-state pools under bf16
activations. The library runs the whole launch; the oracle checks every
channel (each depthwise channel is independent: channel blocks on all host
cores) and every kv group of the fused CCA (a kv group's query and key heads
are coupled: one job per kv group).
"""
import numpy as np
import pytest
import torch

import oracle
from state_cached_causal_gb300 import ops, synth
from tests._util import pool_np, to_np
from tests._full import assert_blocks, channel_blocks, count_out_of_tol, pmap
from tests.test_parity_depthwise import (assert_bits_equal, check_full, gpu_fwd, gpu_upd,
                                         new_err)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda")


def _f32_pool(case, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    case.pool = torch.randn(case.pool.shape, generator=g, device=DEV)
    return case


def test_gdn_mixed_fp32_state_full():
    case = _f32_pool(synth.gdn_mixed(DEV), 3001)
    err = new_err()
    out, pool = gpu_fwd(case, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_full(case, out=out, pool=pool, what="gdn_mixed, fp32 state")


def test_ple_spec_fp32_state_full():
    case = _f32_pool(synth.ple_spec(DEV), 3002)
    err = new_err()
    out, pool = gpu_fwd(case, err=err)
    out_s, pool = gpu_upd(case, pool=pool, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_full(case, out=out, out_s=out_s, pool=pool, what="ple_spec, fp32 state")


def test_ple_fused_full():
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
    xn, resn, outern, gotn = to_np(x), to_np(res), to_np(outer), to_np(got)
    want, want_pool, got_pool = resn.copy(), pool_np(case.pool.clone()), pool_np(pool)
    wn = to_np(case.w)
    sidx, na, ip = to_np(case.spec_state_idx), to_np(case.num_accepted), to_np(idx_s)
    meta, ipp = (to_np(case.state_idx), to_np(case.cu_seqlens), to_np(case.has_init)), to_np(idx_p)

    def block(sl):
        oracle.cconv_update_fused(xn[:, sl], want_pool[:, sl, :], wn[sl], None, sidx,
                                  case.n_spec, na, None, case.width, case.dilation, case.act,
                                  want[:, sl], outern[:, sl], ip)
        oracle.cconv_fwd_varlen_fused(xn[:, sl], wn[sl], None, want_pool[:, sl, :], *meta,
                                      case.width, case.dilation, case.act, want[:, sl],
                                      outern[:, sl], ipp)
        n, e = count_out_of_tol(gotn[:, sl], want[:, sl], True)
        return sl, n, e, int((got_pool[:, sl, :] != want_pool[:, sl, :]).sum())
    assert_blocks(pmap(block, channel_blocks(C)), "ple_fused")


def test_zaya_fused_full():
    # 16 query + 4 key heads: kv group j is query heads 4j .. 4j+3 and key head j;
    # one oracle job per kv group on the host cores, the value half once
    cc = synth.zaya_cca(DEV)
    Hq, Hkv, hd = 16, 4, 128
    kvg = Hq // Hkv
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
    got, got_pool = to_np(out), pool_np(pool)
    qk_all, pool0, ds0 = to_np(cc.qk), pool_np(cc.pool), to_np(cc.delayed_state)
    w_dw, b_dw, w_gr, b_gr = (to_np(t) for t in (cc.w_dw, cc.b_dw, cc.w_gr, cc.b_gr))
    delayed, dinit, vc = to_np(cc.delayed), to_np(cc.delayed_init), to_np(v_cur)
    meta = (to_np(cc.state_idx), to_np(cc.cu_seqlens), to_np(cc.has_init))

    def kv_group(j):
        heads = list(range(j * kvg, (j + 1) * kvg)) + [Hq + j]
        chans = np.concatenate([np.arange(h * hd, (h + 1) * hd) for h in heads])
        sub = lambda a: None if a is None else np.ascontiguousarray(a[chans])
        qk = np.ascontiguousarray(qk_all[:, chans])
        p = pool0[:, chans, :].copy()
        ds = ds0.copy()
        conv, dprev = np.zeros_like(qk), np.zeros_like(delayed)
        oracle.cca_qk_conv(qk, sub(w_dw), sub(b_dw), sub(w_gr), sub(b_gr), len(heads), cc.t0,
                           cc.t1, delayed, dinit, p, ds, *meta, conv, dprev)
        want = np.zeros((T, len(heads) * hd + 2 * (hd // 2)), dtype=np.uint16)
        oracle.cca_project_epilogue(qk, conv, vc, dprev, kvg, 1, want)
        n, e = count_out_of_tol(got[:, chans], want[:, :len(heads) * hd], True)
        neq = int((got_pool[:, chans, :] != p).sum())
        return chans, n, e, neq, dprev, ds
    res = pmap(kv_group, range(Hkv))
    assert_blocks([r[:4] for r in res], "zaya fused query|key")
    assert_bits_equal(got[:, cc.Cqk:cc.Cqk + cc.Dv], vc, "v_current")
    assert_bits_equal(got[:, cc.Cqk + cc.Dv:], res[0][4], "delayed_prev")
    assert_bits_equal(to_np(dstate), res[0][5], "delayed_state")
