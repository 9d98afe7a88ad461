"""GPU parity: cca_qk_conv (through the C ABI) vs the oracle.

q/k outputs within |err| <= 2e-2 + 2e-2*|ref| (bf16); the delayed half of v,
the raw-history state and the delayed state bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from state_cached_causal_gb300 import ops, synth
from tests._full import assert_blocks, count_out_of_tol, pmap
from tests._util import pool_np, to_np
from tests.test_parity_depthwise import assert_bits_equal, assert_out_close, new_err

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def gpu_cca(case, err=None, num_tokens=None, out=None, dprev=None):
    pool = case.pool.clone()
    dstate = case.delayed_state.clone()
    out = torch.zeros_like(case.qk) if out is None else out
    dprev = torch.zeros_like(case.delayed) if dprev is None else dprev
    ops.cca_qk_conv(case.qk, case.w_dw, case.b_dw, case.w_gr, case.b_gr, case.groups, case.t0,
                    case.t1, case.delayed, case.delayed_init, pool, dstate, case.state_idx,
                    case.cu_seqlens, case.has_init, out, dprev, dev_err=err,
                    num_tokens=num_tokens)
    return out, dprev, pool, dstate


def oracle_cca(case, groups=None):
    """Oracle over all groups, or over the listed groups only (they are independent)."""
    qk = to_np(case.qk)
    pool = pool_np(case.pool)
    dstate = to_np(case.delayed_state).copy()
    w_dw, b_dw, w_gr, b_gr = (to_np(case.w_dw), to_np(case.b_dw), to_np(case.w_gr),
                              to_np(case.b_gr))
    gs = case.Cqk // case.groups
    sel = list(range(case.groups)) if groups is None else list(groups)
    chans = np.concatenate([np.arange(g * gs, (g + 1) * gs) for g in sel])
    sub = lambda a: None if a is None else np.ascontiguousarray(a[chans])
    q = np.ascontiguousarray(qk[:, chans])
    p = pool[:, chans, :].copy()
    out = np.zeros_like(q)
    dprev = np.zeros_like(to_np(case.delayed))
    oracle.cca_qk_conv(q, sub(w_dw), sub(b_dw), sub(w_gr), sub(b_gr), len(sel), case.t0,
                       case.t1, to_np(case.delayed), to_np(case.delayed_init), p, dstate,
                       to_np(case.state_idx), to_np(case.cu_seqlens), to_np(case.has_init),
                       out, dprev)
    return chans, out, dprev, p, dstate


def check(case, groups=None):
    err = new_err()
    out, dprev, pool, dstate = gpu_cca(case, err=err)
    chans, w_out, w_dprev, w_pool, w_dstate = oracle_cca(case, groups)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, int(err.item())
    assert_out_close(to_np(out)[:, chans], w_out, torch.bfloat16, "qk")
    assert_bits_equal(to_np(dprev), w_dprev, "delayed_prev")
    assert_bits_equal(pool_np(pool)[:, chans, :], w_pool, "conv_state")
    assert_bits_equal(to_np(dstate), w_dstate, "delayed_state")


LENS = [1, 1, 1, 0, 2, 3, 1, 5, 126, 127, 128, 129, 1, 300, 255, 7]


@pytest.mark.parametrize("t0,t1", [(2, 2), (1, 1), (2, 1), (3, 1), (4, 1), (1, 2), (3, 2),
                                   (4, 2)])
def test_cca_fuzz(t0, t1):
    case = synth.cca_case(400 + 10 * t0 + t1, DEV, lens=LENS, decode_prefix=3, Hq=4, Hkv=2,
                          t0=t0, t1=t1, padding_every=6)
    check(case)


@pytest.mark.parametrize("layout", ["DS", "SD"])
def test_cca_layouts_and_no_bias(layout):
    case = synth.cca_case(431, DEV, lens=LENS, decode_prefix=3, Hq=2, Hkv=1, layout=layout,
                          bias=False)
    check(case)


def test_cca_all_decodes_and_long_prefill():
    case = synth.cca_case(432, DEV, lens=[1] * 300 + [1000], decode_prefix=300, Hq=3, Hkv=1)
    check(case)


def test_cca_empty_requests_only():
    case = synth.cca_case(433, DEV, lens=[0, 0, 0], decode_prefix=0, Hq=1, Hkv=1)
    case.has_init = torch.tensor([1, 0, 1], dtype=torch.uint8, device=DEV)
    case.state_idx[2] = -1
    check(case)


def test_cca_untouched_rows_and_bad_slot():
    case = synth.cca_case(434, DEV, lens=[3, 40, 2], decode_prefix=0, Hq=1, Hkv=1,
                          num_slots=6, has_init="all")
    T = int(case.qk.shape[0])
    out = torch.full((T + 5, case.Cqk), 5.0, device=DEV, dtype=torch.bfloat16)
    dprev = torch.full((T + 5, case.Dv), 5.0, device=DEV, dtype=torch.bfloat16)
    qk = torch.zeros((T + 5, case.Cqk), device=DEV, dtype=torch.bfloat16)
    qk[:T] = case.qk
    dl = torch.zeros((T + 5, case.Dv), device=DEV, dtype=torch.bfloat16)
    dl[:T] = case.delayed
    good = synth.cca_case(434, DEV, lens=[3, 40, 2], decode_prefix=0, Hq=1, Hkv=1,
                          num_slots=6, has_init="all")
    case.qk, case.delayed = qk, dl
    case.state_idx[1] = 6                              # == num_slots: skipped, flagged
    err = new_err()
    out, dprev, pool, dstate = gpu_cca(case, err=err, out=out, dprev=dprev)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.DERR_SLOT_RANGE
    assert bool((out[T:] == 5.0).all()) and bool((dprev[T:] == 5.0).all())
    cu = case.cu_seqlens.tolist()
    assert bool((out[cu[1]:cu[2]] == 5.0).all())
    chans, w_out, w_dprev, _, _ = oracle_cca(good)
    got = to_np(out)
    for a, b in ((cu[0], cu[1]), (cu[2], cu[3])):
        assert_out_close(got[a:b], w_out[a:b], torch.bfloat16)
        assert_bits_equal(to_np(dprev)[a:b], w_dprev[a:b])


@pytest.mark.parametrize("t0,t1", [(2, 2), (4, 2), (1, 2), (3, 1)])
@pytest.mark.parametrize("L", [1, 2, 5, 130])
def test_cca_one_request_per_call(t0, t1, L):
    """A call holding one request: its tiles are single-request tiles, where the
    token before row 0 comes from the history (and a one-token request also
    rewrites that history in the same pass)."""
    case = synth.cca_case(437 + L, DEV, lens=[L], decode_prefix=0, Hq=2, Hkv=1, t0=t0, t1=t1,
                          has_init="all")
    check(case)


def test_cca_split_invariance_on_gpu_is_bitexact():
    L = 700
    case = synth.cca_case(435, DEV, lens=[L], decode_prefix=0, Hq=2, Hkv=1, has_init="all")
    full = gpu_cca(case)
    pool = case.pool.clone()
    dstate = case.delayed_state.clone()
    out = torch.zeros_like(case.qk)
    dprev = torch.zeros_like(case.delayed)
    one = torch.ones(1, dtype=torch.uint8, device=DEV)
    edges = [0, 1, 130, 131, 500] + list(range(501, L + 1))
    for a, b in zip(edges[:-1], edges[1:]):
        ops.cca_qk_conv(case.qk[a:b], case.w_dw, case.b_dw, case.w_gr, case.b_gr, case.groups,
                        2, 2, case.delayed[a:b], case.delayed_init, pool, dstate,
                        case.state_idx, torch.tensor([0, b - a], dtype=torch.int32,
                                                     device=DEV), one, out[a:b], dprev[a:b])
    torch.cuda.synchronize()
    assert torch.equal(out, full[0])
    assert torch.equal(dprev, full[1])
    assert torch.equal(pool, full[2])
    assert torch.equal(dstate, full[3])


def test_cca_rejects_unsupported():
    case = synth.cca_case(436, DEV, lens=[4], decode_prefix=0, Hq=1, Hkv=1, head_dim=64)
    with pytest.raises(ops.CConvError) as e:
        gpu_cca(case)
    assert e.value.status == ops.ERR_UNSUPPORTED


@pytest.mark.slow
def test_zaya_cca_full():
    """Every group of the zaya_cca launch against the oracle, one group per job
    on all host cores (the groups are independent; each job keeps its own
    delayed state, and the delayed half of v and the delayed state are compared
    once, from group 0's run)."""
    case = synth.zaya_cca(DEV)
    err = new_err()
    out, dprev, pool, dstate = gpu_cca(case, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    qk, got, got_pool = to_np(case.qk), to_np(out), pool_np(pool)
    w_dw, b_dw, w_gr, b_gr = (to_np(case.w_dw), to_np(case.b_dw), to_np(case.w_gr),
                              to_np(case.b_gr))
    want, want_pool = np.zeros_like(got), pool_np(case.pool.clone())
    delayed, dinit, ds0 = to_np(case.delayed), to_np(case.delayed_init), to_np(case.delayed_state)
    meta = (to_np(case.state_idx), to_np(case.cu_seqlens), to_np(case.has_init))
    gs = case.Cqk // case.groups
    opt = lambda a, sl: None if a is None else a[sl]

    def group(g):
        sl = slice(g * gs, (g + 1) * gs)
        ds, dp = ds0.copy(), np.zeros_like(delayed)
        oracle.cca_qk_conv(qk[:, sl], w_dw[sl], opt(b_dw, sl), w_gr[sl], opt(b_gr, sl), 1,
                           case.t0, case.t1, delayed, dinit, want_pool[:, sl, :], ds, *meta,
                           want[:, sl], dp)
        n, e = count_out_of_tol(got[:, sl], want[:, sl], True)
        return sl, n, e, int((got_pool[:, sl, :] != want_pool[:, sl, :]).sum()), dp, ds
    res = pmap(group, range(case.groups))
    assert_blocks([r[:4] for r in res], "zaya_cca")
    assert_bits_equal(to_np(dprev), res[0][4], "delayed_prev")
    assert_bits_equal(to_np(dstate), res[0][5], "delayed_state")


# ---- the fused tail of ZayaCCA.project ----------------------------------------

@pytest.mark.parametrize("Hq,Hkv,t0,t1", [(4, 2, 2, 2), (16, 4, 2, 2), (2, 2, 3, 1),
                                          (6, 2, 1, 2)])
def test_cca_fused_project_tail(Hq, Hkv, t0, t1):
    case = synth.cca_case(460 + Hq + t0, DEV, lens=LENS, decode_prefix=3, Hq=Hq, Hkv=Hkv,
                          t0=t0, t1=t1, padding_every=6)
    T = int(case.qk.shape[0])
    g = torch.Generator(device=DEV).manual_seed(11)
    v_cur = torch.randn(T, case.Dv, generator=g, device=DEV).to(torch.bfloat16)
    out = torch.full((T, case.Cqk + 2 * case.Dv + 8), 9.0, device=DEV, dtype=torch.bfloat16)
    pool = case.pool.clone()
    dstate = case.delayed_state.clone()
    err = new_err()
    ops.cca_qk_conv_fused(case.qk, case.w_dw, case.b_dw, case.w_gr, case.b_gr, case.groups, Hq,
                          t0, t1, case.delayed, case.delayed_init, v_cur, pool, dstate,
                          case.state_idx, case.cu_seqlens, case.has_init,
                          out[:, :case.Cqk + 2 * case.Dv], dev_err=err)
    chans, w_conv, w_dprev, w_pool, w_dstate = oracle_cca(case)
    want = np.zeros((T, case.Cqk + 2 * case.Dv), dtype=np.uint16)
    oracle.cca_project_epilogue(to_np(case.qk), w_conv, to_np(v_cur), w_dprev, Hq, Hkv, want)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = to_np(out)
    assert_out_close(got[:, :case.Cqk], want[:, :case.Cqk], torch.bfloat16, "query|key")
    assert_bits_equal(got[:, case.Cqk:case.Cqk + 2 * case.Dv], want[:, case.Cqk:], "value")
    assert bool((out[:, case.Cqk + 2 * case.Dv:] == 9.0).all())
    assert_bits_equal(pool_np(pool), w_pool, "conv_state")
    assert_bits_equal(to_np(dstate), w_dstate, "delayed_state")
