"""GPU parity: cconv_fwd_varlen / cconv_update (through the C ABI) vs the oracle.

State write-back is compared bit for bit; outputs within max|err| <= 1e-5
(fp32) or |err| <= 2e-2 + 2e-2*|ref| (bf16), element by element on the same
seeded inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from state_cached_causal_gb300 import ops, synth
from tests._full import assert_blocks, channel_blocks, count_out_of_tol, pmap
from tests._util import np_to_f64, pool_np, to_np

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


# ---- comparison --------------------------------------------------------------

def assert_out_close(got, want, dtype, what="out"):
    g, w = np_to_f64(got), np_to_f64(want)
    assert g.shape == w.shape
    err = np.abs(g - w)
    if dtype == torch.float32:
        assert err.max(initial=0.0) <= 1e-5, f"{what}: max|err| {err.max():.3g}"
    else:
        bad = err > 2e-2 + 2e-2 * np.abs(w)
        assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, max {err.max():.3g}"


def assert_bits_equal(got, want, what="state"):
    assert got.shape == want.shape
    neq = got != want
    assert not neq.any(), f"{what}: {int(neq.sum())} elements differ"


def new_err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


# ---- runners ---------------------------------------------------------------

def gpu_fwd(case, pool=None, out=None, err=None):
    pool = case.pool.clone() if pool is None else pool
    out = torch.zeros_like(case.x) if out is None else out
    ops.cconv_fwd_varlen(case.x, case.w, case.bias, pool, case.state_idx, case.cu_seqlens,
                         case.has_init, case.width, case.dilation, case.act, out, dev_err=err)
    return out, pool


def oracle_fwd(case, chans=None):
    sl = slice(None) if chans is None else chans
    x = np.ascontiguousarray(to_np(case.x)[:, sl])
    w = np.ascontiguousarray(to_np(case.w)[sl])
    b = None if case.bias is None else np.ascontiguousarray(to_np(case.bias)[sl])
    pool = pool_np(case.pool)[:, sl, :].copy() if chans is not None else pool_np(case.pool.clone())
    out = np.zeros_like(x)
    oracle.cconv_fwd_varlen(x, w, b, pool, to_np(case.state_idx), to_np(case.cu_seqlens),
                            to_np(case.has_init), case.width, case.dilation, case.act, out)
    return out, pool


def gpu_upd(case, pool=None, err=None):
    pool = case.pool.clone() if pool is None else pool
    out = torch.zeros_like(case.x_spec)
    ops.cconv_update(case.x_spec, pool, case.w, case.bias, case.spec_state_idx, case.n_spec,
                     case.num_accepted if case.n_spec else None, case.spec_has_init,
                     case.width, case.dilation, case.act, out, dev_err=err)
    return out, pool


def oracle_upd(case, pool_np_in=None, chans=None):
    sl = slice(None) if chans is None else chans
    x = np.ascontiguousarray(to_np(case.x_spec)[:, sl])
    w = np.ascontiguousarray(to_np(case.w)[sl])
    b = None if case.bias is None else np.ascontiguousarray(to_np(case.bias)[sl])
    if pool_np_in is None:
        pool = pool_np(case.pool)[:, sl, :].copy() if chans is not None else pool_np(case.pool.clone())
    else:
        pool = pool_np_in
    out = np.zeros_like(x)
    oracle.cconv_update(x, pool, w, b, to_np(case.spec_state_idx), case.n_spec,
                        to_np(case.num_accepted) if case.n_spec else None,
                        to_np(case.spec_has_init), case.width, case.dilation, case.act, out)
    return out, pool


def check_fwd(case):
    err = new_err()
    out, pool = gpu_fwd(case, err=err)
    want_out, want_pool = oracle_fwd(case)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_out_close(to_np(out), want_out, case.dtype)
    assert_bits_equal(pool_np(pool), want_pool)


def check_upd(case):
    err = new_err()
    out, pool = gpu_upd(case, err=err)
    want_out, want_pool = oracle_upd(case)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_out_close(to_np(out), want_out, case.dtype)
    assert_bits_equal(pool_np(pool), want_pool)


# ---- fuzz over width x dilation x dtype --------------------------------------

# widths and dilations above 4 (one runtime-dilation kernel per width): the
# corners and the diagonal of width 2..8 x dilation 1..8, and mixed ones
WIDE = [(8, 1), (2, 8), (8, 8), (5, 5), (6, 6), (7, 7), (5, 1), (2, 5), (3, 6), (6, 2), (7, 8),
        (4, 5)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("W,D", [(w, d) for w in (2, 3, 4) for d in (1, 2, 3, 4)] + WIDE)
def test_fwd_varlen_fuzz(W, D, dtype):
    S = (W - 1) * D
    lens = [1, 1, 1, 0, 2, max(1, S - 1), S, S + 1, 63, 64, 65, 129, 200, 7]
    case = synth.depthwise_case(100 + 10 * W + D, DEV, lens=lens, C=1040 if dtype ==
                                torch.bfloat16 else 520, width=W, dilation=D, act=1,
                                dtype=dtype, w_std=0.5, bias_std=0.1, decode_prefix=3,
                                padding_every=5)
    check_fwd(case)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("W,D", [(w, d) for w in (2, 3, 4) for d in (1, 2, 3, 4)] + WIDE)
@pytest.mark.parametrize("n_spec", [0, 1, 3, 7])
def test_update_fuzz(W, D, dtype, n_spec):
    case = synth.depthwise_case(200 + 10 * W + D + n_spec, DEV, lens=[], C=1040 if dtype ==
                                torch.bfloat16 else 520, width=W, dilation=D, act=1,
                                dtype=dtype, w_std=0.5, bias_std=0.1, spec_requests=37,
                                n_spec=n_spec)
    g = torch.Generator(device=DEV).manual_seed(5)
    case.spec_has_init = (torch.rand(37, generator=g, device=DEV) < 0.8).to(torch.uint8)
    case.spec_state_idx[::6] = -1
    check_upd(case)


@pytest.mark.parametrize("layout", ["DS", "SD", "wide"])
@pytest.mark.parametrize("act,bias", [(0, False), (1, True)])
def test_layouts_and_epilogues(layout, act, bias):
    W, D = 4, 3
    lens = [1, 2, 9, 10, 77, 300]
    kw = dict(lens=lens, C=2048, width=W, dilation=D, act=act, dtype=torch.bfloat16, w_std=0.3,
              bias_std=0.1 if bias else None, spec_requests=9, n_spec=3)
    if layout == "wide":
        # the PLE view: last cap columns of a wider channel-first cache
        case = synth.depthwise_case(301, DEV, cap=15, **kw)
        case.pool = case.pool[:, :, 3:]
    else:
        case = synth.depthwise_case(301, DEV, layout=layout, **kw)
    check_fwd(case)
    check_upd(case)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_update_decode_of_wide_buffer_keeps_extra_columns(dtype):
    """n_spec == 0 on a channel-first buffer wider than S: columns >= S are
    neither read nor changed, with or without history."""
    case = synth.depthwise_case(309, DEV, lens=[], C=1032 if dtype == torch.bfloat16 else 516,
                                width=4, dilation=2, act=1, dtype=dtype, w_std=0.5,
                                bias_std=0.1, spec_requests=23, n_spec=0, cap=11)
    g = torch.Generator(device=DEV).manual_seed(6)
    case.spec_has_init = (torch.rand(23, generator=g, device=DEV) < 0.5).to(torch.uint8)
    case.spec_state_idx[::5] = -1
    check_upd(case)
    _, pool = gpu_upd(case)
    torch.cuda.synchronize()
    assert torch.equal(pool[:, :, 6:], case.pool[:, :, 6:])


def test_row_strides_and_untouched_rows():
    C = 1024
    case = synth.depthwise_case(302, DEV, lens=[5, 70, 3], C=C, width=4, dilation=1, act=1,
                                dtype=torch.bfloat16, w_std=0.5, bias_std=0.1)
    T = case.num_tokens
    xbig = torch.randn(T + 4, C + 64, device=DEV).to(torch.bfloat16)
    xbig[:T, :C] = case.x
    case.x = xbig[:T, :C]                              # row stride C + 64
    obig = torch.full((T + 4, C + 32), 7.0, device=DEV, dtype=torch.bfloat16)
    out = obig[:, :C]                                  # more rows than tokens
    pool = case.pool.clone()
    ops.cconv_fwd_varlen(case.x, case.w, case.bias, pool, case.state_idx, case.cu_seqlens,
                         case.has_init, 4, 1, 1, out, num_tokens=T + 4)
    want_out, want_pool = oracle_fwd(case)
    torch.cuda.synchronize()
    assert_out_close(to_np(out[:T]), want_out, torch.bfloat16)
    assert bool((obig[T:] == 7.0).all()) and bool((obig[:, C:] == 7.0).all())
    assert_bits_equal(pool_np(pool), want_pool)


def test_empty_batch_and_empty_sequences():
    case = synth.depthwise_case(303, DEV, lens=[0, 0, 0], C=256, width=4, dilation=2, act=1,
                                dtype=torch.bfloat16, w_std=0.5)
    case.has_init = torch.tensor([1, 0, 1], dtype=torch.uint8, device=DEV)
    case.state_idx[2] = -1
    check_fwd(case)
    # num_seqs == 0 is a no-op
    pool = case.pool.clone()
    ops.cconv_fwd_varlen(case.x, case.w, None, pool, case.state_idx[:0], case.cu_seqlens[:1],
                         None, 4, 2, 1, torch.zeros_like(case.x))
    torch.cuda.synchronize()
    assert torch.equal(pool, case.pool)


def test_split_invariance_on_gpu_is_bitexact():
    """One 300-token sequence == prefill(100) + prefill(150) + 50 decodes."""
    W, D, L, C = 4, 3, 300, 2048
    case = synth.depthwise_case(304, DEV, lens=[L], C=C, width=W, dilation=D, act=1,
                                dtype=torch.bfloat16, w_std=0.3, has_init="all", cap=12)
    full_out, full_pool = gpu_fwd(case)
    pool = case.pool.clone()
    out = torch.zeros_like(case.x)
    sidx, one = case.state_idx, torch.ones(1, dtype=torch.uint8, device=DEV)
    for a, b in ((0, 100), (100, 250)):
        ops.cconv_fwd_varlen(case.x[a:b], case.w, None, pool, sidx,
                             torch.tensor([0, b - a], dtype=torch.int32, device=DEV), one, W, D,
                             1, out[a:b])
    for t in range(250, L):
        ops.cconv_update(case.x[t:t + 1], pool, case.w, None, sidx, 0, None, None, W, D, 1,
                         out[t:t + 1])
    torch.cuda.synchronize()
    assert torch.equal(out, full_out)
    assert torch.equal(pool, full_pool)


# ---- device-detected bad data ----------------------------------------------

def test_bad_slot_sets_flag_and_skips_only_that_sequence():
    case = synth.depthwise_case(305, DEV, lens=[4, 5, 6], C=256, width=4, dilation=1, act=1,
                                dtype=torch.bfloat16, w_std=0.5, num_slots=8)
    case.state_idx[1] = 8                      # == num_slots
    err = new_err()
    out = torch.full_like(case.x, 3.0)
    out, pool = gpu_fwd(case, out=out, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.DERR_SLOT_RANGE
    cu = case.cu_seqlens.tolist()
    assert bool((out[cu[1]:cu[2]] == 3.0).all())
    good = synth.depthwise_case(305, DEV, lens=[4, 5, 6], C=256, width=4, dilation=1, act=1,
                                dtype=torch.bfloat16, w_std=0.5, num_slots=8)
    want_out, _ = oracle_fwd(good)
    got = to_np(out)
    assert_out_close(got[cu[0]:cu[1]], want_out[cu[0]:cu[1]], torch.bfloat16)
    assert_out_close(got[cu[2]:cu[3]], want_out[cu[2]:cu[3]], torch.bfloat16)


def test_decode_bad_slot_sets_flag_and_skips_only_that_request():
    # one-token decodes on a dense channel-first pool of S columns (the one-pass
    # decode kernel): the bad request's output row and every slot stay as they were
    case = synth.depthwise_case(306, DEV, lens=[], C=1040, width=4, dilation=1, act=1,
                                dtype=torch.bfloat16, w_std=0.5, bias_std=0.1, num_slots=12,
                                spec_requests=5, n_spec=0)
    case.spec_state_idx[2] = 12                # == num_slots
    err = new_err()
    pool = case.pool.clone()
    out = torch.full_like(case.x_spec, 3.0)
    ops.cconv_update(case.x_spec, pool, case.w, case.bias, case.spec_state_idx, 0, None, None,
                     4, 1, 1, out, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.DERR_SLOT_RANGE
    assert bool((out[2] == 3.0).all())
    keep = [0, 1, 3, 4]
    x = to_np(case.x_spec)[keep]
    ref_pool = pool_np(case.pool.clone())
    ref_out = np.zeros_like(x)
    oracle.cconv_update(x, ref_pool, to_np(case.w), to_np(case.bias),
                        to_np(case.spec_state_idx)[keep], 0, None, None, 4, 1, 1, ref_out)
    assert_out_close(to_np(out)[keep], ref_out, torch.bfloat16)
    assert_bits_equal(pool_np(pool), ref_pool)


@pytest.mark.parametrize("what", ["w", "bias"])
def test_decode_with_unaligned_weights(what):
    # weights or biases that do not start on 16 bytes cannot take the decode
    # kernel's vector loads; the call still computes the same result
    case = synth.depthwise_case(307, DEV, lens=[], C=1040, width=4, dilation=1, act=1,
                                dtype=torch.bfloat16, w_std=0.5, bias_std=0.1,
                                spec_requests=9, n_spec=0)
    if what == "w":
        buf = torch.zeros(case.w.numel() + 1, dtype=case.w.dtype, device=DEV)
        buf[1:] = case.w.reshape(-1)
        case.w = buf[1:].view(case.w.shape)
    else:
        buf = torch.zeros(case.bias.numel() + 3, dtype=case.bias.dtype, device=DEV)
        buf[3:] = case.bias
        case.bias = buf[3:]
    check_upd(case)


def test_bad_cu_seqlens_sets_flag():
    case = synth.depthwise_case(306, DEV, lens=[4, 5, 6], C=256, width=4, dilation=1, act=1,
                                dtype=torch.bfloat16, w_std=0.5)
    case.cu_seqlens[2] = 2                      # decreasing
    err = new_err()
    gpu_fwd(case, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.DERR_CU_SEQLENS


def test_bad_num_accepted_sets_flag():
    case = synth.depthwise_case(307, DEV, lens=[], C=256, width=4, dilation=3, act=1,
                                dtype=torch.bfloat16, w_std=0.5, spec_requests=4, n_spec=3)
    case.num_accepted[0] = 0
    case.num_accepted[3] = 5
    err = new_err()
    gpu_upd(case, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & ops.DERR_NUM_ACCEPTED


def test_invalid_arguments_raise():
    case = synth.depthwise_case(308, DEV, lens=[4], C=256, width=4, dilation=1, act=1,
                                dtype=torch.bfloat16, w_std=0.5)
    flat = torch.zeros(4 * 256 + 1, dtype=torch.bfloat16, device=DEV)
    mis = flat[1:].view(4, 256)                 # 2-byte offset: not 16-byte aligned
    with pytest.raises(ops.CConvError) as e:
        ops.cconv_fwd_varlen(mis, case.w, None, case.pool, case.state_idx, case.cu_seqlens,
                             None, 4, 1, 1, torch.zeros_like(case.x))
    assert e.value.status == ops.ERR_INVALID
    with pytest.raises(ops.CConvError) as e:
        ops.cconv_update(case.x[:1], case.pool, case.w, None, case.state_idx, 1,
                         torch.ones(1, dtype=torch.int32, device=DEV), None, 4, 1, 1,
                         torch.zeros_like(case.x[:1]))
    assert e.value.status == ops.ERR_INVALID       # cap 3 < S + n_spec


# ---- the five workloads at full size ----------------------------------------

def test_single_prefill_full():
    for hi in ("none", "all"):
        case = synth.single_prefill(DEV, has_init=hi)
        check_fwd(case)
    a_out, a_pool = gpu_fwd(synth.single_prefill(DEV, has_init="none"))
    b_out, b_pool = gpu_fwd(synth.single_prefill(DEV, has_init="all"))
    torch.cuda.synchronize()
    assert torch.equal(a_out, b_out) and torch.equal(a_pool, b_pool)


def test_gdn_decode_full():
    check_upd(synth.gdn_decode(DEV))


def _slices(C):
    return [slice(0, 64), slice(C // 2 - 40, C // 2 + 24), slice(C - 64, C)]


def check_full(case, out=None, out_s=None, pool=None, what=""):
    """Every channel of a full-size launch against the oracle: the varlen outputs
    (out), then the update outputs (out_s) on the pool the varlen call left, both
    within the tolerance, and the whole pool -- used and unused slots -- bit for
    bit. The oracle runs on channel blocks on all host cores."""
    bf16 = case.dtype == torch.bfloat16
    w = to_np(case.w)
    b = None if case.bias is None else to_np(case.bias)
    want_pool = pool_np(case.pool.clone())
    got_pool = pool_np(pool)
    jobs = []
    if out is not None:
        x, got = to_np(case.x), to_np(out)
        want = np.zeros_like(got)
        meta = (to_np(case.state_idx), to_np(case.cu_seqlens), to_np(case.has_init))
        jobs.append(lambda sl: (oracle.cconv_fwd_varlen(
            x[:, sl], w[sl], None if b is None else b[sl], want_pool[:, sl, :], *meta,
            case.width, case.dilation, case.act, want[:, sl]), (got, want))[1])
    if out_s is not None:
        xs, got_s = to_np(case.x_spec), to_np(out_s)
        want_s = np.zeros_like(got_s)
        na = to_np(case.num_accepted) if case.n_spec else None
        sidx, shi = to_np(case.spec_state_idx), to_np(case.spec_has_init)
        jobs.append(lambda sl: (oracle.cconv_update(
            xs[:, sl], want_pool[:, sl, :], w[sl], None if b is None else b[sl], sidx,
            case.n_spec, na, shi, case.width, case.dilation, case.act, want_s[:, sl]),
            (got_s, want_s))[1])

    def block(sl):
        bad, worst = 0, 0.0
        for job in jobs:                       # varlen first, then the update
            g, wnt = job(sl)
            n, e = count_out_of_tol(g[:, sl], wnt[:, sl], bf16)
            bad, worst = bad + n, max(worst, e)
        return sl, bad, worst, int((got_pool[:, sl, :] != want_pool[:, sl, :]).sum())
    assert_blocks(pmap(block, channel_blocks(case.C)), what)


@pytest.mark.slow
def test_gdn_mixed_full():
    case = synth.gdn_mixed(DEV)
    err = new_err()
    out, pool = gpu_fwd(case, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_full(case, out=out, pool=pool, what="gdn_mixed")


@pytest.mark.slow
def test_ple_spec_full():
    case = synth.ple_spec(DEV)
    err = new_err()
    out, pool = gpu_fwd(case, err=err)
    out_s, pool = gpu_upd(case, pool=pool, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    check_full(case, out=out, out_s=out_s, pool=pool, what="ple_spec")
