"""Pins for the oracle: checks against things other than the oracle itself.

* torch.nn.functional.conv1d in fp64 (a library routine) on tiny inputs -- pins
  tap orientation, dilation, bias, the history window and the grouped-conv
  weight layout ([out, in/groups, taps]);
* torch's own bf16 rounding -- pins the oracle's round-to-nearest-even;
* special cases with a closed form: an identity tap gives y == x, zero weights
  give y = act(bias);
* invariants the pages state: the stored state is a copy of the last
  (width-1)*dilation inputs; a full sequence equals any prefill/decode split
  through the pool; a dilated conv is d interleaved undilated ones; the spec
  rolling buffer resumed at num_accepted = a equals recomputing from the
  history that ends at draft token a-1;
* the Zaya profile-run path (zero padding, no metadata) equals the state path
  of one request without history.

No CUDA is involved; everything here runs on the CPU.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from state_cached_causal_gb300 import synth
from tests._util import np_to_f64, pool_np, to_np

CPU = torch.device("cpu")


# ---- fp64 library references ------------------------------------------------

def conv_ref(hist, xs, w, bias, D, act):
    """[C,S] history + [L,C] tokens -> [L,C] fp64 via F.conv1d (depthwise)."""
    C, W = w.shape
    inp = torch.cat([torch.as_tensor(hist), torch.as_tensor(xs).T], dim=1)[None]
    y = F.conv1d(inp, torch.as_tensor(w)[:, None, :],
                 None if bias is None else torch.as_tensor(bias), dilation=D, groups=C)[0].T
    if act:
        y = y * torch.sigmoid(y)
    return y.numpy()


def tol_ok(got, ref, atol, rtol):
    err = np.abs(got - ref)
    return bool(np.all(err <= atol + rtol * np.abs(ref))), float(err.max(initial=0.0))


def run_fwd(case, out=None):
    x = to_np(case.x)
    pool = pool_np(case.pool.clone())
    out = np.zeros_like(x) if out is None else out
    oracle.cconv_fwd_varlen(x, to_np(case.w), to_np(case.bias), pool, to_np(case.state_idx),
                            to_np(case.cu_seqlens), to_np(case.has_init), case.width,
                            case.dilation, case.act, out)
    return out, pool


# ---- bf16 rounding -----------------------------------------------------------

def test_bf16_rounding_matches_torch():
    g = torch.Generator().manual_seed(7)
    vals = torch.randn(4000, generator=g) * torch.exp(torch.randn(4000, generator=g) * 4)
    # exact ties: bf16 value plus half an ulp, both parities
    base = torch.randn(200, generator=g).to(torch.bfloat16).float()
    ulp_half = torch.ldexp(torch.ones(200), torch.frexp(base).exponent - 9)
    vals = torch.cat([vals, base + ulp_half, base - ulp_half, torch.tensor([0.0, -0.0])])
    want = vals.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.oracle_f32_to_bf16_scalar(float(v)) for v in vals.tolist()],
                   dtype=np.uint16)
    assert np.array_equal(got, want)


# ---- depthwise varlen vs F.conv1d ----------------------------------------------

CASES = [(w, d) for w in (2, 3, 4) for d in (1, 2, 3)]
# widths and dilations to 8: corners and the diagonal of the accepted range
WIDE = [(8, 1), (2, 8), (8, 8), (5, 5), (6, 3), (7, 7), (3, 6)]


@pytest.mark.parametrize("W,D", CASES + WIDE)
@pytest.mark.parametrize("act,use_bias", [(0, False), (1, True)])
def test_fwd_varlen_fp32_matches_conv1d(W, D, act, use_bias):
    S = (W - 1) * D
    lens = [0, 1, max(1, S - 1), S, S + 1, 7, 20]
    case = synth.depthwise_case(11 + W * 10 + D, CPU, lens=lens, C=12, width=W,
                                dilation=D, act=act, dtype=torch.float32, w_std=0.5,
                                bias_std=0.3 if use_bias else None, cap=S + 2)
    pool0 = pool_np(case.pool.clone())
    out, pool = run_fwd(case)
    x = to_np(case.x).astype(np.float64)
    w = to_np(case.w).astype(np.float64)
    b = None if case.bias is None else to_np(case.bias).astype(np.float64)
    cu = to_np(case.cu_seqlens)
    for s, slot in enumerate(to_np(case.state_idx)):
        h = bool(to_np(case.has_init)[s])
        hist = pool0[slot, :, :S].astype(np.float64) if h else np.zeros((12, S))
        xs = x[cu[s]:cu[s + 1]]
        if len(xs):
            ref = conv_ref(hist, xs, w, b, D, act)
            ok, err = tol_ok(out[cu[s]:cu[s + 1]].astype(np.float64), ref, 2e-6, 2e-6)
            assert ok, (s, err)
        # stored state == last S inputs of [history, tokens]; wider columns untouched
        ext = np.concatenate([hist, xs.T], axis=1)
        assert np.array_equal(pool[slot, :, :S], ext[:, ext.shape[1] - S:].astype(np.float32))
        assert np.array_equal(pool[slot, :, S:], pool0[slot, :, S:])


@pytest.mark.parametrize("layout", ["DS", "SD"])
def test_fwd_varlen_bf16_matches_conv1d(layout):
    W, D = 4, 3
    S = 9
    lens = [1, 5, 9, 10, 33]
    case = synth.depthwise_case(5, CPU, lens=lens, C=16, width=W, dilation=D, act=1,
                                dtype=torch.bfloat16, w_std=0.3, bias_std=0.1, layout=layout)
    pool0 = pool_np(case.pool.clone())
    out, pool = run_fwd(case)
    x = np_to_f64(to_np(case.x))
    w = np_to_f64(to_np(case.w))
    b = np_to_f64(to_np(case.bias))
    cu = to_np(case.cu_seqlens)
    for s, slot in enumerate(to_np(case.state_idx)):
        h = bool(to_np(case.has_init)[s])
        hist = np_to_f64(pool0[slot, :, :S]) if h else np.zeros((16, S))
        ref = conv_ref(hist, x[cu[s]:cu[s + 1]], w, b, D, 1)
        got = np_to_f64(out[cu[s]:cu[s + 1]])
        ok, err = tol_ok(got, ref, 1e-5, 2.0 ** -8)  # one bf16 rounding of the output
        assert ok, (s, err)
        ext = np.concatenate([pool0[slot, :, :S] if h else np.zeros((16, S), np.uint16),
                              to_np(case.x)[cu[s]:cu[s + 1]].T], axis=1)
        assert np.array_equal(pool[slot, :, :S], ext[:, -S:])


def test_identity_tap_gives_input_bitexact():
    for dtype in (torch.float32, torch.bfloat16):
        case = synth.depthwise_case(3, CPU, lens=[4, 17], C=8, width=4, dilation=2, act=0,
                                    dtype=dtype, w_std=1.0)
        case.w.zero_()
        case.w[:, -1] = 1.0
        out, _ = run_fwd(case)
        assert np.array_equal(out, to_np(case.x))


def test_zero_weights_give_act_of_bias():
    case = synth.depthwise_case(4, CPU, lens=[3, 6], C=8, width=3, dilation=1, act=1,
                                dtype=torch.float32, w_std=1.0, bias_std=2.0)
    case.w.zero_()
    out, _ = run_fwd(case)
    b = to_np(case.bias).astype(np.float64)
    want = b * (1.0 / (1.0 + np.exp(-b)))
    assert np.allclose(out, np.broadcast_to(want, out.shape), rtol=1e-6, atol=1e-7)


def test_dilation_is_interleaved_undilated_convs():
    W, D, L, C = 3, 3, 23, 8
    S = (W - 1) * D
    case = synth.depthwise_case(9, CPU, lens=[L], C=C, width=W, dilation=D, act=1,
                                dtype=torch.float32, w_std=0.5, bias_std=0.2, has_init="all")
    pool0 = pool_np(case.pool.clone())
    slot = int(case.state_idx[0])
    out, _ = run_fwd(case)
    ext = np.concatenate([pool0[slot, :, :S], to_np(case.x).T], axis=1)  # [C, S+L]
    for r in range(D):
        sub = ext[:, r::D]                   # residue class r of [history, tokens]
        hist_r, xs_r = sub[:, :W - 1], sub[:, W - 1:].T.copy()
        pool_r = np.ascontiguousarray(hist_r[None])
        out_r = np.zeros_like(xs_r)
        oracle.cconv_fwd_varlen(xs_r, to_np(case.w), to_np(case.bias), pool_r,
                                np.array([0], np.int32), np.array([0, len(xs_r)], np.int32),
                                np.array([1], np.uint8), W, 1, 1, out_r)
        assert np.array_equal(out[r::D], out_r)


def _split_fwd(case, cuts):
    """Process the single sequence of ``case`` in pieces at ``cuts`` through the pool."""
    x = to_np(case.x)
    pool = pool_np(case.pool.clone())
    out = np.zeros_like(x)
    edges = [0] + list(cuts) + [x.shape[0]]
    hi0 = to_np(case.has_init)[0]
    for i, (a, b) in enumerate(zip(edges[:-1], edges[1:])):
        xs = np.ascontiguousarray(x[a:b])
        o = np.zeros_like(xs)
        oracle.cconv_fwd_varlen(xs, to_np(case.w), to_np(case.bias), pool,
                                to_np(case.state_idx), np.array([0, b - a], np.int32),
                                np.array([hi0 if i == 0 else 1], np.uint8), case.width,
                                case.dilation, case.act, o)
        out[a:b] = o
    return out, pool


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("h", ["all", "none"])
def test_split_invariance_prefill_chunks_and_decodes(dtype, h):
    W, D, L = 4, 3, 40
    case = synth.depthwise_case(21, CPU, lens=[L], C=16, width=W, dilation=D, act=1,
                                dtype=dtype, w_std=0.4, bias_std=0.1, has_init=h, cap=12)
    full_out, full_pool = run_fwd(case)
    for cuts in ([1], [5, 9, 10], [20, 30], list(range(31, 40))):
        out, pool = _split_fwd(case, cuts)
        assert np.array_equal(out, full_out), cuts
        assert np.array_equal(pool, full_pool), cuts
    # tail as one-token decodes through the update entry point
    x = to_np(case.x)
    pool = pool_np(case.pool.clone())
    out = np.zeros_like(x)
    k = 25
    oracle.cconv_fwd_varlen(np.ascontiguousarray(x[:k]), to_np(case.w), to_np(case.bias),
                            pool, to_np(case.state_idx), np.array([0, k], np.int32),
                            to_np(case.has_init), W, D, 1, out[:k])
    for t in range(k, L):
        o = np.zeros_like(x[t:t + 1])
        oracle.cconv_update(np.ascontiguousarray(x[t:t + 1]), pool, to_np(case.w),
                            to_np(case.bias), to_np(case.state_idx), 0, None, None, W, D, 1, o)
        out[t] = o[0]
    assert np.array_equal(out, full_out)
    assert np.array_equal(pool, full_pool)


def test_padding_slot_reads_zero_history_and_writes_nothing():
    case = synth.depthwise_case(8, CPU, lens=[3, 5, 2], C=8, width=4, dilation=1, act=1,
                                dtype=torch.bfloat16, w_std=0.5, bias_std=0.1,
                                has_init="all", padding_every=2)
    pool0 = pool_np(case.pool.clone())
    out, pool = run_fwd(case)
    assert int(case.state_idx[1]) == -1
    # the padding sequence equals the same tokens with has_init = 0 in a scratch slot
    cu = to_np(case.cu_seqlens)
    xs = np.ascontiguousarray(to_np(case.x)[cu[1]:cu[2]])
    scratch = np.zeros((1, 8, 3), np.uint16)
    o = np.zeros_like(xs)
    oracle.cconv_fwd_varlen(xs, to_np(case.w), to_np(case.bias), scratch,
                            np.array([0], np.int32), np.array([0, len(xs)], np.int32),
                            np.array([0], np.uint8), 4, 1, 1, o)
    assert np.array_equal(out[cu[1]:cu[2]], o)
    used = set(int(v) for v in to_np(case.state_idx) if v >= 0)
    for s in range(pool.shape[0]):
        if s not in used:
            assert np.array_equal(pool[s], pool0[s])


def test_empty_sequence_state_rule():
    case = synth.depthwise_case(12, CPU, lens=[0, 0], C=8, width=3, dilation=2, act=0,
                                dtype=torch.float32, w_std=0.5)
    case.has_init = torch.tensor([1, 0], dtype=torch.uint8)
    pool0 = pool_np(case.pool.clone())
    x = np.zeros((0, 8), np.float32)
    pool = pool_np(case.pool.clone())
    oracle.cconv_fwd_varlen(x, to_np(case.w), None, pool, to_np(case.state_idx),
                            to_np(case.cu_seqlens), to_np(case.has_init), 3, 2, 0,
                            np.zeros((0, 8), np.float32))
    s0, s1 = (int(v) for v in to_np(case.state_idx))
    assert np.array_equal(pool[s0], pool0[s0])          # h: state kept
    assert not pool[s1, :, :4].any()                     # !h: history is zero
    assert np.array_equal(pool[s1, :, 4:], pool0[s1, :, 4:])


# ---- decode / spec -----------------------------------------------------------

def _spec_setup(seed, dtype, W=4, D=3, n_spec=3, C=8, R=5):
    case = synth.depthwise_case(seed, CPU, lens=[], C=C, width=W, dilation=D, act=1,
                                dtype=dtype, w_std=0.4, bias_std=0.1, spec_requests=R,
                                n_spec=n_spec)
    return case


def test_decode_update_equals_one_token_varlen():
    case = synth.depthwise_case(31, CPU, lens=[1] * 6, C=16, width=4, dilation=2, act=1,
                                dtype=torch.bfloat16, w_std=0.4, bias_std=0.1,
                                has_init="all", cap=9)
    out_v, pool_v = run_fwd(case)
    pool_u = pool_np(case.pool.clone())
    out_u = np.zeros_like(out_v)
    oracle.cconv_update(to_np(case.x), pool_u, to_np(case.w), to_np(case.bias),
                        to_np(case.state_idx), 0, None, None, 4, 2, 1, out_u)
    assert np.array_equal(out_u, out_v)
    assert np.array_equal(pool_u, pool_v)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_spec_outputs_match_conv1d_over_prior_window(dtype):
    W, D, n_spec = 4, 3, 3
    S, q = 9, 4
    case = _spec_setup(41, dtype, W, D, n_spec)
    pool0 = pool_np(case.pool.clone())
    pool = pool_np(case.pool.clone())
    x = to_np(case.x_spec)
    out = np.zeros_like(x)
    oracle.cconv_update(x, pool, to_np(case.w), to_np(case.bias), to_np(case.spec_state_idx),
                        n_spec, to_np(case.num_accepted), None, W, D, 1, out)
    w, b = np_to_f64(to_np(case.w)), np_to_f64(to_np(case.bias))
    for r, slot in enumerate(to_np(case.spec_state_idx)):
        off = int(to_np(case.num_accepted)[r]) - 1
        prior = np_to_f64(pool0[slot, :, off:off + S])
        ref = conv_ref(prior, np_to_f64(x[r * q:(r + 1) * q]), w, b, D, 1)
        ok, err = tol_ok(np_to_f64(out[r * q:(r + 1) * q]), ref, 2e-6,
                         2e-6 if dtype == torch.float32 else 2.0 ** -8)
        assert ok, err
        # rolled buffer: drop accepted history, append the q new tokens
        cap = pool.shape[2]
        want = np.concatenate([pool0[slot, :, off + 1:off + 1 + cap - q],
                               x[r * q:(r + 1) * q].T], axis=1)
        assert np.array_equal(pool[slot], want)


def test_spec_first_step_equals_sequential_decodes():
    W, D, n_spec = 4, 3, 3
    q = 4
    case = _spec_setup(42, torch.bfloat16, W, D, n_spec)
    case.num_accepted.fill_(1)   # fresh from prefill: the history sits at column 0
    x = to_np(case.x_spec)
    pool = pool_np(case.pool.clone())
    out = np.zeros_like(x)
    oracle.cconv_update(x, pool, to_np(case.w), to_np(case.bias), to_np(case.spec_state_idx),
                        n_spec, to_np(case.num_accepted), None, W, D, 1, out)
    pool_d = pool_np(case.pool.clone())
    out_d = np.zeros_like(x)
    R = len(to_np(case.spec_state_idx))
    for i in range(q):
        rows = np.ascontiguousarray(x[i::q])
        o = np.zeros_like(rows)
        oracle.cconv_update(rows, pool_d, to_np(case.w), to_np(case.bias),
                            to_np(case.spec_state_idx), 0, None, None, W, D, 1, o)
        out_d[i::q] = o
    assert np.array_equal(out, out_d)
    assert R == out.shape[0] // q


@pytest.mark.parametrize("a", [1, 2, 3, 4])
def test_spec_rollback_equals_recompute_from_accepted_prefix(a):
    """Step 1 drafts x1 (q tokens); step 2 resumes at num_accepted = a. Its outputs
    must equal decoding step 2's tokens from the history that ends at x1[a-1]."""
    W, D, n_spec = 4, 2, 3
    q = 4
    case = _spec_setup(43 + a, torch.float32, W, D, n_spec, R=3)
    case.num_accepted.fill_(1)
    w, b, sidx = to_np(case.w), to_np(case.bias), to_np(case.spec_state_idx)
    x1 = to_np(case.x_spec)
    g = torch.Generator().manual_seed(99 + a)
    x2 = torch.randn(x1.shape, generator=g).numpy()
    pool = pool_np(case.pool.clone())
    o1 = np.zeros_like(x1)
    oracle.cconv_update(x1, pool, w, b, sidx, n_spec, to_np(case.num_accepted), None, W, D,
                        1, o1)
    o2 = np.zeros_like(x2)
    oracle.cconv_update(x2, pool, w, b, sidx, n_spec, np.full(len(sidx), a, np.int32), None,
                        W, D, 1, o2)
    # recompute: original history + the a accepted draft tokens, then x2 as decodes
    pool_r = pool_np(case.pool.clone())
    acc = np.ascontiguousarray(np.concatenate([x1[r * q:r * q + a] for r in range(len(sidx))]))
    cu = np.arange(0, len(sidx) * a + 1, a, dtype=np.int32)
    oracle.cconv_fwd_varlen(acc, w, b, pool_r, sidx, cu, np.ones(len(sidx), np.uint8), W, D,
                            1, np.zeros_like(acc))
    o2r = np.zeros_like(x2)
    for i in range(q):
        rows = np.ascontiguousarray(x2[i::q])
        o = np.zeros_like(rows)
        oracle.cconv_update(rows, pool_r, w, b, sidx, 0, None, None, W, D, 1, o)
        o2r[i::q] = o
    assert np.array_equal(o2, o2r)


# ---- Zaya CCA ------------------------------------------------------------------

def cca_ref(hist, xs, w_dw, b_dw, w_gr, b_gr, G, t0, t1, bf16):
    """fp64 two-stage conv of one request via F.conv1d; u stored as bf16 when asked."""
    inp = torch.cat([torch.as_tensor(hist), torch.as_tensor(xs).T], dim=1)[None]
    C = inp.shape[1]
    u = F.conv1d(inp, torch.as_tensor(w_dw)[:, None, :], torch.as_tensor(b_dw), groups=C)
    if bf16:
        u = u.to(torch.bfloat16).to(torch.float64)
    v = F.conv1d(u, torch.as_tensor(w_gr), torch.as_tensor(b_gr), groups=G)
    return v[0].T.numpy()


def run_cca(case):
    qk = to_np(case.qk)
    pool = pool_np(case.pool.clone())
    dstate = to_np(case.delayed_state.clone()).copy()
    out = np.zeros_like(qk)
    dprev = np.zeros_like(to_np(case.delayed))
    oracle.cca_qk_conv(qk, to_np(case.w_dw), to_np(case.b_dw), to_np(case.w_gr),
                       to_np(case.b_gr), case.groups, case.t0, case.t1, to_np(case.delayed),
                       to_np(case.delayed_init), pool, dstate, to_np(case.state_idx),
                       to_np(case.cu_seqlens), to_np(case.has_init), out, dprev)
    return out, dprev, pool, dstate


@pytest.mark.parametrize("t0,t1", [(2, 2), (3, 1), (1, 2), (3, 2)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_cca_matches_two_conv1d(t0, t1, dtype):
    lens = [1, 1, 2, 5, 9]
    case = synth.cca_case(61, CPU, lens=lens, decode_prefix=2, Hq=2, Hkv=1, head_dim=8,
                          t0=t0, t1=t1, dtype=dtype)
    pool0 = pool_np(case.pool.clone())
    dstate0 = to_np(case.delayed_state).copy()
    out, dprev, pool, dstate = run_cca(case)
    n = t0 + t1 - 2
    bf = dtype == torch.bfloat16
    f = np_to_f64
    cu = to_np(case.cu_seqlens)
    for s, slot in enumerate(to_np(case.state_idx)):
        h = bool(to_np(case.has_init)[s])
        hist = f(pool0[slot, :, :n]) if h else np.zeros((case.Cqk, n))
        xs = f(to_np(case.qk)[cu[s]:cu[s + 1]])
        ref = cca_ref(hist, xs, f(to_np(case.w_dw)), f(to_np(case.b_dw)), f(to_np(case.w_gr)),
                      f(to_np(case.b_gr)), case.groups, t0, t1, bf)
        got = f(out[cu[s]:cu[s + 1]])
        ok, err = tol_ok(got, ref, 2e-3 if bf else 2e-6, 2.0 ** -7 if bf else 2e-6)
        assert ok, (s, err)
        # delayed half of v: first token sees the state (or the initial value)
        d = to_np(case.delayed)
        first = dstate0[slot] if h else to_np(case.delayed_init)
        assert np.array_equal(dprev[cu[s]], first)
        assert np.array_equal(dprev[cu[s] + 1:cu[s + 1]], d[cu[s]:cu[s + 1] - 1])
        assert np.array_equal(dstate[slot], d[cu[s + 1] - 1])
        ext = np.concatenate([pool0[slot, :, :n] if h else np.zeros_like(pool0[slot, :, :n]),
                              to_np(case.qk)[cu[s]:cu[s + 1]].T], axis=1)
        assert np.array_equal(pool[slot, :, :n], ext[:, ext.shape[1] - n:])


def test_cca_profile_path_equals_state_path_without_history():
    """Profile run: conv of the zero-padded batch (one request) == has_init = 0."""
    case = synth.cca_case(62, CPU, lens=[13], decode_prefix=0, Hq=2, Hkv=2, head_dim=8,
                          has_init="none")
    out, _, _, _ = run_cca(case)
    n = case.t0 + case.t1 - 2
    qk = torch.as_tensor(np_to_f64(to_np(case.qk)))
    f = lambda t: torch.as_tensor(np_to_f64(to_np(t)))
    u = F.conv1d(F.pad(qk.T[None], (n, 0)), f(case.w_dw)[:, None, :], f(case.b_dw),
                 groups=case.Cqk).to(torch.bfloat16).double()
    v = F.conv1d(u, f(case.w_gr), f(case.b_gr), groups=case.groups)[0].T.numpy()
    ok, err = tol_ok(np_to_f64(out), v, 2e-3, 2.0 ** -7)
    assert ok, err


@pytest.mark.parametrize("cuts", [[1], [1, 2], [4, 5, 6, 7], [2, 9]])
def test_cca_split_invariance(cuts):
    L = 12
    case = synth.cca_case(63, CPU, lens=[L], decode_prefix=0, Hq=2, Hkv=2, head_dim=8,
                          has_init="all")
    full = run_cca(case)
    qk, dl = to_np(case.qk), to_np(case.delayed)
    pool = pool_np(case.pool.clone())
    dstate = to_np(case.delayed_state.clone()).copy()
    out = np.zeros_like(qk)
    dprev = np.zeros_like(dl)
    edges = [0] + cuts + [L]
    for a, b in zip(edges[:-1], edges[1:]):
        o = np.zeros_like(qk[a:b])
        dp = np.zeros_like(dl[a:b])
        oracle.cca_qk_conv(np.ascontiguousarray(qk[a:b]), to_np(case.w_dw), to_np(case.b_dw),
                           to_np(case.w_gr), to_np(case.b_gr), case.groups, 2, 2,
                           np.ascontiguousarray(dl[a:b]), to_np(case.delayed_init), pool,
                           dstate, to_np(case.state_idx), np.array([0, b - a], np.int32),
                           np.array([1], np.uint8), o, dp)
        out[a:b] = o
        dprev[a:b] = dp
    assert np.array_equal(out, full[0])
    assert np.array_equal(dprev, full[1])
    assert np.array_equal(pool, full[2])
    assert np.array_equal(dstate, full[3])


def test_cca_padding_and_empty_requests():
    case = synth.cca_case(64, CPU, lens=[2, 0, 3, 0], decode_prefix=0, Hq=1, Hkv=1,
                          head_dim=8, has_init="all")
    case.state_idx[2] = -1
    case.has_init[3] = 0
    pool0 = pool_np(case.pool.clone())
    dstate0 = to_np(case.delayed_state).copy()
    out, dprev, pool, dstate = run_cca(case)
    s1, s3 = int(case.state_idx[1]), int(case.state_idx[3])
    assert np.array_equal(pool[s1], pool0[s1]) and np.array_equal(dstate[s1], dstate0[s1])
    assert not pool[s3].any()
    assert np.array_equal(dstate[s3], to_np(case.delayed_init))
    # the padding request's first token sees the initial delayed value
    cu = to_np(case.cu_seqlens)
    assert np.array_equal(dprev[cu[2]], to_np(case.delayed_init))
