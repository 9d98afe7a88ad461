"""Pins for the oracle's fused epilogue (residual additions and logical row
order of the "Qwen4ExpPLELayer" short conv), against things other than the
oracle itself:

* torch.nn.functional.conv1d in fp64 plus the two residual terms, on tiny
  fp32 inputs with a random logical -> physical row permutation;
* reduction to the plain operation: a zero residual, no outer residual and the
  identity row order give the plain output bit for bit;
* permutation invariance: moving the rows of x, residual and outer by a
  permutation and passing it as token_indices moves the result with them;
* rejection of a row index outside the physical rows.

No CUDA is involved.
"""
import numpy as np
import pytest
import torch

import oracle
from state_cached_causal_gb300 import synth
from tests._util import pool_np, to_np
from tests.test_oracle_pins import conv_ref

CPU = torch.device("cpu")


def _case(seed, dtype, lens=(5, 1, 0, 9, 3), W=4, D=2, n_spec=0, spec=0):
    return synth.depthwise_case(seed, CPU, lens=list(lens), C=16, width=W, dilation=D, act=1,
                                dtype=dtype, w_std=0.5, bias_std=0.1, padding_every=4,
                                spec_requests=spec, n_spec=n_spec)


def _rand_rows(rows, C, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    return to_np(torch.randn(rows, C, generator=g).to(dtype))


def _f64(a):
    return oracle.bf16_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(
        np.float64)


def test_fused_fwd_fp32_matches_conv1d_plus_residuals():
    case = _case(901, torch.float32)
    T, C = case.x.shape
    perm = np.random.default_rng(3).permutation(T).astype(np.int32)
    x_log = to_np(case.x)
    x_phys = np.empty_like(x_log)
    x_phys[perm] = x_log                                  # logical row i lives at perm[i]
    res = _rand_rows(T, C, 11, torch.float32)
    outer = _rand_rows(T, C, 12, torch.float32)
    pool = pool_np(case.pool.clone())
    got = res.copy()
    oracle.cconv_fwd_varlen_fused(x_phys, to_np(case.w), to_np(case.bias), pool,
                                  to_np(case.state_idx), to_np(case.cu_seqlens),
                                  to_np(case.has_init), case.width, case.dilation, case.act,
                                  got, outer, perm)
    want = res.astype(np.float64).copy()
    cu = to_np(case.cu_seqlens)
    pool0 = pool_np(case.pool)
    S = (case.width - 1) * case.dilation
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if b == a:
            continue
        slot = int(case.state_idx[s])
        h = slot >= 0 and int(case.has_init[s]) != 0
        hist = pool0[slot, :, :S].astype(np.float64) if h else np.zeros((C, S))
        y = conv_ref(hist, x_log[a:b].astype(np.float64), to_np(case.w).astype(np.float64),
                     to_np(case.bias).astype(np.float64), case.dilation, case.act)
        for i in range(a, b):
            want[perm[i]] = res[perm[i]] + y[i - a] + outer[perm[i]]
    assert np.abs(got - want).max() <= 1e-5


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fused_fwd_reduces_to_plain(dtype):
    case = _case(902, dtype)
    x = to_np(case.x)
    out = np.zeros_like(x)
    pool_a = pool_np(case.pool.clone())
    oracle.cconv_fwd_varlen(x, to_np(case.w), to_np(case.bias), pool_a, to_np(case.state_idx),
                            to_np(case.cu_seqlens), to_np(case.has_init), case.width,
                            case.dilation, case.act, out)
    res = np.zeros_like(x)
    pool_b = pool_np(case.pool.clone())
    oracle.cconv_fwd_varlen_fused(x, to_np(case.w), to_np(case.bias), pool_b,
                                  to_np(case.state_idx), to_np(case.cu_seqlens),
                                  to_np(case.has_init), case.width, case.dilation, case.act,
                                  res)
    assert np.array_equal(res, out)
    assert np.array_equal(pool_a, pool_b)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fused_fwd_row_order_is_a_permutation(dtype):
    case = _case(903, dtype)
    T, C = case.x.shape
    perm = np.random.default_rng(4).permutation(T).astype(np.int32)
    x, res, outer = to_np(case.x), _rand_rows(T, C, 13, dtype), _rand_rows(T, C, 14, dtype)
    args = (to_np(case.w), to_np(case.bias))
    meta = (to_np(case.state_idx), to_np(case.cu_seqlens), to_np(case.has_init), case.width,
            case.dilation, case.act)
    r_id = res.copy()
    p_id = pool_np(case.pool.clone())
    oracle.cconv_fwd_varlen_fused(x, *args, p_id, *meta, r_id, outer)
    xp, rp, op = (np.empty_like(a) for a in (x, res, outer))
    xp[perm], rp[perm], op[perm] = x, res, outer
    p_pm = pool_np(case.pool.clone())
    oracle.cconv_fwd_varlen_fused(xp, *args, p_pm, *meta, rp, op, perm)
    assert np.array_equal(rp[perm], r_id)
    assert np.array_equal(p_pm, p_id)


def test_fused_update_fp32_matches_conv1d_plus_residuals():
    n_spec, W, D = 3, 4, 2
    case = _case(904, torch.float32, lens=(), W=W, D=D, n_spec=n_spec, spec=6)
    q = 1 + n_spec
    R, C = case.x_spec.shape
    perm = np.random.default_rng(5).permutation(R).astype(np.int32)
    x_log = to_np(case.x_spec)
    x_phys = np.empty_like(x_log)
    x_phys[perm] = x_log
    res = _rand_rows(R, C, 15, torch.float32)
    outer = _rand_rows(R, C, 16, torch.float32)
    pool = pool_np(case.pool.clone())
    got = res.copy()
    oracle.cconv_update_fused(x_phys, pool, to_np(case.w), to_np(case.bias),
                              to_np(case.spec_state_idx), n_spec, to_np(case.num_accepted),
                              to_np(case.spec_has_init), W, D, case.act, got, outer, perm)
    S = (W - 1) * D
    pool0 = pool_np(case.pool)
    want = res.astype(np.float64).copy()
    for s in range(R // q):
        slot = int(case.spec_state_idx[s])
        hi = case.spec_has_init
        h = slot >= 0 and (hi is None or int(hi[s]) != 0)
        off = int(case.num_accepted[s]) - 1
        B = pool0[slot].astype(np.float64) if h else np.zeros((C, pool0.shape[2]))
        y = conv_ref(B[:, off:off + S], x_log[s * q:(s + 1) * q].astype(np.float64),
                     to_np(case.w).astype(np.float64), to_np(case.bias).astype(np.float64),
                     D, case.act)
        for i in range(q):
            p = perm[s * q + i]
            want[p] = res[p] + y[i] + outer[p]
    assert np.abs(got - want).max() <= 1e-5


@pytest.mark.parametrize("n_spec", [0, 3])
def test_fused_update_reduces_to_plain(n_spec):
    case = _case(905, torch.bfloat16, lens=(), W=4, D=3, n_spec=n_spec, spec=7)
    x = to_np(case.x_spec)
    na = to_np(case.num_accepted) if n_spec else None
    out = np.zeros_like(x)
    pool_a = pool_np(case.pool.clone())
    oracle.cconv_update(x, pool_a, to_np(case.w), to_np(case.bias), to_np(case.spec_state_idx),
                        n_spec, na, to_np(case.spec_has_init), 4, 3, case.act, out)
    res = np.zeros_like(x)
    pool_b = pool_np(case.pool.clone())
    oracle.cconv_update_fused(x, pool_b, to_np(case.w), to_np(case.bias),
                              to_np(case.spec_state_idx), n_spec, na,
                              to_np(case.spec_has_init), 4, 3, case.act, res)
    assert np.array_equal(res, out)
    assert np.array_equal(pool_a, pool_b)


def test_fused_rejects_row_index_outside_rows():
    case = _case(906, torch.float32)
    T, C = case.x.shape
    idx = np.arange(T, dtype=np.int32)
    idx[3] = T                                            # one past the last row
    with pytest.raises(ValueError):
        oracle.cconv_fwd_varlen_fused(to_np(case.x), to_np(case.w), to_np(case.bias),
                                      pool_np(case.pool.clone()), to_np(case.state_idx),
                                      to_np(case.cu_seqlens), to_np(case.has_init), case.width,
                                      case.dilation, case.act, np.zeros((T, C), np.float32),
                                      None, idx)


# ---- prefill checkpoint export ----------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("layout", ["DS", "SD"])
def test_checkpoint_equals_state_after_prefilling_to_the_offset(dtype, layout):
    """The window exported at offset k is the state a prefill of the request's
    first k tokens leaves in the pool (whatever its history, since k >= S)."""
    W, D = 4, 3
    S = (W - 1) * D
    lens = [40, 9, 25]
    case = synth.depthwise_case(907, CPU, lens=lens, C=16, width=W, dilation=D, act=1,
                                dtype=dtype, w_std=0.5, layout=layout, num_slots=12)
    cu = to_np(case.cu_seqlens)
    cks = [(0, 9), (0, 27), (0, 40), (1, 9), (2, 18)]
    slots = [6, 7, 8, 9, 10]
    pool = pool_np(case.pool.clone())
    oracle.cconv_checkpoint_export(to_np(case.x), pool, [c[0] for c in cks],
                                   [c[1] for c in cks], slots, cu, W, D)
    for (s, k), d in zip(cks, slots):
        x_pre = np.ascontiguousarray(to_np(case.x)[cu[s]:cu[s] + k])
        p2 = pool_np(case.pool.clone())
        oracle.cconv_fwd_varlen(x_pre, to_np(case.w), None, p2, np.array([d], np.int32),
                                np.array([0, k], np.int32), np.array([1], np.uint8), W, D, 1,
                                np.zeros_like(x_pre))
        assert np.array_equal(pool[d, :, :S], p2[d, :, :S])
    untouched = [i for i in range(pool.shape[0]) if i not in slots]
    assert np.array_equal(pool[untouched], pool_np(case.pool)[untouched])


def test_checkpoint_follows_token_indices_and_rejects_bad_offsets():
    W, D = 3, 2
    S = (W - 1) * D
    case = synth.depthwise_case(908, CPU, lens=[12, 7], C=8, width=W, dilation=D, act=0,
                                dtype=torch.float32, w_std=0.5, num_slots=4)
    T = case.num_tokens
    perm = np.random.default_rng(9).permutation(T).astype(np.int32)
    xp = np.empty_like(to_np(case.x))
    xp[perm] = to_np(case.x)
    cu = to_np(case.cu_seqlens)
    p1 = pool_np(case.pool.clone())
    p2 = pool_np(case.pool.clone())
    oracle.cconv_checkpoint_export(to_np(case.x), p1, [0, 1], [8, 7], [2, 3], cu, W, D)
    oracle.cconv_checkpoint_export(xp, p2, [0, 1], [8, 7], [2, 3], cu, W, D, perm)
    assert np.array_equal(p1, p2)
    # slicing by hand
    assert np.array_equal(p1[2, :, :S].T, to_np(case.x)[8 - S:8])
    for bad in ([0], [S - 1], [2]), ([1], [8], [2]), ([2], [4], [2]):
        with pytest.raises(ValueError):
            oracle.cconv_checkpoint_export(to_np(case.x), pool_np(case.pool.clone()), bad[0],
                                           bad[1], bad[2], cu, W, D)


# ---- Zaya q/k residual mix and value assembly -------------------------------

def _torch_project_tail(qk, conv, v_cur, dprev, Hq, Hkv):
    """The tail of ZayaCCA.project on the Zaya page, run with torch's own ops in
    the tensors' dtype (an implementation independent of the oracle's C)."""
    T = qk.shape[0]
    hd = qk.shape[1] // (Hq + Hkv)
    qdim, kvg = Hq * hd, Hq // Hkv
    heads = (T, -1, hd)
    queries, keys = qk[:, :qdim], qk[:, qdim:]
    query_residual = 0.5 * (queries.reshape(heads)
                            + keys.reshape(heads).repeat_interleave(kvg, dim=1))
    key_residual = query_residual.reshape(T, -1, kvg, hd).mean(dim=2)
    query = conv[:, :qdim].reshape(heads) + query_residual
    key = conv[:, qdim:].reshape(heads) + key_residual
    value = torch.cat([v_cur, dprev], dim=-1)
    return torch.cat([query, key, value.reshape(heads)], dim=1).flatten(1)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("Hq,Hkv", [(4, 2), (3, 1), (2, 2)])
def test_cca_project_tail_matches_torch(dtype, Hq, Hkv):
    hd, T = 16, 11
    g = torch.Generator().manual_seed(Hq * 10 + Hkv)
    C = (Hq + Hkv) * hd
    qk = torch.randn(T, C, generator=g).to(dtype)
    conv = torch.randn(T, C, generator=g).to(dtype)
    v_cur = torch.randn(T, Hkv * hd // 2, generator=g).to(dtype)
    dprev = torch.randn(T, Hkv * hd // 2, generator=g).to(dtype)
    want = _torch_project_tail(qk, conv, v_cur, dprev, Hq, Hkv)
    out = np.zeros((T, Hq * hd + 2 * Hkv * hd), dtype=to_np(qk).dtype)
    oracle.cca_project_epilogue(to_np(qk), to_np(conv), to_np(v_cur), to_np(dprev), Hq, Hkv,
                                out)
    got, ref = _f64(out), _f64(to_np(want))
    if dtype == torch.float32:
        assert np.abs(got - ref).max() <= 1e-6
    else:
        # bf16 results agree except where the fp32 mean's summation order flips a rounding
        ulp = np.abs(ref) * 2.0 ** -7 + 1e-30
        assert np.all(np.abs(got - ref) <= ulp)
    vcols = slice(Hq * hd + Hkv * hd, None)
    assert np.array_equal(out[:, vcols], to_np(torch.cat([v_cur, dprev], dim=-1)))


def test_cca_project_tail_one_query_head_per_kv_head():
    """With one query head per kv head the key residual is the query residual of
    the same head: key = conv_k + 0.5 * (q + k) as well."""
    Hq = Hkv = 3
    hd, T = 8, 5
    g = torch.Generator().manual_seed(3)
    qk = torch.randn(T, 2 * Hq * hd, generator=g)
    conv = torch.randn(T, 2 * Hq * hd, generator=g)
    v = torch.zeros(T, Hkv * hd // 2)
    out = np.zeros((T, 3 * Hq * hd), np.float32)
    oracle.cca_project_epilogue(to_np(qk), to_np(conv), to_np(v), to_np(v), Hq, Hkv, out)
    res = 0.5 * (qk[:, :Hq * hd] + qk[:, Hq * hd:])
    assert np.allclose(out[:, :Hq * hd], to_np(conv[:, :Hq * hd] + res), atol=1e-6)
    assert np.allclose(out[:, Hq * hd:2 * Hq * hd], to_np(conv[:, Hq * hd:] + res), atol=1e-6)
