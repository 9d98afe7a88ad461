"""cca_qk_conv_noalloc on the GPU: the CCA entry point that allocates nothing.

Some callers may not allocate device memory while they call this library: a
host framework that owns all device memory and hands its kernels only inputs
and outputs (an inference engine's plugin), code recording a CUDA graph, a
latency-critical serving loop. For them cca_qk_conv_noalloc keeps the kernel's
scratch -- the two counters of its dynamic work split -- in a fixed array
inside the library instead of anywhere the caller would have to provide.

The test calls it through the C ABI twice in a row, a mixed prefill/decode
batch and then a one-token decode step that continues from the state the
first call wrote, and checks each call against cca_qk_conv on the same inputs:
q/k outputs within the bf16 tolerance of the other CCA tests, the delayed half
of v and both states bit for bit, no device error. The second call shows that
what the first one left in the shared scratch does not carry over.

(The file name makes pytest collect it last.)
"""
import pytest
import torch

from state_cached_causal_gb300 import ops, synth
from tests._util import pool_np, to_np
from tests.test_parity_depthwise import assert_bits_equal, assert_out_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _run(fn, inputs, pool, dstate):
    """One call of `fn` (cca_qk_conv or cca_qk_conv_noalloc) on the inputs,
    updating pool and dstate in place; returns (out, delayed_prev, dev_err)."""
    c = inputs
    out = torch.zeros_like(c["qk"])
    dprev = torch.zeros_like(c["delayed"])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    fn(c["qk"], c["w_dw"], c["b_dw"], c["w_gr"], c["b_gr"], c["groups"], 2, 2, c["delayed"],
       c["delayed_init"], pool, dstate, c["state_idx"], c["cu_seqlens"], c["has_init"], out,
       dprev, dev_err=err)
    return out, dprev, err


def _compare(got, want, pool_g, pool_w, ds_g, ds_w, what):
    out_g, dprev_g, err_g = got
    out_w, dprev_w, err_w = want
    torch.cuda.synchronize()
    assert int(err_g.item()) == 0 and int(err_w.item()) == 0, what
    assert_out_close(to_np(out_g), to_np(out_w), torch.bfloat16, f"{what}: qk")
    assert_bits_equal(to_np(dprev_g), to_np(dprev_w), f"{what}: delayed_prev")
    assert_bits_equal(pool_np(pool_g), pool_np(pool_w), f"{what}: conv_state")
    assert_bits_equal(to_np(ds_g), to_np(ds_w), f"{what}: delayed_state")


def test_noalloc_matches_cca_qk_conv_on_two_calls_in_a_row():
    # Zaya heads (16 q + 4 kv of 128: 20 groups); 64 decodes and three
    # prefills, 4264 tokens: 34 token tiles x 20 groups = 680 work units, so
    # the work split has a static and a dynamic (counter-driven) part
    lens = [1] * 64 + [1500, 2000, 700]
    case = synth.cca_case(9100, DEV, lens=lens, decode_prefix=64, num_slots=160)
    first = dict(qk=case.qk, w_dw=case.w_dw, b_dw=case.b_dw, w_gr=case.w_gr, b_gr=case.b_gr,
                 groups=case.groups, delayed=case.delayed, delayed_init=case.delayed_init,
                 state_idx=case.state_idx, cu_seqlens=case.cu_seqlens, has_init=case.has_init)
    pool_w, ds_w = case.pool.clone(), case.delayed_state.clone()
    pool_g, ds_g = case.pool.clone(), case.delayed_state.clone()
    want = _run(ops.cca_qk_conv, first, pool_w, ds_w)
    got = _run(ops.cca_qk_conv_noalloc, first, pool_g, ds_g)
    _compare(got, want, pool_g, pool_w, ds_g, ds_w, "first call")

    # second call: one new token per request, continuing from the state each
    # entry point wrote in the first call
    B = len(lens)
    g = torch.Generator(device=DEV).manual_seed(9101)
    second = dict(first)
    second["qk"] = torch.randn(B, case.Cqk, generator=g, device=DEV).to(torch.bfloat16)
    second["delayed"] = torch.randn(B, case.Dv, generator=g, device=DEV).to(torch.bfloat16)
    second["cu_seqlens"] = torch.arange(B + 1, dtype=torch.int32, device=DEV)
    second["has_init"] = torch.ones(B, dtype=torch.uint8, device=DEV)
    want = _run(ops.cca_qk_conv, second, pool_w, ds_w)
    got = _run(ops.cca_qk_conv_noalloc, second, pool_g, ds_g)
    _compare(got, want, pool_g, pool_w, ds_g, ds_w, "second call")
