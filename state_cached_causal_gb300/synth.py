"""Seeded synthetic inputs for the state-cached causal short convolution.

This module only draws random tensors and batch metadata; it holds none of the
convolution's arithmetic, so both the oracle tests and the CUDA path can use
it. Every generator takes a seed and a device; the same seed on the same
device gives the same tensors.

Workloads (one per batch shape the hybrid layers serve):

* ``single_prefill``  -- 1 sequence x 32 tokens, 64 channels, fp32, width 4,
  dilation 1, no bias, no activation; w ~ N(0, 0.25^2), x ~ N(0, 1); one
  zero-initialised state slot.
* ``gdn_decode``      -- 64 requests x 1 token, 8192 channels, bf16, width 4,
  bias ~ N(0, 0.02^2), SiLU; pool 256 x 8192 x 3 ~ N(0, 1); state indices are
  the first 64 entries of a seeded permutation of the pool.
* ``gdn_mixed``       -- 128 one-token decodes then 16 prefills with lengths
  uniform in [1, 2048]; 8192 channels, bf16, width 4, bias, SiLU;
  has_initial_state ~ Bernoulli(0.5) for prefills; pool of 512 slots.
* ``zaya_cca``        -- 256 decodes then 8 prefills x 4096 tokens; 16 q + 4 kv
  heads of 128 -> 2560 q/k channels; depthwise width 2 then grouped width 2
  with 20 groups of 128; 256 delayed v channels; weights ~ N(0, 1/fan_in),
  biases ~ N(0, 0.02^2); pool of 512 slots.
* ``ple_spec``        -- 32 prefills x 2048 tokens then 512 speculative
  requests x (1 + 3) tokens; 16384 channels, bf16, width 4, dilation 3, no
  bias, SiLU, w ~ N(0, 0.1^2); pool of 1024 slots x 12 columns;
  num_accepted ~ U{1..4}.

Pools are returned as a ``[slot, channel, column]`` view over storage laid out
either channel-first ("DS", ``[slots, C, cap]`` contiguous) or column-first
("SD", ``[slots, cap, C]`` contiguous), the two cache layouts the layers use.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

SEED_BASE = 1000
WORKLOADS = ("single_prefill", "gdn_decode", "gdn_mixed", "zaya_cca", "ple_spec")


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std, g, device, dtype):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def make_pool(num_slots, C, cap, dtype, g, device, layout="DS", zero=False):
    """Conv-state pool; returns the [slot, channel, column] view."""
    if layout == "DS":
        shape = (num_slots, C, cap)
    elif layout == "SD":
        shape = (num_slots, cap, C)
    else:
        raise ValueError(layout)
    if zero:
        store = torch.zeros(shape, device=device, dtype=dtype)
    else:
        store = normal(shape, 1.0, g, device, dtype)
    return store if layout == "DS" else store.transpose(1, 2)


def randperm(n, g, device):
    return torch.randperm(n, generator=g, device=device)


def cu_from_lens(lens, device):
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    if len(lens):
        cu[1:] = torch.cumsum(torch.as_tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return cu.to(device)


@dataclass
class DepthwiseCase:
    """Inputs of one varlen (prefill/decode) call and/or one spec call."""
    C: int
    width: int
    dilation: int
    act: int
    dtype: torch.dtype
    w: torch.Tensor
    bias: torch.Tensor | None
    pool: torch.Tensor
    # varlen part
    x: torch.Tensor | None = None
    state_idx: torch.Tensor | None = None
    cu_seqlens: torch.Tensor | None = None
    has_init: torch.Tensor | None = None
    # spec part
    x_spec: torch.Tensor | None = None
    spec_state_idx: torch.Tensor | None = None
    num_accepted: torch.Tensor | None = None
    n_spec: int = 0
    spec_has_init: torch.Tensor | None = None
    meta: dict = field(default_factory=dict)

    @property
    def num_tokens(self):
        return 0 if self.x is None else int(self.x.shape[0])


@dataclass
class CCACase:
    Cqk: int
    groups: int
    t0: int
    t1: int
    Dv: int
    dtype: torch.dtype
    qk: torch.Tensor
    w_dw: torch.Tensor
    b_dw: torch.Tensor | None
    w_gr: torch.Tensor
    b_gr: torch.Tensor | None
    delayed: torch.Tensor
    delayed_init: torch.Tensor
    pool: torch.Tensor
    delayed_state: torch.Tensor
    state_idx: torch.Tensor
    cu_seqlens: torch.Tensor
    has_init: torch.Tensor
    meta: dict = field(default_factory=dict)


def depthwise_case(seed, device, *, lens, C, width, dilation, act, dtype, w_std,
                   bias_std=None, num_slots=None, cap=None, layout="DS",
                   has_init="bernoulli", decode_prefix=0, zero_pool=False,
                   spec_requests=0, n_spec=0, padding_every=0):
    """Generic varlen (+ optional spec) case.

    ``lens``: lengths of the varlen sequences (the first ``decode_prefix`` of
    them are one-token decodes whose history is always their slot). ``has_init``:
    "bernoulli" (p = 0.5 for non-decodes), "all", "none". ``spec_requests``
    speculative requests with q = 1 + n_spec tokens each use slots disjoint
    from the varlen sequences. ``padding_every`` > 0 marks every k-th varlen
    sequence as a padding row (state index -1).
    """
    g = generator(seed, device)
    S = (width - 1) * dilation
    if cap is None:
        cap = S + n_spec
    B = len(lens)
    if num_slots is None:
        num_slots = max(1, 2 * (B + spec_requests))
    assert num_slots >= B + spec_requests
    w = normal((C, width), w_std, g, device, dtype)
    bias = normal((C,), bias_std, g, device, dtype) if bias_std is not None else None
    pool = make_pool(num_slots, C, cap, dtype, g, device, layout, zero=zero_pool)
    perm = randperm(num_slots, g, device).to(torch.int32)
    case = DepthwiseCase(C=C, width=width, dilation=dilation, act=act, dtype=dtype, w=w,
                         bias=bias, pool=pool, n_spec=n_spec)
    T = int(sum(lens))
    if B:
        case.x = normal((T, C), 1.0, g, device, dtype)
        sidx = perm[:B].clone()
        if padding_every:
            sidx[padding_every - 1::padding_every] = -1
        case.state_idx = sidx
        case.cu_seqlens = cu_from_lens(lens, device)
        if has_init == "all":
            hi = torch.ones(B, dtype=torch.uint8, device=device)
        elif has_init == "none":
            hi = torch.zeros(B, dtype=torch.uint8, device=device)
        else:
            hi = (torch.rand(B, generator=g, device=device) < 0.5).to(torch.uint8)
            hi[:decode_prefix] = 1
        case.has_init = hi
    if spec_requests:
        q = 1 + n_spec
        case.x_spec = normal((spec_requests * q, C), 1.0, g, device, dtype)
        case.spec_state_idx = perm[B:B + spec_requests].clone()
        case.num_accepted = torch.randint(1, q + 1, (spec_requests,), generator=g,
                                          device=device, dtype=torch.int32)
    case.meta = dict(lens=list(lens), T=T, S=S, cap=cap, num_slots=num_slots,
                     layout=layout, decode_prefix=decode_prefix)
    return case


def cca_case(seed, device, *, lens, decode_prefix, Hq=16, Hkv=4, head_dim=128, t0=2, t1=2,
             dtype=torch.bfloat16, num_slots=None, layout="DS", has_init="bernoulli",
             bias=True, padding_every=0, zero_pool=False):
    g = generator(seed, device)
    G = Hq + Hkv
    Cqk = G * head_dim
    Dv = Hkv * head_dim // 2
    n = t0 + t1 - 2
    B = len(lens)
    if num_slots is None:
        num_slots = max(1, 2 * B)
    T = int(sum(lens))
    qk = normal((T, Cqk), 1.0, g, device, dtype)
    w_dw = normal((Cqk, t0), (1.0 / t0) ** 0.5, g, device, dtype)
    b_dw = normal((Cqk,), 0.02, g, device, dtype) if bias else None
    w_gr = normal((Cqk, head_dim, t1), (1.0 / (head_dim * t1)) ** 0.5, g, device, dtype)
    b_gr = normal((Cqk,), 0.02, g, device, dtype) if bias else None
    delayed = normal((T, Dv), 1.0, g, device, dtype)
    delayed_init = normal((Dv,), 0.02, g, device, dtype)
    pool = make_pool(num_slots, Cqk, max(n, 1), dtype, g, device, layout, zero=zero_pool)
    if zero_pool:
        dstate = torch.zeros((num_slots, Dv), device=device, dtype=dtype)
    else:
        dstate = normal((num_slots, Dv), 1.0, g, device, dtype)
    perm = randperm(num_slots, g, device).to(torch.int32)
    sidx = perm[:B].clone()
    if padding_every:
        sidx[padding_every - 1::padding_every] = -1
    if has_init == "all":
        hi = torch.ones(B, dtype=torch.uint8, device=device)
    elif has_init == "none":
        hi = torch.zeros(B, dtype=torch.uint8, device=device)
    else:
        hi = (torch.rand(B, generator=g, device=device) < 0.5).to(torch.uint8)
        hi[:decode_prefix] = 1
    return CCACase(Cqk=Cqk, groups=G, t0=t0, t1=t1, Dv=Dv, dtype=dtype, qk=qk, w_dw=w_dw,
                   b_dw=b_dw, w_gr=w_gr, b_gr=b_gr, delayed=delayed,
                   delayed_init=delayed_init, pool=pool, delayed_state=dstate,
                   state_idx=sidx, cu_seqlens=cu_from_lens(lens, device), has_init=hi,
                   meta=dict(lens=list(lens), T=T, n=n, num_slots=num_slots, layout=layout,
                             decode_prefix=decode_prefix))


# ---- the five named workloads ------------------------------------------------

def _seed(name):
    return SEED_BASE + WORKLOADS.index(name)


def single_prefill(device, has_init="none"):
    return depthwise_case(_seed("single_prefill"), device, lens=[32], C=64, width=4,
                          dilation=1, act=0, dtype=torch.float32, w_std=0.25,
                          num_slots=1, has_init=has_init, zero_pool=True)


def gdn_decode(device):
    return depthwise_case(_seed("gdn_decode"), device, lens=[], C=8192, width=4, dilation=1,
                          act=1, dtype=torch.bfloat16, w_std=0.5, bias_std=0.02,
                          num_slots=256, spec_requests=64, n_spec=0)


def gdn_mixed_lens(seed=None):
    g = torch.Generator()
    g.manual_seed(_seed("gdn_mixed") if seed is None else seed)
    pre = torch.randint(1, 2049, (16,), generator=g).tolist()
    return [1] * 128 + pre


def gdn_mixed(device):
    return depthwise_case(_seed("gdn_mixed"), device, lens=gdn_mixed_lens(), C=8192,
                          width=4, dilation=1, act=1, dtype=torch.bfloat16, w_std=0.5,
                          bias_std=0.02, num_slots=512, decode_prefix=128)


def zaya_cca(device):
    return cca_case(_seed("zaya_cca"), device, lens=[1] * 256 + [4096] * 8,
                    decode_prefix=256, num_slots=512)


def ple_spec(device):
    return depthwise_case(_seed("ple_spec"), device, lens=[2048] * 32, C=16384, width=4,
                          dilation=3, act=1, dtype=torch.bfloat16, w_std=0.1,
                          num_slots=1024, spec_requests=512, n_spec=3)


def workload(name, device):
    return {"single_prefill": single_prefill, "gdn_decode": gdn_decode,
            "gdn_mixed": gdn_mixed, "zaya_cca": zaya_cca, "ple_spec": ple_spec}[name](device)
