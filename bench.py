#!/usr/bin/env python
"""Benchmark of the state-cached causal short convolution on GB300.

One step = one pass of the whole hot path over one batch of each serving
shape, all through the C ABI of libcconv.so:
  gdn_decode  64 requests x 1 token x 8192 channels        (cconv_update)
  gdn_mixed   128 decodes + 16 prefills (seeded), 8192 ch   (cconv_fwd_varlen)
  zaya_cca    256 decodes + 8 x 4096 prefill, 2560 q/k ch   (cca_qk_conv)
  ple_spec    32 x 2048 prefill + 512 x 4 spec, 16384 ch    (cconv_fwd_varlen
              and cconv_update with 3 speculative tokens)
Every input is seeded and synthetic and resident in HBM before timing; the
step moves about 5.7 GB, far more than the 129 MB L2, so no flush is needed.
`value` is tokens*channels processed per second (whole job) over K replays of
the step captured as one CUDA graph (the same launches as the stream path),
`per_call` the per-launch times from a second pass launched on the stream with
events around every launch, `e2e` the same metric with the inputs copied from
pinned host memory and the outputs copied back inside the timed region. `roofline` reports the dominant kernel's
achieved HBM bandwidth (algorithmic bytes / CUDA-event duration) against the
measured copy bandwidth. `cpu_baseline` times the plain-C oracle on a bounded
channel/request sample of the same step on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload hybrid_step|ple_fused|ple_prefill_small|cca_small|...]
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("causal-conv G(tokens·channels)/s and achieved HBM GB/s vs GB300 peak, 1 GPU")
UNIT = "G(tokens*channels)/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0    # GB300 HBM3e data-sheet bandwidth (context beside the measured peak)
LEAD_CYCLES = 2_000_000     # device-side wait (about 1 ms) queued ahead of a timed region


# ---- workloads ---------------------------------------------------------------

class Call:
    """One launch of the hot path with its algorithmic byte/flop counts."""

    def __init__(self, name, kernel, fn, units, nbytes, flops=0.0, h2d=None, d2h=None):
        self.name, self.kernel, self.fn = name, kernel, fn
        self.units, self.bytes, self.flops = units, nbytes, flops
        self.h2d = h2d or []     # (device tensor, pinned host tensor): inputs
        self.d2h = d2h or []     # (device tensor, pinned host tensor): outputs


def _e(t):
    return t.element_size()


def depthwise_calls(name, case, dev_err):
    from state_cached_causal_gb300 import ops
    calls = []
    e, C, W, S = _e(case.w), case.C, case.width, case.meta["S"]
    es = _e(case.pool)                                # the pool's own storage type
    wbytes = C * W * e + (C * e if case.bias is not None else 0)
    if case.x is not None:
        out = torch.empty_like(case.x)
        hi = case.has_init.to(torch.int64).cpu()
        valid = (case.state_idx.cpu() >= 0).to(torch.int64)
        nread = int((hi * valid).sum())
        nwrite = int(valid.sum())
        T = case.num_tokens
        nbytes = 2 * T * C * e + wbytes + C * es * S * (nread + nwrite)

        def f(case=case, out=out):
            ops.cconv_fwd_varlen(case.x, case.w, case.bias, case.pool, case.state_idx,
                                 case.cu_seqlens, case.has_init, case.width, case.dilation,
                                 case.act, out, dev_err=dev_err)
        calls.append(Call(f"{name}.fwd_varlen", "cconv_fwd_varlen", f, T * C, nbytes,
                          h2d=[case.x], d2h=[out]))
    if case.x_spec is not None:
        out = torch.empty_like(case.x_spec)
        R = int(case.spec_state_idx.numel())
        q = 1 + case.n_spec
        cols_w = case.meta["cap"] if case.n_spec else S
        nbytes = 2 * R * q * C * e + wbytes + R * C * es * (S + cols_w)
        na = case.num_accepted if case.n_spec else None

        def g(case=case, out=out, na=na):
            ops.cconv_update(case.x_spec, case.pool, case.w, case.bias, case.spec_state_idx,
                             case.n_spec, na, case.spec_has_init, case.width, case.dilation,
                             case.act, out, dev_err=dev_err)
        calls.append(Call(f"{name}.update", "cconv_update", g, R * q * C, nbytes,
                          h2d=[case.x_spec], d2h=[out]))
    return calls


def fused_calls(name, case, dev_err, seed=2100):
    """The PLE layer's dispatch on one mixed batch kept in arrival order: the
    spec requests (cconv_update_fused) and the prefills (cconv_fwd_varlen_fused)
    read x and update residual (+ outer residual) at their own physical rows,
    found through token_indices."""
    from state_cached_causal_gb300 import ops
    e, C, W, S = _e(case.w), case.C, case.width, case.meta["S"]
    q = 1 + case.n_spec
    lens_p = (case.cu_seqlens[1:] - case.cu_seqlens[:-1]).cpu().tolist()
    Rs = int(case.spec_state_idx.numel())
    blocks = [("p", i, L) for i, L in enumerate(lens_p)] + [("s", i, q) for i in range(Rs)]
    g = torch.Generator().manual_seed(seed)
    order = torch.randperm(len(blocks), generator=g).tolist()
    T, Rtot = case.num_tokens, case.num_tokens + Rs * q
    idx_p = torch.empty(T, dtype=torch.int32)
    idx_s = torch.empty(Rs * q, dtype=torch.int32)
    cu = case.cu_seqlens.cpu().tolist()
    row = 0
    for k in order:
        kind, i, L = blocks[k]
        if kind == "p":
            idx_p[cu[i]:cu[i] + L] = torch.arange(row, row + L, dtype=torch.int32)
        else:
            idx_s[i * q:(i + 1) * q] = torch.arange(row, row + q, dtype=torch.int32)
        row += L
    idx_p, idx_s = idx_p.to(case.x.device), idx_s.to(case.x.device)
    x = torch.empty(Rtot, C, dtype=case.x.dtype, device=case.x.device)
    x[idx_p.long()] = case.x
    x[idx_s.long()] = case.x_spec
    case.x, case.x_spec = None, None                  # only the physical copy stays
    res = torch.randn(Rtot, C, device=x.device).to(x.dtype)
    outer = torch.randn(Rtot, C, device=x.device).to(x.dtype)
    wbytes = C * W * e
    hi = case.has_init.to(torch.int64).cpu()
    valid = (case.state_idx.cpu() >= 0).to(torch.int64)
    nread, nwrite = int((hi * valid).sum()), int(valid.sum())
    nb_p = 4 * T * C * e + wbytes + C * e * S * (nread + nwrite) + 4 * T
    nb_s = 4 * Rs * q * C * e + wbytes + Rs * C * e * (S + case.meta["cap"]) + 4 * Rs * q

    def f(case=case):
        ops.cconv_fwd_varlen_fused(x, case.w, case.bias, case.pool, case.state_idx,
                                   case.cu_seqlens, case.has_init, W, case.dilation, case.act,
                                   res, outer, idx_p, dev_err=dev_err, num_tokens=T)

    def u(case=case):
        ops.cconv_update_fused(x, case.pool, case.w, case.bias, case.spec_state_idx,
                               case.n_spec, case.num_accepted, case.spec_has_init, W,
                               case.dilation, case.act, res, outer, idx_s, dev_err=dev_err)
    return [Call(f"{name}.update_fused", "cconv_update_fused", u, Rs * q * C, nb_s,
                 h2d=[x, res, outer], d2h=[res]),
            Call(f"{name}.fwd_varlen_fused", "cconv_fwd_varlen_fused", f, T * C, nb_p)]


def cca_calls(name, cc, dev_err):
    from state_cached_causal_gb300 import ops
    out = torch.empty_like(cc.qk)
    dprev = torch.empty_like(cc.delayed)
    e, T, Cqk, Dv, n = _e(cc.qk), int(cc.qk.shape[0]), cc.Cqk, cc.Dv, cc.meta["n"]
    es = _e(cc.pool)
    hi = cc.has_init.to(torch.int64).cpu()
    valid = (cc.state_idx.cpu() >= 0).to(torch.int64)
    nread, nwrite = int((hi * valid).sum()), int(valid.sum())
    wbytes = sum(_e(t) * t.numel() for t in (cc.w_dw, cc.b_dw, cc.w_gr, cc.b_gr)
                 if t is not None)
    nbytes = (2 * T * Cqk * e + 2 * T * Dv * e + wbytes + Dv * e
              + (nread + nwrite) * (n * Cqk * es + Dv * es))
    flops = 2.0 * T * Cqk * (Cqk // cc.groups) * cc.t1 + 2.0 * (T + 1) * Cqk * cc.t0

    def f(cc=cc, out=out, dprev=dprev):
        ops.cca_qk_conv(cc.qk, cc.w_dw, cc.b_dw, cc.w_gr, cc.b_gr, cc.groups, cc.t0, cc.t1,
                        cc.delayed, cc.delayed_init, cc.pool, cc.delayed_state, cc.state_idx,
                        cc.cu_seqlens, cc.has_init, out, dprev, dev_err=dev_err)
    return [Call(f"{name}.cca_qk_conv", "cca_qk_conv", f, T * Cqk, nbytes, flops,
                 h2d=[cc.qk, cc.delayed], d2h=[out, dprev])]


def cca_fused_calls(name, cc, Hq, dev_err):
    """cca_qk_conv_fused: the conv plus ZayaCCA.project's residual mix and value
    assembly into the [query | key | value] output rows."""
    from state_cached_causal_gb300 import ops
    e, T, Cqk, Dv, n = _e(cc.qk), int(cc.qk.shape[0]), cc.Cqk, cc.Dv, cc.meta["n"]
    v_cur = torch.randn(T, Dv, device=cc.qk.device).to(cc.qk.dtype)
    out = torch.empty(T, Cqk + 2 * Dv, device=cc.qk.device, dtype=cc.qk.dtype)
    hi = cc.has_init.to(torch.int64).cpu()
    valid = (cc.state_idx.cpu() >= 0).to(torch.int64)
    nread, nwrite = int((hi * valid).sum()), int(valid.sum())
    wbytes = sum(_e(t) * t.numel() for t in (cc.w_dw, cc.b_dw, cc.w_gr, cc.b_gr)
                 if t is not None)
    # qk, delayed and v_current read once; the [query | key | value] rows written once
    nbytes = (T * Cqk * e + 2 * T * Dv * e + T * (Cqk + 2 * Dv) * e + wbytes + Dv * e
              + (nread + nwrite) * (n * Cqk * e + Dv * e))
    flops = 2.0 * T * Cqk * (Cqk // cc.groups) * cc.t1 + 2.0 * (T + 1) * Cqk * cc.t0

    def f(cc=cc):
        ops.cca_qk_conv_fused(cc.qk, cc.w_dw, cc.b_dw, cc.w_gr, cc.b_gr, cc.groups, Hq, cc.t0,
                              cc.t1, cc.delayed, cc.delayed_init, v_cur, cc.pool,
                              cc.delayed_state, cc.state_idx, cc.cu_seqlens, cc.has_init, out,
                              dev_err=dev_err)
    return [Call(f"{name}.cca_qk_conv_fused", "cca_qk_conv_fused", f, T * Cqk, nbytes, flops,
                 h2d=[cc.qk, cc.delayed, v_cur], d2h=[out])]


def build_workload(name, dev, dev_err):
    from state_cached_causal_gb300 import synth
    if name == "hybrid_step":
        calls = []
        calls += depthwise_calls("gdn_decode", synth.gdn_decode(dev), dev_err)
        calls += depthwise_calls("gdn_mixed", synth.gdn_mixed(dev), dev_err)
        calls += cca_calls("zaya_cca", synth.zaya_cca(dev), dev_err)
        calls += depthwise_calls("ple_spec", synth.ple_spec(dev), dev_err)
        desc = ("hybrid_step: gdn_decode 64x1 tok x 8192 ch (cconv_update) + gdn_mixed "
                "128 decodes + 16 prefills U[1,2048] x 8192 ch (cconv_fwd_varlen) + "
                "zaya_cca 256 decodes + 8x4096 prefill, 20 groups x 128 ch, t0=t1=2 "
                "(cca_qk_conv) + ple_spec 32x2048 prefill + 512x(1+3) spec x 16384 ch, "
                "width 4 dilation 3 (cconv_fwd_varlen + cconv_update)")
        return calls, desc
    if name == "hybrid_step_f32state":
        # the same step with fp32 conv-state pools (and CCA delayed state) under
        # the bf16 activations: random fp32 state, so both conversions are live
        def f32(case, seed):
            g = torch.Generator(device=dev).manual_seed(seed)
            case.pool = torch.randn(case.pool.shape, generator=g, device=dev)
            if hasattr(case, "delayed_state"):
                case.delayed_state = torch.randn(case.delayed_state.shape, generator=g,
                                                 device=dev)
            return case
        calls = []
        calls += depthwise_calls("gdn_decode", f32(synth.gdn_decode(dev), 1), dev_err)
        calls += depthwise_calls("gdn_mixed", f32(synth.gdn_mixed(dev), 2), dev_err)
        calls += cca_calls("zaya_cca", f32(synth.zaya_cca(dev), 3), dev_err)
        calls += depthwise_calls("ple_spec", f32(synth.ple_spec(dev), 4), dev_err)
        return calls, ("hybrid_step_f32state: the hybrid_step batches with fp32 conv-state "
                       "pools (channel-first) and fp32 CCA delayed state under bf16 "
                       "activations")
    # small single-kernel cases for profiling (a few GB at most, > L2)
    if name == "ple_prefill_small":
        case = synth.depthwise_case(2001, dev, lens=[2048] * 8, C=16384, width=4, dilation=3,
                                    act=1, dtype=torch.bfloat16, w_std=0.1, num_slots=64)
        return depthwise_calls("ple_prefill_small", case, dev_err), \
            "ple prefill 8x2048 tok x 16384 ch, width 4 dilation 3"
    if name == "ple_spec_small":
        case = synth.depthwise_case(2002, dev, lens=[], C=16384, width=4, dilation=3, act=1,
                                    dtype=torch.bfloat16, w_std=0.1, num_slots=1024,
                                    spec_requests=512, n_spec=3)
        return depthwise_calls("ple_spec_small", case, dev_err), \
            "ple spec 512x(1+3) tok x 16384 ch"
    if name == "ple_spec_small_f32state":
        case = synth.depthwise_case(2002, dev, lens=[], C=16384, width=4, dilation=3, act=1,
                                    dtype=torch.bfloat16, w_std=0.1, num_slots=1024,
                                    spec_requests=512, n_spec=3)
        g = torch.Generator(device=dev).manual_seed(2005)
        case.pool = torch.randn(case.pool.shape, generator=g, device=dev)
        return depthwise_calls("ple_spec_small_f32state", case, dev_err), \
            "ple spec 512x(1+3) tok x 16384 ch, fp32 conv-state pool under bf16 activations"
    if name == "gdn_mixed":
        return depthwise_calls("gdn_mixed", synth.gdn_mixed(dev), dev_err), "gdn_mixed"
    if name == "ple_spec":
        return depthwise_calls("ple_spec", synth.ple_spec(dev), dev_err), "ple_spec"
    if name == "gdn_decode":
        return depthwise_calls("gdn_decode", synth.gdn_decode(dev), dev_err), "gdn_decode"
    if name == "cca_small":
        cc = synth.cca_case(2003, dev, lens=[1] * 256 + [4096] * 2, decode_prefix=256,
                            num_slots=512)
        return cca_calls("cca_small", cc, dev_err), "zaya cca 256 decodes + 2x4096"
    if name == "zaya_cca":
        return cca_calls("zaya_cca", synth.zaya_cca(dev), dev_err), "zaya_cca"
    if name == "zaya_fused":
        return cca_fused_calls("zaya_fused", synth.zaya_cca(dev), 16, dev_err), (
            "zaya_fused: the zaya_cca batch through cca_qk_conv_fused (conv + q/k residual "
            "mix + [query | key | value] assembly, 16 q + 4 kv heads)")
    if name == "ple_fused_small":
        case = synth.depthwise_case(2004, dev, lens=[2048] * 8, C=16384, width=4, dilation=3,
                                    act=1, dtype=torch.bfloat16, w_std=0.1, num_slots=256,
                                    spec_requests=128, n_spec=3)
        return fused_calls("ple_fused_small", case, dev_err), \
            "ple fused 8x2048 prefill + 128x(1+3) spec x 16384 ch, random request order"
    if name == "ple_fused":
        return fused_calls("ple_fused", synth.ple_spec(dev), dev_err), (
            "ple_fused: the ple_spec batch (32x2048 prefill + 512x(1+3) spec x 16384 ch, "
            "width 4 dilation 3) in one physical tensor in a random request order, "
            "residual += conv + outer residual through token_indices "
            "(cconv_update_fused + cconv_fwd_varlen_fused)")
    raise SystemExit(f"unknown workload {name}")


# ---- measurement helpers -----------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# Sources that make up each entry point's kernels (a recorded DRAM traffic
# figure stays valid while these files are unchanged).
KERNEL_SOURCES = {
    "cconv_fwd_varlen": ["depthwise.cuh", "depthwise.cu", "depthwise_wide.cu", "common.cuh",
                         "update.cuh"],
    "cconv_update": ["depthwise.cuh", "depthwise.cu", "depthwise_wide.cu", "update_bulk.cuh",
                     "update_bulk.cu", "update_bulk_f32.cu", "update_bulk_wide.cu", "update.cuh",
                     "async.cuh", "common.cuh"],
    "cca_qk_conv": ["cca.cuh", "cca_qk_conv.cu", "async.cuh", "common.cuh"],
    "cca_qk_conv_fused": ["cca.cuh", "cca_fused.cu", "async.cuh", "common.cuh"],
    "cconv_fwd_varlen_fused": ["depthwise.cuh", "depthwise_fused.cu", "depthwise_wide.cu",
                               "common.cuh"],
    "cconv_update_fused": ["depthwise.cuh", "depthwise_fused.cu", "depthwise_wide.cu",
                           "update_bulk.cuh", "update_bulk.cu", "update_bulk_f32.cu",
                           "update_bulk_wide.cu", "update.cuh", "async.cuh", "common.cuh"],
}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    d = os.path.join(ROOT, "state_cached_causal_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES.get(kernel, os.listdir(d))):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch from a committed ncu summary, if it still matches the code."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        rec = d[kernel]
        if rec.get("source_hash") != kernel_source_hash(kernel):
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


# ---- CPU oracle sample ---------------------------------------------------------

# channels (groups for CCA) of each workload in the oracle sample: about 10 s of
# single-core work on the GPU host; `light` is the reference arm's per-step sample
SAMPLE_CHANNELS = {"gdn_decode": 8192, "gdn_mixed": 8192, "zaya_cca": 20, "ple_spec": 12288}
LIGHT_CHANNELS = {"gdn_decode": 512, "gdn_mixed": 64, "zaya_cca": 1, "ple_spec": 64}


def cpu_sample(dev, light=False, parts=1):
    """Bounded sample of the hybrid step for the oracle: channel (group) subsets of
    each workload, all tokens of the sampled requests. Each workload's channels are
    split into `parts` disjoint blocks (independent jobs, for the all-cores run)."""
    import numpy as np
    from state_cached_causal_gb300 import synth
    from oracle.torch_io import pool_np, to_np
    import oracle
    jobs = []
    nch = LIGHT_CHANNELS if light else SAMPLE_CHANNELS

    def blocks(total, unit):
        n = max(1, min(parts, total // unit))
        edges = [(k * (total // unit) // n) * unit for k in range(n + 1)]
        return [(edges[k], edges[k + 1]) for k in range(n)]

    def dw(name, case, chans):
        for lo, hi in blocks(chans, 8):
            sl = slice(lo, hi)
            w = np.ascontiguousarray(to_np(case.w)[sl])
            b = None if case.bias is None else np.ascontiguousarray(to_np(case.bias)[sl])
            pool = pool_np(case.pool[:, sl, :].contiguous())
            if case.x is not None:
                x = np.ascontiguousarray(to_np(case.x[:, sl].contiguous()))
                args = (to_np(case.state_idx), to_np(case.cu_seqlens), to_np(case.has_init))

                def run(x=x, w=w, b=b, pool=pool, args=args, case=case):
                    oracle.cconv_fwd_varlen(x, w, b, pool.copy(), *args, case.width,
                                            case.dilation, case.act, np.zeros_like(x))
                jobs.append((f"{name}.fwd_varlen", run, x.shape[0] * (hi - lo)))
            if case.x_spec is not None:
                xs = np.ascontiguousarray(to_np(case.x_spec[:, sl].contiguous()))
                na = to_np(case.num_accepted) if case.n_spec else None

                def run2(xs=xs, w=w, b=b, pool=pool, case=case, na=na):
                    oracle.cconv_update(xs, pool.copy(), w, b, to_np(case.spec_state_idx),
                                        case.n_spec, na, None, case.width, case.dilation,
                                        case.act, np.zeros_like(xs))
                jobs.append((f"{name}.update", run2, xs.shape[0] * (hi - lo)))

    dw("gdn_decode", synth.gdn_decode(dev), nch["gdn_decode"])
    dw("gdn_mixed", synth.gdn_mixed(dev), nch["gdn_mixed"])
    cc = synth.zaya_cca(dev)
    nreq = 257   # the 256 decodes and the first 4096-token prefill
    T = int(cc.cu_seqlens[nreq].item())
    dl = np.ascontiguousarray(to_np(cc.delayed[:T].contiguous()))
    ds = to_np(cc.delayed_state).copy()
    meta = (to_np(cc.state_idx[:nreq]), to_np(cc.cu_seqlens[:nreq + 1]),
            to_np(cc.has_init[:nreq]))
    for g0, g1 in blocks(nch["zaya_cca"], 1):
        sl = slice(g0 * 128, g1 * 128)
        qk = np.ascontiguousarray(to_np(cc.qk[:T, sl].contiguous()))
        wts = [np.ascontiguousarray(to_np(t)[sl]) for t in (cc.w_dw, cc.b_dw, cc.w_gr, cc.b_gr)]
        pool = pool_np(cc.pool[:, sl, :].contiguous())

        def run3(qk=qk, wts=wts, pool=pool, ng=g1 - g0):
            oracle.cca_qk_conv(qk, *wts, ng, 2, 2, dl, to_np(cc.delayed_init), pool.copy(),
                               ds.copy(), *meta, np.zeros_like(qk), np.zeros_like(dl))
        jobs.append(("zaya_cca.cca_qk_conv", run3, T * (g1 - g0) * 128))
    dw("ple_spec", synth.ple_spec(dev), nch["ple_spec"])
    units = sum(j[2] for j in jobs)
    desc = (f"oracle on: gdn_decode {nch['gdn_decode']} ch, gdn_mixed {nch['gdn_mixed']} ch, "
            f"zaya_cca {nch['zaya_cca']} group(s) x {nreq} requests ({T} tokens), ple_spec "
            f"{nch['ple_spec']} ch; all tokens of the sampled requests; {units} "
            "tokens*channels")
    return jobs, units, desc


def run_cpu_parallel(jobs, threads):
    """The jobs on `threads` host threads (the oracle's C calls release the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    order = sorted(jobs, key=lambda j: -j[2])
    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda j: j[1](), order))
    return time.perf_counter() - t0


ARM_PARTS = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1"}


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
                if line.lower().startswith("cpu part"):
                    part = line.split(":", 1)[1].strip()
                    return f"{ARM_PARTS.get(part, 'Arm')} (cpu part {part})"
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def run_cpu_sample(jobs):
    t0 = time.perf_counter()
    for _, fn, _ in jobs:
        fn()
    return time.perf_counter() - t0


# ---- arms ----------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def capture_step(step, stream, dev):
    """One step captured as a CUDA graph, or None when capture is not possible."""
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        torch.cuda.synchronize()
        return g
    except Exception:
        torch.cuda.synchronize()
        return None


def whole_job_value(ws, units_per_step, steps, elapsed):
    """Replicas: every rank runs the whole step on its own GPU (weak scaling), so
    the job processed ws * units_per_step * steps units in the slowest rank's
    time; in G(tokens*channels)/s."""
    return ws * units_per_step * steps / elapsed / 1e9


def reduce_max(value, ws):
    if ws <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def arm_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    dev = torch.device("cuda" if torch.cuda.is_available() else "cpu")
    jobs, units, desc = cpu_sample(dev, light=True)
    for _ in range(args.warmup):
        run_cpu_sample(jobs)
    times = [run_cpu_sample(jobs) for _ in range(args.steps)]
    total = sum(times)
    value = units * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32-accumulate bf16",
        "data": "synthetic",
        "config": {"workload": "hybrid_step (oracle sample)", "sample": desc,
                   "parallelism": "host, 1 thread"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def arm_ours(args):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    from state_cached_causal_gb300 import ops
    ops.load()
    dev_err = torch.zeros(1, dtype=torch.int32, device=dev)
    calls, desc = build_workload(args.workload, dev, dev_err)
    stream = torch.cuda.current_stream(dev)
    units_per_step = sum(c.units for c in calls)
    bytes_per_step = sum(c.bytes for c in calls)

    def step():
        for c in calls:
            c.fn()

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize()
    if int(dev_err.item()) != 0:
        raise SystemExit(f"device error flag {int(dev_err.item())} during warm-up")

    # The step's launches captured once as a CUDA graph: the timed region replays
    # it K times (the same kernels and arguments, without the host's per-launch
    # overhead); if capture fails, the timed region launches the calls on the
    # stream instead.
    graph = capture_step(step, stream, dev)
    if graph is not None:
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()

    # timed region: K steps between two events on the launching stream
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        # a short device-side wait first, so that the host has queued the first
        # launches when the timed region begins (the region then measures the
        # device, not the host's first enqueue)
        torch.cuda._sleep(LEAD_CYCLES)
        start.record(stream)
        for k in range(args.steps):
            if graph is not None:
                graph.replay()
            else:
                step()
        stop.record(stream)
        torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    elapsed = start.elapsed_time(stop) / 1e3

    # per-launch breakdown: a second pass of K steps launched on the stream
    # with events around every launch (the events add about 2 us per launch)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in calls] for _ in range(args.steps)]
    torch.cuda._sleep(LEAD_CYCLES)
    for k in range(args.steps):
        for c, (a, b) in zip(calls, ev[k]):
            a.record(stream)
            c.fn()
            b.record(stream)
    torch.cuda.synchronize()
    events_step_ms = ev[0][0][0].elapsed_time(ev[-1][-1][1]) / args.steps
    elapsed = reduce_max(elapsed, ws)
    per_call = {c.name: sum(ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps))
                / args.steps / 1e3 for i, c in enumerate(calls)}
    if int(dev_err.item()) != 0:
        raise SystemExit(f"device error flag {int(dev_err.item())} in the timed region")

    value = whole_job_value(ws, units_per_step, args.steps, elapsed)
    hbm_peak, bf16_peak, peak_src = measured_peaks()
    dom = max(calls, key=lambda c: per_call[c.name])
    t_dom = per_call[dom.name]
    achieved = dom.bytes / t_dom / 1e9
    traffic = recorded_traffic(dom.kernel)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": traffic, "kernel": dom.name,
                "algorithmic_bytes": dom.bytes, "ms_per_launch": t_dom * 1e3,
                "peak_source": f"{peak_src} hbm_gbs"}
    breakdown = {}
    for c in calls:
        t = per_call[c.name]
        d = {"ms": t * 1e3, "Gtokch_per_s": c.units / t / 1e9, "GB_per_s": c.bytes / t / 1e9,
             "hbm_frac": c.bytes / t / 1e9 / hbm_peak,
             "hbm_frac_of_nominal": c.bytes / t / 1e9 / NOMINAL_HBM_GBS, "bytes": c.bytes}
        if c.flops:
            d["TFLOP_per_s"] = c.flops / t / 1e12
            d["tensor_frac_of_bf16_peak"] = c.flops / t / 1e12 / bf16_peak
        breakdown[c.name] = d

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": desc, "l2": "inputs larger than L2 each step "
                   f"({bytes_per_step / 1e9:.2f} GB algorithmic), no flush",
                   "parallelism": "replicas" if ws > 1 else "1 GPU"},
        "hbm_GBps": bytes_per_step * args.steps / elapsed / 1e9,
        "gpu_launches": len(calls) * args.steps,
        "launch": ("one CUDA graph of the step's %d launches per step" % len(calls)
                   if graph is not None else "stream launches"),
        "ms_per_step_stream_with_call_events": events_step_ms,
        "roofline": roofline,
        "clocks": clk.summary(),
        "per_call": breakdown,
    }

    if not args.no_e2e:
        line["e2e"] = e2e_run(args, calls, stream, dev, ws)
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        ncores = os.cpu_count() or 1
        jobs, units, sdesc = cpu_sample(dev, parts=ncores)
        t = run_cpu_sample(jobs)
        tp = min(run_cpu_parallel(jobs, ncores) for _ in range(2))
        line["cpu_baseline"] = {"value": units / t / 1e9, "unit": UNIT, "cores": 1,
                                "kind": "oracle", "sample": sdesc + " (1 thread)",
                                "seconds_per_sample": t,
                                "all_cores": {"value": units / tp / 1e9, "cores": ncores,
                                              "seconds_per_sample": tp,
                                              "cpu": cpu_model()}}
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def e2e_run(args, calls, stream, dev, ws):
    """Same step through the C ABI with the inputs copied in from pinned host
    memory and the outputs copied out, all inside the timed region. Copies run
    on their own streams, call by call, so that host-to-device, kernels and
    device-to-host overlap; events keep a call's inputs from being overwritten
    before its previous launch has read them and its outputs from being
    rewritten before they have been copied out."""
    ins, outs = [], []
    for c in calls:
        ins.append([(t, torch.empty(t.shape, dtype=t.dtype, pin_memory=True)) for t in c.h2d])
        outs.append([(t, torch.empty(t.shape, dtype=t.dtype, pin_memory=True)) for t in c.d2h])
    for pairs in ins:
        for d, h in pairs:
            h.copy_(d)
    h2d = sum(d.numel() * d.element_size() for pairs in ins for d, _ in pairs)
    d2h = sum(d.numel() * d.element_size() for pairs in outs for d, _ in pairs)
    steps = max(3, min(args.steps, 20))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n = len(calls)
    ev = lambda: torch.cuda.Event()
    done_k = [None] * n      # kernel k of the previous step finished
    out_k = [None] * n       # outputs of call k of the previous step copied out

    def step():
        for k, c in enumerate(calls):
            with torch.cuda.stream(s_in):
                if done_k[k] is not None:
                    s_in.wait_event(done_k[k])
                for d, h in ins[k]:
                    d.copy_(h, non_blocking=True)
                e_in = ev()
                e_in.record(s_in)
            stream.wait_event(e_in)
            if out_k[k] is not None:
                stream.wait_event(out_k[k])
            with torch.cuda.stream(stream):
                c.fn()
            e_c = ev()
            e_c.record(stream)
            done_k[k] = e_c
            with torch.cuda.stream(s_out):
                s_out.wait_event(e_c)
                for d, h in outs[k]:
                    h.copy_(d, non_blocking=True)
                e_o = ev()
                e_o.record(s_out)
            out_k[k] = e_o

    step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(LEAD_CYCLES)
    a.record(stream)
    s_in.wait_event(a)
    s_out.wait_event(a)
    for _ in range(steps):
        step()
    for s_ in (s_in, s_out):
        e = ev()
        e.record(s_)
        stream.wait_event(e)
    b.record(stream)
    torch.cuda.synchronize()
    el = reduce_max(a.elapsed_time(b) / 1e3, ws)
    units = sum(c.units for c in calls)
    return {"value": ws * units * steps / el / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "overlap": "per call: h2d, kernel and d2h on three streams"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="hybrid_step")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 0 or args.steps < 1:
        raise SystemExit("--steps >= 1 and --warmup >= 0")
    if args.impl == "reference":
        return arm_reference(args)
    return arm_ours(args)


if __name__ == "__main__":
    sys.exit(main())
