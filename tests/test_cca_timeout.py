"""The CCA kernel's timeout path, on the GPU, without hanging or faulting it.

Every pipeline wait of the CCA kernel is bounded: when one runs out, the kernel
sets CCONV_DERR_TIMEOUT, the other roles stop at their next wait, copies and
MMAs in flight are drained, TMEM is freed and the kernel returns. With the
normal limit (about a second) no test can make a wait run out, so this test
builds the CCA entry point a second time with a limit of zero cycles and polls
that never suspend the thread: any wait not satisfied at its first poll gives
up. The drain keeps its normal limit. The test checks that such a launch returns with the error bit set and
that the same process then runs a normal call correctly.
"""
import ctypes

import pytest
import torch

from state_cached_causal_gb300 import build as cbuild
from state_cached_causal_gb300 import ops, synth
from tests.test_parity_cca import check, gpu_cca

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def test_cca_wait_timeout_returns_with_the_error_bit(tmp_path):
    short = ctypes.CDLL(cbuild.build_cca_variant(str(tmp_path), ["-DCCA_WAIT_CYCLES=0", "-DCCA_WAIT_POLL_NS=20"]))
    short.cca_qk_conv.argtypes = ops.load().cca_qk_conv.argtypes
    short.cca_qk_conv.restype = ctypes.c_int
    short.cconv_status_string.argtypes = [ctypes.c_int]
    short.cconv_status_string.restype = ctypes.c_char_p
    case = synth.cca_case(4700, DEV, lens=[1, 1, 1, 40, 200, 130], decode_prefix=3, Hq=2, Hkv=1)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    saved = ops._lib
    ops._lib = short                      # the binding's calls go to the short-wait build
    try:
        gpu_cca(case, err=err)            # raises if the launch itself failed
        torch.cuda.synchronize()          # the aborted kernel has returned
    finally:
        ops._lib = saved
    assert int(err.item()) & ops.DERR_TIMEOUT
    # the context is intact: a normal call on the same process is correct
    check(case)
