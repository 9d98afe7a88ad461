"""The ctypes binding's marshalling (state_cached_causal_gb300/ops.py), on the
CPU: pool views become the right base, strides, sizes and storage type, rows
and dtypes are checked, host tensors and a missing library are refused, and
the CCA wrappers insist on one storage type for both state tensors. No kernel
runs here."""
import pytest
import torch

from state_cached_causal_gb300 import ops


def test_pool_view_of_each_layout():
    ds = torch.zeros(5, 16, 3, dtype=torch.bfloat16)
    p = ops._pool(ds)
    assert (p.s_slot, p.s_chan, p.s_col, p.num_slots, p.cap, p.dtype) == (48, 3, 1, 5, 3,
                                                                           ops.DTYPE_BF16)
    assert p.p == ds.data_ptr()
    sd = torch.zeros(5, 3, 16, dtype=torch.float32).transpose(1, 2)   # column-first storage
    p = ops._pool(sd)
    assert (p.s_slot, p.s_chan, p.s_col, p.cap, p.dtype) == (48, 1, 16, 3, ops.DTYPE_F32)
    wide = torch.zeros(5, 16, 12, dtype=torch.bfloat16)[:, :, -9:]      # last cap columns
    p = ops._pool(wide)
    assert (p.s_slot, p.s_chan, p.s_col, p.cap) == (192, 12, 1, 9)
    assert p.p == wide.data_ptr()                                   # the view's first element
    with pytest.raises(ValueError):
        ops._pool(torch.zeros(5, 16))


def test_rows_and_dtypes():
    x = torch.zeros(4, 32, dtype=torch.bfloat16)
    assert ops._rows(x) == 32
    assert ops._rows(torch.zeros(8, 64)[:, :32]) == 64           # row stride, not width
    with pytest.raises(ValueError):
        ops._rows(torch.zeros(32, 4).t())                         # rows not contiguous
    assert ops._dtype_code(x) == ops.DTYPE_BF16
    assert ops._dtype_code(torch.zeros(1)) == ops.DTYPE_F32
    with pytest.raises(TypeError):
        ops._dtype_code(torch.zeros(1, dtype=torch.float16))


def test_host_tensors_are_refused():
    with pytest.raises(ValueError):
        ops._ptr(torch.zeros(4))
    assert ops._ptr(None) is None


def test_index_types_are_checked():
    with pytest.raises(TypeError):
        ops._i32(torch.zeros(3, dtype=torch.int64), "state_idx")
    with pytest.raises(TypeError):
        ops._u8(torch.zeros(3, dtype=torch.int32), "has_init")
    assert ops._u8(torch.zeros(3, dtype=torch.bool), "has_init") is not None


def test_cca_state_tensors_share_one_storage_type():
    pool = torch.zeros(4, 256, 2, dtype=torch.float32)
    dstate = torch.zeros(4, 64, dtype=torch.bfloat16)
    z = torch.zeros(1)
    with pytest.raises(TypeError):
        ops.cca_qk_conv(z, z, z, z, z, 2, 2, 2, z, z, pool, dstate, z, z, z, z, z)
    with pytest.raises(TypeError):
        ops.cca_qk_conv_fused(z, z, z, z, z, 2, 1, 2, 2, z, z, z, pool, dstate, z, z, z, z)


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(ops, "_lib", None)
    monkeypatch.setattr(ops, "LIB_PATH", str(tmp_path / "libcconv.so"))
    with pytest.raises(RuntimeError):
        ops.load()
