"""Test helpers (re-exported from the oracle's torch/numpy conversion module)."""
from oracle.torch_io import np_to_f64, pool_np, to_np  # noqa: F401
