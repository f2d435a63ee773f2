"""Host logic of the per-layer precision policy (no GPU): which layers keep
BF16 (the pages' first and last two), overrides, and per-layer constants."""
import pytest

import ue8m0_kv_cache_gb300 as uq
from ue8m0_kv_cache_gb300.policy import LayerPolicy


def test_boundary_layers_are_bf16():
    p = LayerPolicy(32)
    assert [l for l in range(32) if p.dtype(l) == uq.BF16] == [0, 1, 30, 31]
    assert p.count(uq.FP4_UE8M0) == 28


def test_small_stacks_and_no_boundary():
    assert LayerPolicy(3, boundary=2).dtypes == [uq.BF16] * 3
    assert LayerPolicy(4, boundary=0).dtypes == [uq.FP4_UE8M0] * 4


def test_overrides_and_constants():
    p = LayerPolicy(8, overrides={5: uq.FP8_E4M3}, fp4_c=[0.0, 0.0, 0.2, 0.17, 0.0, 0.3, 0.0, 0.0])
    assert p.dtype(5) == uq.FP8_E4M3
    assert p.fp4_c(2) == 0.2 and p.fp4_c(3) == 0.17
    assert p.fp4_c(5) == 0.0 and p.fp4_c(0) == 0.0  # not FP4 layers
    with pytest.raises(ValueError):
        LayerPolicy(4, fp4_c=[0.1, 0.2])
    with pytest.raises(ValueError):
        LayerPolicy(0)
