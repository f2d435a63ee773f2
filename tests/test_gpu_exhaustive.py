"""Exhaustive checks of the append's two scalar stages through their stage
hooks (the same device functions the append kernels call): the E2M1
conversion (R3) on every fp32 bit pattern, and the UE8M0 scale byte (R2) on
every non-negative fp32 bit pattern.  The device generates each chunk of bit
patterns itself; the oracle enumerates the same range on the host cores."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import ue8m0_kv_cache_gb300 as uq

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
CHUNK = 1 << 26           # bit patterns per device call
SUB = 1 << 22             # per oracle call
THREADS = max(1, os.cpu_count() or 1)


def _patterns(first, n):
    """fp32 tensor on the device holding bit patterns first .. first + n - 1
    (first a multiple of n, so a chunk never crosses 2^31)."""
    signed = first - (1 << 32) if first >= 1 << 31 else first
    return torch.arange(signed, signed + n, dtype=torch.int32, device=DEV).view(torch.float32)


def _sweep(first_all, end_all, gpu_fn, oracle_fn):
    bad = 0
    with ThreadPoolExecutor(THREADS) as ex:
        for first in range(first_all, end_all, CHUNK):
            subs = [ex.submit(oracle_fn, first + o, SUB) for o in range(0, CHUNK, SUB)]
            got = gpu_fn(_patterns(first, CHUNK)).cpu().numpy()
            want = np.concatenate([f.result() for f in subs])
            yield first, got, want


def test_e2m1_conversion_on_every_fp32_pattern():
    checked = 0
    for first, got, want in _sweep(0, 1 << 32, uq.uq_test_cvt_e2m1, oracle.e2m1_codes_of_bits):
        live = want != 0xFF  # NaN patterns carry no E2M1 code
        if not np.array_equal(got[live], want[live]):
            i = int(np.flatnonzero(live & (got != want))[0])
            pytest.fail("pattern 0x%08x: GPU code %d, oracle %d" % (first + i, got[i], want[i]))
        checked += int(live.sum())
    assert uq.uq_check_device_status() == 0
    assert checked == (1 << 32) - 2 * ((1 << 23) - 1)  # every pattern but the NaNs


def test_scale_byte_on_every_non_negative_fp32_pattern():
    for first, got, want in _sweep(0, 1 << 31, uq.uq_test_scale_byte, oracle.scale_bytes_of_bits):
        if not np.array_equal(got, want):
            i = int(np.flatnonzero(got != want)[0])
            pytest.fail("pattern 0x%08x: GPU byte %d, oracle %d" % (first + i, got[i], want[i]))
    assert uq.uq_check_device_status() == 0
