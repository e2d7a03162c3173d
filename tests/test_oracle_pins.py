"""The CPU oracle against closed forms, invariants of the method, a brute-force
sequential decoder and library routines (see oracle_pins.py)."""
import pytest

import oracle.cpu_blend as ob
import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(ob)


def test_bf16_storage_mode_rounds_once():
    """With bf16 storage every stored K/V value is a bfloat16 number, and the r=1 blend
    stays within a few bf16 ulps of the float64-storage blend."""
    import numpy as np
    _, chunks, _, toks = pins.micro_request()
    caches = ob.round_bf16(pins.brute_caches())
    got = ob.blend(pins.MICRO_CFG, pins.micro_weights(), toks, caches, chunks, 1.0, "bf16")
    kv = got["out_kv"].astype(np.float64)
    assert np.array_equal(ob.round_bf16(kv), kv)
    exact = ob.blend(pins.MICRO_CFG, pins.micro_weights(), toks, pins.brute_caches(), chunks, 1.0, "f64")
    scale = np.abs(exact["out_kv"]).max()
    assert np.abs(kv - exact["out_kv"]).max() < 0.02 * scale
