"""CPU checks of the seeded input generators' 16-bit helpers (input
generation only: the oracle consumes the values they produce)."""
import numpy as np

import workloads


def test_round_to_bf16_is_nearest_ties_to_even():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(20000).astype(np.float32)
    # add exact halfway cases: a bf16 value plus half an ulp
    base = workloads.round_to_bf16(rng.standard_normal(2000).astype(np.float32))
    ulp = np.abs(base) * 2.0 ** -7
    x = np.concatenate([x, (base + np.float32(0.5) * ulp.astype(np.float32))])
    r = workloads.round_to_bf16(x)
    bits = r.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0)                    # representable in bf16
    lo = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)  # truncation toward zero
    hi = ((x.view(np.uint32) & 0xFFFF0000) + 0x10000).view(np.float32)
    dlo, dhi = np.abs(x.astype(np.float64) - lo), np.abs(hi.astype(np.float64) - x)
    nearest = np.where(dlo < dhi, lo, hi)
    tie = dlo == dhi
    even = np.where((lo.view(np.uint32) >> 16) & 1 == 0, lo, hi)
    want = np.where(tie, even, nearest)
    assert np.array_equal(r, want)


def test_half_bits_round_trip():
    rng = np.random.default_rng(1)
    x = workloads.round_to_bf16(rng.uniform(-4, 4, 1000).astype(np.float32))
    b = workloads.half_bits(x, "bf16")
    assert np.array_equal((b.astype(np.uint32) << 16).view(np.float32), x)
    y = rng.uniform(-4, 4, 1000).astype(np.float16).astype(np.float32)
    h = workloads.half_bits(y, "fp16")
    assert np.array_equal(h.view(np.float16).astype(np.float32), y)
