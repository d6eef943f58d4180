"""The GPU INT4 quantizer over every finite bf16 value, bit-exact against the
oracle (page "Persistent input/output feedback", quantization paragraph:
round half to even, saturate to the code range; page "Custom, quantized, and
persistent values": blocked affine, two codes per byte, least-significant bits
first).

Fixed parameters: all 65,280 finite bf16 patterns, in rows of 128, through
ol_int4kv_append with several fp16 scales (a power of two, an inexact one, a
subnormal one, a large one) and zero points 0, 7, 8 and 15 (an odd zero point
separates rounding before the zero point is added from rounding after).
Dynamic parameters: the same patterns in blocks of 32 neighbouring patterns,
plus blocks built so that x / scale lands exactly halfway between integers
(with even and odd zero points), the all-zero block, blocks of one sign, and
blocks whose range underflows or overflows fp16. Codes, scales and zero points
must equal the oracle's bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle as O
import place_kv_cache_gb300 as ol
from workloads import bf16_from_f32
from tests.gpu_util import to_dev, to_host

pytestmark = pytest.mark.gpu

D = 128


def finite_bf16():
    u = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return u[(u & 0x7F80) != 0x7F80]                          # exponent all ones: inf and NaN


def rows_of(values_u16):
    """[2, B, 1, 1, 128] values (planes and rows filled in order), zero-padded."""
    n = -(-values_u16.size // (2 * D)) * 2 * D
    v = np.zeros(n, np.uint16)
    v[:values_u16.size] = values_u16
    return np.ascontiguousarray(v.reshape(2, n // (2 * D), 1, 1, D))


def run_both(values, mode, fixed_scale=0.25, fixed_zp=8):
    B = values.shape[1]
    planes = O.int4_planes(B, 1, 1, D)
    pos = np.zeros(B, np.int32)
    O.int4_append(*planes, values, pos, mode=mode, fixed_scale=fixed_scale, fixed_zp=fixed_zp)
    dev = tuple(to_dev(np.zeros_like(p)) for p in planes)
    desc = ol.int4_kv(*dev, head_dim=D, quant_mode=mode, fixed_scale=fixed_scale, fixed_zp=fixed_zp)
    ol.ol_int4kv_append(desc, dev[0], to_dev(values), pos, to_dev(pos))
    torch.cuda.synchronize()
    for name, g, r in zip(("codes", "scales", "zero points"), dev, planes):
        got = to_host(g)
        bad = np.argwhere(got != r)
        assert bad.size == 0, f"{len(bad)} {name} differ, first at {bad[0].tolist()}: {got[tuple(bad[0])]} vs " \
                              f"{r[tuple(bad[0])]}"


@pytest.mark.parametrize("zp", [0, 7, 8, 15])
@pytest.mark.parametrize("scale", [0.25, 0.1, 3.0e-5, 1000.0])
def test_fixed_parameters_every_finite_bf16(scale, zp):
    run_both(rows_of(finite_bf16()), O.Q_FIXED, fixed_scale=scale, fixed_zp=zp)


def tie_blocks():
    """Blocks whose scale is exact and whose other values sit exactly halfway
    between codes: range [-8s, 7s] (zero point 8) and [-7s, 8s] (zero point 7)
    for power-of-two s, so (hi - lo) / 15 = s exactly."""
    out = []
    for e in (-20, -10, -3, 0, 5, 12):
        s = np.float32(2.0 ** e)
        for lo_k, hi_k in ((-8, 7), (-7, 8)):
            ties = [(k + 0.5) * s for k in range(lo_k, hi_k)]            # 15 halfway values
            grid = [k * s for k in range(lo_k + 1, hi_k)]                # 14 grid values
            block = [lo_k * s, hi_k * s] + ties + grid + [0.0]
            out.append(np.array(block[:32], np.float32))
    return out


def special_blocks(rng):
    out = [np.zeros(32, np.float32),                                    # all zero: scale 1, zero point 0
           np.abs(rng.standard_normal(32)).astype(np.float32),          # one sign: lo = 0
           -np.abs(rng.standard_normal(32)).astype(np.float32),         # the other: hi = 0
           np.full(32, -0.0, np.float32),
           (rng.standard_normal(32) * 1e-39).astype(np.float32),        # bf16 subnormals: the range underflows fp16
           (rng.standard_normal(32) * 1e30).astype(np.float32),         # the range overflows fp16
           np.array([3.0e38, -3.0e38] + [1.0] * 30, np.float32)]
    return out


def test_dynamic_parameters_every_finite_bf16_and_built_blocks():
    rng = np.random.default_rng(90)
    neighbours = finite_bf16()                                  # blocks of 32 consecutive patterns
    built = np.concatenate([bf16_from_f32(b) for b in tie_blocks() + special_blocks(rng)])
    run_both(rows_of(np.concatenate([neighbours, built])), O.Q_DYNAMIC)
