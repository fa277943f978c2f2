"""The oracle's fp16 and e4m3 converters over every fp32 input (all 2^32 bit patterns).

The int4 quantiser's fp16 offset (rounded toward -inf) and scale (toward +inf), and the FP8
window cache's e4m3 codes (nearest-even, saturating at +-448), carry every bit that the
bit-exactness of the cache rests on ("Serving Kolibri-1 with a 4-bit KV cache", section "What
we do": one fp16 scale and one fp16 offset per token and head; the sliding-window layers keep
an FP8 cache). Here each converter is compared, input by input, with an independent one:
  - nearest-even fp16: torch's float32 -> float16 cast (numpy's on one chunk as well);
  - toward -inf / +inf: the nearest-even result, stepped by one fp16 ulp (integer arithmetic on
    the bit pattern) when it lies on the wrong side of the input, which also gives IEEE overflow
    (the inward direction stops at +-65504, the outward one goes to infinity);
  - e4m3: torch's float32 -> float8_e4m3fn cast wherever that is finite; torch's cast does not
    saturate, so where it gives NaN for a finite input the oracle must give +-448.
NaN inputs must give a NaN pattern. CPU only.
"""

import concurrent.futures

import numpy as np
import pytest
import torch

CHUNK = 1 << 21


def _reference(bits):
    """(x, rn, rd, ru, e4) for a uint32 numpy array of fp32 bit patterns; fp16 results as int16
    tensors of bit patterns. The directed results step the nearest-even pattern by one ulp where
    it lies on the wrong side of x: +1 on the pattern moves a positive value up and a negative one
    down. (A zero result never needs the step across the sign: a -0 nearest result comes from
    x <= -0, a +0 from x >= +0.) e4 is torch's non-saturating cast, NaN where it overflows."""
    xt = torch.from_numpy(bits.view(np.float32))
    rn16 = xt.to(torch.float16)
    rn = rn16.view(torch.int16)
    h = rn16.to(torch.float32)  # exact
    away = 1 - 2 * (rn < 0).to(torch.int16)  # +1 for a positive pattern, -1 for a negative one
    rd = rn - (h > xt).to(torch.int16) * away
    ru = rn + (h < xt).to(torch.int16) * away
    e4 = xt.to(torch.float8_e4m3fn).view(torch.uint8)
    return xt, rn, rd, ru, e4


def _first_mismatch(xt, bits, name, got, want):
    i = int(torch.nonzero(got != want)[0])
    raise AssertionError(f"{name} of {float(xt[i])!r} (bits {int(bits[i]):#010x}): oracle "
                         f"{int(got[i]) & 0xFFFF:#06x}, reference {int(want[i]) & 0xFFFF:#06x}")


def _compare(orc, first, n, got=None):
    """Compare the oracle on bit patterns first .. first+n-1 (got: its convert_range output, if
    already computed) with the references."""
    bits = np.arange(first, first + n, dtype=np.uint32)
    xt, rn, rd, ru, e4 = _reference(bits)
    o_rn, o_rd, o_ru, o_e4 = got or orc.convert_range(first, n)
    o16 = [torch.from_numpy(a.view(np.int16)) for a in (o_rn, o_rd, o_ru)]
    o_e4 = torch.from_numpy(o_e4)
    # torch's e4m3 cast gives NaN (0x7F / 0xFF) where the saturating conversion gives +-448
    e4_sat = torch.where((e4 & 0x7F) == 0x7F, (e4 & 0x80) | 0x7E, e4)
    nan = torch.isnan(xt)
    if not bool(nan.any()):
        for name, g, want in zip(("fp16 nearest", "fp16 down", "fp16 up"), o16, (rn, rd, ru)):
            if not torch.equal(g, want):
                _first_mismatch(xt, bits, name, g, want)
        if not torch.equal(o_e4, e4_sat):
            _first_mismatch(xt, bits, "e4m3", o_e4.to(torch.int32), e4_sat.to(torch.int32))
        return
    ok = ~nan
    for name, g, want in zip(("fp16 nearest", "fp16 down", "fp16 up"), o16, (rn, rd, ru)):
        if not torch.equal(g[ok], want[ok]):
            _first_mismatch(xt[ok], bits[ok.numpy()], name, g[ok], want[ok])
        gn = g[nan].to(torch.int32) & 0xFFFF
        assert bool((((gn & 0x7C00) == 0x7C00) & ((gn & 0x03FF) != 0)).all()), f"{name} of a NaN is not NaN"
    assert torch.equal(o_e4[ok], e4_sat[ok]), "e4m3 differs"
    assert bool(((o_e4[nan] & 0x7F) == 0x7F).all()), "e4m3 of a NaN is not NaN"


def test_converters_spot_values(orc):
    """Hand-checked values, including the IEEE overflow rules and signed zeros."""
    cases = [  # x, nearest, down, up
        (65504.0, 0x7BFF, 0x7BFF, 0x7BFF),
        (65519.996, 0x7BFF, 0x7BFF, 0x7C00),
        (65520.0, 0x7C00, 0x7BFF, 0x7C00),
        (-65520.0, 0xFC00, 0xFC00, 0xFBFF),
        (float("inf"), 0x7C00, 0x7C00, 0x7C00),
        (1e-9, 0x0000, 0x0000, 0x0001),
        (-1e-9, 0x8000, 0x8001, 0x8000),
        (-0.0, 0x8000, 0x8000, 0x8000),
        (1.3, 0x3D33, 0x3D33, 0x3D34),
    ]
    for x, n, d, u in cases:
        got = tuple(orc.fp16_round_bits(np.float32(x), k) for k in (0, -1, 1))
        assert got == (n, d, u), (x, [hex(v) for v in got])
    for x, c in ((448.0, 0x7E), (464.0, 0x7E), (465.0, 0x7E), (1e30, 0x7E), (-1e30, 0xFE), (2.0 ** -9, 0x01),
                 (2.0 ** -10, 0x00), (0.0009765625 * 1.5, 0x01)):
        assert orc.e4m3_encode(np.float32(x)) == c, (x, hex(orc.e4m3_encode(np.float32(x))))


def test_reference_agrees_with_numpy_on_one_chunk():
    """The torch nearest-even cast used below agrees with numpy's on a chunk with normal,
    subnormal and overflowing fp16 results."""
    for first in (0x33000000, 0x47000000):
        x = np.arange(first, first + CHUNK, dtype=np.uint32).view(np.float32)
        with np.errstate(over="ignore"):
            a = x.astype(np.float16).view(np.uint16).astype(np.int64)
        b = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().astype(np.int64) & 0xFFFF
        assert np.array_equal(a, b)


@pytest.mark.parametrize("part", range(4), ids=lambda p: f"quarter{p}")
def test_converters_all_fp32_inputs(orc, part):
    """Every fp32 bit pattern of one quarter of the 2^32 (sign and top exponent bit fixed)."""
    first = part << 30
    starts = list(range(first, first + (1 << 30), CHUNK))
    # the oracle evaluates the next chunk on a worker thread (ctypes drops the GIL) while the
    # references of the current one are computed
    with concurrent.futures.ThreadPoolExecutor(1) as pool:
        nxt = pool.submit(orc.convert_range, starts[0], CHUNK)
        for i, a in enumerate(starts):
            got = nxt.result()
            if i + 1 < len(starts):
                nxt = pool.submit(orc.convert_range, starts[i + 1], CHUNK)
            _compare(orc, a, CHUNK, got)
