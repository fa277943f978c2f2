"""GPU parity of the cache formats at their edge cases, through the C ABI.

"Serving Kolibri-1 with a 4-bit KV cache", section "What we do": every token and head gets
4-bit codes with one fp16 scale and one fp16 offset; the sliding-window layers keep a stock
FP8 cache. The value rows of kvq_rotate_quant_append go straight into the int4 quantiser (no
prologue), so hand-built rows reach its corners on the GPU: the golden cases of
tests/golden/quantizer_cases.txt (ramp, exact constant, fp16-subnormal scale, ties at .5,
offset rounded down), offsets and spans beyond the fp16 range (saturated, KVQ_DEVERR_RANGE),
a minimum of -0 and rows of signed zeros (a zero offset or scale is stored as +0), tiny and huge
magnitudes; an append past the cache's capacity (KVQ_DEVERR_POS, nothing written); e4m3 codes
of values beyond +-448 (saturated), subnormal e4m3 codes and signed zeros.
Codes, scale bits and offset bits must equal the oracle's; the error word must match the
oracle's flags.
"""

import numpy as np
import pytest
import torch

import pins
from gpu_util import unpack_int4
from quantized_kv_cache_fold_gb300 import (DEVERR_POS, DEVERR_RANGE, alloc_fp8_ring, alloc_int4_cache,
                                           kvq_fp8_append, kvq_rotate_quant_append)

pytestmark = pytest.mark.gpu

HKV = 4


def _edge_rows():
    """name -> fp32 value row (128) beyond the golden cases."""
    i = np.arange(128, dtype=np.float64)
    rows = {
        "min_neg_zero": np.concatenate([[-0.0], np.linspace(0.25, 3.0, 127)]).astype(np.float32),
        "all_neg_zero": np.full(128, -0.0, np.float32),
        "mixed_zeros": np.where(np.arange(128) % 3 == 0, -0.0, 0.0).astype(np.float32),
        "tiny_subnormal": (i * 2.0 ** -27).astype(np.float32),  # span below the smallest fp16 step
        "huge_positive": np.full(128, 1.0e6, np.float32) + i.astype(np.float32),  # offset rounds down to 65504
        "wide_span": np.linspace(-60000.0, 900000.0, 128).astype(np.float32),  # scale 64000: in range
        "negative_only": (-1.0 - i / 7.0).astype(np.float32),
        "alternating": np.where(i % 2 == 0, -3.3, 7.7).astype(np.float32),
    }
    return rows


def _range_rows():
    """Rows whose offset or scale leaves the fp16 range (oracle flag 2, KVQ_DEVERR_RANGE)."""
    i = np.arange(128, dtype=np.float64)
    return {
        "offset_below_fp16": np.concatenate([[-1.0e6], np.zeros(127)]).astype(np.float32),
        "span_above_fp16": np.linspace(0.0, 16 * 65504.0, 128).astype(np.float32),
        "both": np.where(i % 2 == 0, -7.0e7, 7.0e7).astype(np.float32),
    }


def _append_values(v_rows, positions, max_pages=1):
    """Append value rows (each at its own position of sequence 0, every KV head the same row) with
    random keys; returns (tensors, error word)."""
    T = len(v_rows)
    bt = torch.arange(max_pages, dtype=torch.int32).reshape(1, max_pages)
    tensors, cache = alloc_int4_cache(max_pages, HKV, bt)
    rng = np.random.default_rng(7)
    k = torch.from_numpy(rng.standard_normal((T, HKV, 128)).astype(np.float32)).cuda()
    v = torch.from_numpy(np.repeat(np.stack(v_rows)[:, None, :], HKV, axis=1)).cuda()
    seq = torch.zeros(T, dtype=torch.int32, device="cuda")
    pos = torch.tensor(positions, dtype=torch.int32, device="cuda")
    Mk = torch.eye(128, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq_rotate_quant_append(cache, Mk, k, v, seq, pos, err)
    torch.cuda.synchronize()
    return tensors, int(err.item())


def _check_rows(orc, names, rows, tensors):
    c, sb, ob, fl = orc.quantize_int4(np.stack(rows))
    for h in range(HKV):
        got = unpack_int4(tensors, 0, h, len(rows))
        for i, name in enumerate(names):
            assert np.array_equal(got["vc"][i], c[i]), f"{name} head {h}: codes {got['vc'][i][:8]} vs {c[i][:8]}"
            assert int(got["vs"][i]) == int(sb[i]), f"{name} head {h}: scale {int(got['vs'][i]):#06x} vs {int(sb[i]):#06x}"
            assert int(got["vo"][i]) == int(ob[i]), f"{name} head {h}: offset {int(got['vo'][i]):#06x} vs {int(ob[i]):#06x}"
    return c, sb, ob, fl


def test_golden_and_edge_rows_bit_exact(orc):
    golden = pins.quantizer_case_rows()
    want = pins.golden_quantizer_cases()
    rows = dict(golden)
    rows.update(_edge_rows())
    names = list(rows)
    tensors, err = _append_values([rows[n] for n in names], list(range(len(names))))
    c, sb, ob, fl = _check_rows(orc, names, [rows[n] for n in names], tensors)
    assert err == 0 and not fl.any(), f"error word {err:#x}, oracle flags {fl}"
    for i, name in enumerate(names):
        if name in want:  # the file's hand-worked bits, independently of the oracle
            assert (int(sb[i]), int(ob[i])) == want[name], name
    i_sub = names.index("const_1p3")
    assert int(sb[i_sub]) == 0x00DB  # an fp16 subnormal scale
    for n in ("min_neg_zero", "all_neg_zero", "mixed_zeros"):
        assert int(ob[names.index(n)]) == 0x0000, f"{n}: a zero offset is stored as +0"
    for n in ("all_neg_zero", "mixed_zeros"):
        assert int(sb[names.index(n)]) == 0x0000, f"{n}: a zero scale is stored as +0"
    assert int(ob[names.index("huge_positive")]) == 0x7BFF  # rounded down to 65504, not saturated


@pytest.mark.parametrize("name", sorted(_range_rows()))
def test_range_saturation_flagged(orc, name):
    row = _range_rows()[name]
    tensors, err = _append_values([row], [5])
    c, sb, ob, fl = orc.quantize_int4(row[None])
    assert fl[0] == 2, f"oracle flags {fl[0]}"
    assert err == DEVERR_RANGE, f"error word {err:#x}"
    got = unpack_int4(tensors, 0, 1, 6)
    assert np.array_equal(got["vc"][5], c[0])
    assert (int(got["vs"][5]), int(got["vo"][5])) == (int(sb[0]), int(ob[0]))
    assert int(sb[0]) in (0x7BFF, 0x0000) or int(ob[0]) == 0xFBFF  # saturated at the fp16 limit


def test_append_past_capacity_flagged_and_skipped():
    row = pins.quantizer_case_rows()["ramp"]
    tensors, err = _append_values([row, row], [63, 64])  # capacity is one page: 64 positions
    assert err == DEVERR_POS, f"error word {err:#x}"
    pages = tensors["pages"].cpu().numpy()
    assert pages.shape[0] == 1  # position 64 has no page: only slot 63 may have been written
    written = np.zeros(pages.shape[2], bool)
    for lo, hi in ((63 * 64, 64 * 64), (4096 + 63 * 64, 4096 + 64 * 64), (8192 + 4 * 63, 8192 + 4 * 64),
                   (8448 + 4 * 63, 8448 + 4 * 64)):
        written[lo:hi] = True
    assert not pages[:, :, ~written].any(), "a byte outside slot 63 was written"


def test_e4m3_saturation_and_signed_zero(orc):
    """Window cache: code = e4m3(x / scale), nearest even, saturating to +-448 (stock FP8 format)."""
    scale = 0.5
    i = np.arange(128, dtype=np.float64)
    small = (i - 64) * 2.0 ** -12  # x / scale = (i - 64) 2^-11: zeros and subnormal e4m3 codes
    small[::5] = -0.0
    rows = np.stack([
        np.where(i % 2 == 0, 1.0, -1.0) * (200.0 + 30.0 * i),  # x / scale from 400 to 8000
        small,
        np.full(128, 1.0e30),
    ]).astype(np.float32)
    T = rows.shape[0]
    tensors, ring = alloc_fp8_ring(1, HKV, 576)
    k = torch.from_numpy(np.repeat(rows[:, None, :], HKV, axis=1)).cuda()
    v = torch.from_numpy(np.repeat(-rows[:, None, :], HKV, axis=1)).cuda()
    seq = torch.zeros(T, dtype=torch.int32, device="cuda")
    pos = torch.arange(T, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq_fp8_append(ring, k, v, seq, pos, scale, scale, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    from gpu_util import unpack_fp8
    want_k = orc.quantize_fp8(rows, scale)
    want_v = orc.quantize_fp8(-rows, scale)
    assert (want_k[0][np.abs(rows[0] / scale) > 464] & 0x7F == 0x7E).all()  # the oracle saturates
    for h in range(HKV):
        gk, gv = unpack_fp8(tensors, 0, h, np.arange(T))
        assert np.array_equal(gk, want_k), f"K codes head {h}"
        assert np.array_equal(gv, want_v), f"V codes head {h}"
