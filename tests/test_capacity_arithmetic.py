"""Bytes per session of the capacity sweep (bench.session_bytes), against the arithmetic of the
pages' capacity claim ("Serving Kolibri-1 with a 4-bit KV cache", section "Benchmarks": the
rotated int4 cache fits +82% more sessions at 64k and +95% at 256k than the FP8 stock cache on
2x H100, since the 10 full-attention layers drop from 256 to 136 bytes per token and head and the
40 window-513 layers stay FP8). CPU only."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_session_bytes_at_the_window():
    # 10 layers x 4 heads x L x (136 or 256) B + 40 layers x 4 heads x 513 x 256 B
    assert bench.session_bytes("fp8", 65536, 513) == 671_088_640 + 21_012_480        # 692.1 MB
    assert bench.session_bytes("int4", 65536, 513) == 356_515_840 + 21_012_480       # 377.5 MB
    assert bench.session_bytes("fp8", 262144, 513) == 2_684_354_560 + 21_012_480     # 2705.4 MB
    assert bench.session_bytes("int4", 262144, 513) == 1_426_063_360 + 21_012_480    # 1447.1 MB
    for ctx, mb_fp8, mb_int4 in ((65536, 692, 378), (262144, 2705, 1447)):
        assert round(bench.session_bytes("fp8", ctx, 513) / 1e6) == mb_fp8
        assert round(bench.session_bytes("int4", ctx, 513) / 1e6) == mb_int4


def test_session_gain_shape():
    """Sessions per pool scale as the inverse bytes per session: +83% at 64k, +87% at 256k from
    the cache alone (the page's +82% / +95% are whole-server fills on 2x H100, context only)."""
    g64 = bench.session_bytes("fp8", 65536, 513) / bench.session_bytes("int4", 65536, 513) - 1
    g256 = bench.session_bytes("fp8", 262144, 513) / bench.session_bytes("int4", 262144, 513) - 1
    assert abs(g64 - 0.833) < 0.001 and abs(g256 - 0.870) < 0.001
    # the sweep's rings hold 576 slots (a multiple of 64 pages' worth, >= window + 7 verify rows)
    extra = bench.session_bytes("int4", 65536, 576) - bench.session_bytes("int4", 65536, 513)
    assert extra == 40 * 4 * 63 * 256
