"""C-ABI checks that need no GPU: the library loads and exports every call kvq.h declares,
the host-only steps (rotation, gain fold) match the oracle bit for bit, and host-side
argument checks reject bad calls before any CUDA work."""

import ctypes
import os
import re

import numpy as np
import pytest

import quantized_kv_cache_fold_gb300 as kvq
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "kvq.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", txt)))


def test_exports_every_declared_symbol():
    names = declared_symbols()
    assert len(names) >= 8
    for n in names:
        assert hasattr(kvq.lib, n), f"libkvq.so does not export {n}"


@pytest.mark.parametrize("seed", [0, 1, 1234567, 2**63 + 5])
def test_rotation_matches_oracle(orc, seed):
    R, s = kvq.kvq_build_rotation(seed)
    R64, R32 = orc.rotation(seed)
    assert np.array_equal(R, R32)
    assert np.array_equal(s, orc.signs(seed, 128))


def test_fold_matches_oracle(orc):
    for layer in range(3):
        gq, gk = synth.gains(7, layer)
        R, _ = kvq.kvq_build_rotation(synth.rotation_seed(7, layer))
        Mq, Mk = kvq.kvq_fold_qk(R, gq, gk)
        oMq, oMk = orc.fold(R, gq, gk)
        assert np.array_equal(Mq, oMq) and np.array_equal(Mk, oMk)


def test_status_strings():
    assert kvq.status_string(0) == "ok"
    assert "invalid" in kvq.status_string(1)


def test_workspace_bytes():
    assert kvq.kvq_decode_workspace_bytes(8, 1, 20, 4) > 0
    assert kvq.kvq_decode_workspace_bytes(8, 9, 20, 4) == 0      # S > 8
    assert kvq.kvq_decode_workspace_bytes(8, 8, 56, 4) == 0      # 8*14 rows > 48
    assert kvq.kvq_decode_workspace_bytes(0, 1, 20, 4) == 0
    assert kvq.kvq_decode_workspace_bytes(8, 1, 20, 3) == 0      # 20 % 3


def _fake_cache(**over):
    d = dict(pages=0x10000, block_table=0x50000, num_seqs=4, max_pages_per_seq=8, num_pages=32, num_kv_heads=4,
             page_size=64, head_dim=128)
    d.update(over)
    return kvq.Int4Cache(**d)


def _attn(cache, **over):
    a = dict(Mq=0x60000, Mk=0x70000, q=0x80000, dtype=1, B=2, S=1, Hq=20, ctx=0x90000, k_new=None, v_new=None,
             sm=0.088, eps=1e-6, out=0xA0000, ws=0xB0000, ws_bytes=1 << 30, qrot=None, err=0xC0000, stream=None)
    a.update(over)
    return kvq.lib.kvq_decode_attn_int4(ctypes.byref(cache), a["Mq"], a["Mk"], a["q"], a["dtype"], a["B"], a["S"],
                                        a["Hq"], a["ctx"], a["k_new"], a["v_new"], a["sm"], a["eps"], a["out"],
                                        a["ws"], a["ws_bytes"], a["qrot"], a["err"], a["stream"])


def test_host_validation_rejects_before_launch():
    c = _fake_cache()
    assert _attn(_fake_cache(head_dim=64)) == 2
    assert _attn(_fake_cache(page_size=32)) == 2
    assert _attn(c, S=9) == 2
    assert _attn(c, Hq=21) == 2
    assert _attn(c, B=5) == 1                       # more sequences than block-table rows
    assert _attn(c, ws=0xB0010) == 1                # workspace not 256-byte aligned
    assert _attn(c, ws_bytes=1024) == 1             # workspace too small
    assert _attn(c, k_new=0xD0000) == 1             # k_new without v_new
    assert _attn(c, q=0) == 1
    assert _attn(c, err=0) == 1
    assert _attn(c, sm=float("nan")) == 1
    assert _attn(_fake_cache(pages=0x10008)) == 1  # cache array not 16-byte aligned
    ring = kvq.Fp8Ring(0x10000, 4, 4, 576, 128)
    f = kvq.lib.kvq_decode_attn_fp8_swa
    assert f(ctypes.byref(ring), 0x80000, 1, 2, 1, 20, 0x90000, 600, None, None, 0.01, 0.01, 0.088, 0xA0000,
             0xB0000, 1 << 30, 0xC0000, None) == 1  # window larger than the ring
    bad_ring = kvq.Fp8Ring(0x10000, 4, 4, 500, 128)
    assert f(ctypes.byref(bad_ring), 0x80000, 1, 2, 1, 20, 0x90000, 400, None, None, 0.01, 0.01, 0.088, 0xA0000,
             0xB0000, 1 << 30, 0xC0000, None) == 1  # capacity not a multiple of 64
    shape = (ctypes.c_int32 * 4)()
    plan = kvq.lib.kvq_fp8_swa_plan
    assert plan(500, 8, 1, 20, 4, shape) == 1       # capacity not a multiple of 64
    assert plan(576, 8, 9, 20, 4, shape) == 2       # more than 8 rows
    assert plan(576, 8, 1, 21, 4, shape) == 2       # query heads not a multiple of KV heads
    assert plan(576, 0, 1, 20, 4, shape) == 1
    assert plan(576, 8, 1, 20, 4, None) == 1
    assert kvq.lib.kvq_build_rotation(1, 64, None, 0x1000) == 2
    assert kvq.lib.kvq_rotate_quant_append(ctypes.byref(c), 0x1000, 0x2000, 0x3000, 1, 0, None, None, 1e-6, None,
                                           None) == 0  # T == 0 is a no-op


def test_stream_k_split_arithmetic():
    """The device maps page p to CTA ((p+1)n-1)//P for ranges [iP//n, (i+1)P//n); check by brute force,
    and that slot = cta + segment is injective over (cta, segment) pairs that share pages."""
    rng = np.random.default_rng(0)
    for _ in range(200):
        B = int(rng.integers(1, 9))
        Hkv = int(rng.integers(1, 5))
        np_b = rng.integers(1, 40, B)
        P = int(Hkv * np_b.sum())
        n = int(min(rng.integers(1, 64), P))
        starts = [i * P // n for i in range(n + 1)]
        owner = np.empty(P, np.int64)
        for i in range(n):
            assert starts[i + 1] > starts[i]
            owner[starts[i]:starts[i + 1]] = i
        assert all(((p + 1) * n - 1) // P == owner[p] for p in range(P))
        used = set()
        pre = np.concatenate([[0], np.cumsum(np_b)])
        for b in range(B):
            for h in range(Hkv):
                seg = b * Hkv + h
                first = Hkv * pre[b] + h * np_b[b]
                for c in sorted(set(owner[first:first + np_b[b]])):
                    slot = c + seg
                    assert slot not in used
                    used.add(slot)
        assert max(used) < n + B * Hkv


def _noalloc(cache, **over):
    a = dict(Mq=0x60000, Mk=0x70000, q=0x80000, dtype=1, B=2, S=1, Hq=20, ctx=0x90000, k_new=None, v_new=None,
             sm=0.088, eps=1e-6, out=0xA0000, qrot=None, err=0xC0000, stream=None)
    a.update(over)
    return kvq.lib.kvq_decode_attn_int4_noalloc(ctypes.byref(cache), a["Mq"], a["Mk"], a["q"], a["dtype"], a["B"],
                                                a["S"], a["Hq"], a["ctx"], a["k_new"], a["v_new"], a["sm"], a["eps"],
                                                a["out"], a["qrot"], a["err"], a["stream"])


def test_noalloc_rejects_like_the_workspace_call():
    """The allocation-free entry point returns the same status as kvq_decode_attn_int4 for the same
    bad argument, before its scratch-size check and before any CUDA call."""
    big = _fake_cache(num_seqs=1024, max_pages_per_seq=8)
    for cache, over in ((_fake_cache(), dict(B=0)), (_fake_cache(), dict(B=5)), (big, dict(B=1025)),
                        (_fake_cache(head_dim=64), {}), (_fake_cache(), dict(S=9)), (_fake_cache(), dict(q=0x80004)),
                        (_fake_cache(), dict(dtype=7)), (_fake_cache(pages=0), {}), (big, dict(B=1024, q=None))):
        want = _attn(cache, **over)
        assert want in (1, 2)
        assert _noalloc(cache, **over) == want, over
    assert _noalloc(_fake_cache(), B=0) == 1  # KVQ_ERR_INVALID_ARG
