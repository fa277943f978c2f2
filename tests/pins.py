"""Pins of the oracle against things other than itself.

Each check takes an oracle.Oracle and raises AssertionError when the oracle
disagrees with a closed form, an invariant, a hand-worked case, an independent
library routine, or a claim of "Serving Kolibri-1 with a 4-bit KV cache". The
checks are plain functions so that tests/test_oracle_mutations.py can run them
against builds of the oracle with a planted mistake and see that one fails.
"""

from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
SM = 1.0 / math.sqrt(128.0)


def _rng(seed=0):
    return np.random.default_rng(seed)


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.rstrip("\n") for ln in f if ln.strip() and not ln.lstrip().startswith("#")]


def _fwht(x):
    """Fast Walsh-Hadamard transform (unnormalised, Sylvester order) along the last axis."""
    x = np.array(x, dtype=np.float64, copy=True)
    h = 1
    n = x.shape[-1]
    while h < n:
        y = x.reshape(x.shape[:-1] + (n // (2 * h), 2, h))
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        x = y.reshape(x.shape)
        h *= 2
    return x


# ------------------------------------------------------------------ rotation

def check_hadamard(O):
    """Section "What we do": H is the 128x128 Hadamard matrix (Sylvester order)."""
    H = O.hadamard(128).astype(np.int64)
    assert set(np.unique(H)) == {-1, 1}
    assert np.array_equal(H @ H.T, 128 * np.eye(128, dtype=np.int64)), "H H^T != 128 I"
    H4 = np.array([[int(v) for v in ln.split()] for ln in _golden_lines("hadamard4.txt")])
    assert np.array_equal(H[:4, :4], H4)
    i = np.arange(128)
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i[:, None] & i[None, :])
    assert np.array_equal(H, np.where(pc % 2 == 0, 1, -1)), "not Sylvester ordering"


def check_signs(O):
    """Sign vector: top bit of successive splitmix64 outputs (published test vector)."""
    ref = [int(x) for x in _golden_lines("splitmix64_seed1234567.txt")]
    s = O.signs(1234567, 5)
    assert list(s) == [-1 if (v >> 63) else 1 for v in ref]
    for seed in (1, 2, 99):
        s = O.signs(seed, 128)
        assert set(np.unique(s)) <= {-1, 1} and 32 < int((s < 0).sum()) < 96


def check_rotation(O):
    """R = H diag(s)/sqrt(128) is orthogonal; R x equals FWHT(s*x)/sqrt(128); columns carry s."""
    for seed in (5, 77):
        R64, R32 = O.rotation(seed)
        assert np.abs(R64 @ R64.T - np.eye(128)).max() < 1e-14
        assert np.array_equal(R32, R64.astype(np.float32))
        s = O.signs(seed, 128).astype(np.float64)
        x = _rng(seed).standard_normal((6, 128))
        Rx = x @ R64.T
        assert np.abs(Rx - _fwht(x * s) / math.sqrt(128)).max() < 1e-12, "FWHT closed form"
        H = O.hadamard(128).astype(np.float64)
        for j in (0, 3, 127):  # diag(s) on the right scales column j by s_j
            assert np.allclose(R64[:, j], s[j] * H[:, j] / math.sqrt(128), atol=0, rtol=1e-15)


def check_fold(O):
    """Section "What we do": q.k is unchanged by the rotation and by moving g_k to the query.
    (M_q n(q)) . (M_k n(k)) == (g_q n(q)) . (g_k n(k)); the cache holds R n(k) (no gain)."""
    rng = _rng(3)
    R64, R32 = O.rotation(11)
    gq = rng.uniform(0.5, 1.5, 128).astype(np.float32)
    gk = rng.uniform(0.5, 1.5, 128).astype(np.float32)
    Mq, Mk = O.fold(R32, gq, gk)
    assert np.array_equal(Mk, R32), "keys are cached as R n(k)"
    q = rng.standard_normal((8, 128)).astype(np.float32)
    k = rng.standard_normal((8, 128)).astype(np.float32)
    nq = q.astype(np.float64) / np.sqrt((q.astype(np.float64) ** 2).mean(1, keepdims=True) + 1e-6)
    nk = k.astype(np.float64) / np.sqrt((k.astype(np.float64) ** 2).mean(1, keepdims=True) + 1e-6)
    lhs = (nq @ Mq.astype(np.float64).T) @ (nk @ Mk.astype(np.float64).T).T
    rhs = (nq * gq) @ (nk * gk).T
    assert np.abs(lhs - rhs).max() <= 1e-5 * np.abs(rhs).max(), "fold changes q.k"


# ------------------------------------------------------------------ prologue

def check_prologue(O):
    """fp32 prologue close to the fp64 value M x/sqrt(mean x^2 + eps); exact for power-of-2 rescaling."""
    rng = _rng(4)
    _, R32 = O.rotation(21)
    M = R32 * rng.uniform(0.5, 1.5, 128).astype(np.float32)[None, :]
    x = rng.standard_normal((64, 128)).astype(np.float32)
    x[:, 7] *= 9.0
    y = O.prologue(M, x, 1e-6)
    xd = x.astype(np.float64)
    ref = (xd / np.sqrt((xd ** 2).mean(1, keepdims=True) + 1e-6)) @ M.astype(np.float64).T
    assert np.abs(y - ref).max() <= 2e-6 * np.abs(ref).max(), "prologue far from M n(x)"
    y0 = O.prologue(M, x, 0.0)
    y4 = O.prologue(M, x * np.float32(4.0), 0.0)
    assert np.array_equal(y0, y4), "RMS norm must remove a power-of-two scale exactly"
    ones = O.prologue(np.eye(128, dtype=np.float32), np.full((1, 128), 3.0, np.float32), 0.0)
    assert np.array_equal(ones, np.ones((1, 128), np.float32)), "n(c 1) = 1 for eps 0"


def check_prologue_fwht(O):
    """Second prologue specification, R n(x) = H (s n(x)) / sqrt(128) through the FWHT:
    a one-hot input reproduces s_k times column k of the (independently built) Hadamard matrix
    with equal magnitudes; random inputs stay within fp32 error of the fp64 products R n(x) and
    R diag(g_q g_k) n(x); the multipliers are s and fp32(s g_q g_k)."""
    H = O.hadamard(128).astype(np.int64)
    for seed, k in ((5, 0), (5, 77), (31, 126)):
        s = O.signs(seed, 128)
        wq, wk = O.fold_fwht(s, np.ones(128, np.float32), np.ones(128, np.float32))
        assert np.array_equal(wk, s.astype(np.float32)), "key multipliers are the signs"
        x = np.zeros((1, 128), np.float32)
        x[0, k] = 3.0
        y = O.prologue_fwht(wk, x, 0.0)[0]
        assert np.array_equal(np.sign(y).astype(np.int64), int(s[k]) * H[:, k]), "butterflies != Hadamard column"
        assert np.all(np.abs(y) == np.abs(y[0])), "one-hot transform has unequal magnitudes"
        assert abs(float(np.abs(y[0])) - 1.0) < 1e-6, "n(3 e_k) = sqrt(128) e_k, so |R n| = 1"
    rng = _rng(6)
    x = rng.standard_normal((32, 128)).astype(np.float32)
    x[:, 3] *= 9.0
    xd = x.astype(np.float64)
    nd = xd / np.sqrt((xd ** 2).mean(1, keepdims=True) + 1e-6)
    R64, _ = O.rotation(41)
    s = O.signs(41, 128)
    gq = rng.uniform(0.5, 1.5, 128).astype(np.float32)
    gk = rng.uniform(0.5, 1.5, 128).astype(np.float32)
    wq, wk = O.fold_fwht(s, gq, gk)
    assert np.array_equal(wq, (s.astype(np.float64) * gq.astype(np.float64) * gk.astype(np.float64)).astype(np.float32))
    for w, M in ((wk, R64), (wq, R64 * (gq.astype(np.float64) * gk.astype(np.float64))[None, :])):
        y = O.prologue_fwht(w, x, 1e-6)
        ref = nd @ M.T
        assert np.abs(y - ref).max() <= 2e-6 * np.abs(ref).max(), "FWHT prologue far from its fp64 value"
    y0 = O.prologue_fwht(wk, x, 0.0)
    y4 = O.prologue_fwht(wk, x * np.float32(4.0), 0.0)
    assert np.array_equal(y0, y4), "RMS norm must remove a power-of-two scale exactly"


# ------------------------------------------------------------------ quantiser

def _golden_quant_cases():
    cases = {}
    for ln in _golden_lines("quantizer_cases.txt"):
        name, how, sb, ob, codes = [p.strip() for p in ln.split("|")]
        cases[name] = (int(sb, 16), int(ob, 16), codes)
    return cases


def quantizer_case_rows():
    """The 128-vectors of tests/golden/quantizer_cases.txt, built as the file's second column says."""
    i = np.arange(128)
    return {
        "ramp": (0.5 * (i % 16)).astype(np.float32),
        "const_exact": np.full(128, 1.5, np.float32),
        "const_1p3": np.full(128, 1.3, np.float32),
        "ties": np.array([0, 15] + [k + 0.5 for k in range(15)] + [0] * 111, np.float32),
        "neg_offset": np.array([-1.0001] + [0] * 127, np.float32),
    }


def golden_quantizer_cases():
    """name -> (scale bits, offset bits) from tests/golden/quantizer_cases.txt."""
    return {k: v[:2] for k, v in _golden_quant_cases().items()}


def check_quantizer_cases(O):
    g = _golden_quant_cases()
    i = np.arange(128)
    ys = quantizer_case_rows()
    expect_codes = {
        "ramp": i % 16,
        "const_exact": np.zeros(128),
        "const_1p3": np.full(128, 15),
        "ties": np.array([0, 15, 0, 2, 2, 4, 4, 6, 6, 8, 8, 10, 10, 12, 12, 14, 14] + [0] * 111),
        "neg_offset": np.array([0] + [15] * 127),
    }
    for name, y in ys.items():
        c, s, o, f = O.quantize_int4(y[None])
        sb, ob, _ = g[name]
        assert int(s[0]) == sb and int(o[0]) == ob, (name, hex(int(s[0])), hex(int(o[0])))
        assert np.array_equal(c[0], expect_codes[name].astype(np.uint8)), name
        assert int(f[0]) == 0


def check_quantizer_bounds(O):
    """Every dequantised value within s/2 of its input; offset rounded down, scale up."""
    rng = _rng(5)
    y = (rng.standard_normal((2000, 128)) * rng.uniform(0.01, 30, (2000, 1))).astype(np.float32)
    y[:50] += 1000.0
    c, sb, ob, f = O.quantize_int4(y)
    assert (f == 0).all() and c.max() <= 15
    s = np.array([O.fp16_value(int(v)) for v in sb])
    o = np.array([O.fp16_value(int(v)) for v in ob])
    yd = y.astype(np.float64)
    mn, mx = yd.min(1), yd.max(1)
    assert (o <= mn).all(), "offset must not exceed min"
    assert (s * 15 >= (mx - o) * (1 - 2 ** -23)).all(), "scale must cover the span"
    deq = O.dequant_int4(c, sb, ob)
    slack = s / 2 + 4 * np.spacing(np.maximum(np.abs(yd).max(1), np.abs(o)).astype(np.float32)).astype(np.float64)
    assert (np.abs(deq - yd).max(1) <= slack).all(), "dequant error above s/2"
    # the largest element maps to the top code
    top = c[np.arange(len(c)), yd.argmax(1)]
    assert (top == 15).all()


def check_quantizer_flags(O):
    y = np.zeros((3, 128), np.float32)
    y[0, 5] = np.nan
    y[1, 9] = -1e6          # offset below -65504 -> saturated
    y[2, :] = np.linspace(-3e5, 3e5, 128)
    _, _, _, f = O.quantize_int4(y)
    assert f[0] & 1 and f[1] & 2 and f[2] & 2


# ------------------------------------------------------------------ converters

def check_fp16_converter(O):
    rng = _rng(6)
    bits = rng.integers(0, 2 ** 32, 3000, dtype=np.uint64).astype(np.uint32)
    xs = list(bits.view(np.float32))
    xs += list(np.float32([0.0, -0.0, 65504, 65519.99, 65520, 65536, -70000, 6e-8, 2.98e-8, 1e-9, -1e-9,
                           1.0001, -1.0001, 3.0e-5, np.inf, -np.inf]))
    for x in xs:
        x = np.float32(x)
        if np.isnan(x):
            continue
        with np.errstate(over="ignore"):
            rn = np.float16(x)
        b_rn = int(np.array([rn], np.float16).view(np.uint16)[0])
        assert O.fp16_round_bits(x, 0) == b_rn, ("RN", x)
        # directed rounding from RN and one fp16 step
        x64 = float(x)
        r = float(rn)
        down = rn if r <= x64 else np.nextafter(rn, np.float16(-np.inf))
        with np.errstate(over="ignore"):
            up = rn if r >= x64 else np.nextafter(rn, np.float16(np.inf))
        if np.isinf(rn) and not np.isinf(x):
            down = np.float16(65504) if x > 0 else np.float16(-np.inf)
            up = np.float16(np.inf) if x > 0 else np.float16(-65504)
        for d, want in ((-1, down), (1, up)):
            wb = int(np.array([want], np.float16).view(np.uint16)[0])
            got = O.fp16_round_bits(x, d)
            if want == 0 and got in (0, 0x8000):  # sign of a zero result is not pinned here
                continue
            assert got == wb, ("dir", d, x, hex(got), hex(wb))
    for h in range(0, 65536, 7):
        v = np.array([h], np.uint16).view(np.float16)[0]
        if np.isnan(v):
            continue
        assert O.fp16_value(h) == float(v)


def check_e4m3_converter(O):
    import torch
    codes = torch.arange(256, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        if np.isnan(vals[c]):
            assert math.isnan(O.e4m3_value(c))
        else:
            assert O.e4m3_value(c) == float(vals[c]), c
    rng = _rng(7)
    xs = np.concatenate([rng.uniform(-448, 448, 3000), rng.standard_normal(2000) * 0.01,
                         rng.standard_normal(500) * 1e-3]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, r in zip(xs, ref):
        assert O.e4m3_encode(x) == int(r), (x, O.e4m3_encode(x), int(r))
    for x in (448.0, 460.0, 464.0, 500.0, 1e9, float("inf")):  # saturating conversion
        assert O.e4m3_encode(x) == 0x7E and O.e4m3_encode(-x) == 0xFE, x


# ------------------------------------------------------------------ attention

def _int4_record(codes_row, s_bits, o_bits, L):
    kc = np.tile(np.asarray(codes_row, np.uint8), (L, 1))
    return kc, np.full(L, s_bits, np.uint16), np.full(L, o_bits, np.uint16)


def check_attention_closed_forms(O):
    rng = _rng(8)
    L = 37
    kc = rng.integers(0, 16, (L, 128)).astype(np.uint8)
    vc = rng.integers(0, 16, (L, 128)).astype(np.uint8)
    ks = np.full(L, 0x3800, np.uint16)    # 0.5
    ko = np.full(L, 0xBC00, np.uint16)    # -1
    vs = np.full(L, 0x3400, np.uint16)    # 0.25
    vo = np.full(L, 0xC000, np.uint16)    # -2
    q = rng.standard_normal((3, 128)).astype(np.float32)
    vhat = vc.astype(np.float64) * 0.25 - 2.0
    # one visible key: the output is that key's value
    out = O.attention_int4(q, [1, 1, 1], kc, ks, ko, vc, vs, vo, SM)
    assert np.abs(out - vhat[0]).max() < 1e-12, "L=1 -> o = v0"
    # all keys identical: uniform weights -> mean of values
    kce = np.tile(kc[:1], (L, 1))
    out = O.attention_int4(q, [L, L, L], kce, ks, ko, vc, vs, vo, SM)
    assert np.abs(out - vhat.mean(0)).max() < 1e-12, "equal keys -> mean"
    # 2-token hand case: k0 = 0, k1 = 1-vector, q = (a,0,..) with sm*a = ln 2 -> p = (1/3, 2/3);
    # v0 = 0, v1 = 2 -> o = 4/3
    a = np.float32(math.log(2.0) / SM)
    qq = np.zeros((1, 128), np.float32)
    qq[0, 0] = a
    k2 = np.zeros((2, 128), np.uint8)
    k2[1] = 1
    v2 = np.zeros((2, 128), np.uint8)
    v2[1] = 2
    one = np.full(2, 0x3C00, np.uint16)
    zero = np.zeros(2, np.uint16)
    out = O.attention_int4(qq, [2], k2, one, zero, v2, one, zero, SM)
    assert np.abs(out - 4.0 / 3.0).max() < 1e-6, out[0, :3]
    # offsets enter the dequantised values: shifting every key by a constant along q's orthogonal
    # complement leaves scores unchanged; shifting values by c shifts the output by c.
    vo2 = np.full(L, 0x4000, np.uint16)  # +2 instead of -2
    o1 = O.attention_int4(q, [L] * 3, kc, ks, ko, vc, vs, vo, SM)
    o2 = O.attention_int4(q, [L] * 3, kc, ks, ko, vc, vs, vo2, SM)
    assert np.abs((o2 - o1) - 4.0).max() < 1e-11, "value offset"
    # a dominant key: huge score gap -> that key's value
    qd = np.zeros((1, 128), np.float32)
    qd[0] = 50.0
    kd = np.zeros((L, 128), np.uint8)
    kd[13] = 15
    out = O.attention_int4(qd, [L], kd, np.full(L, 0x3C00, np.uint16), np.zeros(L, np.uint16), vc, vs, vo, SM)
    assert np.abs(out[0] - vhat[13]).max() < 1e-9, "dominant key"


def check_attention_structure(O):
    rng = _rng(9)
    L = 50
    kc = rng.integers(0, 16, (L, 128)).astype(np.uint8)
    vc = rng.integers(0, 16, (L, 128)).astype(np.uint8)
    ks = rng.integers(0x2C00, 0x3C00, L).astype(np.uint16)
    ko = rng.integers(0xBC00, 0xC200, L).astype(np.uint16)
    vs = rng.integers(0x2C00, 0x3C00, L).astype(np.uint16)
    vo = rng.integers(0xBC00, 0xC200, L).astype(np.uint16)
    q = rng.standard_normal((4, 128)).astype(np.float32)
    vis = np.array([L, 1, 17, 33])
    out = O.attention_int4(q, vis, kc, ks, ko, vc, vs, vo, SM)
    # causal prefix: row with vis=v equals a full attention over the first v positions
    for r in range(4):
        v = int(vis[r])
        o = O.attention_int4(q[r:r + 1], [v], kc[:v], ks[:v], ko[:v], vc[:v], vs[:v], vo[:v], SM)
        assert np.array_equal(o[0], out[r])
    # permutation of the cache positions does not change a full-visibility row
    p = rng.permutation(L)
    o = O.attention_int4(q[:1], [L], kc[p], ks[p], ko[p], vc[p], vs[p], vo[p], SM)
    assert np.abs(o[0] - out[0]).max() < 1e-12
    # rotation invariance of the fp64 attention (nothing is rotated back)
    R64, _ = O.rotation(3)
    K = rng.standard_normal((L, 128))
    V = rng.standard_normal((L, 128))
    qq = rng.standard_normal((2, 128))
    a = O.attention_f64(qq, K, V, SM)
    b = O.attention_f64(qq @ R64.T, K @ R64.T, V, SM)
    assert np.abs(a - b).max() < 1e-12


def check_attention_fp8(O):
    rng = _rng(10)
    L = 40
    kc = rng.integers(0, 0x7E, (L, 128)).astype(np.uint8)
    vc = rng.integers(0, 0x7E, (L, 128)).astype(np.uint8)
    q = rng.standard_normal((2, 128)).astype(np.float32)
    lo = np.array([5, 0])
    hi = np.array([20, 0])
    out = O.attention_fp8(q, lo, hi, kc, vc, 0.05, 0.1, SM)
    vals = np.array([O.e4m3_value(c) for c in range(256)])
    assert np.abs(out[1] - vals[vc[0]] * 0.1).max() < 1e-12, "single key"
    kc2 = kc.copy()
    kc2[:5] = 0x55
    kc2[21:] = 0x22
    vc2 = vc.copy()
    vc2[:5] = 0x11
    out2 = O.attention_fp8(q, lo, hi, kc2, vc2, 0.05, 0.1, SM)
    assert np.array_equal(out[0], out2[0]), "keys outside the window must not matter"
    kce = np.tile(kc[:1], (L, 1))
    out3 = O.attention_fp8(q, lo, hi, kce, vc, 0.05, 0.1, SM)
    assert np.abs(out3[0] - (vals[vc[5:21]] * 0.1).mean(0)).max() < 1e-12, "equal keys -> mean"


# ------------------------------------------------------------------ claims of the page

def check_channel_ratio(O):
    """Section "What we do": the largest key channel against the average one. The hand-worked
    matrix of tests/golden/channel_ratio.txt has the exact ratio 8/3; the statistic ignores signs,
    the order of tokens and channels and a common scale, and is 1 for a single channel."""
    lines = _golden_lines("channel_ratio.txt")
    rows = [[float(v) for v in ln.split()] for ln in lines if not ln.startswith("ratio")]
    num, den = (int(v) for v in [ln for ln in lines if ln.startswith("ratio")][0].split()[1].split("/"))
    k = np.array(rows, np.float64)
    assert abs(O.channel_ratio(k) - num / den) < 1e-12, ("hand-worked ratio", O.channel_ratio(k))
    rng = _rng(12)
    x = rng.standard_normal((33, 16))
    x[:, 5] *= 6.0
    r = O.channel_ratio(x)
    assert abs(O.channel_ratio(-x) - r) < 1e-12
    assert abs(O.channel_ratio(x[rng.permutation(33)][:, rng.permutation(16)]) - r) < 1e-12
    assert abs(O.channel_ratio(0.25 * x) - r) < 1e-12
    assert abs(O.channel_ratio(x[:, :1]) - 1.0) < 1e-15


def check_claims(O):
    """Section "What we do": rotation lowers the max/mean key channel ratio (<= 2.2 after),
    and 4-bit keys move attention less with the rotation; FP8 keys move it least."""
    import synth
    seed = 1
    gq, gk = synth.gains(seed, 0)
    q = synth.q_rows(seed, 0, 0, 4096, 1, 64, False).reshape(-1, 128)
    k = synth.kv_rows(seed, 0, 0, 0, 4096, 1, "k", False).reshape(-1, 128)
    v = synth.kv_rows(seed, 0, 0, 0, 4096, 1, "v", False).reshape(-1, 128)
    _, R32 = O.rotation(synth.rotation_seed(seed, 0))
    c = O.claim_errors(q, k, v, gq, gk, R32)
    assert c["ratio_unrotated"] > 5.0 and c["ratio_rotated"] <= 2.2, c
    assert c["int4_rotated"] < c["int4_unrotated"], c
    assert c["fp8"] < c["int4_rotated"], c
    return c


ALL_CHECKS = [
    check_hadamard, check_signs, check_rotation, check_fold, check_prologue, check_prologue_fwht,
    check_quantizer_cases,
    check_quantizer_bounds, check_quantizer_flags, check_fp16_converter, check_e4m3_converter,
    check_attention_closed_forms, check_attention_structure, check_attention_fp8, check_channel_ratio,
    check_claims,
]
