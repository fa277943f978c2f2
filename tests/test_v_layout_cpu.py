"""The int4 cache's V code layout (host logic, no GPU).

V records store each token's codes of dims 4l..4l+3 in one 16-bit element as sign/magnitude
fields of c - 7.5 so that the attention kernels read them as exact f16 subnormals with integer
ops alone (see v_encode4 / unpack8_v in the CUDA sources). This test restates the encoding,
checks that the test-side decoder used by the parity tests inverts it for all 65,536 4-code
elements, and emulates the kernels' four bit views (mask, shift, byte swap) to confirm each
gives (c - 7.5) 2^(k - 23) with k = 0, 4, 2, 6 in both halves of a 32-bit register.
"""

import itertools

import numpy as np

from gpu_util import _v_codes

K_OF_DIM = (0, 4, 2, 6)


def _enc(c):
    s = [int(x < 8) for x in c]
    e = [(7 - x) if x < 8 else x - 8 for x in c]
    return (e[0] << 1) | (s[0] << 15) | (e[1] << 4) | (s[1] << 14) | (e[2] << 11) | (s[2] << 7) | (e[3] << 8) | s[3]


def _view(x, i):
    m = 0xFFFFFFFF
    if i == 0:
        return (x & 0x800E800E) | 0x00010001
    if i == 1:
        return (((x << 1) & m) & 0x80E080E0) | 0x00100010
    r = ((x & 0xFF) << 8) | ((x >> 8) & 0xFF) | (((x >> 16) & 0xFF) << 24) | (((x >> 24) & 0xFF) << 16)
    if i == 2:
        return (r & 0x80388038) | 0x00040004
    return (((r << 7) & m) & 0x83808380) | 0x00400040


def test_v_layout_roundtrip_and_views():
    allc = np.array(list(itertools.product(range(16), repeat=4)))
    u = np.array([_enc(c) for c in allc], np.uint64)
    assert len(set(u.tolist())) == 65536
    rec = np.zeros((65536, 64), np.uint8)
    rec[:, 0] = u & 255
    rec[:, 1] = u >> 8
    assert (_v_codes(rec)[:, :4] == allc).all()
    x = u | (u[::-1] << 16)  # a register holding two elements
    for i in range(4):
        h = _view(x, i)
        lo = (h & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
        hi = (h >> 16).astype(np.uint16).view(np.float16).astype(np.float64)
        scale = 2.0 ** (K_OF_DIM[i] - 23)
        assert np.array_equal(lo, (allc[:, i] - 7.5) * scale)
        assert np.array_equal(hi, (allc[::-1, i] - 7.5) * scale)
