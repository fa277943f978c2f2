"""ORACLE -- test infrastructure, not part of the product.

Plain fp64 C++ CPU restatement of the rotated 4-bit KV-cache decode path of
"Serving Kolibri-1 with a 4-bit KV cache" (section "What we do"), used only by
tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg. It shares no
code with the CUDA library in quantized_kv_cache_fold_gb300/ and neither side
imports the other.

Functions and what pins them (tests/test_oracle_pins.py):
  rotation / hadamard / signs  H H^T = 128 I in integers, R R^T = I, FWHT closed form
  fold                          (M_q n(q)).(M_k n(k)) == (g_q n(q)).(g_k n(k))
  prologue                      fp32 spec vs an fp64 evaluation (error bound), scale invariance
  quantize_int4                 |y^ - y| <= s/2 bound, ramp and tie hand cases, constant vector
  fp16 / e4m3 converters        numpy/torch float16 and torch float8_e4m3fn, nextafter for RD/RU,
                                over all 2^32 fp32 inputs (tests/test_oracle_converters.py)
  channel_ratio                 a hand-worked matrix with an exact ratio (tests/golden/channel_ratio.txt)
  attention_int4 / fp8 / f64    L=1, equal keys, dominant key, 2-token closed form, permutation
  claim_errors                  ordering claims of the page; its percentages stay unpinned
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build_cmd(out_path: str = _LIB_PATH, defines: tuple = ()) -> list:
    return (["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-ffp-contract=off", "-fno-fast-math",
             "-pthread"] + [f"-D{d}" for d in defines] +
            [os.path.join(_HERE, "oracle.cpp"), "-o", out_path])


def build(verbose: bool = False) -> str:
    subprocess.run(build_cmd(), check=True, capture_output=not verbose)
    return _LIB_PATH


def threads_default() -> int:
    return max(1, os.cpu_count() or 1)


def _bind(L):
    vp, i64, u64, f32, f64, i32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float,
                                   ctypes.c_double, ctypes.c_int)
    L.orc_hadamard.argtypes = [i32, vp]
    L.orc_signs.argtypes = [u64, i32, vp]
    L.orc_rotation.argtypes = [u64, i32, vp, vp]
    L.orc_fold.argtypes = [vp, vp, vp, i32, vp, vp]
    L.orc_prologue.argtypes = [vp, vp, i64, f32, vp, i32]
    L.orc_fold_fwht.argtypes = [vp, vp, vp, i32, vp, vp]
    L.orc_prologue_fwht.argtypes = [vp, vp, i64, f32, vp, i32]
    L.orc_quantize_int4.argtypes = [vp, i64, vp, vp, vp, vp, i32]
    L.orc_dequant_int4.argtypes = [vp, vp, vp, i64, vp]
    L.orc_convert_range.argtypes = [ctypes.c_uint32, i64, vp, vp, vp, vp, i32]
    L.orc_fp16_round_bits.argtypes = [f32, i32]
    L.orc_fp16_round_bits.restype = ctypes.c_uint16
    L.orc_fp16_value.argtypes = [ctypes.c_uint16]
    L.orc_fp16_value.restype = f64
    L.orc_e4m3_encode.argtypes = [f32]
    L.orc_e4m3_encode.restype = ctypes.c_uint8
    L.orc_e4m3_value.argtypes = [ctypes.c_uint8]
    L.orc_e4m3_value.restype = f64
    L.orc_quantize_fp8.argtypes = [vp, i64, f32, vp, i32]
    L.orc_attention_int4.argtypes = [vp, i64, vp, vp, vp, vp, vp, vp, vp, i64, f64, vp, i32]
    L.orc_attention_fp8.argtypes = [vp, i64, vp, vp, vp, vp, i64, f64, f64, f64, vp, i32]
    L.orc_attention_f64.argtypes = [vp, i64, vp, vp, i64, f64, vp, i32]
    L.orc_channel_ratio.argtypes = [vp, i64, i32]
    L.orc_channel_ratio.restype = f64
    L.orc_claim_errors.argtypes = [vp, i64, vp, vp, i64, vp, vp, vp, f32, vp, vp, i32]
    return L


def load(path: str | None = None):
    """Load liboracle.so (building it if absent). A custom path loads a variant build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """numpy-facing wrappers around one loaded build of the oracle."""

    def __init__(self, lib=None, threads: int | None = None):
        self.L = lib if lib is not None else load()
        self.threads = threads or threads_default()

    # -- rotation and fold
    def hadamard(self, n=128):
        H = np.empty((n, n), np.int8)
        self.L.orc_hadamard(n, H.ctypes.data)
        return H

    def signs(self, seed, n=128):
        s = np.empty(n, np.int8)
        self.L.orc_signs(seed & (2**64 - 1), n, s.ctypes.data)
        return s

    def rotation(self, seed, n=128):
        R64 = np.empty((n, n), np.float64)
        R32 = np.empty((n, n), np.float32)
        self.L.orc_rotation(seed & (2**64 - 1), n, R64.ctypes.data, R32.ctypes.data)
        return R64, R32

    def fold(self, R32, gq, gk):
        n = R32.shape[0]
        R32, gq, gk = _c(R32, np.float32), _c(gq, np.float32), _c(gk, np.float32)
        Mq = np.empty((n, n), np.float32)
        Mk = np.empty((n, n), np.float32)
        self.L.orc_fold(R32.ctypes.data, gq.ctypes.data, gk.ctypes.data, n, Mq.ctypes.data, Mk.ctypes.data)
        return Mq, Mk

    def fold_fwht(self, s, gq, gk):
        """Multipliers of the FWHT prologue: (w_q, w_k) = (fp32(s g_q g_k), s)."""
        s = _c(s, np.int8)
        gq, gk = _c(gq, np.float32), _c(gk, np.float32)
        n = s.shape[0]
        wq = np.empty(n, np.float32)
        wk = np.empty(n, np.float32)
        self.L.orc_fold_fwht(s.ctypes.data, gq.ctypes.data, gk.ctypes.data, n, wq.ctypes.data, wk.ctypes.data)
        return wq, wk

    def prologue_fwht(self, w, x, eps=1e-6):
        """Second specification of the prologue: c * FWHT(w * n(x)), fp32 (see oracle.cpp)."""
        w, x = _c(w, np.float32), _c(x, np.float32)
        shp = x.shape
        x2 = x.reshape(-1, 128)
        y = np.empty_like(x2)
        self.L.orc_prologue_fwht(w.ctypes.data, x2.ctypes.data, x2.shape[0], float(eps), y.ctypes.data, self.threads)
        return y.reshape(shp)

    # -- codec
    def prologue(self, M, x, eps=1e-6):
        M, x = _c(M, np.float32), _c(x, np.float32)
        shp = x.shape
        x2 = x.reshape(-1, 128)
        y = np.empty_like(x2)
        self.L.orc_prologue(M.ctypes.data, x2.ctypes.data, x2.shape[0], eps, y.ctypes.data, self.threads)
        return y.reshape(shp)

    def quantize_int4(self, y):
        y = _c(y, np.float32)
        shp = y.shape[:-1]
        y2 = y.reshape(-1, 128)
        n = y2.shape[0]
        codes = np.empty((n, 128), np.uint8)
        sb = np.empty(n, np.uint16)
        ob = np.empty(n, np.uint16)
        fl = np.empty(n, np.int32)
        self.L.orc_quantize_int4(y2.ctypes.data, n, codes.ctypes.data, sb.ctypes.data, ob.ctypes.data,
                                 fl.ctypes.data, self.threads)
        return codes.reshape(shp + (128,)), sb.reshape(shp), ob.reshape(shp), fl.reshape(shp)

    def dequant_int4(self, codes, sb, ob):
        codes, sb, ob = _c(codes, np.uint8), _c(sb, np.uint16), _c(ob, np.uint16)
        shp = codes.shape
        n = codes.reshape(-1, 128).shape[0]
        out = np.empty((n, 128), np.float64)
        self.L.orc_dequant_int4(codes.ctypes.data, sb.ctypes.data, ob.ctypes.data, n, out.ctypes.data)
        return out.reshape(shp)

    def fp16_round_bits(self, x: float, direction: int) -> int:
        """direction 0 nearest-even, -1 toward -inf, +1 toward +inf."""
        return int(self.L.orc_fp16_round_bits(float(x), int(direction)))

    def convert_range(self, first: int, n: int):
        """(rn, rd, ru, e4) of the n fp32 bit patterns first, first+1, ...: fp16 bits rounded to
        nearest-even, toward -inf and toward +inf, and the saturating e4m3 code."""
        rn = np.empty(n, np.uint16)
        rd = np.empty(n, np.uint16)
        ru = np.empty(n, np.uint16)
        e4 = np.empty(n, np.uint8)
        self.L.orc_convert_range(first & 0xFFFFFFFF, n, rn.ctypes.data, rd.ctypes.data, ru.ctypes.data,
                                 e4.ctypes.data, self.threads)
        return rn, rd, ru, e4

    def fp16_value(self, h: int) -> float:
        return float(self.L.orc_fp16_value(int(h)))

    def e4m3_encode(self, x: float) -> int:
        return int(self.L.orc_e4m3_encode(float(x)))

    def e4m3_value(self, c: int) -> float:
        return float(self.L.orc_e4m3_value(int(c)))

    def quantize_fp8(self, x, scale: float):
        x = _c(x, np.float32)
        out = np.empty(x.shape, np.uint8)
        self.L.orc_quantize_fp8(x.ctypes.data, x.size, float(scale), out.ctypes.data, self.threads)
        return out

    # -- attention
    def attention_int4(self, q, vis_len, kc, ks, ko, vc, vs, vo, sm_scale):
        q = _c(q, np.float32).reshape(-1, 128)
        vis = _c(vis_len, np.int64)
        kc, vc = _c(kc, np.uint8), _c(vc, np.uint8)
        ks, ko, vs, vo = (_c(a, np.uint16) for a in (ks, ko, vs, vo))
        L = kc.shape[0]
        assert int(vis.max()) <= L and vis.shape[0] == q.shape[0]
        out = np.empty((q.shape[0], 128), np.float64)
        self.L.orc_attention_int4(q.ctypes.data, q.shape[0], vis.ctypes.data, kc.ctypes.data, ks.ctypes.data,
                                  ko.ctypes.data, vc.ctypes.data, vs.ctypes.data, vo.ctypes.data, L,
                                  float(sm_scale), out.ctypes.data, self.threads)
        return out

    def attention_fp8(self, q, lo, hi, kc, vc, k_scale, v_scale, sm_scale):
        q = _c(q, np.float32).reshape(-1, 128)
        lo, hi = _c(lo, np.int64), _c(hi, np.int64)
        kc, vc = _c(kc, np.uint8), _c(vc, np.uint8)
        L = kc.shape[0]
        assert int(hi.max()) < L and int(lo.min()) >= 0
        out = np.empty((q.shape[0], 128), np.float64)
        self.L.orc_attention_fp8(q.ctypes.data, q.shape[0], lo.ctypes.data, hi.ctypes.data, kc.ctypes.data,
                                 vc.ctypes.data, L, float(k_scale), float(v_scale), float(sm_scale),
                                 out.ctypes.data, self.threads)
        return out

    def attention_f64(self, q, K, V, sm_scale):
        q, K, V = _c(q, np.float64).reshape(-1, 128), _c(K, np.float64), _c(V, np.float64)
        out = np.empty((q.shape[0], 128), np.float64)
        self.L.orc_attention_f64(q.ctypes.data, q.shape[0], K.ctypes.data, V.ctypes.data, K.shape[0],
                                 float(sm_scale), out.ctypes.data, self.threads)
        return out

    # -- claims
    def channel_ratio(self, keys):
        keys = _c(keys, np.float64)
        return float(self.L.orc_channel_ratio(keys.ctypes.data, keys.shape[0], keys.shape[1]))

    def claim_errors(self, q, k, v, gq, gk, R32, eps=1e-6):
        q, k, v = _c(q, np.float32), _c(k, np.float32), _c(v, np.float32)
        gq, gk, R32 = _c(gq, np.float32), _c(gk, np.float32), _c(R32, np.float32)
        err = np.empty(3, np.float64)
        ratio = np.empty(2, np.float64)
        self.L.orc_claim_errors(q.ctypes.data, q.shape[0], k.ctypes.data, v.ctypes.data, k.shape[0],
                                gq.ctypes.data, gk.ctypes.data, R32.ctypes.data, eps, err.ctypes.data,
                                ratio.ctypes.data, self.threads)
        return {"int4_unrotated": err[0], "int4_rotated": err[1], "fp8": err[2],
                "ratio_unrotated": ratio[0], "ratio_rotated": ratio[1]}
