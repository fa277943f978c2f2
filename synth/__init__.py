"""Seeded synthetic inputs shared by the oracle's tests and the CUDA path's bench.

This package draws numbers and nothing else: it contains none of the method's
arithmetic. It wraps ``libkvqsynth.so`` (built from ``synth.cu``), which
implements one counter-based generator (splitmix64) on the host and on the
device with the same definition, so a GPU-filled cache and a CPU oracle input
hold the same bits.

Recipe (shapes follow the decode workloads of "Serving Kolibri-1 with a 4-bit KV
cache", section "Benchmarks": head_dim 128, 20 query / 4 KV heads):

* element index of a K/V input: ((((layer*1024 + seq) << 20) + pos) * n_kv + head) * 128 + dim
* element index of a query:     ((((layer*1024 + seq) << 20) + pos) * n_q  + head) * 128 + dim
* normals: Irwin-Hall-12 on 16-bit integer uniforms, support [-6, 6], variance 1
* keys of full-attention layers: normal x alpha on 4 fixed channels per layer,
  alpha = 930/98 so that largest/mean channel magnitude is 7.5 (the ratio quoted
  in section "What we do")
* gains g_q, g_k ~ U(0.5, 1.5) per channel and layer
* FP8 sliding-window layers: keys, values and queries plain normals
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libkvqsynth.so")
_lib = None

HEAD_DIM = 128
ALPHA = np.float32(930.0 / 98.0)

# stream ids
S_KEYS, S_VALUES, S_QUERIES, S_GQ, S_GK, S_OUTLIERS, S_CTXLEN, S_PAGEPERM = 1, 2, 3, 4, 5, 6, 7, 8
S_SWA_K, S_SWA_V, S_SWA_Q, S_ROTSEED = 9, 10, 11, 12
S_ALIGN = 13


def build(verbose: bool = False) -> str:
    """Compile libkvqsynth.so next to this file (host + sm_103a device code)."""
    cmd = [
        "nvcc", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
        "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
        os.path.join(_HERE, "synth.cu"), "-o", _LIB_PATH,
    ]
    subprocess.run(cmd, check=True, capture_output=not verbose)
    return _LIB_PATH


def build_cmd() -> list:
    return [
        "nvcc", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
        "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
        os.path.join(_HERE, "synth.cu"), "-o", _LIB_PATH,
    ]


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            build()
        L = ctypes.CDLL(_LIB_PATH)
        u64, i64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        L.synth_key.restype = u64
        L.synth_key.argtypes = [u64, u64]
        L.synth_draw.restype = u64
        L.synth_draw.argtypes = [u64, u64]
        L.synth_normal_host.argtypes = [u64, u64, i64, vp, ctypes.c_int, vp]
        L.synth_uniform_host.argtypes = [u64, u64, i64, vp]
        L.synth_draw_host.argtypes = [u64, u64, i64, vp]
        L.synth_permutation_host.argtypes = [u64, i64, vp]
        L.synth_normal_device.restype = ctypes.c_int
        L.synth_normal_device.argtypes = [u64, u64, i64, vp, ctypes.c_int, vp, vp]
        _lib = L
    return _lib


def key(seed: int, stream: int) -> int:
    return int(lib().synth_key(seed & (2**64 - 1), stream))


def draws(k: int, start: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint64)
    lib().synth_draw_host(k, start, n, out.ctypes.data)
    return out


def normals(k: int, start: int, n: int, mult: np.ndarray | None = None, bf16: bool = False) -> np.ndarray:
    """n normals from element index `start`; bf16=True returns raw bf16 bits (uint16)."""
    if mult is not None:
        mult = np.ascontiguousarray(mult, np.float32)
        assert mult.shape == (HEAD_DIM,)
    out = np.empty(n, np.uint16 if bf16 else np.float32)
    lib().synth_normal_host(k, start, n, None if mult is None else mult.ctypes.data, 1 if bf16 else 0,
                            out.ctypes.data)
    return out


def uniforms(k: int, start: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float32)
    lib().synth_uniform_host(k, start, n, out.ctypes.data)
    return out


def permutation(k: int, n: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    lib().synth_permutation_host(k, n, out.ctypes.data)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- recipe helpers

def kv_index(layer: int, seq: int, pos: int, n_kv: int) -> int:
    """Element index of (layer, seq, pos, head 0, dim 0) for K/V inputs."""
    return (((layer * 1024 + seq) << 20) + pos) * n_kv * HEAD_DIM


def q_index(layer: int, seq: int, pos: int, n_q: int) -> int:
    return (((layer * 1024 + seq) << 20) + pos) * n_q * HEAD_DIM


def outlier_channels(seed: int, layer: int, count: int = 4) -> list:
    k = key(seed, S_OUTLIERS)
    picked = []
    n = 0
    while len(picked) < count:
        c = int(draws(k, layer * 64 + n, 1)[0] % HEAD_DIM)
        n += 1
        if c not in picked:
            picked.append(c)
    return picked


def key_multiplier(seed: int, layer: int) -> np.ndarray:
    m = np.ones(HEAD_DIM, np.float32)
    m[outlier_channels(seed, layer)] = ALPHA
    return m


def gains(seed: int, layer: int):
    """(g_q, g_k), each float32[128] in [0.5, 1.5)."""
    gq = np.float32(0.5) + uniforms(key(seed, S_GQ), layer * HEAD_DIM, HEAD_DIM)
    gk = np.float32(0.5) + uniforms(key(seed, S_GK), layer * HEAD_DIM, HEAD_DIM)
    return gq.astype(np.float32), gk.astype(np.float32)


def rotation_seed(seed: int, layer: int) -> int:
    return int(draws(key(seed, S_ROTSEED), layer, 1)[0])


def kv_rows(seed: int, layer: int, seq: int, pos0: int, T: int, n_kv: int, which: str, bf16: bool,
            outliers: bool = True):
    """Pre-norm keys or values for positions pos0..pos0+T-1 of one sequence: [T, n_kv, 128].

    which: 'k' / 'v' (full-attention layers) or 'swa_k' / 'swa_v' (FP8 sliding-window layers).
    Returns float32 (bf16=False) or bf16 bits as uint16 (bf16=True).
    """
    stream = {"k": S_KEYS, "v": S_VALUES, "swa_k": S_SWA_K, "swa_v": S_SWA_V}[which]
    mult = key_multiplier(seed, layer) if (which == "k" and outliers) else None
    x = normals(key(seed, stream), kv_index(layer, seq, pos0, n_kv), T * n_kv * HEAD_DIM, mult, bf16)
    return x.reshape(T, n_kv, HEAD_DIM)


def q_rows(seed: int, layer: int, seq: int, pos0: int, S: int, n_q: int, bf16: bool, swa: bool = False):
    stream = S_SWA_Q if swa else S_QUERIES
    x = normals(key(seed, stream), q_index(layer, seq, pos0, n_q), S * n_q * HEAD_DIM, None, bf16)
    return x.reshape(S, n_q, HEAD_DIM)


def aligned_rows(seed: int, seq: int, L: int, S: int, n_q: int, n_kv: int, theta0: float = 1.4,
                 v_scale: float = 1.0):
    """Inputs whose scores climb through the context, for exercising the online softmax.

    Per KV head a direction u_h; the key at position t is cos(a_t) u_h + sin(a_t) |u_h| w_t / |w_t|
    with a normal draw w_t and a_t = theta0 (1 - t / (L - 1)), so its alignment with u_h rises
    towards the end. Query rows (S of them per head, the last S positions) are u_h of their KV
    head (hq // (n_q / n_kv)) plus 0.05 x a normal draw. Values are normal draws x v_scale.
    Returns (keys [L, n_kv, 128], values [L, n_kv, 128], queries [S, n_q, 128]), float32."""
    k = key(seed, S_ALIGN)
    u = normals(k, kv_index(1, seq, 0, n_kv), n_kv * HEAD_DIM).reshape(n_kv, HEAD_DIM).astype(np.float64)
    w = normals(k, kv_index(0, seq, 0, n_kv), L * n_kv * HEAD_DIM).reshape(L, n_kv, HEAD_DIM).astype(np.float64)
    a = theta0 * (1.0 - np.arange(L, dtype=np.float64) / max(L - 1, 1))
    un = np.linalg.norm(u, axis=-1)
    wn = np.linalg.norm(w, axis=-1, keepdims=True)
    keys = np.cos(a)[:, None, None] * u[None] + (np.sin(a)[:, None] * un[None])[..., None] * w / wn
    vals = normals(k, kv_index(2, seq, 0, n_kv), L * n_kv * HEAD_DIM).reshape(L, n_kv, HEAD_DIM) * np.float32(v_scale)
    noise = normals(k, q_index(3, seq, 0, n_q), S * n_q * HEAD_DIM).reshape(S, n_q, HEAD_DIM).astype(np.float64)
    qs = u[np.arange(n_q) // (n_q // n_kv)][None] + 0.05 * noise
    return keys.astype(np.float32), vals.astype(np.float32), qs.astype(np.float32)


def context_lengths(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] (inclusive), from 24-bit draws."""
    d = draws(key(seed, S_CTXLEN), 0, n)
    u24 = (d >> np.uint64(40)).astype(np.int64)
    return (lo + ((u24 * (hi - lo + 1)) >> 24)).astype(np.int64)


def page_permutation(seed: int, layer: int, n: int) -> np.ndarray:
    return permutation(key(seed, S_PAGEPERM) ^ (layer * 0x10001), n)


# ---------------------------------------------------------------- device fill

def normals_device(k: int, start: int, n: int, out_ptr: int, mult: np.ndarray | None, bf16: bool,
                   stream_ptr: int = 0) -> None:
    """Same numbers as normals(), written by a CUDA kernel into device memory at out_ptr."""
    if mult is not None:
        mult = np.ascontiguousarray(mult, np.float32)
    rc = lib().synth_normal_device(k, start, n, None if mult is None else mult.ctypes.data,
                                   1 if bf16 else 0, out_ptr, stream_ptr)
    if rc != 0:
        raise RuntimeError(f"synth_normal_device failed with CUDA error {rc}")


def kv_rows_device(seed: int, layer: int, seq: int, pos0: int, T: int, n_kv: int, which: str, bf16: bool,
                   out_ptr: int, stream_ptr: int = 0, outliers: bool = True) -> None:
    stream = {"k": S_KEYS, "v": S_VALUES, "swa_k": S_SWA_K, "swa_v": S_SWA_V}[which]
    mult = key_multiplier(seed, layer) if (which == "k" and outliers) else None
    normals_device(key(seed, stream), kv_index(layer, seq, pos0, n_kv), T * n_kv * HEAD_DIM, out_ptr, mult,
                   bf16, stream_ptr)


def q_rows_device(seed: int, layer: int, seq: int, pos0: int, S: int, n_q: int, bf16: bool, out_ptr: int,
                  stream_ptr: int = 0, swa: bool = False) -> None:
    stream = S_SWA_Q if swa else S_QUERIES
    normals_device(key(seed, stream), q_index(layer, seq, pos0, n_q), S * n_q * HEAD_DIM, out_ptr, None, bf16,
                   stream_ptr)
