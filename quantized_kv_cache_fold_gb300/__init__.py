"""Rotated 4-bit KV-cache decode path for GB300 (sm_103a): Python binding of libkvq.so.

The functions here carry the C-ABI names of include/kvq.h and only marshal arguments:
torch tensors (device memory) and numpy arrays (host memory) become raw pointers, every
computation runs in the CUDA kernels of libkvq.so. A non-zero kvq_status raises KvqError.
There is no CPU fallback: importing fails loudly when the library is missing.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvq.so")

HEAD_DIM = 128
PAGE_SIZE = 64
MAX_SEQS = 1024
F32, BF16 = 0, 1
DEVERR_PAGE, DEVERR_POS, DEVERR_NONFINITE, DEVERR_RANGE, DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8, 0x10


class KvqError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


INT4_BLOCK_BYTES = 8704  # one (page, KV head): K codes 4096, V codes 4096, K meta 256, V meta 256
FP8_BLOCK_BYTES = 16384  # 64 ring slots of one head: K 8192, V 8192


class Int4Cache(ctypes.Structure):
    _fields_ = [("pages", ctypes.c_void_p), ("block_table", ctypes.c_void_p), ("num_seqs", ctypes.c_int32),
                ("max_pages_per_seq", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("page_size", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class Fp8Ring(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("num_seqs", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, f32, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_size_t
    L.kvq_status_string.restype = ctypes.c_char_p
    L.kvq_status_string.argtypes = [i32]
    L.kvq_build_rotation.restype = i32
    L.kvq_build_rotation.argtypes = [u64, i32, vp, vp]
    L.kvq_fold_qk.restype = i32
    L.kvq_fold_qk.argtypes = [vp, vp, vp, i32, vp, vp]
    L.kvq_fold_qk_fwht.restype = i32
    L.kvq_fold_qk_fwht.argtypes = [vp, vp, vp, i32, vp, vp]
    for name in ("kvq_rotate_quant_append", "kvq_rotate_quant_append_fwht"):
        getattr(L, name).restype = i32
        getattr(L, name).argtypes = [ctypes.POINTER(Int4Cache), vp, vp, vp, i32, i32, vp, vp, f32, vp, vp]
    L.kvq_decode_workspace_bytes.restype = sz
    L.kvq_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.kvq_fp8_swa_plan.restype = i32
    L.kvq_fp8_swa_plan.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_int32)]
    for name in ("kvq_decode_attn_int4", "kvq_decode_attn_int4_fwht"):
        getattr(L, name).restype = i32
        getattr(L, name).argtypes = [ctypes.POINTER(Int4Cache), vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, f32,
                                     f32, vp, vp, sz, vp, vp, vp]
    L.kvq_fp8_append.restype = i32
    L.kvq_fp8_append.argtypes = [ctypes.POINTER(Fp8Ring), vp, vp, i32, i32, vp, vp, f32, f32, vp, vp]
    L.kvq_decode_attn_int4_noalloc.restype = i32
    L.kvq_decode_attn_int4_noalloc.argtypes = [ctypes.POINTER(Int4Cache), vp, vp, vp, i32, i32, i32, i32, vp, vp, vp,
                                               f32, f32, vp, vp, vp, vp]
    L.kvq_set_stage_wait_limit_ns.restype = i32
    L.kvq_set_stage_wait_limit_ns.argtypes = [u64]
    L.kvq_decode_attn_fp8_swa.restype = i32
    L.kvq_decode_attn_fp8_swa.argtypes = [ctypes.POINTER(Fp8Ring), vp, i32, i32, i32, i32, vp, i32, vp, vp, f32,
                                          f32, f32, vp, vp, sz, vp, vp]
    return L


lib = _load()


def _ptr(x):
    """Device/host address of a torch tensor, numpy array, raw int or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, status):
    if status != 0:
        raise KvqError(fn, status)


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def status_string(status: int) -> str:
    return lib.kvq_status_string(int(status)).decode()


# ---------------------------------------------------------------- host-side steps

def kvq_build_rotation(seed: int, head_dim: int = HEAD_DIM):
    """R = H diag(s)/sqrt(128) as float32[128,128] and the signs s as int8[128] (numpy)."""
    R = np.empty((head_dim, head_dim), np.float32)
    s = np.empty(head_dim, np.int8)
    _check("kvq_build_rotation", lib.kvq_build_rotation(seed & (2**64 - 1), head_dim, s.ctypes.data, R.ctypes.data))
    return R, s


def kvq_fold_qk(R, g_q, g_k):
    """(M_q, M_k) = (R diag(g_q g_k), R) as float32[128,128] numpy arrays."""
    R = np.ascontiguousarray(R, np.float32)
    g_q = np.ascontiguousarray(g_q, np.float32)
    g_k = np.ascontiguousarray(g_k, np.float32)
    n = R.shape[0]
    Mq = np.empty((n, n), np.float32)
    Mk = np.empty((n, n), np.float32)
    _check("kvq_fold_qk", lib.kvq_fold_qk(R.ctypes.data, g_q.ctypes.data, g_k.ctypes.data, n, Mq.ctypes.data,
                                          Mk.ctypes.data))
    return Mq, Mk


# ---------------------------------------------------------------- cache descriptors

def int4_cache(pages, block_table) -> Int4Cache:
    """Descriptor over caller-owned device tensors: pages uint8 [num_pages, num_kv_heads, 8704]
    and block_table int32 [num_seqs, max_pages_per_seq] (see kvq.h for the block layout)."""
    num_seqs, max_pages = block_table.shape
    num_pages, num_kv_heads, nbytes = pages.shape
    assert nbytes == INT4_BLOCK_BYTES
    return Int4Cache(_ptr(pages), _ptr(block_table), num_seqs, max_pages, num_pages, num_kv_heads, PAGE_SIZE,
                     HEAD_DIM)


def fp8_ring(data) -> Fp8Ring:
    """data uint8 [num_seqs, num_kv_heads, capacity/64, 16384]."""
    num_seqs, num_kv, nblk, nbytes = data.shape
    assert nbytes == FP8_BLOCK_BYTES
    return Fp8Ring(_ptr(data), num_seqs, num_kv, nblk * PAGE_SIZE, HEAD_DIM)


def alloc_int4_cache(num_pages: int, num_kv_heads: int, block_table, device="cuda"):
    """Device tensors for an int4 cache (plumbing only: torch allocates, kernels fill)."""
    import torch
    pages = torch.zeros((num_pages, num_kv_heads, INT4_BLOCK_BYTES), dtype=torch.uint8, device=device)
    bt = block_table.to(device=device, dtype=torch.int32).contiguous()
    return {"pages": pages, "block_table": bt}, int4_cache(pages, bt)


def alloc_fp8_ring(num_seqs: int, num_kv_heads: int, capacity: int, device="cuda"):
    import torch
    assert capacity % PAGE_SIZE == 0
    data = torch.zeros((num_seqs, num_kv_heads, capacity // PAGE_SIZE, FP8_BLOCK_BYTES), dtype=torch.uint8,
                       device=device)
    return {"data": data}, fp8_ring(data)


# ---------------------------------------------------------------- device calls

def kvq_fold_qk_fwht(s, g_q, g_k):
    """(w_q, w_k) = (s g_q g_k, s) as float32[128] numpy arrays: the multipliers of the FWHT prologue."""
    s = np.ascontiguousarray(s, np.int8)
    g_q = np.ascontiguousarray(g_q, np.float32)
    g_k = np.ascontiguousarray(g_k, np.float32)
    n = s.shape[0]
    wq = np.empty(n, np.float32)
    wk = np.empty(n, np.float32)
    _check("kvq_fold_qk_fwht", lib.kvq_fold_qk_fwht(s.ctypes.data, g_q.ctypes.data, g_k.ctypes.data, n,
                                                    wq.ctypes.data, wk.ctypes.data))
    return wq, wk


def kvq_rotate_quant_append(cache: Int4Cache, Mk, k, v, seq_ids, positions, dev_err, eps: float = 1e-6,
                            stream=None, fwht: bool = False):
    """fwht=False: Mk is the 128x128 matrix; fwht=True: Mk is the multiplier vector w_k."""
    T = k.shape[0]
    name = "kvq_rotate_quant_append_fwht" if fwht else "kvq_rotate_quant_append"
    _check(name, getattr(lib, name)(ctypes.byref(cache), _ptr(Mk), _ptr(k), _ptr(v), _dtype_code(k), T,
                                    _ptr(seq_ids), _ptr(positions), eps, _ptr(dev_err), _stream(stream)))


def kvq_decode_workspace_bytes(B: int, S: int, num_q_heads: int, num_kv_heads: int) -> int:
    return int(lib.kvq_decode_workspace_bytes(B, S, num_q_heads, num_kv_heads))


def kvq_fp8_swa_plan(capacity: int, B: int, S: int, num_q_heads: int, num_kv_heads: int) -> tuple:
    """(CTAs per pair or 0 for the split-K path, streams per CTA, stages, units per stream)."""
    out = (ctypes.c_int32 * 4)()
    _check("kvq_fp8_swa_plan", lib.kvq_fp8_swa_plan(capacity, B, S, num_q_heads, num_kv_heads, out))
    return tuple(int(x) for x in out)


def kvq_decode_attn_int4(cache: Int4Cache, Mq, Mk, q, ctx_len, out, workspace, dev_err, k_new=None, v_new=None,
                         sm_scale: float = HEAD_DIM ** -0.5, eps: float = 1e-6, q_rot_out=None, stream=None,
                         fwht: bool = False):
    """fwht=False: Mq, Mk are the folded matrices; fwht=True: the multiplier vectors w_q, w_k."""
    B, S, Hq, _ = q.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    name = "kvq_decode_attn_int4_fwht" if fwht else "kvq_decode_attn_int4"
    _check(name, getattr(lib, name)(ctypes.byref(cache), _ptr(Mq), _ptr(Mk), _ptr(q), _dtype_code(q), B, S, Hq,
                                    _ptr(ctx_len), _ptr(k_new), _ptr(v_new), sm_scale, eps, _ptr(out),
                                    _ptr(workspace), ws_bytes, _ptr(q_rot_out), _ptr(dev_err), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 16 << 20
ERR_SCRATCH_TOO_SMALL = 4


def kvq_decode_attn_int4_noalloc(cache: Int4Cache, Mq, Mk, q, ctx_len, out, dev_err, k_new=None, v_new=None,
                                 sm_scale: float = HEAD_DIM ** -0.5, eps: float = 1e-6, q_rot_out=None, stream=None):
    """kvq_decode_attn_int4 without a caller workspace: for callers that cannot allocate device
    memory while decoding. Uses the library's fixed scratch (NOALLOC_SCRATCH_BYTES per device);
    calls that overlap on the GPU race on it. The first call on a device must precede any
    stream capture."""
    B, S, Hq, _ = q.shape
    _check("kvq_decode_attn_int4_noalloc",
           lib.kvq_decode_attn_int4_noalloc(ctypes.byref(cache), _ptr(Mq), _ptr(Mk), _ptr(q), _dtype_code(q), B, S,
                                            Hq, _ptr(ctx_len), _ptr(k_new), _ptr(v_new), sm_scale, eps, _ptr(out),
                                            _ptr(q_rot_out), _ptr(dev_err), _stream(stream)))


STAGE_WAIT_DEFAULT_NS = 2_000_000_000


def kvq_set_stage_wait_limit_ns(ns: int):
    """Test hook: the split-K attention kernel's stage-wait limit for later launches (default 2 s)."""
    _check("kvq_set_stage_wait_limit_ns", lib.kvq_set_stage_wait_limit_ns(int(ns)))


def kvq_fp8_append(ring: Fp8Ring, k, v, seq_ids, positions, k_scale: float, v_scale: float, dev_err, stream=None):
    T = k.shape[0]
    _check("kvq_fp8_append",
           lib.kvq_fp8_append(ctypes.byref(ring), _ptr(k), _ptr(v), _dtype_code(k), T, _ptr(seq_ids),
                              _ptr(positions), k_scale, v_scale, _ptr(dev_err), _stream(stream)))


def kvq_decode_attn_fp8_swa(ring: Fp8Ring, q, pos0, window: int, k_scale: float, v_scale: float, out, workspace,
                            dev_err, k_new=None, v_new=None, sm_scale: float = HEAD_DIM ** -0.5, stream=None):
    B, S, Hq, _ = q.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("kvq_decode_attn_fp8_swa",
           lib.kvq_decode_attn_fp8_swa(ctypes.byref(ring), _ptr(q), _dtype_code(q), B, S, Hq, _ptr(pos0), window,
                                       _ptr(k_new), _ptr(v_new), k_scale, v_scale, sm_scale, _ptr(out),
                                       _ptr(workspace), ws_bytes, _ptr(dev_err), _stream(stream)))


def alloc_workspace(B: int, S: int, num_q_heads: int, num_kv_heads: int, device="cuda"):
    import torch
    n = kvq_decode_workspace_bytes(B, S, num_q_heads, num_kv_heads)
    if n == 0:
        raise KvqError("kvq_decode_workspace_bytes", 2)
    return torch.empty(n, dtype=torch.uint8, device=device)
