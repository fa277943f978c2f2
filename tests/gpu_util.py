"""Helpers for the GPU parity tests: unpack the library's physical cache layouts into
logical (code, scale, offset) triplets, build synthetic workloads on the GPU through the
C ABI, and compute the oracle's view of the same (sequence, KV head) on the CPU.

Both sides take their inputs from the synth module only; the oracle never reads a value
produced by the CUDA path.
"""

from __future__ import annotations

import numpy as np
import torch

import synth
from synth.workloads import SWA_K_SCALE, SWA_V_SCALE

ATOL = 2e-3    # max-abs tolerance of attention outputs
RTOL_L2 = 1e-3  # relative L2 tolerance of attention outputs
SM = 128 ** -0.5


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    mx = float(np.abs(got - ref).max())
    rl = rel_l2(got, ref)
    assert mx <= ATOL and rl <= RTOL_L2, f"{what}: max-abs {mx:.3e} rel-L2 {rl:.3e}"
    return mx, rl


# ---------------------------------------------------------------- layout unpacking

def _nibbles(rec):
    """[..., 64] bytes -> [..., 128] codes (code 2b in the low nibble of byte b)."""
    rec = rec.astype(np.uint8)
    out = np.empty(rec.shape[:-1] + (128,), np.uint8)
    out[..., 0::2] = rec & 15
    out[..., 1::2] = rec >> 4
    return out


def _v_codes(rec):
    """[..., 64] bytes of V records (chunk swizzle undone) -> [..., 128] codes. Each 16-bit element
    (little endian) holds dims 4l..4l+3 as (e, sign) fields: dim 0 e bits 1-3 / sign 15, dim 1
    4-6 / 14, dim 2 11-13 / 7, dim 3 8-10 / 0; code = sign ? 7 - e : 8 + e."""
    u = rec.astype(np.uint16).reshape(rec.shape[:-1] + (32, 2))
    u = (u[..., 0] | (u[..., 1] << 8)).astype(np.int64)
    out = np.empty(rec.shape[:-1] + (32, 4), np.uint8)
    for i, (eb, sb) in enumerate(((1, 15), (4, 14), (11, 7), (8, 0))):
        e = (u >> eb) & 7
        sg = (u >> sb) & 1
        out[..., i] = np.where(sg == 1, 7 - e, 8 + e)
    return out.reshape(rec.shape[:-1] + (128,))


def unpack_int4(tensors, b, h, L):
    """Logical K/V codes and fp16 scale/offset bits of positions 0..L-1 of sequence b, head h."""
    bt = tensors["block_table"][b].cpu().numpy()
    pos = np.arange(L)
    dev = tensors["pages"].device
    pages = torch.from_numpy(bt[pos // 64].astype(np.int64)).to(dev)
    blk = tensors["pages"][pages, h].cpu().numpy()          # [L, 8704]: each position's page-head block
    slot = pos % 64
    rows = np.arange(L)
    # K chunk c of slot s sits at physical chunk c ^ (((s >> 1) & 1) | ((s >> 2) & 2))
    ksw = ((slot >> 1) & 1) | ((slot >> 2) & 2)
    kbyte = np.arange(64)[None, :]
    kc = blk[rows[:, None], slot[:, None] * 64 + 16 * ((kbyte >> 4) ^ ksw[:, None]) + (kbyte & 15)]
    vc = blk[rows[:, None], 4096 + slot[:, None] * 64 + np.arange(64)[None, :]]
    meta = blk[:, 8192:8704].copy().view(np.uint32)          # [L, 128]: K meta 0..63, V meta 64..127
    km = meta[rows, slot]
    vm = meta[rows, 64 + slot]
    # undo the V chunk swizzle: logical chunk c sits at physical chunk c ^ ((slot >> 1) & 3)
    sw = (slot >> 1) & 3
    vlog = np.empty_like(vc)
    for c in range(4):
        idx = ((c ^ sw)[:, None] * 16 + np.arange(16)[None, :])
        vlog[:, c * 16:(c + 1) * 16] = np.take_along_axis(vc, idx, axis=1)
    return {
        "kc": _nibbles(kc), "ks": (km & 0xFFFF).astype(np.uint16), "ko": (km >> 16).astype(np.uint16),
        "vc": _v_codes(vlog), "vs": (vm & 0xFFFF).astype(np.uint16), "vo": (vm >> 16).astype(np.uint16),
    }


def unpack_fp8(tensors, b, h, positions):
    """Logical e4m3 K/V bytes [n, 128] of the given positions of sequence b, head h."""
    data = tensors["data"][b, h].cpu().numpy()              # [cap/64, 16384]
    cap = data.shape[0] * 64
    slots = np.asarray(positions) % cap
    blk = data[slots // 64]
    within = slots % 64
    rows = np.arange(len(slots))
    k = blk[rows[:, None], within[:, None] * 128 + np.arange(128)[None, :]]
    v = blk[rows[:, None], 8192 + within[:, None] * 128 + np.arange(128)[None, :]]
    sw = slots & 7
    out = []
    for x in (k, v):
        lg = np.empty_like(x)
        for c in range(8):
            idx = ((c ^ sw)[:, None] * 16 + np.arange(16)[None, :])
            lg[:, c * 16:(c + 1) * 16] = np.take_along_axis(x, idx, axis=1)
        out.append(lg)
    return out[0], out[1]


# ---------------------------------------------------------------- synthetic inputs

def torch_dtype(bf16):
    return torch.bfloat16 if bf16 else torch.float32


def host_rows(arr_bits, bf16):
    """synth output (bf16 bits or float32) -> float32 numpy."""
    return synth.bf16_bits_to_f32(arr_bits) if bf16 else arr_bits


def device_kv(w, layer, b, pos0, T, which, kbuf=None):
    """Device tensor [T, Hkv, 128] of synthetic keys/values (same numbers as synth.kv_rows)."""
    out = kbuf if kbuf is not None else torch.empty((T, w.Hkv, 128), dtype=torch_dtype(w.bf16), device="cuda")
    synth.kv_rows_device(w.seed, layer, b, pos0, T, w.Hkv, which, w.bf16, out.data_ptr(),
                         torch.cuda.current_stream().cuda_stream)
    return out


def device_q(w, layer, S, pos_of_b, swa=False):
    """Device tensor [B, S, Hq, 128] of the queries at positions pos_of_b[b] .. +S-1."""
    q = torch.empty((w.B, S, w.Hq, 128), dtype=torch_dtype(w.bf16), device="cuda")
    for b in range(w.B):
        synth.q_rows_device(w.seed, layer, b, int(pos_of_b[b]), S, w.Hq, w.bf16, q[b].data_ptr(),
                            torch.cuda.current_stream().cuda_stream, swa=swa)
    return q


def device_new_kv(w, layer, S, pos_of_b, which):
    x = torch.empty((w.B, S, w.Hkv, 128), dtype=torch_dtype(w.bf16), device="cuda")
    for b in range(w.B):
        synth.kv_rows_device(w.seed, layer, b, int(pos_of_b[b]), S, w.Hkv, which, w.bf16, x[b].data_ptr(),
                             torch.cuda.current_stream().cuda_stream)
    return x


# ---------------------------------------------------------------- oracle views

def oracle_layer_params(O, w, layer, prologue="matrix"):
    """The oracle's own R, M_q, M_k for an int4 layer (from the same seeds); for the FWHT
    prologue ("fwht", w_q, w_k)."""
    seed = synth.rotation_seed(w.seed, layer)
    gq, gk = synth.gains(w.seed, layer)
    if prologue == "fwht":
        wq, wk = O.fold_fwht(O.signs(seed, 128), gq, gk)
        return "fwht", wq, wk
    _, R32 = O.rotation(seed)
    Mq, Mk = O.fold(R32, gq, gk)
    return R32, Mq, Mk


def oracle_int4_seq(O, w, layer, b, h, S, ctx_b, params=None):
    """Oracle codes of positions 0..ctx_b+S-1 and attention output of rows 0..S-1 for the G query
    heads of KV head h of sequence b. Returns (codes dict, q~ [S, G, 128], out [S, G, 128])."""
    params = params if params is not None else oracle_layer_params(O, w, layer)
    fwht = isinstance(params[0], str) and params[0] == "fwht"  # ("fwht", w_q, w_k): second prologue specification
    _, Mq, Mk = params
    Ltot = ctx_b + S
    k = host_rows(synth.kv_rows(w.seed, layer, b, 0, Ltot, w.Hkv, "k", w.bf16), w.bf16)[:, h]
    v = host_rows(synth.kv_rows(w.seed, layer, b, 0, Ltot, w.Hkv, "v", w.bf16), w.bf16)[:, h]
    y = O.prologue_fwht(Mk, k) if fwht else O.prologue(Mk, k)
    kc, ks, ko, kf = O.quantize_int4(y)
    vc, vs, vo, vf = O.quantize_int4(v)
    q = host_rows(synth.q_rows(w.seed, layer, b, ctx_b, S, w.Hq, w.bf16), w.bf16)
    qg = q[:, h * w.G:(h + 1) * w.G].reshape(-1, 128)
    qt = O.prologue_fwht(Mq, qg) if fwht else O.prologue(Mq, qg)
    vis = np.repeat(ctx_b + 1 + np.arange(S), w.G)
    out = O.attention_int4(qt, vis, kc, ks, ko, vc, vs, vo, SM)
    codes = {"kc": kc, "ks": ks, "ko": ko, "vc": vc, "vs": vs, "vo": vo, "kflags": kf, "vflags": vf}
    return codes, qt.reshape(S, w.G, 128), out.reshape(S, w.G, 128)


def oracle_swa_seq(O, w, layer, b, h, S, pos0_b, window):
    """Oracle e4m3 codes of the window positions and output rows of KV head h of sequence b."""
    lo_all = max(0, pos0_b - window + 1)
    hi_all = pos0_b + S - 1
    n = hi_all - lo_all + 1
    k = host_rows(synth.kv_rows(w.seed, layer, b, lo_all, n, w.Hkv, "swa_k", w.bf16), w.bf16)[:, h]
    v = host_rows(synth.kv_rows(w.seed, layer, b, lo_all, n, w.Hkv, "swa_v", w.bf16), w.bf16)[:, h]
    kc = O.quantize_fp8(k, SWA_K_SCALE)
    vc = O.quantize_fp8(v, SWA_V_SCALE)
    q = host_rows(synth.q_rows(w.seed, layer, b, pos0_b, S, w.Hq, w.bf16, swa=True), w.bf16)
    qg = q[:, h * w.G:(h + 1) * w.G].reshape(-1, 128)
    rows_pos = np.repeat(pos0_b + np.arange(S), w.G)
    lo = np.maximum(0, rows_pos - window + 1) - lo_all
    hi = rows_pos - lo_all
    out = O.attention_fp8(qg, lo, hi, kc, vc, SWA_K_SCALE, SWA_V_SCALE, SM)
    return kc, vc, np.arange(lo_all, hi_all + 1), out.reshape(S, w.G, 128)
