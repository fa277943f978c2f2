"""Decode-step runtime over a stack of attention layers.

Holds, per layer, the device state of the rotated int4 path (page pool, block table,
M_q/M_k) or of the FP8 sliding-window path (ring), plus one shared workspace and error
word; `decode_step` runs every layer of one decode step through the C ABI, in model
order (Kolibri-1: 50 layers, every fifth one full attention; "Serving Kolibri-1 with a
4-bit KV cache", section "What we do"). Torch is used for device memory only.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import (HEAD_DIM, PAGE_SIZE, alloc_fp8_ring, alloc_int4_cache, alloc_workspace, kvq_build_rotation,
               kvq_decode_attn_fp8_swa, kvq_decode_attn_int4, kvq_fold_qk, kvq_fold_qk_fwht, kvq_rotate_quant_append)


@dataclass
class Int4Layer:
    tensors: dict
    cache: object
    Mq: torch.Tensor  # folded query matrix, or the FWHT multipliers w_q
    Mk: torch.Tensor  # R, or the FWHT multipliers w_k = s
    R: np.ndarray
    fwht: bool = False


@dataclass
class SwaLayer:
    tensors: dict
    ring: object
    k_scale: float
    v_scale: float
    window: int


class DecodeStack:
    """Layers l = 0..n_layers-1; layer l is full attention (int4) when l % full_every == full_every-1."""

    def __init__(self, B, Hq, Hkv, S, max_pages, n_layers=1, full_every=1, ring_capacity=576, window=513,
                 swa_k_scale=1.0, swa_v_scale=1.0, page_perm=None, device="cuda"):
        self.B, self.Hq, self.Hkv, self.S = B, Hq, Hkv, S
        self.max_pages = max_pages
        self.device = device
        self.layers = []
        for l in range(n_layers):
            if l % full_every == full_every - 1:
                npages = B * max_pages
                perm = page_perm(l, npages) if page_perm is not None else np.arange(npages, dtype=np.int32)
                bt = torch.from_numpy(np.ascontiguousarray(perm.reshape(B, max_pages), dtype=np.int32))
                tensors, cache = alloc_int4_cache(npages, Hkv, bt, device)
                self.layers.append(Int4Layer(tensors, cache, None, None, None))
            else:
                tensors, ring = alloc_fp8_ring(B, Hkv, ring_capacity, device)
                self.layers.append(SwaLayer(tensors, ring, swa_k_scale, swa_v_scale, window))
        self.workspace = alloc_workspace(B, S, Hq, Hkv, device)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=device)

    def int4_layers(self):
        return [i for i, L in enumerate(self.layers) if isinstance(L, Int4Layer)]

    def swa_layers(self):
        return [i for i, L in enumerate(self.layers) if isinstance(L, SwaLayer)]

    def set_int4_params(self, l, rot_seed, g_q, g_k, rotate=True, prologue="matrix"):
        """Build R from the seed and fold the gains (host), upload M_q and M_k. rotate=False folds
        R = I instead: the unrotated int4 baseline (M_q = diag(g_q g_k), M_k = I).
        prologue="fwht": the same rotation through the fast Walsh-Hadamard prologue (uploads the
        multipliers w_q = s g_q g_k and w_k = s); set it before filling the layer's cache."""
        L = self.layers[l]
        if prologue == "fwht":
            R, s = kvq_build_rotation(rot_seed)
            wq, wk = kvq_fold_qk_fwht(s, g_q, g_k)
            L.R, L.fwht = R, True
            L.Mq = torch.from_numpy(wq).to(self.device)
            L.Mk = torch.from_numpy(wk).to(self.device)
            return
        assert prologue == "matrix", prologue
        R = kvq_build_rotation(rot_seed)[0] if rotate else np.eye(HEAD_DIM, dtype=np.float32)
        Mq, Mk = kvq_fold_qk(R, g_q, g_k)
        L.R, L.fwht = R, False
        L.Mq = torch.from_numpy(Mq).to(self.device)
        L.Mk = torch.from_numpy(Mk).to(self.device)

    def append_int4(self, l, k, v, seq_ids, positions, stream=None):
        L = self.layers[l]
        kvq_rotate_quant_append(L.cache, L.Mk, k, v, seq_ids, positions, self.dev_err, stream=stream, fwht=L.fwht)

    def prefill_int4(self, l, ctx, fill, chunk_tokens=16384, bf16=True):
        """Append positions 0..ctx[b]-1 of every sequence; fill(b, pos0, T, k_out, v_out) writes the
        pre-norm keys and values of those positions into device buffers [T, Hkv, 128]."""
        dt = torch.bfloat16 if bf16 else torch.float32
        kbuf = torch.empty((chunk_tokens, self.Hkv, HEAD_DIM), dtype=dt, device=self.device)
        vbuf = torch.empty_like(kbuf)
        for b in range(self.B):
            for p0 in range(0, int(ctx[b]), chunk_tokens):
                T = min(chunk_tokens, int(ctx[b]) - p0)
                fill(b, p0, T, kbuf, vbuf)
                seq = torch.full((T,), b, dtype=torch.int32, device=self.device)
                pos = torch.arange(p0, p0 + T, dtype=torch.int32, device=self.device)
                self.append_int4(l, kbuf[:T], vbuf[:T], seq, pos)

    def decode_layer(self, l, q, ctx, out, k_new=None, v_new=None, q_rot_out=None, stream=None):
        L = self.layers[l]
        if isinstance(L, Int4Layer):
            kvq_decode_attn_int4(L.cache, L.Mq, L.Mk, q, ctx, out, self.workspace, self.dev_err, k_new=k_new,
                                 v_new=v_new, q_rot_out=q_rot_out, stream=stream, fwht=L.fwht)
        else:
            kvq_decode_attn_fp8_swa(L.ring, q, ctx, L.window, L.k_scale, L.v_scale, out, self.workspace,
                                    self.dev_err, k_new=k_new, v_new=v_new, stream=stream)

    def decode_step(self, qs, ctx, outs, k_news=None, v_news=None, stream=None):
        """One decode step over all layers: qs[l], outs[l], k_news[l], v_news[l] per layer."""
        for l in range(len(self.layers)):
            self.decode_layer(l, qs[l], ctx, outs[l], None if k_news is None else k_news[l],
                              None if v_news is None else v_news[l], stream=stream)

    def read_error(self) -> int:
        return int(self.dev_err.item())


def pages_needed(ctx_max: int, extra_positions: int) -> int:
    return (ctx_max + extra_positions + PAGE_SIZE - 1) // PAGE_SIZE
