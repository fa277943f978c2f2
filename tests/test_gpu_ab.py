"""A/B baselines of the full-attention layers, on the GPU through the C ABI.

"Serving Kolibri-1 with a 4-bit KV cache", section "What we do": the rotated 4-bit keys are the
method; plain (unrotated) 4-bit keys and the stock FP8 e4m3 cache are the two formats it is
weighed against, for bytes and for attention-output error. Three variants of one layer:

  rotated int4    M_k = R, M_q = R diag(g_q g_k)          136 B per token-head
  unrotated int4  M_k = I, M_q = diag(g_q g_k)            136 B per token-head
  FP8 e4m3        keys g_k n(k), values v, per-tensor scales max|x| / 448, queries g_q n(q),
                  full attention through the window kernel (capacity and window above the
                  context)                                256 B per token-head

On the outlier key generator (4 channels x 930/98) each variant's stored codes are bit-exact with
the oracle and its output within the usual tolerance of the oracle's attention over those codes;
and the error of the output against exact attention on unquantised keys and values orders the
formats as the page does: unrotated int4 > rotated int4 > FP8.
"""

import numpy as np
import pytest
import torch

import synth
from gpu_util import (SM, assert_close, device_new_kv, device_q, host_rows, oracle_int4_seq, unpack_fp8,
                      unpack_int4)
from quantized_kv_cache_fold_gb300 import kvq_fp8_append
from quantized_kv_cache_fold_gb300.runner import DecodeStack
from synth.workloads import Workload
from test_gpu_parity import build_int4

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _norm(x):
    """n(x) = x / sqrt(mean(x^2) + eps) in float32 (an input of the FP8 variant, the same array
    for the GPU and the oracle)."""
    x = np.asarray(x, np.float32)
    ms = np.mean(x * x, axis=-1, keepdims=True, dtype=np.float32)
    return (x / np.sqrt(ms + np.float32(EPS))).astype(np.float32)


def _rel(got, ref):
    return float(np.mean([np.linalg.norm(got[i] - ref[i]) / np.linalg.norm(ref[i]) for i in range(len(ref))]))


def test_ab_variants_match_oracle_and_order_their_errors(orc):
    w = Workload("ab", 41, 2, 20, 4, 1, np.array([3000, 4100]), True)
    layer, S = 2, 1
    gq, gk = synth.gains(w.seed, layer)
    ctx = torch.from_numpy(w.ctx.astype(np.int32)).cuda()
    q_dev = device_q(w, layer, S, w.ctx)
    kn_dev = device_new_kv(w, layer, S, w.ctx, "k")
    vn_dev = device_new_kv(w, layer, S, w.ctx, "v")

    # ---- host rows of every position 0..ctx (the appended row included), per sequence
    K, V, Q = [], [], []
    for b in range(w.B):
        L = int(w.ctx[b]) + S
        K.append(host_rows(synth.kv_rows(w.seed, layer, b, 0, L, w.Hkv, "k", w.bf16), w.bf16))
        V.append(host_rows(synth.kv_rows(w.seed, layer, b, 0, L, w.Hkv, "v", w.bf16), w.bf16))
        Q.append(host_rows(synth.q_rows(w.seed, layer, b, int(w.ctx[b]), S, w.Hq, w.bf16), w.bf16)[0])

    # ---- exact reference: attention of g_q n(q) over g_k n(k) and v, in fp64
    kp = [_norm(k) * gk for k in K]
    qp = [_norm(q) * gq for q in Q]
    exact = {}
    for b in range(w.B):
        for h in range(w.Hkv):
            exact[b, h] = orc.attention_f64(qp[b][h * w.G:(h + 1) * w.G], kp[b][:, h].astype(np.float64),
                                            V[b][:, h].astype(np.float64), SM)

    errs = {}
    # ---- rotated and unrotated int4 (same kernels; only the folded matrices differ)
    for name, rotate in (("int4_rotated", True), ("int4_unrotated", False)):
        st = build_int4(w, layer, S, rotate=rotate)
        out = torch.empty((w.B, S, w.Hq, 128), dtype=torch.float32, device="cuda")
        st.decode_layer(0, q_dev, ctx, out, k_new=kn_dev, v_new=vn_dev)
        torch.cuda.synchronize()
        assert st.read_error() == 0
        out = out.cpu().numpy()
        if rotate:
            _, R32 = orc.rotation(synth.rotation_seed(w.seed, layer))
        else:
            R32 = np.eye(128, dtype=np.float32)
        Mq, Mk = orc.fold(R32, gq, gk)
        e = []
        for b in range(w.B):
            for h in range(w.Hkv):
                codes, _, ref = oracle_int4_seq(orc, w, layer, b, h, S, int(w.ctx[b]), (R32, Mq, Mk))
                got = unpack_int4(st.layers[0].tensors, b, h, int(w.ctx[b]) + S)
                for key in ("kc", "ks", "ko", "vc", "vs", "vo"):
                    assert np.array_equal(got[key], codes[key]), f"{name}: {key} differs seq {b} head {h}"
                o = out[b, 0, h * w.G:(h + 1) * w.G]
                assert_close(o, ref[0], f"{name} seq {b} head {h}")
                e.append(_rel(o, exact[b, h]))
        errs[name] = float(np.mean(e))
        del st

    # ---- FP8 e4m3 keys and values for the whole context (window kernel, window above the context)
    cap = int(-(-(int(w.ctx.max()) + S) // 64) * 64)
    window = cap - S + 1
    ks8 = float(max(np.abs(k).max() for k in kp)) / 448.0
    vs8 = float(max(np.abs(v).max() for v in V)) / 448.0
    st = DecodeStack(w.B, w.Hq, w.Hkv, S, 1, n_layers=1, full_every=2, ring_capacity=cap, window=window,
                     swa_k_scale=ks8, swa_v_scale=vs8)
    Lr = st.layers[0]
    for b in range(w.B):
        cb = int(w.ctx[b])
        k = torch.from_numpy(kp[b][:cb]).cuda()
        v = torch.from_numpy(np.ascontiguousarray(V[b][:cb])).cuda()
        seq = torch.full((cb,), b, dtype=torch.int32, device="cuda")
        pos = torch.arange(0, cb, dtype=torch.int32, device="cuda")
        kvq_fp8_append(Lr.ring, k, v, seq, pos, ks8, vs8, st.dev_err)
    q8 = torch.from_numpy(np.stack([qp[b] for b in range(w.B)])[:, None]).cuda()
    kn8 = torch.from_numpy(np.stack([kp[b][int(w.ctx[b]):int(w.ctx[b]) + S] for b in range(w.B)])).cuda()
    vn8 = torch.from_numpy(np.stack([V[b][int(w.ctx[b]):int(w.ctx[b]) + S] for b in range(w.B)])).cuda()
    out = torch.empty((w.B, S, w.Hq, 128), dtype=torch.float32, device="cuda")
    st.decode_layer(0, q8, ctx, out, k_new=kn8, v_new=vn8)
    torch.cuda.synchronize()
    assert st.read_error() == 0
    out = out.cpu().numpy()
    e = []
    for b in range(w.B):
        L = int(w.ctx[b]) + S
        for h in range(w.Hkv):
            kc = orc.quantize_fp8(kp[b][:, h], ks8)
            vc = orc.quantize_fp8(V[b][:, h], vs8)
            gk8, gv8 = unpack_fp8(Lr.tensors, b, h, np.arange(L))
            assert np.array_equal(gk8, kc) and np.array_equal(gv8, vc), f"fp8 codes differ seq {b} head {h}"
            ref = orc.attention_fp8(qp[b][h * w.G:(h + 1) * w.G], np.zeros(w.G, np.int64),
                                    np.full(w.G, L - 1, np.int64), kc, vc, ks8, vs8, SM)
            o = out[b, 0, h * w.G:(h + 1) * w.G]
            assert_close(o, ref, f"fp8 seq {b} head {h}")
            e.append(_rel(o, exact[b, h]))
    errs["fp8"] = float(np.mean(e))

    assert errs["int4_unrotated"] > errs["int4_rotated"] > errs["fp8"], errs
