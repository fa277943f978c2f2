"""Online softmax of the int4 attention kernels under climbing scores, on the GPU through the C ABI.

"Serving Kolibri-1 with a 4-bit KV cache", section "What we do": decode attention reads the
packed codes and keeps an online softmax over the context. The kernels hold the exponent base
until a page has a score more than 8 (log2 units) above it, and on pages with a V scale of 255
or more until any score passes it. The synthetic workloads, with their near-uniform attention,
move the base only near the start of a segment; these inputs (synth.aligned_rows) turn the keys
towards the queries along the context, and large gains stretch the scores over about 100 log2
units, so the base moves again and again, P reaches 2^8 in between, and with v_scale = 3000 the
V scales pass 255. Each case compares every output row with the oracle's attention over the same
codes: S = 1 and 2 (split kernel, one and two row tiles) and 8 (the shared-tile kernel).
Attention is linear in V, so errors are judged on out / v_scale.
"""

import numpy as np
import pytest
import torch

import synth
from gpu_util import SM, assert_close
from quantized_kv_cache_fold_gb300.runner import DecodeStack

pytestmark = pytest.mark.gpu

SEED = 77
HQ, HKV = 20, 4
G = HQ // HKV


def _inputs(ctx, S, v_scale):
    return [synth.aligned_rows(SEED, b, int(ctx[b]) + S, S, HQ, HKV, v_scale=v_scale) for b in range(len(ctx))]


@pytest.mark.parametrize("S,v_scale", [(1, 1.0), (2, 1.0), (8, 1.0), (1, 3000.0), (8, 3000.0)])
def test_climbing_scores_match_oracle(orc, S, v_scale):
    ctx = np.array([2900, 4700], np.int64)
    B = len(ctx)
    data = _inputs(ctx, S, v_scale)
    max_pages = int(-(-(int(ctx.max()) + S) // 64))
    gq = np.full(128, 2.5, np.float32)
    gk = np.full(128, 2.5, np.float32)
    rot_seed = 12345

    st = DecodeStack(B, HQ, HKV, S, max_pages, 1, 1)
    st.set_int4_params(0, rot_seed, gq, gk)

    def fill(b, p0, T, kb, vb):
        kb[:T].copy_(torch.from_numpy(data[b][0][p0:p0 + T]))
        vb[:T].copy_(torch.from_numpy(data[b][1][p0:p0 + T]))

    st.prefill_int4(0, ctx + S, fill, bf16=False)  # the S query positions are already cached
    q = torch.from_numpy(np.stack([data[b][2] for b in range(B)])).cuda()
    out = torch.empty((B, S, HQ, 128), dtype=torch.float32, device="cuda")
    st.decode_layer(0, q, torch.from_numpy(ctx.astype(np.int32)).cuda(), out)
    torch.cuda.synchronize()
    assert st.read_error() == 0
    out = out.cpu().numpy()

    _, R32 = orc.rotation(rot_seed)
    Mq, Mk = orc.fold(R32, gq, gk)
    for b in range(B):
        keys, vals, qs = data[b]
        L = int(ctx[b]) + S
        for h in range(HKV):
            kc, ks, ko, _ = orc.quantize_int4(orc.prologue(Mk, keys[:, h]))
            vc, vs, vo, _ = orc.quantize_int4(vals[:, h])
            if v_scale > 1.0:
                assert float(np.max(vs.view(np.float16))) >= 255.0  # large V scales are exercised
            qt = orc.prologue(Mq, qs[:, h * G:(h + 1) * G].reshape(-1, 128))
            vis = np.repeat(int(ctx[b]) + 1 + np.arange(S), G)
            ref = orc.attention_int4(qt, vis, kc, ks, ko, vc, vs, vo, SM).reshape(S, G, 128)
            got = out[b, :, h * G:(h + 1) * G]
            assert_close(got / v_scale, ref / v_scale, f"S={S} v_scale={v_scale} seq {b} head {h}")
            assert L == kc.shape[0]
