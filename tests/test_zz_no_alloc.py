"""The allocation-free decode entry point (kvq_decode_attn_int4_noalloc).

It serves callers that cannot allocate device memory while decoding (for example an
engine that gave all free GPU memory to its KV pool at start-up): the workspace comes
from a fixed scratch array inside the library instead of from the caller. This file is
collected last on purpose, and it must pass both on its own in a fresh process (where its
first call performs the per-device scratch set-up) and after every other test.

The check: through the C ABI, the new entry point gives the same attention output as
kvq_decode_attn_int4 with a caller workspace, within the tolerance of the other GPU tests and
in fact bit for bit (the same kernels run on the same inputs), on two consecutive rounds with
different queries and contexts (so a stale scratch from the previous call would show); and a
request larger than the scratch is refused.
"""

import ctypes

import numpy as np
import pytest
import torch

import quantized_kv_cache_fold_gb300 as kvq
from gpu_util import assert_close, device_q
from synth.workloads import Workload
from test_gpu_parity import build_int4

pytestmark = pytest.mark.gpu


def _noalloc(cache, Mq, Mk, q, ctx, out, err):
    B, S, Hq, _ = q.shape
    return kvq.lib.kvq_decode_attn_int4_noalloc(
        ctypes.byref(cache), Mq.data_ptr(), Mk.data_ptr(), q.data_ptr(), kvq.BF16, B, S, Hq, ctx.data_ptr(), None,
        None, 128 ** -0.5, 1e-6, out.data_ptr(), None, err.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _with_workspace(cache, Mq, Mk, q, ctx, out, ws, err):
    B, S, Hq, _ = q.shape
    return kvq.lib.kvq_decode_attn_int4(
        ctypes.byref(cache), Mq.data_ptr(), Mk.data_ptr(), q.data_ptr(), kvq.BF16, B, S, Hq, ctx.data_ptr(), None,
        None, 128 ** -0.5, 1e-6, out.data_ptr(), ws.data_ptr(), ws.numel(), None, err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_twice():
    w = Workload("noalloc", 31, 4, 20, 4, 2, np.array([100, 1000, 64, 3000]), True)
    S = 2
    st = build_int4(w, 0, S)
    L = st.layers[0]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rounds = [(w.ctx - 2, 0), (w.ctx - 40, 7)]  # different context lengths and queries per round
    for ctx_np, qshift in rounds:
        ctx = torch.from_numpy(ctx_np.astype(np.int32)).cuda()
        q = device_q(w, qshift, S, ctx_np)
        ref = torch.empty((w.B, S, w.Hq, 128), dtype=torch.float32, device="cuda")
        got = torch.full_like(ref, float("nan"))
        ws = kvq.alloc_workspace(w.B, S, w.Hq, w.Hkv)
        assert _with_workspace(L.cache, L.Mq, L.Mk, q, ctx, ref, ws, err) == 0
        assert _noalloc(L.cache, L.Mq, L.Mk, q, ctx, got, err) == 0
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        g, r = got.cpu().numpy(), ref.cpu().numpy()
        assert_close(g, r, "noalloc vs workspace entry point")
        # the same kernels on the same inputs with a workspace of the same layout: bit for bit
        assert np.array_equal(g, r), "noalloc output differs in some bit from the workspace entry point's"


def test_noalloc_rejects_requests_beyond_its_scratch():
    need = kvq.kvq_decode_workspace_bytes(512, 8, 40, 8)
    assert need > kvq.NOALLOC_SCRATCH_BYTES
    cache = kvq.Int4Cache(0x10000, 0x20000, 512, 8, 64, 8, 64, 128)
    out = torch.empty(16, dtype=torch.float32, device="cuda")
    q = torch.empty((512, 8, 40, 128), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = kvq.lib.kvq_decode_attn_int4_noalloc(ctypes.byref(cache), 0x30000, 0x40000, q.data_ptr(), kvq.BF16, 512, 8,
                                              40, 0x50000, None, None, 0.088, 1e-6, out.data_ptr(), None,
                                              err.data_ptr(), None)
    assert rc == kvq.ERR_SCRATCH_TOO_SMALL
    assert "scratch" in kvq.status_string(rc)
