"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Codes, fp16 scales/offsets and rotated queries must be bit-exact; attention outputs within
max-abs 2e-3 and relative L2 1e-3 of the oracle's fp64 attention on its own (identical)
dequantised cache. Inputs come from the synth generator on both sides.
"""

import numpy as np
import pytest
import torch

import synth
from gpu_util import (assert_close, device_kv, device_new_kv, device_q, oracle_int4_seq, oracle_layer_params,
                      oracle_swa_seq, unpack_fp8, unpack_int4)
from quantized_kv_cache_fold_gb300 import DEVERR_NONFINITE, DEVERR_PAGE, DEVERR_POS, KvqError, kvq_fp8_swa_plan
from quantized_kv_cache_fold_gb300.runner import DecodeStack
from synth.workloads import SWA_K_SCALE, SWA_V_SCALE, Workload, config

pytestmark = pytest.mark.gpu


def build_int4(w, layer, S, page_perm=True, rotate=True, prologue="matrix"):
    max_pages = w.max_pages()
    perm = None
    if page_perm and w.page_order == "random":
        perm = lambda l, n: synth.page_permutation(w.seed, layer, n)  # noqa: E731
    st = DecodeStack(w.B, w.Hq, w.Hkv, S, max_pages, 1, 1, page_perm=perm)
    gq, gk = synth.gains(w.seed, layer)
    st.set_int4_params(0, synth.rotation_seed(w.seed, layer), gq, gk, rotate=rotate, prologue=prologue)

    def fill(b, p0, T, kb, vb):
        device_kv(w, layer, b, p0, T, "k", kb[:T])
        device_kv(w, layer, b, p0, T, "v", vb[:T])

    st.prefill_int4(0, w.ctx, fill, bf16=w.bf16)
    return st


def run_int4_step(st, w, layer, S):
    ctx = torch.from_numpy(w.ctx.astype(np.int32)).cuda()
    q = device_q(w, layer, S, w.ctx)
    k_new = device_new_kv(w, layer, S, w.ctx, "k")
    v_new = device_new_kv(w, layer, S, w.ctx, "v")
    out = torch.empty((w.B, S, w.Hq, 128), dtype=torch.float32, device="cuda")
    qrot = torch.empty_like(out)
    st.decode_layer(0, q, ctx, out, k_new=k_new, v_new=v_new, q_rot_out=qrot)
    torch.cuda.synchronize()
    return out.cpu().numpy(), qrot.cpu().numpy()


def check_int4(orc, w, layer, S, seqs, heads=None, st=None, prologue="matrix"):
    st = st or build_int4(w, layer, S, prologue=prologue)
    out, qrot = run_int4_step(st, w, layer, S)
    assert st.read_error() == 0, f"device error word {st.read_error():#x}"
    params = oracle_layer_params(orc, w, layer, prologue)
    errs = []
    for b in seqs:
        cb = int(w.ctx[b])
        for h in (heads if heads is not None else range(w.Hkv)):
            codes, qt, ref = oracle_int4_seq(orc, w, layer, b, h, S, cb, params)
            got = unpack_int4(st.layers[0].tensors, b, h, cb + S)
            for key in ("kc", "ks", "ko", "vc", "vs", "vo"):
                if not np.array_equal(got[key], codes[key]):
                    bad = np.argwhere(got[key] != codes[key])[:3]
                    raise AssertionError(f"{key} differs for seq {b} head {h} at {bad.tolist()}")
            g = w.G
            assert np.array_equal(qrot[b, :, h * g:(h + 1) * g], qt), f"q~ differs seq {b} head {h}"
            errs.append(assert_close(out[b, :, h * g:(h + 1) * g], ref, f"seq {b} head {h}"))
    return st, out, errs


def test_generator_device_matches_host():
    for bf16 in (False, True):
        mult = synth.key_multiplier(5, 3)
        k = synth.key(5, synth.S_KEYS)
        for start, n in ((0, 1000), (123456789, 4099), (2**40 + 7, 777)):
            host = synth.normals(k, start, n, mult, bf16)
            dev = torch.empty(n, dtype=torch.int16 if bf16 else torch.float32, device="cuda")
            synth.normals_device(k, start, n, dev.data_ptr(), mult, bf16, torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            assert dev.cpu().numpy().tobytes() == host.tobytes()


def test_config1_tiny(orc):
    w = config(1)
    check_int4(orc, w, 0, 1, [0])


@pytest.mark.parametrize("S", [1, 2, 3, 5, 8])
def test_ragged_page_edges(orc, S):
    """Contexts around page boundaries (0, 1, 63, 64, 65, 127, 200), fp32 inputs, random pages."""
    ctx = np.array([0, 1, 63, 64, 65, 127, 200], np.int64)
    w = Workload("edges", 11, len(ctx), 20, 4, S, ctx, False)
    check_int4(orc, w, 2, S, range(len(ctx)))


def test_gqa_group_sizes(orc):
    """Other head groupings: G = 8 (S=6 -> 48 rows) and G = 1."""
    w = Workload("g8", 12, 3, 16, 2, 6, np.array([300, 77, 1000]), True)
    check_int4(orc, w, 1, 6, range(3))
    w = Workload("g1", 13, 2, 4, 4, 1, np.array([500, 129]), True)
    check_int4(orc, w, 1, 1, range(2))


def test_config2_all(orc):
    w = config(2)
    _, _, errs = check_int4(orc, w, 0, 1, range(w.B))
    print("config2 worst max-abs %.2e rel-L2 %.2e" % (max(e[0] for e in errs), max(e[1] for e in errs)))


def test_verify_rows_match_single_row(orc):
    """Row r of an S-block equals the single-row decode at context L + r over the same cache."""
    w = Workload("verify", 14, 4, 20, 4, 4, np.array([1000, 1023, 64, 4000]), True)
    st, out_blk, _ = check_int4(orc, w, 3, 4, range(4))
    ctx0 = torch.from_numpy(w.ctx.astype(np.int32)).cuda()
    for r in range(4):
        q = device_q(w, 3, 4, w.ctx)[:, r:r + 1].contiguous()
        out = torch.empty((w.B, 1, w.Hq, 128), dtype=torch.float32, device="cuda")
        st.decode_layer(0, q, ctx0 + r, out)  # cache already holds the block rows
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy()[:, 0], out_blk[:, r], f"row {r}")


def test_deterministic(orc):
    w = Workload("det", 15, 3, 20, 4, 2, np.array([5000, 70, 900]), True)
    st = build_int4(w, 0, 2)
    ctx = torch.from_numpy(w.ctx.astype(np.int32)).cuda()
    q = device_q(w, 0, 2, w.ctx)
    outs = []
    for _ in range(2):
        out = torch.empty((w.B, 2, w.Hq, 128), dtype=torch.float32, device="cuda")
        st.decode_layer(0, q, ctx, out)
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


def test_bad_page_and_nonfinite_flagged():
    w = Workload("err", 16, 2, 20, 4, 1, np.array([100, 100]), True)
    st = build_int4(w, 0, 1)
    L = st.layers[0]
    # a block-table entry outside the pool: flagged, skipped, no fault
    saved = int(L.tensors["block_table"][1, 0])
    L.tensors["block_table"][1, 0] = L.cache.num_pages + 5
    ctx = torch.from_numpy(w.ctx.astype(np.int32)).cuda()
    q = device_q(w, 0, 1, w.ctx)
    out = torch.empty((w.B, 1, w.Hq, 128), dtype=torch.float32, device="cuda")
    st.decode_layer(0, q, ctx, out)
    torch.cuda.synchronize()
    assert st.read_error() & DEVERR_PAGE
    # a NaN in an appended key: flagged, row skipped
    st.dev_err.zero_()
    L.tensors["block_table"][1, 0] = saved
    k_new = device_new_kv(w, 0, 1, w.ctx, "k")
    k_new[0, 0, 2, 5] = float("nan")
    v_new = device_new_kv(w, 0, 1, w.ctx, "v")
    st.decode_layer(0, q, ctx, out, k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    assert st.read_error() & DEVERR_NONFINITE
    # the context stays usable
    st.dev_err.zero_()
    st.decode_layer(0, q, ctx, out)
    torch.cuda.synchronize()
    assert st.read_error() == 0 and np.isfinite(out.cpu().numpy()).all()


def test_host_errors_raise():
    w = Workload("err", 17, 2, 20, 4, 1, np.array([10, 10]), True)
    st = build_int4(w, 0, 1)
    q = device_q(w, 0, 1, w.ctx)
    out = torch.empty((w.B, 1, w.Hq, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(KvqError):
        st.decode_layer(0, q[:, :, :19].contiguous(), torch.zeros(2, dtype=torch.int32, device="cuda"), out)


@pytest.mark.parametrize("S", [1, 5])
def test_fwht_prologue(orc, S):
    """The second prologue specification (fast Walsh-Hadamard form): codes, fp16 scale/offset
    and q~ bit-exact with the oracle's FWHT prologue, attention within tolerance, for single rows
    and a verify block with its rows appended in the call."""
    w = Workload("fwht", 28, 3, 20, 4, S, np.array([0, 130, 2047]), True)
    _, out, _ = check_int4(orc, w, 3, S, range(w.B), prologue="fwht")
    assert np.isfinite(out).all()


def test_fwht_and_matrix_prologues_agree(orc):
    """Both specifications compute R n(k) and R diag(g_q g_k) n(q): their q~ agree to fp32 rounding."""
    w = Workload("fwht-vs-matrix", 29, 2, 20, 4, 1, np.array([200, 900]), True)
    qr = []
    for prologue in ("matrix", "fwht"):
        st = build_int4(w, 4, 1, prologue=prologue)
        _, qrot = run_int4_step(st, w, 4, 1)
        assert st.read_error() == 0
        qr.append(qrot)
    assert np.abs(qr[0] - qr[1]).max() <= 1e-5 * np.abs(qr[0]).max()


# ---------------------------------------------------------------- FP8 sliding window

def build_swa(w, layer, S, cap=576, window=513):
    st = DecodeStack(w.B, w.Hq, w.Hkv, S, 1, 1, 2, ring_capacity=cap, window=window, swa_k_scale=SWA_K_SCALE,
                     swa_v_scale=SWA_V_SCALE)
    L = st.layers[0]
    from quantized_kv_cache_fold_gb300 import kvq_fp8_append
    for b in range(w.B):
        P = int(w.ctx[b])
        lo = max(0, P - cap)
        if P - lo <= 0:
            continue
        k = device_kv(w, layer, b, lo, P - lo, "swa_k")
        v = device_kv(w, layer, b, lo, P - lo, "swa_v")
        seq = torch.full((P - lo,), b, dtype=torch.int32, device="cuda")
        pos = torch.arange(lo, P, dtype=torch.int32, device="cuda")
        kvq_fp8_append(L.ring, k, v, seq, pos, SWA_K_SCALE, SWA_V_SCALE, st.dev_err)
    return st


def check_swa(orc, w, layer, S, window=513, cap=576, sample=None):
    """Window layer of the call against the oracle: every sequence, or the sequences in
    `sample` (all outputs still checked to be finite)."""
    st = build_swa(w, layer, S, cap, window)
    ctx = torch.from_numpy(w.ctx.astype(np.int32)).cuda()
    q = device_q(w, layer, S, w.ctx, swa=True)
    k_new = device_new_kv(w, layer, S, w.ctx, "swa_k")
    v_new = device_new_kv(w, layer, S, w.ctx, "swa_v")
    out = torch.empty((w.B, S, w.Hq, 128), dtype=torch.float32, device="cuda")
    st.decode_layer(0, q, ctx, out, k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    assert st.read_error() == 0, f"device error word {st.read_error():#x}"
    out = out.cpu().numpy()
    assert np.isfinite(out).all()
    for b in (range(w.B) if sample is None else sample):
        for h in range(w.Hkv):
            kc, vc, positions, ref = oracle_swa_seq(orc, w, layer, b, h, S, int(w.ctx[b]), window)
            gk, gv = unpack_fp8(st.layers[0].tensors, b, h, positions)
            assert np.array_equal(gk, kc) and np.array_equal(gv, vc), f"e4m3 codes differ seq {b} head {h}"
            assert_close(out[b, :, h * w.G:(h + 1) * w.G], ref, f"swa seq {b} head {h}")


@pytest.mark.parametrize("S", [1, 4, 8])
def test_swa_window_wrap(orc, S):
    """Early rings (position < window), exact window, and wrap-around of the 576-slot ring."""
    ctx = np.array([0, 5, 300, 512, 513, 600, 1151, 5000], np.int64)
    w = Workload("swa", 21, len(ctx), 20, 4, S, ctx, True)
    check_swa(orc, w, 0, S)


def test_swa_small_window(orc):
    w = Workload("swa16", 22, 3, 20, 4, 2, np.array([10, 100, 1000]), False)
    check_swa(orc, w, 1, 2, window=16, cap=64)


@pytest.mark.parametrize("cap", [1024, 2048, 4096])
def test_swa_cluster_streams(orc, cap):
    """Rings of 16, 32 and 64 blocks over one 8-CTA cluster per (sequence, KV head): 1, 2 and 4
    blocks per warp stream (one- and two-stage buffers, refills after a patched stage)."""
    w = Workload(f"swa-ring{cap}", 23, 3, 20, 4, 2, np.array([40, cap - 300, 3 * cap + 17]), True)
    check_swa(orc, w, 2, 2, window=cap - 500, cap=cap)


def test_swa_large_ring_general_path(orc):
    """An 8192-slot ring (128 blocks) is beyond one cluster: separate append, split-K path and
    a combine pass."""
    w = Workload("swa-ring8192", 25, 2, 20, 4, 2, np.array([5000, 20000]), True)
    check_swa(orc, w, 3, 2, window=4097, cap=8192)


def test_swa_many_sequences(orc):
    """40 sequences x 4 KV heads: 160 clusters of 3 CTAs, more CTAs than SMs."""
    ctx = (np.arange(40) * 97 % 1500).astype(np.int64)
    w = Workload("swa-many", 26, len(ctx), 20, 4, 1, ctx, True)
    check_swa(orc, w, 4, 1)


ONE_CTA_PER_PAIR = [(420, 1), (300, 1), (160, 1), (110, 1), (55, 1), (200, 4), (120, 8)]


def test_swa_plan_shapes():
    """Window launch shapes: a cluster of several CTAs per (sequence, KV head) for few pairs,
    one CTA per pair once there are as many pairs as SMs (with different stream counts over
    the batches below), the split-K path for a ring beyond one cluster."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    shapes = {(B, S): kvq_fp8_swa_plan(576, B, S, 20, 4) for B, S in ONE_CTA_PER_PAIR}
    for (B, S), (cs, nws, nst, ups) in shapes.items():
        assert (cs == 1) == (4 * B >= sms), (B, S, cs)
        assert nws >= 1 and 1 <= nst <= ups and nws * ups >= 18
    if sms <= 220:
        assert len({sh[1] for sh in shapes.values() if sh[0] == 1}) >= 3
    assert kvq_fp8_swa_plan(576, 8, 1, 20, 4)[0] > 1
    assert kvq_fp8_swa_plan(8192, 2, 2, 20, 4) == (0, 0, 0, 0)


@pytest.mark.parametrize("B,S", ONE_CTA_PER_PAIR)
def test_swa_one_cta_per_pair(orc, B, S):
    """Batches whose (sequence, KV head) pairs fill the GPU unsplit (on 152 SMs): one CTA per
    pair, its 18 ring units over one to a few streams of several units each (ragged when the
    count does not divide 18; S = 8 with two tile groups). Contexts from 0 to 2999: early
    rings, full windows, wrap-around. Every seventh sequence and the last against the oracle."""
    ctx = (np.arange(B) * 389 % 3000).astype(np.int64)
    w = Workload(f"swa-pairs{B}x{S}", 28, B, 20, 4, S, ctx, True)
    check_swa(orc, w, 6, S, sample=sorted(set(range(0, B, 7)) | {B - 1}))


def test_swa_nonfinite_row_one_cta_per_pair(orc):
    """The error paths with one CTA per (sequence, KV head) and a lone stream storing its rows
    directly (300 sequences on 152 SMs): a NaN in one appended window key is flagged, that row
    is neither stored nor attended and the other pairs stay exact; a negative position is
    flagged and clamped."""
    B = 300
    ctx = (np.arange(B) * 389 % 3000).astype(np.int64)
    w = Workload("swa-err-pairs", 29, B, 20, 4, 1, ctx, True)
    st = build_swa(w, 7, 1)
    assert kvq_fp8_swa_plan(576, B, 1, 20, 4)[0] == 1
    dev_ctx = torch.from_numpy(w.ctx.astype(np.int32)).cuda()
    q = device_q(w, 7, 1, w.ctx, swa=True)
    k_new = device_new_kv(w, 7, 1, w.ctx, "swa_k")
    v_new = device_new_kv(w, 7, 1, w.ctx, "swa_v")
    k_new[7, 0, 2, 5] = float("nan")
    out = torch.empty((B, 1, w.Hq, 128), dtype=torch.float32, device="cuda")
    st.decode_layer(0, q, dev_ctx, out, k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    assert st.read_error() == DEVERR_NONFINITE
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    for b, h in [(0, 0), (7, 0), (7, 1), (7, 3), (8, 2), (150, 1), (299, 3)]:
        kc, vc, positions, ref = oracle_swa_seq(orc, w, 7, b, h, 1, int(w.ctx[b]), 513)
        gk, gv = unpack_fp8(st.layers[0].tensors, b, h, positions)
        assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
        assert_close(got[b, :, h * w.G:(h + 1) * w.G], ref, f"swa seq {b} head {h}")
    st.dev_err.zero_()
    bad = dev_ctx.clone()
    bad[3] = -5
    st.decode_layer(0, q, bad, out)
    torch.cuda.synchronize()
    assert st.read_error() == DEVERR_POS
    assert np.isfinite(out.cpu().numpy()).all()


def test_swa_nonfinite_row_and_bad_position_flagged(orc):
    """A NaN in one appended window key is flagged and that row is neither stored nor attended;
    the other (sequence, KV head) pairs stay exact. A negative position is flagged and clamped."""
    w = Workload("swa-err", 27, 2, 20, 4, 1, np.array([700, 900]), True)
    st = build_swa(w, 5, 1)
    ctx = torch.from_numpy(w.ctx.astype(np.int32)).cuda()
    q = device_q(w, 5, 1, w.ctx, swa=True)
    k_new = device_new_kv(w, 5, 1, w.ctx, "swa_k")
    v_new = device_new_kv(w, 5, 1, w.ctx, "swa_v")
    k_new[1, 0, 3, 7] = float("nan")
    out = torch.empty((w.B, 1, w.Hq, 128), dtype=torch.float32, device="cuda")
    st.decode_layer(0, q, ctx, out, k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    assert st.read_error() == DEVERR_NONFINITE
    got = out.cpu().numpy()
    for b, h in [(0, 0), (0, 3), (1, 0), (1, 2)]:
        kc, vc, positions, ref = oracle_swa_seq(orc, w, 5, b, h, 1, int(w.ctx[b]), 513)
        gk, gv = unpack_fp8(st.layers[0].tensors, b, h, positions)
        assert np.array_equal(gk, kc) and np.array_equal(gv, vc)
        assert_close(got[b, :, h * w.G:(h + 1) * w.G], ref, f"swa seq {b} head {h}")
    assert np.isfinite(got).all()
    st.dev_err.zero_()
    bad = torch.tensor([-5, 900], dtype=torch.int32, device="cuda")
    st.decode_layer(0, q, bad, out)
    torch.cuda.synchronize()
    assert st.read_error() == DEVERR_POS
    assert np.isfinite(out.cpu().numpy()).all()


def test_int4_many_segments_single_cta(orc):
    """More (sequence, KV head) segments than CTAs: short contexts, every segment in one CTA."""
    ctx = (np.arange(300) * 7 % 180).astype(np.int64)
    w = Workload("many", 24, len(ctx), 8, 4, 1, ctx, True)
    check_int4(orc, w, 1, 1, [0, 1, 57, 299])
