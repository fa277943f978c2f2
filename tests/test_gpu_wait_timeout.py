"""The failure path of the bounded waits, made to run on purpose.

Every wait of the split-K attention kernel on a shared-memory stage gives up after a time
limit, records KVQ_DEVERR_TIMEOUT in the caller's error word and abandons the call's remaining
pages, so that a stalled copy can never hang the GPU. Here the limit is set to zero through the
test hook kvq_set_stage_wait_limit_ns on a workload with many pages per CTA: the producer's
first wait for a stage to be released (and the consumers' first waits for a page's copy) give up
at once. The call must return, the error word must carry KVQ_DEVERR_TIMEOUT, and with the
default limit restored the next call on the same cache must be parity-exact against the oracle
(codes bit-exact, attention within tolerance). The copies already in flight are still drained
with the full limit before a CTA exits, so no copy lands in a retired CTA's shared memory.
"""

import time

import numpy as np
import pytest
import torch

import quantized_kv_cache_fold_gb300 as kvq
from gpu_util import device_q
from synth.workloads import Workload
from test_gpu_parity import build_int4, check_int4

pytestmark = pytest.mark.gpu


def test_stage_wait_runs_out_then_next_call_is_exact(orc):
    # 4 sequences x 65,536 positions x 4 KV heads = 16,384 page-heads: dozens of pages per CTA,
    # more than the 12 stages of the ring, so the producer has to wait for released stages
    w = Workload("timeout", 41, 4, 20, 4, 1, np.full(4, 65536, np.int64), True)
    st = build_int4(w, 0, 1)
    ctx = torch.from_numpy(w.ctx.astype(np.int32)).cuda()
    q = device_q(w, 0, 1, w.ctx)
    out = torch.empty((w.B, 1, w.Hq, 128), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    assert st.read_error() == 0
    kvq.kvq_set_stage_wait_limit_ns(0)
    try:
        t0 = time.perf_counter()
        st.decode_layer(0, q, ctx, out)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        kvq.kvq_set_stage_wait_limit_ns(kvq.STAGE_WAIT_DEFAULT_NS)
    err = st.read_error()
    assert err & kvq.DEVERR_TIMEOUT, f"error word {err:#x}: no wait gave up"
    assert err & ~kvq.DEVERR_TIMEOUT == 0, f"error word {err:#x}"
    assert elapsed < 10.0, f"the abandoned call took {elapsed:.1f} s"
    st.dev_err.zero_()
    # the same cache, default limit: the append and attention of the next step are exact
    check_int4(orc, w, 0, 1, seqs=[0, 3], heads=[0, 2], st=st)
    assert st.read_error() == 0
