"""Concurrent calls from several host threads (the C ABI is documented thread-safe).

Two Python threads, each with its own DecodeStack (cache, workspace, error word) and CUDA
stream, issue decode calls at the same time; ctypes releases the GIL during the foreign calls,
so the library's launch-configuration caches are shared between the threads. Every thread's
output must equal the one the same call gives when run alone (the kernels are deterministic).
"""

import threading

import numpy as np
import pytest
import torch

from gpu_util import device_q
from synth.workloads import Workload
from test_gpu_parity import build_int4

pytestmark = pytest.mark.gpu


def test_concurrent_decode_calls_from_two_threads():
    cases = [Workload("t0", 61, 2, 20, 4, 1, np.array([3000, 1700]), True),
             Workload("t1", 62, 3, 20, 4, 8, np.array([900, 2500, 1234]), True)]  # S = 8: many-row kernel
    stacks = [build_int4(w, 0, w.S) for w in cases]
    qs = [device_q(w, 0, w.S, w.ctx) for w in cases]
    ctxs = [torch.from_numpy(w.ctx.astype(np.int32)).cuda() for w in cases]
    ref = []
    for st, w, q, c in zip(stacks, cases, qs, ctxs):
        out = torch.empty((w.B, w.S, w.Hq, 128), dtype=torch.float32, device="cuda")
        st.decode_layer(0, q, c, out)
        torch.cuda.synchronize()
        ref.append(out.cpu().numpy())
    results = [None, None]
    errors = []

    def worker(i):
        try:
            st, w, q, c = stacks[i], cases[i], qs[i], ctxs[i]
            s = torch.cuda.Stream()
            outs = []
            with torch.cuda.stream(s):
                for _ in range(20):
                    out = torch.empty((w.B, w.S, w.Hq, 128), dtype=torch.float32, device="cuda")
                    st.decode_layer(0, q, c, out, stream=s.cuda_stream)
                    outs.append(out)
            s.synchronize()
            results[i] = [o.cpu().numpy() for o in outs]
        except Exception as e:  # surfaced below
            errors.append(e)

    ths = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    assert not errors, errors
    for i in range(2):
        assert stacks[i].read_error() == 0
        for o in results[i]:
            assert np.array_equal(o, ref[i])
