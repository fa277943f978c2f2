"""The largest call the C ABI accepts: KVQ_MAX_SEQS (1024) sequences, through the C ABI.

"Serving Kolibri-1 with a 4-bit KV cache", section "What we do": decode over the rotated 4-bit
cache of the full-attention layers and the FP8 ring of the window layers. At 1024 sequences the
kernels meet their largest sizes: the page prefix of 1024 sequences in every attention CTA's
shared memory (the tcgen05 kernel's included), the prologue/append launch past one wave
(several passes per warp), the combine with the most (segment, row) items, and 4096 window
rings (one CTA per sequence and KV head). Short ragged contexts in random page order keep the
oracle's work small; sampled sequences at both ends and in the middle are checked: codes
bit-exact, outputs within the oracle's tolerance.
"""

import numpy as np
import pytest

from test_gpu_parity import check_int4, check_swa
from synth.workloads import Workload

pytestmark = pytest.mark.gpu

KVQ_MAX_SEQS = 1024
SAMPLE = [0, 1, 511, 512, KVQ_MAX_SEQS - 2, KVQ_MAX_SEQS - 1]


@pytest.mark.parametrize("S", [1, 8])
def test_int4_max_sequences(orc, S):
    # S = 1: the split kernel; S = 8 (40 rows per KV head): the tcgen05 kernel
    ctx = np.random.default_rng(2024 + S).integers(0, 200, KVQ_MAX_SEQS).astype(np.int64)
    w = Workload("maxseq", 41 + S, KVQ_MAX_SEQS, 20, 4, S, ctx, True, page_order="random")
    check_int4(orc, w, 0, S, seqs=SAMPLE)


def test_swa_max_sequences(orc):
    ctx = np.random.default_rng(2031).integers(0, 1500, KVQ_MAX_SEQS).astype(np.int64)
    w = Workload("maxseq_swa", 47, KVQ_MAX_SEQS, 20, 4, 1, ctx, True)
    check_swa(orc, w, 0, 1, sample=SAMPLE)
