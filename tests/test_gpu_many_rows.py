"""Many query rows per KV head (speculative-verify blocks), on the GPU through the C ABI.

"Serving Kolibri-1 with a 4-bit KV cache", section "What we do": one decode kernel family serves
1..8 query rows per sequence so that verify blocks reuse each KV byte. These cases repeat the
parity checks at the larger row counts: codes bit-exact, outputs within the tolerance of the
oracle's attention over the same codes, on the synthetic verify workload (S = 3 .. 8 at GQA 5 and
S = 3, 8 at GQA 6, ragged contexts, random page order), on the climbing-score inputs that move the softmax base
repeatedly and put V scales above 255, and on the full-size verify workload.
"""

import numpy as np
import pytest

from test_gpu_parity import check_int4
from test_gpu_softmax_base import test_climbing_scores_match_oracle
from synth.workloads import Workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("S", [3, 4, 6, 7, 8])
def test_many_rows_verify(orc, S):
    # 3 sequences with ragged contexts (page tails, several CTAs per segment), random page order;
    # 15 .. 40 rows per KV head: the split kernel (15) and the tcgen05 kernel's 24, 32 and 40-row
    # variants
    w = Workload("tc", 19, 3, 20, 4, S, np.array([1000, 2345, 777]), True, page_order="random")
    check_int4(orc, w, 0, S, seqs=range(w.B))


@pytest.mark.parametrize("S", [3, 8])
def test_many_rows_gqa6(orc, S):
    # GQA 6: 18 rows (the smallest call of the tcgen05 kernel) and 48 rows (its largest variant)
    w = Workload("tc6", 23, 3, 24, 4, S, np.array([1500, 64, 3001]), False, page_order="random")
    check_int4(orc, w, 0, S, seqs=range(w.B))


@pytest.mark.parametrize("v_scale", [1.0, 3000.0])
def test_many_rows_climbing_scores(orc, v_scale):
    test_climbing_scores_match_oracle(orc, 8, v_scale)


def test_many_rows_config4_verify_full_size(orc):
    # the speculative-verify workload at its full size (64 x 16,384, S = 8), sampled sequences
    from synth.workloads import config
    w = config(4)
    w.S = 8
    _, _, errs = check_int4(orc, w, 0, 8, [0, 37, 63])
    print("config4 S=8 worst max-abs %.2e rel-L2 %.2e" % (max(e[0] for e in errs), max(e[1] for e in errs)))
