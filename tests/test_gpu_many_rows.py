"""The two selectable many-row attention kernels, on the GPU through the C ABI.

"Serving Kolibri-1 with a 4-bit KV cache", section "What we do": one decode kernel family serves
1..8 query rows per sequence so that verify blocks reuse each KV byte. Every call runs the
split-K kernel by default; for more than 32 rows per KV head KVQ_MANY_ROWS_KERNEL selects one of
two other kernels: "tile", which converts each page's codes once into shared f16 tiles read by
every 8-row tile warp (mma.sync), and "tcgen05", whose QK^T and PV products run as tcgen05.mma
with accumulators in tensor memory. These cases repeat the many-row parity checks through each:
codes bit-exact, outputs within the tolerance of the oracle's attention over the same codes, on
the synthetic verify workload (S = 7 and 8, GQA 5, ragged contexts, random page order) and on the
climbing-score inputs that move the softmax base repeatedly and put V scales above 255.
"""

import os

import numpy as np
import pytest

from test_gpu_parity import check_int4
from test_gpu_softmax_base import test_climbing_scores_match_oracle
from synth.workloads import Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["tile", "tcgen05"])
def many_row_kernel(request):
    old = os.environ.get("KVQ_MANY_ROWS_KERNEL")
    os.environ["KVQ_MANY_ROWS_KERNEL"] = request.param
    yield request.param
    if old is None:
        del os.environ["KVQ_MANY_ROWS_KERNEL"]
    else:
        os.environ["KVQ_MANY_ROWS_KERNEL"] = old


@pytest.mark.parametrize("S", [7, 8])
def test_many_row_kernel_verify_rows(orc, many_row_kernel, S):
    # 3 sequences with ragged contexts (page tails, several CTAs per segment), random page order
    w = Workload("tc", 19, 3, 20, 4, S, np.array([1000, 2345, 777]), True, page_order="random")
    check_int4(orc, w, 0, S, seqs=range(w.B))


@pytest.mark.parametrize("v_scale", [1.0, 3000.0])
def test_many_row_kernel_climbing_scores(orc, many_row_kernel, v_scale):
    test_climbing_scores_match_oracle(orc, 8, v_scale)


def test_many_row_kernel_config4_verify_full_size(orc, many_row_kernel):
    # the speculative-verify workload at its full size (64 x 16,384, S = 8), sampled sequences
    from synth.workloads import config
    w = config(4)
    w.S = 8
    _, _, errs = check_int4(orc, w, 0, 8, [0, 37, 63])
    print("%s config4 S=8 worst max-abs %.2e rel-L2 %.2e" % (many_row_kernel, max(e[0] for e in errs),
                                                             max(e[1] for e in errs)))
