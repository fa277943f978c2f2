"""The append and query prologue at every pass shape of the prep launch, through the C ABI.

"Serving Kolibri-1 with a 4-bit KV cache", section "What we do": new keys are normalised,
rotated and quantised to 4-bit codes, values quantised unrotated, and queries carry the
rotation with both QK-norm gains folded in. The prep launch deals these rows to warps in passes
of 1 to 8 query rows and 1 to 4 key/value jobs, chosen from the call's row counts; an odd
count runs its last row as a plain fp32 chain beside the paired ones. On a 152-SM GPU the
cases below take the shapes (query rows, key/value jobs) (1, 1), (2, 1), (2, 2), (3, 2),
(4, 2), (4, 3), (6, 3), (6, 4) and (8, 4) in one wave, and (8, 4) with several passes per warp
(more rows than one wave holds). Every case checks the codes and q~ bit-exact and the
attention within the oracle's tolerance, on short ragged contexts in random page order.
"""

import numpy as np
import pytest

from test_gpu_parity import check_int4
from synth.workloads import Workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,S", [(8, 1), (64, 1), (180, 1), (130, 2), (64, 5), (180, 2), (64, 8), (180, 3),
                                 (190, 3), (128, 8)])
def test_prep_pass_shapes(orc, B, S):
    ctx = np.random.default_rng(1000 + 10 * B + S).integers(0, 260, B).astype(np.int64)
    w = Workload("prep", 31 + S, B, 20, 4, S, ctx, S % 2 == 0, page_order="random")
    # sequences spread over the grid's blocks (first, last, and between); each holds S x 20
    # query rows and S x 4 key/value jobs, so every slot of a pass is among them
    check_int4(orc, w, 0, S, seqs=sorted({0, 1, B // 3, B // 2 + 1, B - 2, B - 1}))
