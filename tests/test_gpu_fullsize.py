"""Parity at the full sizes of the decode workloads, in the launch configuration the bench
times, on sampled sequences (all KV heads of each sampled sequence): codes bit-exact,
attention within max-abs 2e-3 / rel-L2 1e-3 of the oracle."""

import numpy as np
import pytest

from test_gpu_parity import check_int4, check_swa
from synth.workloads import Workload, config

pytestmark = pytest.mark.gpu


def test_config3_ragged_64k(orc):
    w = config(3)
    seqs = sorted({int(np.argmin(w.ctx)), int(np.argmax(w.ctx)), 7, 20})
    _, _, errs = check_int4(orc, w, 0, 1, seqs)
    print("config3 worst max-abs %.2e rel-L2 %.2e" % (max(e[0] for e in errs), max(e[1] for e in errs)))


@pytest.mark.parametrize("S", [4, 8])
def test_config4_verify(orc, S):
    w = config(4)
    w.S = S
    _, _, errs = check_int4(orc, w, 0, S, [0, 37, 63])
    print("config4 S=%d worst max-abs %.2e rel-L2 %.2e" % (S, max(e[0] for e in errs), max(e[1] for e in errs)))


def test_config5_int4_layer_256k(orc):
    w = config(5)
    _, _, errs = check_int4(orc, w, 4, 1, [0, 5])   # model layer 4: the first full-attention layer
    print("config5 int4 worst max-abs %.2e rel-L2 %.2e" % (max(e[0] for e in errs), max(e[1] for e in errs)))


def test_config5_swa_layer_256k(orc):
    w = config(5)
    sw = Workload(w.name, w.seed, w.B, w.Hq, w.Hkv, 1, w.ctx, True)
    check_swa(orc, sw, 0, 1)
