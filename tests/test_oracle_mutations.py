"""Planted mistakes in the oracle must be caught by its pins.

Each case rebuilds the oracle with -DORACLE_MUTATION=n (one deliberate error, see the
MUT(n) sites in oracle/oracle.cpp) into a temporary library and runs the pin checks of
tests/pins.py against it: at least one check must fail. CPU only.
"""

import os
import subprocess
import tempfile

import pytest

import oracle
import pins

MUTATIONS = {
    1: "value/key offset dropped from the dequantised cache",
    2: "softmax scale not applied to the scores",
    3: "sign vector applied to rows instead of columns",
    4: "fp16 scale rounded to nearest instead of up",
    5: "codes rounded half away from zero",
    6: "RMS normalisation skipped",
    7: "g_k not folded into the query matrix",
    8: "causal bound off by one",
    9: "e4m3 conversion not saturating",
    10: "directed fp16 rounding ignores the sign",
    11: "fp16 offset rounded to nearest instead of down",
    12: "gains applied as diag(g) R instead of R diag(g)",
    13: "FWHT butterfly difference taken the wrong way round",
    14: "FWHT prologue without the 1/sqrt(128) scale",
    15: "FWHT query multipliers without the signs",
    16: "softmax without max subtraction",
    17: "key channel statistic as root-mean-square instead of mean |k|",
}


@pytest.fixture(scope="module")
def tmpdir_mut():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("n", sorted(MUTATIONS), ids=lambda n: f"mut{n}")
def test_mutation_is_caught(n, tmpdir_mut):
    path = os.path.join(tmpdir_mut, f"liboracle_mut{n}.so")
    subprocess.run(oracle.build_cmd(path, defines=(f"ORACLE_MUTATION={n}",)), check=True, capture_output=True)
    O = oracle.Oracle(oracle.load(path), threads=4)
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(O)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(check.__name__)
    assert failed, f"mutation {n} ({MUTATIONS[n]}) passed every pin"
