"""The pins catch plausible mistakes: each mutant build of the oracle carries one
deliberate error (a dropped scale, an off-by-one causal limit, a wrong head
grouping, a wrong pooling radius, reversed tie-breaking, a wrong ring slot, invalid
middle slots treated as valid, a transposed value row, a prefill row missing its
diagonal key), and the pin suite run against it must fail.  CPU only."""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
MUTANTS = {
    1: "softmax scale dropped",
    2: "causal row stops one key early",
    3: "query heads grouped across KV heads",
    4: "pooling radius one too wide",
    5: "ties broken toward the higher position",
    6: "ring slot missing the L_sink + K offset",
    7: "unused middle slots treated as valid",
    8: "value row read backwards",
    9: "prefill attention row stops before the query's own key",
}


@pytest.mark.parametrize("k", sorted(MUTANTS))
def test_pins_fail_on_mutant(k, tmp_path):
    lib = oracle.build_mutant(k, str(tmp_path))
    env = dict(os.environ, SNAP_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_pins.py")], env=env, capture_output=True, text=True,
                       cwd=os.path.dirname(HERE))
    assert r.returncode != 0, f"mutant {k} ({MUTANTS[k]}) passed every pin:\n{r.stdout[-2000:]}"
