"""The oracle's pins catch plausible mistakes: every mistake planted by
tests/oracle_mutations.py (one at a time, in a copy of the oracle) makes the
pin tests fail, and the unmodified copy passes them."""

import os
import sys

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import oracle_mutations  # noqa: E402


def test_every_planted_mistake_is_caught(capsys):
    rc = oracle_mutations.main()
    out = capsys.readouterr().out
    assert rc == 0, out
    assert "MISSED" not in out and out.count("CAUGHT") == len(oracle_mutations.MUTATIONS)
