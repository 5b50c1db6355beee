"""The oracle's pins catch plausible mistakes in it.

``tests/_mutants.py`` plants, one at a time, a slip in an oracle module (a
dropped term, a wrong sign, index or rounding, transposed operands, a wrong
order of summation, a wrong ledger term) and runs the pin tests that call
that module; every mutant must make at least one pin fail, and the pins must
pass on the unmodified oracle.  It runs in a child process so that the
re-executed modules never reach this session."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_every_planted_mistake_fails_a_pin():
    r = subprocess.run([sys.executable, "-m", "tests._mutants"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-4000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res.pop("<none>") == 0, "the pins fail on the unmodified oracle"
    from tests._mutants import MUTANTS
    assert set(res) == set(MUTANTS)
    escaped = sorted(k for k, v in res.items() if v == 0)
    broken = sorted(f"{k} (pytest exit {v})" for k, v in res.items() if v not in (0, 1))
    assert not escaped, f"mutants no pin catches: {escaped}"
    assert not broken, f"mutants whose pin run did not complete: {broken}"
