"""The oracle's pins catch plausible mistakes in it.

For every planted mistake in ``tests/oracle_mutants.py`` the pin suite
(``tests/test_oracle_pins.py``, or ``tests/test_oracle_guard.py`` for the
guard band) runs in a child process against the mutated module and must fail; a mutant that every pin lets through is a mistake the
pins cannot see.  The unmutated oracle passing the same suite is the normal
CPU run.  No GPU involved."""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

from tests import oracle_mutants as om

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


ALL = [m[0] for m in om.MUTANTS + om.GUARD_MUTANTS]


def test_every_mutant_applies_to_the_current_oracle():
    for name in ALL:
        compile(om.mutated_source(name), om.target(name)[1], "exec")
    assert len(set(ALL)) == len(ALL)


def _run_pins(name):
    env = dict(os.environ, **{om.ENV: name})
    cmd = [sys.executable, "-m", "pytest", om.target(name)[2], "-x", "-q",
           "-p", "tests.oracle_mutants", "-p", "no:cacheprovider"]
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


@pytest.fixture(scope="module")
def pin_runs():
    """The pin suite against every mutant, several child processes at a time."""
    workers = max(1, min(8, (os.cpu_count() or 2) // 2))
    with ThreadPoolExecutor(workers) as ex:
        return dict(zip(ALL, ex.map(_run_pins, ALL)))


@pytest.mark.parametrize("name", ALL)
def test_pins_catch_mutant(name, pin_runs):
    r = pin_runs[name]
    tail = "\n".join(r.stdout.splitlines()[-15:])
    assert r.returncode != 0, f"no pin fails with the mutant {name}:\n{tail}"
    assert r.returncode == 1 and " failed" in r.stdout, f"mutant {name} broke the run:\n{tail}"
