"""The sampling oracle's pins catch plausible mistakes: each mutant is a copy of
``oracle/sampling.py`` with one planted slip, run against every ``check_*`` pin; at least
one pin must fail for each."""
import os
import types

import pytest

import test_oracle_sampling as pins

SRC_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "sampling.py")
CHECKS = [getattr(pins, n) for n in dir(pins) if n.startswith("check_")]

MUTANTS = {
    "ties by higher index": ("key=lambda i: (-x[i], i)", "key=lambda i: (-x[i], -i)"),
    "temperature multiplies": ("vals = [x[i] / temperature for i in order]", "vals = [x[i] * temperature for i in order]"),
    "top-p keeps one fewer": ("keep = i + 1", "keep = max(1, i)"),
    "greedy takes the last maximum": ("if x[i] > x[best]:", "if x[i] >= x[best]:"),
    "top-k keeps one more": ("order = sorted(range(V), key=lambda i: (-x[i], i))[:k]",
                             "order = sorted(range(V), key=lambda i: (-x[i], i))[:k + 1]"),
    "draw ignores u": ("target = u * total", "target = 0.5 * total"),
}


def _load(src: str):
    mod = types.ModuleType("sampling_mutant")
    exec(compile(src, "sampling_mutant", "exec"), mod.__dict__)
    return mod


def test_the_unmutated_copy_passes_every_pin():
    mod = _load(open(SRC_PATH).read())
    for check in CHECKS:
        check(mod)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_mutant_fails_a_pin(name):
    src = open(SRC_PATH).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site not found: {old}"
    mod = _load(src.replace(old, new))
    failed = []
    for check in CHECKS:
        try:
            check(mod)
        except (AssertionError, ValueError, IndexError):
            failed.append(check.__name__)
    assert failed, f"mutant '{name}' passes every pin"
