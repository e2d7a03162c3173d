"""The oracle's sizing arithmetic against the numbers the pages print."""
import os

import pytest

from oracle import accounting

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_sizing_examples.txt")


def _cases():
    out = []
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, fn, args, expected, rtol, cite = [p.strip() for p in line.split("|", 5)]
        out.append((name, fn, [float(a) for a in args.split(",")], float(expected), float(rtol), cite))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c[0])
def test_page_sizing_example(case):
    name, fn, args, expected, rtol, cite = case
    assert cite
    base, _, field = fn.partition(".")
    val = getattr(accounting, base)(*args)
    if field:
        val = val[field]
    assert abs(val - expected) <= rtol * abs(expected), (name, val, expected)


def test_controller_ratio_floor_and_match():
    # fast storage: recompute would exceed load -> stay at the 15% quality floor
    assert accounting.controller_ratio(t_prefill_s=1.0, t_load_s=0.05) == 0.15
    # slow storage: recompute up to the load time for free
    assert abs(accounting.controller_ratio(t_prefill_s=1.0, t_load_s=0.4) - 0.4) < 1e-12
