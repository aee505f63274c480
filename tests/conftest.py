import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: large oracle work")


@pytest.fixture(scope="session")
def cuda_lib():
    """The C-ABI library through the Python binding; skips without a GPU."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_scaled_moe_sort_gb300 as m
    return m


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Per-case output parity against the oracle: how many compared elements
    needed the rounding-decision budget on top of the plain atol = rtol =
    2e-2 bar, the plain-bar pass fraction and the largest excess. Written as
    JSON to $MOE_PARITY_RECORD when that is set."""
    mc = sys.modules.get("moe_check")
    log = getattr(mc, "PARITY_LOG", None)
    if not log:
        return
    tr = terminalreporter
    tr.write_sep("-", "output parity vs oracle (plain bar: |err| <= 2e-2 + 2e-2*|ref|)")
    for st in log:
        tr.write_line(
            f"{st['case']}: {st['variant']} M={st['M']} bm={st['block_m']} "
            f"elems={st['n_out']} max_abs_err={st['max_abs_err']:.3g} "
            f"over_plain={st['n_needing_budget']} plain_frac={st['plain_bar_frac']:.6f} "
            f"max_excess={st['max_excess_over_plain']:.3g} "
            f"inter_match={st.get('inter_match', float('nan')):.5f}")
    for v in ("a8w4", "a16w4"):
        cases = [st for st in log if st["variant"] == v]
        if cases:
            n_el = sum(st["n_out"] for st in cases)
            n_over = sum(st["n_needing_budget"] for st in cases)
            n_cases_over = sum(1 for st in cases if st["n_needing_budget"])
            tr.write_line(f"parity summary {v}: {len(cases)} cases, {n_el} output elements, "
                          f"{n_over} over the plain bar in {n_cases_over} cases")
    path = os.environ.get("MOE_PARITY_RECORD")
    if path:
        with open(path, "w") as f:
            json.dump(log, f, indent=1)
