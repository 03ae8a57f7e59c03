import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """Report of the bf16 comparisons: how many elements reached |oracle| >= 4 (where bf16
    cannot hold the value within 1e-2) and how many of those needed the widened bound."""
    mod = sys.modules.get("_harness")
    records = getattr(mod, "BF16_RECORDS", None) if mod else None
    if not records:
        return
    total = sum(r[1] for r in records)
    ge4 = sum(r[2] for r in records)
    widened = sum(r[3] for r in records)
    worst = max(r[4] for r in records)
    tr = terminalreporter
    tr.write_line(f"bf16 parity: {len(records)} comparisons, {total} elements; |oracle| >= 4: {ge4}; "
                  f"widened bound used: {widened}; max |gpu - bf16(oracle)|: {worst:.3e}")
    for label, n, g4, wd, mb in records:
        if g4:
            tr.write_line(f"  {label}: {n} elements, |oracle| >= 4: {g4}, widened bound used: {wd}, "
                          f"max |gpu - bf16(oracle)|: {mb:.3e}")


@pytest.fixture(scope="session")
def oracle_pool():
    """The oracle fanned out over every host core (spawned worker processes), for full-size checks."""
    from oracle.parallel import OraclePool

    pool = OraclePool()
    yield pool
    pool.close()
