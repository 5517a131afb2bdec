import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled library")
    config.addinivalue_line(
        "markers", "slow: long-running oracle case")


@pytest.fixture(scope="session")
def oracle_pool():
    """Spawned worker processes that evaluate the oracle for the full-size
    parity tests (created on first use, one per host core)."""
    from oracle_pool import OraclePool
    pool = OraclePool()
    yield pool
    pool.close()


def pytest_terminal_summary(terminalreporter):
    """One line on the flat max-abs error of every bf16 output checked."""
    try:
        from gpu_utils import FLAT_LOG
    except Exception:
        return
    if not FLAT_LOG:
        return
    worst = max(FLAT_LOG, key=lambda x: x[1])
    n = sum(x[2] for x in FLAT_LOG)
    over = sum(x[3] for x in FLAT_LOG)
    checks_over = [x for x in FLAT_LOG if x[3]]
    big = max((x[4] for x in checks_over), default=0.0)
    terminalreporter.write_line(
        f"bf16 outputs: {len(FLAT_LOG)} checks, {n} elements; flat max|O - O_ref| = "
        f"{worst[1]:.3e} ({worst[0]}); {over} elements above 1e-2 in "
        f"{len(checks_over)} checks (largest |O_ref| among them {big:.3f})")
    for what, mx, size, n_over, big_o in sorted(checks_over, key=lambda x: -x[3])[:16]:
        terminalreporter.write_line(
            f"  above 1e-2: {what}: {n_over} of {size} elements, max {mx:.3e}, "
            f"largest |O_ref| among them {big_o:.3f}")
