import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.lib()


def _parity_ledger():
    # the ledger exists only once a GPU parity test has imported it
    mod = sys.modules.get("tests.parity")
    return None if mod is None else mod


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    mod = _parity_ledger()
    if mod is None or not mod.LEDGER:
        return
    tr = terminalreporter
    tr.write_sep("-", "GPU/oracle decisions per workload (mismatches must stay below 1e-4 of decisions)")
    for name, e in sorted(mod.LEDGER.items()):
        tr.write_line(f"{name}: {e['comparisons']} comparisons, {e['requests']} requests, "
                      f"{e['decisions']} decisions, {e['near_margin']} within 1e-5 of their threshold, "
                      f"{e['mismatches']} mismatched"
                      + (f", {e['kseq_flat_zone']} K-SEQ flat-zone nodes" if e.get('kseq_flat_zone') else ""))


def pytest_sessionfinish(session, exitstatus):
    mod = _parity_ledger()
    if mod is None:
        return
    bad = mod.ledger_violations()
    if bad and session.exitstatus == 0:
        session.exitstatus = 1
        for name, e in bad.items():
            print(f"\nparity bar: {name}: {e['mismatches']} mismatches of {e['decisions']} decisions "
                  f"(not below 1e-4)")
