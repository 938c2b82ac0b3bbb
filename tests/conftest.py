import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


@pytest.fixture(autouse=True)
def _parity_label(request):
    """Label every GPU-vs-oracle comparison with the test that made it."""
    from oracle import compare
    compare.LABEL[0] = request.node.nodeid if request.node.get_closest_marker("gpu") else ""
    yield
    compare.LABEL[0] = ""


def pytest_terminal_summary(terminalreporter):
    """Report the near ties every GPU-vs-oracle comparison counted (shown without -s)."""
    from oracle import compare
    reports = [(label, kind, rep) for label, kind, rep in compare.LOG if label]
    if not reports:
        return
    tr = terminalreporter
    tr.section("GPU vs oracle parity: near ties")
    seqs = sum(r.sequences for _, _, r in reports)
    exact = sum(r.exact for _, _, r in reports)
    acc = sum(r.accept_ties for _, _, r in reports)
    inv = sum(r.bonus_ties for _, _, r in reports)
    fails = sum(len(r.failures) for _, _, r in reports)
    tr.write_line("%d comparisons, %d sequences: %d exact, %d acceptance near ties (|u - p/q| < 1e-6), "
                  "%d inverse-CDF near ties (|u - C/W| < 1e-6), %d failures"
                  % (len(reports), seqs, exact, acc, inv, fails))
    for label, kind, rep in reports:
        if rep.accept_ties or rep.bonus_ties or rep.failures:
            tr.write_line("  %s [%s]: %s" % (label, kind, rep.summary()))
