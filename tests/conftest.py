import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_runtest_teardown(item):
    # per-comparison parity records (norm-wise, worst row, max abs) to the
    # file named by LA_PARITY_REPORT, tagged with the test that made them
    import parity_utils
    if parity_utils.RECORDS and os.environ.get("LA_PARITY_REPORT"):
        for r in parity_utils.RECORDS:
            r["test"] = item.nodeid
        parity_utils.write_report()
    parity_utils.RECORDS.clear()
