import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_sessionfinish(session, exitstatus):
    """With FA_PARITY_REPORT=<path>, write every parity comparison of the run
    (achieved max-abs, relative L2, bf16 floor and the gates) to <path>
    (markdown) and <path>.json."""
    path = os.environ.get("FA_PARITY_REPORT")
    if not path:
        return
    import parity
    if parity.REPORT:
        parity.write_report(path)


def read_golden(name):
    """Parse a tests/golden/*.txt fixture: 'key = numbers' lines, '#' comments.

    Rows of a matrix are separated by ';'.
    """
    path = os.path.join(ROOT, "tests", "golden", name)
    out = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            if ";" in val:
                out[key] = [[float(x) for x in r.split()] for r in val.split(";")]
            else:
                nums = [float(x) for x in val.split()]
                out[key] = nums[0] if len(nums) == 1 else nums
    return out
