import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter):
    """Prints the error margins that the full-size parity checks recorded."""
    mod = sys.modules.get("tests.parity")
    margins = getattr(mod, "MARGINS", None) if mod else None
    if not margins:
        return
    terminalreporter.write_line("parity margins vs the f64 oracle (limits: O abs 2e-2, O row rel 2e-2, LSE abs 1e-3):")
    for label, m in margins.items():
        terminalreporter.write_line(f"  {label}: rows={m['rows']} o_max_abs={m['o_max_abs']:.3e} "
                                    f"o_row_rel={m['o_row_rel']:.3e} lse_max_abs={m['lse_max_abs']:.3e}")


def read_golden(name):
    """Parses a `key = value` fixture under tests/golden (lines starting with #
    are the citation)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition("=")
            out[key.strip()] = val.strip()
    return out


def nums(s, typ=float):
    return [typ(x) for x in s.split()]


def letter_matrix(s):
    """'P F . / . P F' -> list of rows of class codes (0 empty, 1 partial, 2 full)."""
    code = {".": 0, "P": 1, "F": 2}
    return [[code[c] for c in row.split()] for row in s.split("/")]
