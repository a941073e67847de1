import json
import math
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


def eval_expr(x):
    """Evaluate a closed-form fixture entry ("1/sqrt(2)", "log(3)/2", 7)."""
    if isinstance(x, (int, float)):
        return float(x)
    return float(eval(x, {"__builtins__": {}}, {"sqrt": math.sqrt, "log": math.log}))


def eval_tree(t):
    if isinstance(t, list):
        return [eval_tree(e) for e in t]
    return eval_expr(t)


@pytest.fixture(scope="session")
def hand_worked():
    with open(os.path.join(GOLDEN, "hand_worked_n4.json")) as f:
        return json.load(f)
