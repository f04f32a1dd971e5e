import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def load_golden(name):
    import json
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def golden_value(x):
    """Evaluate a hand-worked fixture entry: a number or a short closed form."""
    import math
    if isinstance(x, (int, float)):
        return float(x)
    env = {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4), "ln5": math.log(5),
           "ln14": math.log(14), "ln": math.log, "inf": math.inf}
    return float(eval(x, {"__builtins__": {}}, env))
