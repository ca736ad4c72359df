import json
import os
import sys
from fractions import Fraction
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

GOLDEN = Path(__file__).resolve().parent / "golden"


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def load_golden(name):
    with open(GOLDEN / name) as f:
        return json.load(f)


def frac(s):
    return Fraction(s)


@pytest.fixture(scope="session")
def markov():
    """The rayaq.ca three-token Markov tables as Fractions, keyed by token index."""
    g = load_golden("rayaq_markov_example.json")
    voc = g["vocabulary"]
    P = {voc.index(k): [Fraction(x) for x in v] for k, v in g["target_p"].items()}
    Q = {voc.index(k): [Fraction(x) for x in v] for k, v in g["draft_q"].items()}
    return g, voc, P, Q


def gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


os.environ.setdefault("PYTHONHASHSEED", "0")
