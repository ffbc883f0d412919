"""Loads the worked cases of tests/golden/ (inputs and the oracle's stored y, h_last)."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
NAMES = ("exact_integer", "gated_small", "scalar_small")


def load(name: str) -> dict:
    with open(os.path.join(GOLDEN, name + ".json")) as f:
        fx = json.load(f)
    inp = {k: (None if v is None else np.asarray(v, np.float32)) for k, v in fx["inputs"].items()}
    exp = {k: np.vectorize(float.fromhex)(np.asarray(v)).astype(np.float64) for k, v in fx["expected"].items()}
    return {"name": fx["name"], "cite": fx["cite"], "softplus": fx["softplus"], "inputs": inp, "expected": exp}
