"""Loader for the hand-derived JSON fixtures in this folder (expected values are written
by hand in each file's "derivation"; nothing here computes them)."""
import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def load(name: str) -> dict:
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def words(rows_hex) -> np.ndarray:
    return np.array([[int(w, 16) for w in r] for r in rows_hex], dtype=np.uint32)


def halves(rows_hex) -> np.ndarray:
    return np.array([[int(h, 16) for h in r] for r in rows_hex], dtype=np.uint16)


def x_bits(fx: dict) -> np.ndarray:
    x = np.zeros((fx["T"], fx["K"]), np.uint16)
    for e in fx["x_sparse"]:
        if e["k"] == "all":
            x[e["t"], :] = int(e["bf16"], 16)
        else:
            x[e["t"], e["k"]] = int(e["bf16"], 16)
    return x
