"""Loader for the hand-derived worked examples in tests/golden/."""
import json
import os

import numpy as np

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_examples.json")


def cases():
    with open(PATH) as f:
        data = json.load(f)
    out = []
    for c in data["cases"]:
        K, L, V = c["K"], c["L"], c["V"]
        d = dict(c)
        d["target"] = np.asarray(c["target"], np.float32).reshape(1, K, L + 1, V)
        d["draft"] = np.asarray(c["draft"], np.float32).reshape(1, K, L, V)
        d["tokens"] = np.asarray(c["tokens"], np.int32).reshape(1, K, L)
        d["lengths"] = None if c["lengths"] is None else np.asarray(c["lengths"], np.int32)
        d["accept_u"] = (np.zeros((1, K, L), np.float32) if c["accept_u"] is None
                         else np.asarray(c["accept_u"], np.float32).reshape(1, K, L))
        d["sample_u"] = (np.zeros((1, K, L + 1), np.float32) if c["sample_u"] is None
                         else np.asarray(c["sample_u"], np.float32).reshape(1, K, L + 1))
        out.append(d)
    return out
