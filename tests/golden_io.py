"""Readers for the hand-written fixtures in tests/golden/."""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_json(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def load_mask(name):
    """Returns (types int8 [L], times int64 [L], params dict, mask uint8 [L, L])."""
    types = times = None
    params = {}
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("types:"):
                types = np.array([int(x) for x in line.split(":", 1)[1].split()], dtype=np.int8)
            elif line.startswith("times:"):
                times = np.array([int(x) for x in line.split(":", 1)[1].split()], dtype=np.int64)
            elif line.startswith("params:"):
                for kv in line.split(":", 1)[1].split():
                    key, val = kv.split("=")
                    params[key] = val
            else:
                rows.append([int(x) for x in line.split()])
    return types, times, params, np.array(rows, dtype=np.uint8)


def mask_files():
    return sorted(f for f in os.listdir(GOLDEN) if f.startswith("mask_") and f.endswith(".txt"))
