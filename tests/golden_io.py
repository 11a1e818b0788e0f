"""Reads the key = value fixtures under tests/golden/."""

import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (x.strip() for x in line.split("=", 1))
            parts = val.split()
            nums = [float(p) if "." in p else int(p) for p in parts]
            out[key] = nums if len(nums) > 1 else nums[0]
    return out
