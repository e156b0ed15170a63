"""Reader for the small text fixtures in this folder (``key = value`` lines)."""

import os

HERE = os.path.dirname(os.path.abspath(__file__))


def load(name):
    out = {}
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition("=")
            parts = val.split()
            try:
                nums = [int(x) for x in parts]
                out[key.strip()] = nums[0] if len(nums) == 1 else nums
            except ValueError:
                out[key.strip()] = val.strip()
    return out
