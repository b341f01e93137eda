"""Reader for the hand-derived fixtures under ``tests/golden/``.

Each fixture is plain text: ``#`` lines carry the citation and the derivation,
other lines are ``key: value`` with integers or space-separated integer lists.
"""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            parts = val.split()
            try:
                nums = [int(v) for v in parts]
            except ValueError:
                out[key.strip()] = val.strip()
                continue
            k = key.strip()
            out[k] = nums[0] if len(nums) == 1 and not k.startswith("expected") else nums
    return out


def examples(op: str):
    return [n for n in sorted(os.listdir(GOLDEN))
            if n.endswith(".txt") and n.startswith(op + "_")]
