"""Small shared helpers for the tests (no arithmetic of the method)."""
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def golden(name: str) -> dict:
    """key = value pairs of tests/golden/<name> (comments start with #)."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("=", 1))
                out[k] = v
    return out
