"""Readers for the fixture files under tests/golden/ (each cites its source)."""
import os
import shlex

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rows(name):
    """Non-comment rows of a fixture, split on whitespace (quotes respected)."""
    out = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            out.append(shlex.split(line))
    return out
