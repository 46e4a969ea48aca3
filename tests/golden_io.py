"""Readers for the hand-worked fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rows(name):
    """Yield the '|'-separated fields of each non-comment line of a fixture file."""
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            yield [part.strip() for part in line.split("|")]


def ints(field):
    return [int(x) for x in field.split()] if field else []


def floats(field):
    return [float(x) for x in field.split()] if field else []


def bits(field):
    return [int(c) for c in field]
