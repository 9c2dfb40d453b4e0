"""Parsers for the text fixtures under tests/golden (page values typed in by hand)."""
import ast
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def lines(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for raw in f:
            s = raw.strip()
            if s and not s.startswith("#"):
                yield s.split()


def tup(s):
    v = ast.literal_eval(s)
    return v if isinstance(v, tuple) else (v,)


def nested(s):
    """'((4,8),(2,2))' -> nested tuple; a bare integer stays an int."""
    return ast.literal_eval(s)
