"""Reader for the small text fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            s = raw.split("#", 1)[0].strip()
            if s:
                yield s.split()


def table(name):
    """{first token: [remaining tokens]} for key-value fixtures."""
    out = {}
    for toks in lines(name):
        out.setdefault(toks[0], []).append(toks[1:])
    return out
