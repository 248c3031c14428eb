"""Reader for the small text fixtures under tests/golden (``name: values`` lines)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read(name):
    """Returns a list of (key, value-string) pairs in file order."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out.append((k.strip(), v.strip()))
    return out


def ints(s):
    return [int(x, 0) for x in s.split()]
