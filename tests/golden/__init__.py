"""Reader for the small text fixtures in this folder."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def lines(name):
    """Non-comment, non-empty lines of fixture ``name``."""
    with open(os.path.join(HERE, name)) as f:
        return [ln.split("#")[0].strip() for ln in f if ln.split("#")[0].strip()]


def table(name):
    """``key value`` lines of fixture ``name`` as a dict of strings."""
    return dict(ln.split(None, 1) for ln in lines(name))
