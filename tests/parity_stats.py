"""Parity statistics of the GPU tests.

When the environment variable FP4_PARITY_STATS names a file, every
tolerance check appends one JSON line to it: the test, what was compared,
and the observed statistic (for a contraction the relative Frobenius error
and the largest |err| / sum_k |a_k b_k|; for a masked view comparison the
fraction of scale blocks whose inputs differ from the oracle's).  The line is
written before the assertion, so a failing check is recorded too."""
import json
import os


def record(what: str, **stats):
    path = os.environ.get("FP4_PARITY_STATS")
    if not path:
        return
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    with open(path, "a") as f:
        f.write(json.dumps({"test": test, "what": what, **{k: float(v) for k, v in stats.items()}}) + "\n")
