import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libgtms.so")


@pytest.fixture(scope="session")
def golden_worked_example():
    """Parse tests/golden/worked_example.txt (the README's printed worked example)."""
    import numpy as np

    path = os.path.join(ROOT, "tests", "golden", "worked_example.txt")
    seq_lens, masks, outs = None, {}, {}
    cur = None
    with open(path, encoding="utf-8") as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] == "seq_lens":
                seq_lens = [int(t) for t in tok[1:]]
            elif tok[0] == "mask":
                cur = masks.setdefault(int(tok[1]), [])
            elif tok[0] == "output":
                cur = outs.setdefault((int(tok[1]), int(tok[2])), [])
            else:
                cur.append([float(t) for t in tok])
    B, M, S = len(seq_lens), 2, 5
    mask = np.array([masks[b] for b in range(B)], dtype=bool)
    out = np.array([[outs[(b, m)] for m in range(M)] for b in range(B)], dtype=np.float64)
    assert mask.shape == (B, S, S) and out.shape == (B, M, S, S)
    return np.array(seq_lens, dtype=np.int32), mask, out
