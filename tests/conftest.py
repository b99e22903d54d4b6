import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: a long-running test (full-size model on the CPU oracle)")


def read_golden(name: str) -> dict:
    """Parse a ``key = value  # citation`` fixture under tests/golden."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = v
    return out


@pytest.fixture(autouse=True)
def _check_canaries_at_close(request, monkeypatch):
    """Every model a GPU test closes first has the guard words around its
    device buffers checked: a kernel that wrote past either end of a buffer
    fails the test that ran it."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    import qwen2_decoder_forward_gb300 as q2
    close = q2.Qwen2Model.close

    def checked_close(self):
        if getattr(self, "_h", None):
            try:
                self.check_canaries()
            finally:
                close(self)

    monkeypatch.setattr(q2.Qwen2Model, "close", checked_close)
    yield
