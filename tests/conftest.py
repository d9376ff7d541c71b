import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


import pytest  # noqa: E402


@pytest.fixture(autouse=True)
def _guard_bands(request):
    """After a GPU test, every guard band around its outputs must be intact,
    and no bounded wait of a pipelined kernel may have run out (the tests
    that make one run out read and clear the flag themselves): a wait that
    expires leaves correct-looking results only slower, so the flag is the
    only sign of it."""
    if request.node.get_closest_marker("gpu") is None:
        yield
        return
    import gdn_testutil
    gdn_testutil.reset_guards()
    yield
    expired = False
    try:
        import torch
        if torch.cuda.is_available():
            torch.cuda.synchronize()
            import linear_attention_recurrence_step_gb300 as gdn
            expired = gdn.wait_status()
    except Exception:
        pass
    bad = gdn_testutil.broken_guards()
    gdn_testutil.reset_guards()
    assert not bad, "; ".join(bad)
    assert not expired, "a bounded wait of a pipelined kernel ran out during the test"
