import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


# With ULY_CHECKED=1 the binding loads the checked build of the library:
# every GPU test then also fails if its kernels counted an index outside a
# tensor (tests that provoke violations on purpose reset the count).
import pytest  # noqa: E402


@pytest.fixture(autouse=True)
def _no_index_violations(request):
    yield
    if os.environ.get("ULY_CHECKED", "") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    import ulysses_sequence_attention_uly_gb300 as uly
    n = uly.checked_violations(reset=True)
    assert n == 0, "%d index-check violations in the checked build" % n
