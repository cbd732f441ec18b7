import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long CPU test")
    config.addinivalue_line(
        "markers", "small_route: runs with the library's default routing of small products "
                   "(CUDA cores); other GPU tests send every product to the tensor cores")


@pytest.fixture(autouse=True)
def _tensor_route_for_pipeline_tests(request):
    """GPU tests written for the tensor-core pipelines keep them under test at
    small sizes (ragged tiles, global-load modes, split schedules): products
    that the library would send to its CUDA-core route by default go to the
    tensor cores while such a test runs.  Tests marked small_route run with
    the default routing."""
    if request.node.get_closest_marker("gpu") is None or request.node.get_closest_marker("small_route"):
        yield
        return
    import ternary_weight_int8_t3_gb300 as t3
    prev = t3.t3_set_small_product_limit(0)
    try:
        yield
    finally:
        t3.t3_set_small_product_limit(prev)


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    """Non-comment, non-empty lines of a golden fixture, split on whitespace."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out
