import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(session, config, items):
    """Within each module, run the fp32 cases (plain FFMA kernels) before bf16."""
    def dtype_rank(item):
        cs = getattr(item, "callspec", None)
        d = cs.params.get("dtype") if cs is not None else None
        return 0 if d in (None, "f32") else 1

    order = {}
    for i, it in enumerate(items):
        order.setdefault(str(it.fspath), i)
    items.sort(key=lambda it: (order[str(it.fspath)], dtype_rank(it)))
