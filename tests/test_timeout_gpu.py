"""A device wait that runs out (failure handling without a GPU fault).

Every mbarrier wait in the kernels is bounded; when one gives up, the CTA sets
the timeout bit of the block mask's status word, drains its in-flight copies
and MMAs, frees its TMEM and exits, and fa_get_status reports FA_ERR_TIMEOUT.
This test makes that happen on purpose, in a child process bound to a test
build of the library whose producer skips one load (see timeout_child.py),
for the forward and for the backward, and checks that the GPU stays usable:
the next call on the same context passes parity.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_starved_wait_reports_timeout_and_context_survives():
    pytest.importorskip("block_sparse_masked_fa_gb300")
    r = subprocess.run([sys.executable, os.path.join(HERE, "timeout_child.py")], capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, f"child failed:\n{r.stdout[-3000:]}\n{r.stderr[-3000:]}"
    assert "timeout path ok" in r.stdout
