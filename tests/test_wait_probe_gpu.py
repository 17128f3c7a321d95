"""The kernels' bounded waits end with a status, not a hang.

Every wait in the library's kernels polls its mbarrier a bounded number of
times; when the bound runs out the kernel records TOPK_DEV_INTERNAL in the
device status word and goes on.  topk_ragged_wait_probe makes such a wait on
an mbarrier that nothing completes (no fault, no trap: the wait simply runs
out), so these tests can check the whole path -- the status bit, its
clearing on read, and a context that still computes correct selections
afterwards.
"""
import pytest
import torch

import sparse_attention_deterministic_gb300 as pkg
import workloads as W
from helpers import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkg.build()
    pkg.init()


def test_wait_that_never_completes_reports_internal():
    assert pkg.device_status() == 0
    pkg.wait_probe(4096)
    torch.cuda.synchronize()
    assert pkg.device_status() == pkg.TOPK_DEV_INTERNAL
    assert pkg.device_status() == 0          # read clears it


def test_context_still_selects_after_the_probe():
    pkg.wait_probe(1024)
    assert pkg.device_status() == pkg.TOPK_DEV_INTERNAL
    assert_parity(W.make("tiny"))            # also checks that the status word is clear again
    assert_parity(W.make("decode"))


def test_probe_argument_range():
    for bad in (0, (1 << 22) + 1):
        with pytest.raises(pkg.TopkError) as e:
            pkg.wait_probe(bad)
        assert e.value.status == 1           # TOPK_ERR_INVALID_ARG
    assert pkg.device_status() == 0
