"""Device-side failure reporting without a GPU fault: a bounded wait that runs out records
DFLASH2_ERR_TIMEOUT and returns; the context stays usable."""
import pytest

from tests.gpu_util import require_gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports(torch_mod=None):
    torch = require_gpu()
    import dflash2_block_drafter_gb300 as d
    assert d.dflash2_poll_error() == 0
    d.dflash2_selftest_bounded_wait(2000)   # 2 ms on an mbarrier nothing completes
    assert d.dflash2_poll_error() == -5
    assert d.dflash2_poll_error() == 0
    # the context still works afterwards
    x = torch.ones(4, device="cuda")
    assert float(x.sum()) == 4.0
