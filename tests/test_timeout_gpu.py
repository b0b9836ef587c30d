"""The bounded device-side wait on the GPU: a wait that nothing completes ends after its
budget with GDN_ERR_TIMEOUT in the status word, and the context stays usable (a decode
step afterwards is still correct).  Nothing faults, traps or hangs."""
import pytest
import torch

from gated_deltanet_layer_conv1d_gb300 import gdn
from gated_deltanet_layer_conv1d_gb300 import workloads as wl
from tests.gpu_common import require_gpu
from tests.test_decode_gpu import check_against_oracle, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_wait_that_never_completes_reports_timeout_and_returns():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    gdn.gdn_selftest_wait(5_000_000, status)  # 5 ms
    e1.record()
    torch.cuda.synchronize()
    assert int(status.item()) == 19, gdn.status_string(int(status.item()))
    assert 4.0 <= e0.elapsed_time(e1) < 1000.0  # it waited its budget, then gave up
    # first error wins: a second timeout does not overwrite, a fresh word gets it again
    gdn.gdn_selftest_wait(1_000_000, status)
    fresh = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_selftest_wait(1_000_000, fresh)
    torch.cuda.synchronize()
    assert int(status.item()) == 19 and int(fresh.item()) == 19
    # the context is still usable
    w = wl.batched_decode(n=3, steps=2, shape=wl.TINY, seed=61)
    ys, cores, H, conv, _ = run_decode(w)
    check_against_oracle(w, ys, cores, H, conv)
