"""The bounded-wait error path on the GPU: a wait that runs out ends as an
error status the host reads, not as a hung kernel, and the context stays
usable afterwards.  The failure is made by a diagnostic kernel that waits
with a short limit on an mbarrier phase nothing completes."""
import pytest

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_clears(lib):
    import torch

    s = torch.cuda.Stream()
    assert lib.last_device_error(s) == 0          # nothing recorded so far
    lib.selftest_bounded_wait(2_000_000, stream=s)  # 2 ms limit
    assert lib.last_device_error(s, clear=True) == -5   # QLORA_ERR_TIMEOUT
    assert lib.last_device_error(s) == 0          # cleared
    # the context is still usable: a regular call on the same stream works
    x = torch.ones(1024, device="cuda")
    with torch.cuda.stream(s):
        y = x * 2
    s.synchronize()
    assert float(y.sum()) == 2048.0


def test_selftest_rejects_long_limits(lib):
    with pytest.raises(lib.QloraError) as e:
        lib.selftest_bounded_wait(5_000_000_000)
    assert e.value.status == -1
    with pytest.raises(lib.QloraError) as e:
        lib.selftest_bounded_wait(0)
    assert e.value.status == -1
