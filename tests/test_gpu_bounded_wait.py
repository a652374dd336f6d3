"""The bounded waits give up instead of hanging.

Every pipeline wait of the library's kernels (copy and hand-off barriers)
gives up after a wall-clock limit, records NK_STATUS_TIMEOUT in the device
status word and returns.  nk_selftest_bounded_wait runs that same wait on a
barrier phase that can never complete (one arrival short; no copy involved),
with a 1 ms limit, so the timeout path runs without any fault or hang."""

import pytest
import torch

from paged_kv_cache_append_gb300 import nk

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout():
    nk.load()
    s = torch.cuda.current_stream()
    torch.cuda.synchronize()
    assert nk.nk_status_read(clear=True, stream=s.cuda_stream) & 4 == 0
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    nk.nk_selftest_bounded_wait(1000, waited.data_ptr(), s.cuda_stream)
    s.synchronize()                                   # the kernel returned
    st = nk.nk_status_read(clear=True, stream=s.cuda_stream)
    assert st & 4, f"status {st:#x}: NK_STATUS_TIMEOUT not set"
    ns = int(waited.item())
    assert 1_000_000 <= ns < 1_000_000_000, f"waited {ns} ns for a 1 ms limit"
    # the context is still usable and the status word is clear again
    x = torch.arange(16, device="cuda", dtype=torch.float32)
    assert float((x * 2).sum().item()) == 240.0
    assert nk.nk_status_read(clear=False, stream=s.cuda_stream) == 0


def test_bounded_wait_rejects_limits_outside_the_range():
    nk.load()
    for bad in (0, -5, 1_000_001):
        with pytest.raises(nk.NkError) as e:
            nk.nk_selftest_bounded_wait(bad)
        assert e.value.code == -1
