"""Failure detection without a GPU fault: a bounded wait that nothing satisfies
gives up, the kernel returns, and the host reads RA_ERR_TIMEOUT; the context
stays usable afterwards."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import context_ra_forward_gb300 as ra
    st, _ = ra.check_device_status()
    assert st == 0
    ra.debug_wait_timeout(20000)  # 20 ms limit on a barrier nobody arrives on
    st, detail = ra.check_device_status()
    assert st == -5 and detail[0] == -5 and detail[1] == 3
    # the word is cleared by the read and the context still runs kernels
    st, _ = ra.check_device_status()
    assert st == 0
    x = torch.randn(1, 1, 64, 128, device="cuda").to(torch.bfloat16)
    y = ra.zigzag_permute(x, 2, "zigzag")
    assert torch.equal(ra.unpermute(y, 2, "zigzag").view(torch.int16), x.view(torch.int16))
