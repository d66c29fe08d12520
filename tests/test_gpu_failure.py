"""Bounded device waits: a wait on a barrier nobody arrives at runs out,
records its code, and the host reads H3_ERR_TIMEOUT; the context stays
usable afterwards. No fault, trap or hang is involved."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_wait_timeout_reports_status_and_context_survives(h3lib):
    h3lib.check_device_error()  # clean start
    h3lib.debug_wait_timeout(5_000_000)  # 5 ms limit
    with pytest.raises(h3lib.H3Error) as e:
        h3lib.check_device_error()
    assert e.value.status == 6 and "probe" in e.value.msg
    h3lib.check_device_error()  # the word was cleared
    gu = torch.randn(4, 16, device="cuda").to(torch.bfloat16)
    out = torch.empty(4, 8, device="cuda", dtype=torch.bfloat16)
    h3lib.swiglu(gu, out)
    h3lib.check_device_error()
    assert torch.isfinite(out.float()).all()
