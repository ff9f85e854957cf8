"""GPU tests of the bounded waits and of argument handling on a live device."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def txl():
    import transformer_xl_relative_gb300 as m
    return m


def test_bounded_wait_reports_timeout_and_context_survives(txl):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    txl.selftest_wait_timeout(err, 2000)          # nothing signals the barrier: 2 ms limit
    torch.cuda.synchronize()
    assert int(err.item()) == txl.native.TXL_ERR_TIMEOUT
    x = torch.arange(10, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 45.0


def test_rejected_arguments_raise(txl):
    q = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16, device="cuda")
    r = torch.zeros(4, 2, 64, dtype=torch.bfloat16, device="cuda")
    u = torch.zeros(2, 64, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(txl.TxlError) as e:          # n_rows below min(M+L, clamp_len+1)
        txl.rel_attn_fwd(q, None, q, q, u, u, r, 4, 1000, out)
    assert e.value.status == txl.native.TXL_ERR_INVALID_ARG
