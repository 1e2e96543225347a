"""Failure detection without a GPU fault: the bounded pipeline wait every
tensor-core kernel uses gives up on a barrier that nothing arrives on, reports
MOE_DEV_TIMEOUT in the caller's error word, and the context stays usable."""
import pytest
import torch

import combine_softmax_top_expert_b300 as moe

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    moe.lib()
    return torch.device("cuda:0")


@pytest.mark.parametrize("limit_ms", [5, 40])
def test_wait_gives_up_and_reports_timeout(dev, limit_ms):
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    waited = torch.zeros(1, dtype=torch.int32, device=dev)
    moe.moe_selftest_wait_timeout(err, limit_ms * 1_000_000, waited)
    torch.cuda.synchronize()
    assert int(err.item()) == moe.MOE_DEV_TIMEOUT
    # the wait lasted its limit and not much longer (sleep hints are 0.5 ms)
    assert limit_ms <= int(waited.item()) <= limit_ms + 50


def test_timeout_bit_is_ored_into_existing_bits(dev):
    err = torch.full((1,), moe.MOE_DEV_ID_RANGE, dtype=torch.int32, device=dev)
    moe.moe_selftest_wait_timeout(err, 1_000_000)
    torch.cuda.synchronize()
    assert int(err.item()) == moe.MOE_DEV_ID_RANGE | moe.MOE_DEV_TIMEOUT


def test_context_usable_after_timeout(dev):
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    moe.moe_selftest_wait_timeout(err, 2_000_000)
    torch.cuda.synchronize()
    assert int(err.item()) == moe.MOE_DEV_TIMEOUT
    # the next launches on the same context run normally
    g = torch.Generator().manual_seed(5)
    T, E, k = 64, 16, 4
    logits = torch.randn(T, E, generator=g).to(dev)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    err2 = torch.zeros(1, dtype=torch.int32, device=dev)
    moe.moe_route(logits, T, E, k, ids, w, err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    want = torch.topk(torch.softmax(logits.double().cpu(), -1), k, dim=-1).indices
    assert torch.equal(ids.cpu().long().sort(-1).values, want.sort(-1).values)
