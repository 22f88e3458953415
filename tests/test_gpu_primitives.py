"""tcgen05 / TMA operand forms and the bounded-wait path, one tile at a time."""
import pytest

from gpu_common import device, status_ok, torch

import io_aware_exact_15_gb300 as fa

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode,n", [(0, 128), (1, 64), (1, 128), (2, 64), (2, 128), (3, 64),
                                    (3, 128)])
def test_mma_probe_matches_fp32_matmul(mode, n):
    dev = device()
    g = torch.Generator().manual_seed(100 + 10 * mode + n)
    a = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    b = torch.randn(128, n, generator=g).to(torch.bfloat16)
    if mode == 0:
        ref = a.float() @ b.float().T
    elif mode in (1, 3):
        ref = a.float() @ b.float()
    else:
        ref = a.float().T @ b.float()
    c = torch.full((128, ref.shape[1]), float("nan"), dtype=torch.float32, device=dev)
    assert fa.fa_debug_mma_probe(a.to(dev), b.to(dev), c, mode, n) == fa.FA_OK
    status_ok()
    err = (c.cpu() - ref).abs().max().item()
    assert err <= 1e-3 * max(1.0, ref.abs().max().item()), err


def test_wait_timeout_is_reported_and_context_survives():
    dev = device()
    assert fa.fa_debug_wait_timeout(50_000_000) == fa.FA_OK  # 50 ms
    assert fa.fa_get_device_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_get_device_status() == fa.FA_OK  # read-and-clear
    # the context is still usable: a probe MMA runs and is correct
    a = torch.eye(128, dtype=torch.bfloat16)
    b = torch.arange(128 * 64, dtype=torch.float32).reshape(128, 64).remainder(7).to(torch.bfloat16)
    c = torch.empty(128, 64, dtype=torch.float32, device=dev)
    assert fa.fa_debug_mma_probe(a.to(dev), b.to(dev), c, 1, 64) == fa.FA_OK
    status_ok()
    assert torch.equal(c.cpu(), b.float())
