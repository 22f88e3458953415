"""Every tile configuration of the block-size sweep computes the same exact
attention: parity against the oracle for each (rows per CTA, K/V stages)."""
import pytest

from gpu_common import device, status_ok, torch
import parity

import fa_workloads as W
import io_aware_exact_15_gb300 as fa

pytestmark = pytest.mark.gpu

CONFIGS = [(128, 128, 2), (128, 128, 3), (128, 256, 4), (128, 128, 5), (128, 256, 2),
           (64, 128, 2), (64, 256, 4), (64, 128, 8)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,rows,stages", CONFIGS)
def test_forward_config_parity(d, rows, stages, causal):
    dev = device()
    B, H, N = 1, 3, 700
    q, k, v, _ = W.make_qkv(B, H, N, d, seed=rows + stages + d + causal, with_do=False)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    scale = 1.0 / d ** 0.5
    assert fa.fa_debug_forward_config(qd, kd, vd, o, lse, B, H, N, d, scale, causal, rows,
                                      stages) == fa.FA_OK
    status_ok()
    o_ref, lse_ref = parity.oracle_forward(q, k, v, scale, causal)
    parity.check_forward(o.cpu(), lse.cpu(), o_ref, lse_ref, f"d={d} rows={rows} stages={stages}")


def test_forward_config_rejects_unsupported():
    dev = device()
    x = torch.empty(16, dtype=torch.uint8, device=dev)
    p = x.data_ptr()
    assert fa.fa_debug_forward_config(p, p, p, p, p, 1, 1, 128, 128, 0.1, 0, 192, 3) == \
        fa.FA_ERR_UNSUPPORTED
    assert fa.fa_debug_forward_config(p, p, p, p, p, 1, 1, 128, 128, 0.1, 0, 128, 6) == \
        fa.FA_ERR_UNSUPPORTED
    assert fa.fa_debug_forward_config(p, p, p, p, p, 1, 1, 128, 64, 0.1, 0, 128, 3) == \
        fa.FA_ERR_UNSUPPORTED
