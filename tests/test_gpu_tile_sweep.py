"""Every tile configuration of the block-size sweep computes the same exact
attention: parity against the oracle for each (rows per CTA, key tile B_c,
K/V stages), dense and causal, at a length that is a multiple of none of
the key tiles (700 = 5 x 128 + 60 = 10 x 64 + 60 = 2 x 256 + 188)."""
import pytest

from gpu_common import device, status_ok, torch
import parity

import fa_workloads as W
import io_aware_exact_15_gb300 as fa

pytestmark = pytest.mark.gpu

# (d, key tile) -> K/V ring stages the library builds
STAGES = {(128, 128): (2, 3, 4, 5), (128, 64): (4, 8), (128, 256): (2,),
          (64, 128): (2, 4, 8), (64, 64): (8, 16), (64, 256): (2, 4)}
CONFIGS = [(d, rows, bc, st) for (d, bc), sts in STAGES.items() for st in sts
           for rows in ((128,) if bc == 256 else (128, 256))]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d,rows,bc,stages", CONFIGS)
def test_forward_config_parity(d, rows, bc, stages, causal):
    dev = device()
    B, H, N = 1, 3, 700
    q, k, v, _ = W.make_qkv(B, H, N, d, seed=rows + bc + stages + d + causal, with_do=False)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    scale = 1.0 / d ** 0.5
    assert fa.fa_debug_forward_config(qd, kd, vd, o, lse, B, H, N, d, scale, causal, rows, bc,
                                      stages) == fa.FA_OK
    status_ok()
    o_ref, lse_ref = parity.oracle_forward(q, k, v, scale, causal)
    parity.check_forward(o.cpu(), lse.cpu(), o_ref, lse_ref,
                         f"d={d} rows={rows} key tile={bc} stages={stages} causal={causal}")


def test_forward_config_rejects_unsupported():
    dev = device()
    x = torch.empty(16, dtype=torch.uint8, device=dev)
    p = x.data_ptr()
    bad = [(128, 192, 128, 3), (128, 128, 128, 6), (64, 128, 128, 3), (128, 256, 256, 2),
           (128, 128, 32, 4), (128, 128, 256, 3), (64, 128, 64, 4)]
    for d, rows, bc, st in bad:
        assert fa.fa_debug_forward_config(p, p, p, p, p, 1, 1, 128, d, 0.1, 0, rows, bc, st) == \
            fa.FA_ERR_UNSUPPORTED, (d, rows, bc, st)
