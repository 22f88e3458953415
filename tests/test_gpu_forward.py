"""Forward parity: CUDA path vs the fp64 oracle on the same seeded bf16 inputs."""
import numpy as np
import pytest

from gpu_common import device, status_ok, torch
import parity

import fa_workloads as W
import io_aware_exact_15_gb300 as fa

pytestmark = pytest.mark.gpu


def run_forward(q, k, v, scale, causal, dev):
    B, H, N, d = q.shape
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    assert fa.fa_forward(qd, kd, vd, o, lse, B, H, N, d, scale, causal) == fa.FA_OK
    status_ok()
    return o.cpu(), lse.cpu()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_forward_running_max_jumps(d, causal):
    # Later key tiles score far above the running max: tile 2 (keys 256-383)
    # x4, so that many rows' weights exceed 2^8 against the max of tiles
    # 0-1 and m must be rescaled, and tile 4 (keys 512-639) x60, whose
    # weights against the earlier max overflow fp32.  Both cases take the
    # forward's exact path after its speculative pass; checked in the form
    # fa_forward picks and in the two-tile form.
    dev = device()
    B, H, N = 1, 2, 700
    q, k, v, _ = W.make_qkv(B, H, N, d, seed=900 + d + causal, with_do=False)
    kf = k.float()
    kf[:, :, 256:384] *= 4.0
    kf[:, :, 512:640] *= 60.0
    k = kf.to(torch.bfloat16)
    scale = 1.0 / d ** 0.5
    o_ref, lse_ref = parity.oracle_forward(q, k, v, scale, causal)
    o, lse = run_forward(q, k, v, scale, causal, dev)
    parity.check_forward(o, lse, o_ref, lse_ref, f"max jumps d={d} causal={causal}")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o2 = torch.full_like(qd, float("nan"))
    lse2 = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    assert fa.fa_debug_forward_config(qd, kd, vd, o2, lse2, B, H, N, d, scale, causal, 256, 128,
                                      8 if d == 64 else 5) == fa.FA_OK
    status_ok()
    parity.check_forward(o2.cpu(), lse2.cpu(), o_ref, lse_ref,
                         f"max jumps, two-tile form, d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 100, 128, 129, 255, 300, 513])
def test_forward_small_full(N, d, causal):
    dev = device()
    q, k, v, _ = W.make_qkv(2, 2, N, d, seed=N * 7 + d + causal, with_do=False)
    scale = 1.0 / d ** 0.5
    o, lse = run_forward(q, k, v, scale, causal, dev)
    o_ref, lse_ref = parity.oracle_forward(q, k, v, scale, causal)
    parity.check_forward(o, lse, o_ref, lse_ref, f"N={N} d={d} causal={causal}")
    # grids this small run the compact one-tile form; the two-tile form of
    # long sequences (same ring depth) on the same ragged lengths
    B, H = 2, 2
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o2 = torch.full_like(qd, float("nan"))
    lse2 = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    assert fa.fa_debug_forward_config(qd, kd, vd, o2, lse2, B, H, N, d, scale, causal, 256, 128,
                                      8 if d == 64 else 5) == fa.FA_OK
    status_ok()
    parity.check_forward(o2.cpu(), lse2.cpu(), o_ref, lse_ref,
                         f"two-tile form N={N} d={d} causal={causal}")


def test_forward_scale_and_peaked_keys():
    dev = device()
    q, k, v, _ = W.make_qkv(1, 3, 384, 128, seed=5, peaked_frac=0.02, mask_seed=6, with_do=False)
    for scale in (0.02, 0.3):
        o, lse = run_forward(q, k, v, scale, True, dev)
        o_ref, lse_ref = parity.oracle_forward(q, k, v, scale, True)
        parity.check_forward(o, lse, o_ref, lse_ref, f"scale={scale}")


@pytest.mark.parametrize("name", ["single_head_fwd", "bert_large", "gpt2_causal"])
def test_forward_named_workload_full(name):
    dev = device()
    w = W.WORKLOADS[name]
    q, k, v, _, _ = W.make_inputs(w, with_do=False)
    o, lse = run_forward(q, k, v, w.scale, w.causal, dev)
    o_ref, lse_ref = parity.oracle_forward(q, k, v, w.scale, w.causal)
    parity.check_forward(o, lse, o_ref, lse_ref, name)
