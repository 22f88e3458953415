"""fa_backward_noalloc: the backward for callers that cannot allocate device
memory (no workspace from their host framework, or no cudaMalloc allowed
while running).  Its scratch is a fixed 32 MiB array inside the library.

Checked through the C ABI against fa_backward (caller workspace) on the same
inputs, within the parity tolerance of the other GPU tests, on consecutive
calls that share the array.  Collected last on purpose (file name), and
independent of every other test: it passes alone in a fresh process too.
"""
import pytest

from gpu_common import device, status_ok, torch
import parity

import fa_workloads as W
import io_aware_exact_15_gb300 as fa

pytestmark = pytest.mark.gpu


def _forward(q, k, v, scale, causal):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    assert fa.fa_forward(q, k, v, o, lse, B, H, N, d, scale, causal) == fa.FA_OK
    return o, lse


def _with_workspace(q, k, v, o, do, lse, scale, causal):
    B, H, N, d = q.shape
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    nbytes = fa.fa_backward_workspace_size(B, H, N, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    assert fa.fa_backward(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, scale, causal, ws,
                          nbytes) == fa.FA_OK
    status_ok()
    return dq, dk, dv


def _no_alloc(q, k, v, o, do, lse, scale, causal):
    B, H, N, d = q.shape
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    assert fa.fa_backward_noalloc(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, scale,
                                  causal) == fa.FA_OK
    status_ok()
    return dq, dk, dv


@pytest.mark.parametrize("shape,causal", [((2, 4, 600, 64), True), ((1, 3, 1000, 128), False)])
def test_noalloc_matches_workspace_backward_twice(shape, causal):
    dev = device()
    B, H, N, d = shape
    q, k, v, do = (t.to(dev) for t in W.make_qkv(B, H, N, d, seed=B * N + d))
    scale = 1.0 / d ** 0.5
    o, lse = _forward(q, k, v, scale, causal)
    ref = _with_workspace(q, k, v, o, do, lse, scale, causal)
    for call in range(2):  # consecutive calls share (and reuse) the scratch array
        got = _no_alloc(q, k, v, o, do, lse, scale, causal)
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            parity.check_grad(g.cpu(), parity.f64(r), name, f"no-alloc call {call}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    dev = device()
    A = torch.empty(16, dtype=torch.uint8, device=dev)
    p = A.data_ptr()
    # d = 128, 2^17 rows: workspace 2^19 + 2^26 bytes > 32 MiB
    assert fa.fa_backward_noalloc(p, p, p, p, p, p, p, p, p, 1, 32, 4096, 128, 0.1,
                                  0) == fa.FA_ERR_WORKSPACE
    assert fa.fa_backward_noalloc(p, p, p, p, p, p, p, p, p, 0, 1, 128, 64, 0.1,
                                  0) == fa.FA_ERR_INVALID_ARG
