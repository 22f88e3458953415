"""Out-of-bounds writes, checked without a sanitizer: every output and
workspace of every entry point sits inside a larger buffer whose margins
(4 KiB before, 4 KiB after) hold a sentinel byte pattern; after the call the
margins must be untouched and the inputs unchanged.  Ragged lengths put the
last tile partly past the end of each tensor, which is where a missing row
guard on a store or a TMA reduce-add would write."""
import numpy as np
import pytest

from gpu_common import device, status_ok, torch

import fa_workloads as W
import io_aware_exact_15_gb300 as fa

pytestmark = pytest.mark.gpu

MARGIN = 4096
SENTINEL = 0xA5


class Guarded:
    """Tensors carved out of sentinel-filled buffers with margins."""

    def __init__(self, dev):
        self.dev = dev
        self.bufs = []

    def tensor(self, shape, dtype, name):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        buf = torch.full((MARGIN + n + MARGIN,), SENTINEL, dtype=torch.uint8, device=self.dev)
        self.bufs.append((name, buf, n))
        return buf[MARGIN:MARGIN + n].view(dtype).view(shape)

    def workspace(self, nbytes, name="workspace"):
        return self.tensor((nbytes,), torch.uint8, name)

    def check(self, what):
        status_ok()
        for name, buf, n in self.bufs:
            head = buf[:MARGIN]
            tail = buf[MARGIN + n:]
            assert bool((head == SENTINEL).all()), f"{what}: write before {name}"
            assert bool((tail == SENTINEL).all()), f"{what}: write past the end of {name}"


def _inputs(shape, dev, seed):
    g = torch.Generator().manual_seed(seed)
    return [W.randn_bf16(shape, g).to(dev) for _ in range(4)]


def _unchanged(inputs, copies, what):
    for a, b in zip(inputs, copies):
        assert torch.equal(a, b), f"{what}: an input was modified"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 7, 129, 255])
def test_equal_length_entry_points_stay_in_bounds(N, d):
    dev = device()
    B, H, Hkv = 2, 4, 2
    scale = 1.0 / d ** 0.5
    q, k, v, do = _inputs((B, H, N, d), dev, 50 + N + d)
    kg, vg = k[:, :Hkv].contiguous(), v[:, :Hkv].contiguous()
    copies = [t.clone() for t in (q, k, v, do, kg, vg)]
    nT = (N + 127) // 128
    mask = torch.from_numpy(W.random_block_mask(1, nT, seed=N, density=0.7)).to(dev)
    mask[0, :, 0] = 1
    for causal in (0, 1):
        for kind in ("plain", "gqa", "dropout", "sparse", "deterministic", "noalloc"):
            what = f"{kind} N={N} d={d} causal={causal}"
            g = Guarded(dev)
            kv_h = Hkv if kind == "gqa" else H
            kk, vv = (kg, vg) if kind == "gqa" else (k, v)
            o = g.tensor((B, H, N, d), torch.bfloat16, "O")
            lse = g.tensor((B, H, N), torch.float32, "lse")
            dq = g.tensor((B, H, N, d), torch.bfloat16, "dQ")
            dk = g.tensor((B, kv_h, N, d), torch.bfloat16, "dK")
            dv = g.tensor((B, kv_h, N, d), torch.bfloat16, "dV")
            drop = (0.25, 99 + N, 3)
            if kind == "sparse":
                nb = fa.fa_blocksparse_workspace_size(B, H, N, d, 1)
                ws = g.workspace(nb)
                assert fa.fa_blocksparse_forward(q, k, v, o, lse, B, H, N, d, scale, causal, mask,
                                                 1, ws, nb) == fa.FA_OK
                g.check(what + " forward")
                assert fa.fa_blocksparse_backward(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d,
                                                  scale, causal, mask, 1, ws, nb) == fa.FA_OK
            else:
                if kind == "gqa":
                    st = fa.fa_forward_gqa(q, kk, vv, o, lse, B, H, Hkv, N, d, scale, causal)
                elif kind == "dropout":
                    st = fa.fa_forward_dropout(q, k, v, o, lse, B, H, N, d, scale, causal, *drop)
                else:
                    st = fa.fa_forward(q, k, v, o, lse, B, H, N, d, scale, causal)
                assert st == fa.FA_OK
                g.check(what + " forward")
                nb = fa.fa_backward_workspace_size(B, H, N, d)
                ws = g.workspace(nb)
                if kind == "gqa":
                    st = fa.fa_backward_gqa(q, kk, vv, o, do, lse, dq, dk, dv, B, H, Hkv, N, d,
                                            scale, causal, ws, nb)
                elif kind == "dropout":
                    st = fa.fa_backward_dropout(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d,
                                                scale, causal, *drop, ws, nb)
                elif kind == "deterministic":
                    st = fa.fa_backward_deterministic(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d,
                                                      scale, causal, ws, nb)
                elif kind == "noalloc":
                    st = fa.fa_backward_noalloc(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d,
                                                scale, causal)
                else:
                    st = fa.fa_backward(q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, scale,
                                        causal, ws, nb)
                assert st == fa.FA_OK
            g.check(what + " backward")
            for t in (o, dq, dk, dv):
                assert bool(torch.isfinite(t.float()).all()), f"{what}: non-finite output"
            _unchanged((q, k, v, do, kg, vg), copies, what)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("lengths", [(1, 0, 7), (129, 255, 3), (255,)])
def test_variable_length_entry_points_stay_in_bounds(lengths, d):
    dev = device()
    H, Hkv = 4, 2
    scale = 1.0 / d ** 0.5
    cu = W.cu_seqlens(lengths)
    T, B, L = int(cu[-1]), len(lengths), max(lengths)
    g0 = torch.Generator().manual_seed(7 + T + d)
    q, do = (W.randn_bf16((H, T, d), g0).to(dev) for _ in range(2))
    k, v = (W.randn_bf16((Hkv, T, d), g0).to(dev) for _ in range(2))
    copies = [t.clone() for t in (q, k, v, do)]
    for causal in (0, 1):
        for p in (0.0, 0.3):
            what = f"varlen {lengths} d={d} causal={causal} p={p}"
            g = Guarded(dev)
            cud = g.tensor((B + 1,), torch.int32, "cu_seqlens")
            cud.copy_(torch.from_numpy(cu))
            o = g.tensor((H, T, d), torch.bfloat16, "O")
            lse = g.tensor((H, T), torch.float32, "lse")
            dq = g.tensor((H, T, d), torch.bfloat16, "dQ")
            dk = g.tensor((Hkv, T, d), torch.bfloat16, "dK")
            dv = g.tensor((Hkv, T, d), torch.bfloat16, "dV")
            assert fa.fa_forward_varlen(q, k, v, o, lse, cud, B, L, T, H, Hkv, d, scale, causal,
                                        p, 5, 0) == fa.FA_OK
            g.check(what + " forward")
            nb = fa.fa_backward_workspace_size(1, H, T, d)
            ws = g.workspace(nb)
            assert fa.fa_backward_varlen(q, k, v, o, do, lse, dq, dk, dv, cud, B, L, T, H, Hkv, d,
                                         scale, causal, p, 5, 0, ws, nb) == fa.FA_OK
            g.check(what + " backward")
            assert torch.equal(cud.cpu(), torch.from_numpy(cu)), f"{what}: cu_seqlens modified"
            _unchanged((q, k, v, do), copies, what)
