"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds random number generation and workload descriptions only:
no attention arithmetic.  Both the CUDA path and the CPU oracle receive the
same host bytes produced here.

Recipe (one per workload):
  * Q, K, V and the upstream gradient dO are drawn in that order from one
    ``torch.Generator`` on the CPU seeded with ``1000 + k`` for workload k:
    i.i.d. N(0, 1) in fp32, then rounded to bf16 (round to nearest even).
  * Masks and the "peaked key" choice use a second generator seeded with
    ``2000 + k``.
  * Peaked keys: in every (batch, head), round(frac * N) key rows chosen
    without replacement are multiplied by 8 (exact in bf16).
  * Block mask over 128 x 128 tiles: the diagonal band |i - j| <= 1, block
    column 0, and exactly round(density * R) of the R remaining tiles chosen
    by a seeded permutation; one mask shared by every head.
  * Variable-length batch (padding mask as lengths): B lengths drawn i.i.d.
    uniform on the integers [N/4, N] from the mask generator; the sequences
    are packed back to back, tensors [H, total, d] (K, V: [Hkv, total, d]),
    drawn like the equal-length ones.
  * Grouped heads: K and V have Hkv heads instead of H.
  * Dropout: probability p on P, generator seed DROPOUT_SEED, offset 0.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

TILE = 128
DROPOUT_SEED = 0x5EED0F00D


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool = False
    backward: bool = True
    peaked_frac: float = 0.0
    sparse_density: float | None = None  # block-sparse when not None
    Hkv: int | None = None  # grouped key/value heads when set (H % Hkv == 0)
    varlen: bool = False    # packed batch of lengths in [N/4, N]
    dropout: float = 0.0    # dropout probability on P
    seed_index: int = 0
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / float(self.d) ** 0.5

    @property
    def kv_heads(self) -> int:
        return self.H if self.Hkv is None else self.Hkv

    @property
    def seed(self) -> int:
        return 1000 + self.seed_index

    @property
    def mask_seed(self) -> int:
        return 2000 + self.seed_index


def _sweep():
    out = {}
    for d in (64, 128):
        for N in (2048, 4096, 8192, 16384):
            B = 16384 // N
            out[f"longseq_causal_n{N}_d{d}"] = Workload(
                f"longseq_causal_n{N}_d{d}", B, 16, N, d, causal=True, peaked_frac=0.01,
                seed_index=4, note="B*N = 16384 tokens, H=16, 1% of keys x8, causal")
            out[f"longseq_dense_n{N}_d{d}"] = Workload(
                f"longseq_dense_n{N}_d{d}", B, 16, N, d, causal=False, peaked_frac=0.01,
                seed_index=4, note="same shapes and inputs as the causal sweep, no mask")
    return out


WORKLOADS = {
    "single_head_fwd": Workload("single_head_fwd", 1, 1, 128, 64, backward=False, seed_index=1,
                                note="B=1 H=1 N=128 d=64 forward only"),
    "bert_large": Workload("bert_large", 8, 16, 512, 64, seed_index=2,
                           note="BERT-large-shaped self-attention, B=8 H=16 N=512 d=64"),
    "gpt2_causal": Workload("gpt2_causal", 8, 12, 1024, 64, causal=True, seed_index=3,
                            note="GPT-2-shaped causal self-attention, B=8 H=12 N=1024 d=64"),
    **_sweep(),
    "blocksparse_64k": Workload("blocksparse_64k", 1, 8, 65536, 64, sparse_density=0.05,
                                seed_index=5,
                                note="B=1 H=8 N=65536 d=64, band + column 0 + 5% random tiles"),
    "bert_large_varlen": Workload("bert_large_varlen", 8, 16, 512, 64, varlen=True, seed_index=6,
                                  note="BERT-large shapes with a padding mask: 8 packed "
                                       "sequences of 128..512 tokens, H=16 d=64"),
    "bert_large_varlen_dropout": Workload(
        "bert_large_varlen_dropout", 8, 16, 512, 64, varlen=True, dropout=0.1, seed_index=6,
        note="the section 4.4 benchmark setting (dropout + padding mask) at BERT-large shapes: "
             "8 packed sequences of 128..512 tokens, H=16 d=64, p=0.1"),
    "longseq_dense_n4096_d128_dropout": Workload(
        "longseq_dense_n4096_d128_dropout", 4, 16, 4096, 128, peaked_frac=0.01, dropout=0.1,
        seed_index=4, note="longseq_dense_n4096_d128 with dropout p=0.1 on P"),
    "gqa_causal_n4096_d128": Workload("gqa_causal_n4096_d128", 4, 16, 4096, 128, causal=True,
                                      Hkv=4, seed_index=7,
                                      note="grouped heads: 16 query heads over 4 K/V heads, "
                                           "B=4 N=4096 d=128 causal"),
}


def randn_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def make_qkv(B, H, N, d, seed, peaked_frac=0.0, mask_seed=None, with_do=True):
    """Seeded bf16 CPU tensors q, k, v (and dO) of shape [B, H, N, d]."""
    g = torch.Generator().manual_seed(int(seed))
    q = randn_bf16((B, H, N, d), g)
    k = randn_bf16((B, H, N, d), g)
    v = randn_bf16((B, H, N, d), g)
    do = randn_bf16((B, H, N, d), g) if with_do else None
    if peaked_frac > 0.0:
        gm = torch.Generator().manual_seed(int(mask_seed if mask_seed is not None else seed + 1000))
        npk = int(round(peaked_frac * N))
        if npk > 0:
            for b in range(B):
                for h in range(H):
                    idx = torch.randperm(N, generator=gm)[:npk]
                    k[b, h, idx] = k[b, h, idx] * 8
    return q, k, v, do


def band_random_block_mask(N, seed, density=0.05, band=1, tile=TILE, col0=True):
    """uint8 block mask [1, nT, nT]: |i-j| <= band, column 0, and a seeded
    round(density * R) of the R remaining tiles (without replacement)."""
    nT = (N + tile - 1) // tile
    m = np.zeros((nT, nT), dtype=np.uint8)
    ii, jj = np.meshgrid(np.arange(nT), np.arange(nT), indexing="ij")
    m[np.abs(ii - jj) <= band] = 1
    if col0:
        m[:, 0] = 1
    rest = np.flatnonzero(m.reshape(-1) == 0)
    g = torch.Generator().manual_seed(int(seed))
    nsel = int(round(density * len(rest)))
    pick = torch.randperm(len(rest), generator=g)[:nsel].numpy()
    flat = m.reshape(-1)
    flat[rest[pick]] = 1
    return flat.reshape(1, nT, nT)


def random_block_mask(H, nT, seed, density):
    """uint8 mask [H, nT, nT] with i.i.d. Bernoulli(density) tiles (tests)."""
    g = torch.Generator().manual_seed(int(seed))
    return (torch.rand((H, nT, nT), generator=g) < density).to(torch.uint8).numpy()


def sample_rows(N, n, seed):
    """Sorted seeded sample of min(n, N) distinct row indices."""
    g = torch.Generator().manual_seed(int(seed))
    n = min(int(n), int(N))
    return np.sort(torch.randperm(N, generator=g)[:n].numpy().astype(np.int64))


def varlen_lengths(w: Workload) -> np.ndarray:
    """The B sequence lengths of a variable-length workload (int64)."""
    g = torch.Generator().manual_seed(int(w.mask_seed))
    return torch.randint(w.N // 4, w.N + 1, (w.B,), generator=g).numpy().astype(np.int64)


def cu_seqlens(lengths) -> np.ndarray:
    """int32 offsets [B+1] of sequences packed back to back."""
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int32)


def make_varlen_inputs(w: Workload, with_do=None):
    """q, dO [H, total, d], k, v [Hkv, total, d] (bf16 CPU) and cu_seqlens."""
    if with_do is None:
        with_do = w.backward
    cu = cu_seqlens(varlen_lengths(w))
    T = int(cu[-1])
    g = torch.Generator().manual_seed(int(w.seed))
    q = randn_bf16((w.H, T, w.d), g)
    k = randn_bf16((w.kv_heads, T, w.d), g)
    v = randn_bf16((w.kv_heads, T, w.d), g)
    do = randn_bf16((w.H, T, w.d), g) if with_do else None
    return q, k, v, do, cu


def make_inputs(w: Workload, with_do=None):
    """q, k, v, dO (bf16 CPU) and the block mask (numpy uint8 or None)."""
    if with_do is None:
        with_do = w.backward
    if w.varlen:
        raise ValueError("variable-length workloads: use make_varlen_inputs")
    q, k, v, do = make_qkv(w.B, w.H, w.N, w.d, w.seed, w.peaked_frac, w.mask_seed, with_do)
    if w.Hkv is not None and w.Hkv != w.H:
        # grouped heads: K and V keep the first Hkv heads' draws
        k, v = k[:, :w.Hkv].contiguous(), v[:, :w.Hkv].contiguous()
    mask = None
    if w.sparse_density is not None:
        mask = band_random_block_mask(w.N, w.mask_seed, w.sparse_density)
    return q, k, v, do, mask


def fwd_flops(w: Workload, mask=None) -> float:
    """Algorithmic forward FLOPs: 4*B*H*N^2*d, halved when causal; block-
    sparse counts 4*d*128^2 per kept tile per head; a variable-length batch
    sums 4*H*n^2*d over its sequence lengths n."""
    if w.varlen:
        n = varlen_lengths(w).astype(np.float64)
        f = 4.0 * w.H * w.d * float(np.sum(n * n))
        return f / 2 if w.causal else f
    if mask is not None:
        nnz = int(np.count_nonzero(mask))
        per_head = 4.0 * w.d * TILE * TILE * nnz / mask.shape[0]
        return per_head * w.B * w.H
    f = 4.0 * w.B * w.H * w.N * w.N * w.d
    return f / 2 if w.causal else f


def fwd_bwd_flops(w: Workload, mask=None) -> float:
    """Forward + backward: the backward is five matmuls (2.5x forward)."""
    return 3.5 * fwd_flops(w, mask)
