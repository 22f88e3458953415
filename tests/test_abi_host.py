"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every entry point include/fa.h declares, sizes its
workspaces as documented, and rejects bad arguments before launching
anything (every case below returns before the first CUDA call)."""
import ctypes
import os
import re

import pytest

import io_aware_exact_15_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = fa.load()
    names = _declared()
    assert "fa_forward" in names and "fa_backward" in names and "fa_blocksparse_forward" in names
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(fa.EXPORTS) == names


def test_status_strings():
    for s in range(7):
        assert fa.fa_status_string(s)
    assert fa.fa_status_string(99) == "unknown status"


def test_workspace_sizes():
    B, H, N, d = 2, 3, 300, 64
    rows = B * H * N
    a256 = lambda x: (x + 255) // 256 * 256
    # D, the fp32 dQ accumulator, one counter word (the block-sparse backward's
    # next unit)
    assert fa.fa_backward_workspace_size(B, H, N, d) == a256(4 * rows) + a256(4 * rows * d) + 256
    nT = (N + 127) // 128
    lists = a256(4 * 1 * (2 * (nT + 1) + 2 * nT * nT + nT + 1))
    assert fa.fa_blocksparse_workspace_size(B, H, N, d, 1) == lists + \
        fa.fa_backward_workspace_size(B, H, N, d)
    assert fa.fa_backward_workspace_size(0, 1, 1, 64) == 0
    # Theorem 1: extra memory linear in N (no N^2 term outside the tile lists)
    w1 = fa.fa_backward_workspace_size(1, 1, 4096, 128)
    w2 = fa.fa_backward_workspace_size(1, 1, 8192, 128)
    assert abs(w2 - 2 * w1) <= 512
    # d = 128 beyond 64 key tiles: min(tiles / 2, 96) split slots of two
    # 128 x d fp32 partial sums and two int counters each
    for (B, H, N), ns in (((2, 8, 2048), 96), ((1, 5, 2048), 40), ((1, 4, 2048), 0)):
        rows = B * H * N
        assert fa.fa_backward_workspace_size(B, H, N, 128) == \
            a256(4 * rows) + a256(4 * rows * 128) + a256(ns * 2 * 128 * 128 * 4) + \
            a256(8 * ns + 4)
    rows = 2 * 8 * 2048
    assert fa.fa_backward_workspace_size(2, 8, 2048, 64) == \
        a256(4 * rows) + a256(4 * rows * 64) + 256


def test_noalloc_scratch_row_limits():
    """The scratch of fa_backward_noalloc (32 MiB) holds the workspace of
    about 129k rows B*H*N at d = 64 and about 40k at d = 128 (whose
    workspace adds the split last round's partial sums): the largest N, in
    steps of one 128-row tile, of a single head whose workspace fits."""
    def max_rows(d):
        n = 128
        while fa.fa_backward_workspace_size(1, 1, n + 128, d) <= 32 << 20:
            n += 128
        return n
    assert 125_000 <= max_rows(64) <= 131_072
    assert 39_000 <= max_rows(128) <= 41_000


ALIGNED = 1 << 20          # fake, never dereferenced: every case fails validation first
MIS = ALIGNED + 8


@pytest.mark.parametrize("B,H,N,d,scale,expect", [
    (0, 1, 128, 64, 0.125, fa.FA_ERR_INVALID_ARG),
    (1, 0, 128, 64, 0.125, fa.FA_ERR_INVALID_ARG),
    (1, 1, 0, 64, 0.125, fa.FA_ERR_INVALID_ARG),
    (1, 1, 128, 64, 0.0, fa.FA_ERR_INVALID_ARG),
    (1, 1, 128, 64, -1.0, fa.FA_ERR_INVALID_ARG),
    (1, 1, 128, 64, float("inf"), fa.FA_ERR_INVALID_ARG),
    (1, 1, 128, 64, float("nan"), fa.FA_ERR_INVALID_ARG),
    (1, 1, 128, 96, 0.125, fa.FA_ERR_UNSUPPORTED),
    (1, 1, 128, 256, 0.125, fa.FA_ERR_UNSUPPORTED),
    (1024, 1024, 4096, 128, 0.125, fa.FA_ERR_UNSUPPORTED),
])
def test_forward_rejects_bad_shapes(B, H, N, d, scale, expect):
    assert fa.fa_forward(ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, B, H, N, d, scale, 0, 0) \
        == expect


def test_forward_rejects_null_and_misaligned():
    A = ALIGNED
    assert fa.fa_forward(None, A, A, A, A, 1, 1, 128, 64, 0.1, 0, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_forward(A, A, A, A, None, 1, 1, 128, 64, 0.1, 0, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_forward(MIS, A, A, A, A, 1, 1, 128, 64, 0.1, 0, 0) == fa.FA_ERR_MISALIGNED
    assert fa.fa_forward(A, A, MIS, A, A, 1, 1, 128, 64, 0.1, 0, 0) == fa.FA_ERR_MISALIGNED
    assert fa.fa_forward(A, A, A, MIS, A, 1, 1, 128, 64, 0.1, 0, 0) == fa.FA_ERR_MISALIGNED
    assert fa.fa_forward(A, A, A, A, A + 2, 1, 1, 128, 64, 0.1, 0, 0) == fa.FA_ERR_MISALIGNED


def test_backward_rejects_bad_workspace():
    A = ALIGNED
    need = fa.fa_backward_workspace_size(1, 1, 128, 64)
    args = (A, A, A, A, A, A, A, A, A, 1, 1, 128, 64, 0.1, 0)
    assert fa.fa_backward(*args, A, need - 1, 0) == fa.FA_ERR_WORKSPACE
    assert fa.fa_backward(*args, None, need, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_backward(*args, A + 16, need, 0) == fa.FA_ERR_MISALIGNED
    assert fa.fa_backward(A, A, A, A, A, A, MIS, A, A, 1, 1, 128, 64, 0.1, 0, A, need, 0) \
        == fa.FA_ERR_MISALIGNED


def test_blocksparse_rejects_bad_mask_args():
    A = ALIGNED
    ws = fa.fa_blocksparse_workspace_size(1, 4, 256, 64, 1)
    base = (A, A, A, A, A, 1, 4, 256, 64, 0.1, 0)
    assert fa.fa_blocksparse_forward(*base, None, 1, A, ws, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_blocksparse_forward(*base, A, 2, A, ws, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_blocksparse_forward(*base, A, 1, A, 0, 0) == fa.FA_ERR_WORKSPACE
    assert fa.fa_blocksparse_build_lists(A, 1, 256, A, 0, 0) == fa.FA_ERR_WORKSPACE
    assert fa.fa_blocksparse_build_lists(None, 1, 256, A, 1 << 20, 0) == fa.FA_ERR_INVALID_ARG


def test_debug_entry_points_validate():
    assert fa.fa_debug_wait_timeout(0, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_debug_mma_probe(ALIGNED, ALIGNED, ALIGNED, 4, 64, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_debug_mma_probe(ALIGNED, ALIGNED, ALIGNED, 1, 96, 0) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_set_wait_limit_ns(0) == fa.FA_OK


def test_product_package_does_not_reference_oracle():
    pkg = os.path.join(ROOT, "io_aware_exact_15_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text and "fa_oracle" not in text, f


def test_gqa_rejects_bad_groups():
    A = ALIGNED
    need = fa.fa_backward_workspace_size(1, 6, 128, 64)
    for Hkv in (0, 4, 7, -1):
        assert fa.fa_forward_gqa(A, A, A, A, A, 1, 6, Hkv, 128, 64, 0.1, 0, 0) == \
            fa.FA_ERR_INVALID_ARG
        assert fa.fa_backward_gqa(A, A, A, A, A, A, A, A, A, 1, 6, Hkv, 128, 64, 0.1, 0, A, need,
                                  0) == fa.FA_ERR_INVALID_ARG


def test_varlen_rejects_bad_args():
    A = ALIGNED
    need = fa.fa_backward_workspace_size(1, 4, 1000, 64)
    # (cu, B, max_seqlen, total, H, Hkv, d, scale) -> status
    cases = [
        ((None, 2, 512, 1000, 4, 4, 64, 0.1), fa.FA_ERR_INVALID_ARG),
        ((A + 2, 2, 512, 1000, 4, 4, 64, 0.1), fa.FA_ERR_MISALIGNED),
        ((A, 0, 512, 1000, 4, 4, 64, 0.1), fa.FA_ERR_INVALID_ARG),
        ((A, 2, 0, 1000, 4, 4, 64, 0.1), fa.FA_ERR_INVALID_ARG),
        ((A, 2, 1001, 1000, 4, 4, 64, 0.1), fa.FA_ERR_INVALID_ARG),
        ((A, 2, 512, -1, 4, 4, 64, 0.1), fa.FA_ERR_INVALID_ARG),
        ((A, 2, 512, 1000, 4, 3, 64, 0.1), fa.FA_ERR_INVALID_ARG),
        ((A, 2, 512, 1000, 4, 4, 96, 0.1), fa.FA_ERR_UNSUPPORTED),
        ((A, 2, 512, 1000, 4, 4, 64, 0.0), fa.FA_ERR_INVALID_ARG),
        ((A, 2, 512, 1 << 24, 1024, 1024, 128, 0.1), fa.FA_ERR_UNSUPPORTED),
    ]
    for (cu, B, ms, T, H, Hkv, d, sc), want in cases:
        assert fa.fa_forward_varlen(A, A, A, A, A, cu, B, ms, T, H, Hkv, d, sc, 0, 0.0, 0, 0,
                                    0) == want, \
            (cu, B, ms, T)
        assert fa.fa_backward_varlen(A, A, A, A, A, A, A, A, A, cu, B, ms, T, H, Hkv, d, sc, 0,
                                     0.0, 0, 0, A,
                                     need, 0) == want
    base = (A, 2, 512, 1000, 4, 4, 64, 0.1, 0, 0.0, 0, 0)
    assert fa.fa_forward_varlen(MIS, A, A, A, A, *base, 0) == fa.FA_ERR_MISALIGNED
    assert fa.fa_backward_varlen(A, A, A, A, A, A, A, A, A, *base, A, need - 1, 0) == \
        fa.FA_ERR_WORKSPACE
    assert fa.fa_backward_varlen(A, A, A, A, A, A, A, A, A, *base, A + 16, need, 0) == \
        fa.FA_ERR_MISALIGNED


def test_dropout_rejects_bad_probability():
    A = ALIGNED
    need = fa.fa_backward_workspace_size(1, 2, 256, 64)
    for p in (-0.1, 1.0, 0.999, float("nan"), float("inf")):
        assert fa.fa_forward_dropout(A, A, A, A, A, 1, 2, 256, 64, 0.1, 0, p, 1, 0, 0) == \
            fa.FA_ERR_INVALID_ARG, p
        assert fa.fa_backward_dropout(A, A, A, A, A, A, A, A, A, 1, 2, 256, 64, 0.1, 0, p, 1, 0, A,
                                      need, 0) == fa.FA_ERR_INVALID_ARG, p
        assert fa.fa_forward_varlen(A, A, A, A, A, A, 2, 128, 256, 2, 2, 64, 0.1, 0, p, 1, 0,
                                    0) == fa.FA_ERR_INVALID_ARG, p
    # shape checks come first, as for fa_forward
    assert fa.fa_forward_dropout(A, A, A, A, A, 1, 2, 256, 96, 0.1, 0, 0.1, 1, 0, 0) == \
        fa.FA_ERR_UNSUPPORTED
    assert fa.fa_backward_dropout(A, A, A, A, A, A, A, A, A, 1, 2, 256, 64, 0.1, 0, 0.1, 1, 0, A,
                                  need - 1, 0) == fa.FA_ERR_WORKSPACE


def test_deterministic_backward_validates():
    A = ALIGNED
    need = (1 * 2 * 300 * 4 + 255) // 256 * 256
    args = (A, A, A, A, A, A, A, A, A, 1, 2, 300, 64, 0.1, 0)
    assert fa.fa_backward_deterministic(*args, A, need - 1, 0) == fa.FA_ERR_WORKSPACE
    assert fa.fa_backward_deterministic(*args, None, need, 0) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_backward_deterministic(A, A, A, A, A, A, MIS, A, A, 1, 2, 300, 64, 0.1, 0, A,
                                        need, 0) == fa.FA_ERR_MISALIGNED
    assert fa.fa_backward_deterministic(A, A, A, A, A, A, A, A, A, 1, 2, 300, 96, 0.1, 0, A,
                                        need, 0) == fa.FA_ERR_UNSUPPORTED
