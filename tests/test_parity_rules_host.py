"""Host checks of the sampling rules the GPU parity tests use (no GPU)."""
import numpy as np

import parity

import fa_workloads as W


def test_check_rows_cover_every_tile():
    for N in (2048, 4096, 16384, 1000):
        rows = parity.check_rows(N, 7)
        assert np.all(np.diff(rows) > 0) and rows[0] >= 0 and rows[-1] < N
        tiles = set((rows // 128).tolist())
        assert tiles == set(range((N + 127) // 128))
        assert len(rows) >= min(N, 256)


def test_last_round_heads_follow_the_unit_numbering():
    # B4 H16 N4096: 2048 units; 152 SMs leave units 1976..2047 for the last
    # round.  Dense units are head-major (u // 32 = 61..63); causal ones are
    # key-tile-major (kt 30 for heads 56..63, kt 31 for all 64 heads).
    assert parity.last_round_heads(4, 16, 4096, False, 152) == [(3, 13), (3, 14), (3, 15)]
    assert len(parity.last_round_heads(4, 16, 4096, True, 152)) == 64
    assert parity.last_round_heads(1, 16, 16384, False, 152) == [(0, 15)]
    # fewer units than SMs: one round, every unit in it
    assert parity.last_round_heads(1, 2, 256, False, 152) == [(0, 0), (0, 1)]


def test_backward_heads_budget_and_required_heads():
    for name in ("longseq_dense_n16384_d128", "longseq_dense_n4096_d128",
                 "longseq_causal_n2048_d64", "longseq_dense_n8192_d64"):
        w = W.WORKLOADS[name]
        heads = parity.backward_heads(w, 152)
        per_head = 4.0 * w.N ** 2 * w.d / (2 if w.causal else 1)
        assert len(heads) == len(set(heads))
        assert len(heads) == min(w.B * w.H, max(4, int(parity.ORACLE_BUDGET // per_head)))
        if len(heads) < w.B * w.H:
            last = parity.last_round_heads(w.B, w.H, w.N, w.causal, 152)
            for x in ((0, 0), (w.B - 1, w.H - 1), last[0], last[-1]):
                assert x in heads
    # the smallest shape fits the budget: every head
    w = W.WORKLOADS["longseq_causal_n2048_d64"]
    assert len(parity.backward_heads(w, 152)) == w.B * w.H
