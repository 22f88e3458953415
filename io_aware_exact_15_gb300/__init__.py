"""Exact IO-aware attention for one NVIDIA GB300 (sm_103a).

Python binding of ``libfa_gb300.so``: the functions below carry the C ABI's
names (include/fa.h) and only marshal arguments.  Every step of the
attention path runs in the library's CUDA kernels; PyTorch supplies device
memory and streams.  There is no fallback: if the library cannot be built or
loaded, the first call raises.

Raw calls (``fa_forward``, ``fa_backward`` ...) take tensors or integer
device pointers, the sizes, and a stream (``None`` = PyTorch's current
stream); they return the ``fa_status`` code.  ``attention_forward`` and
``attention_backward`` allocate outputs and raise ``FaError`` on failure.
"""
from __future__ import annotations

import ctypes
import os
import threading

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_WORKSPACE = 4
FA_ERR_CUDA = 5
FA_ERR_TIMEOUT = 6

EXPORTS = (
    "fa_status_string", "fa_forward", "fa_backward_workspace_size", "fa_backward",
    "fa_backward_preprocess", "fa_backward_main", "fa_backward_dq_convert", "fa_backward_noalloc",
    "fa_blocksparse_workspace_size", "fa_blocksparse_build_lists", "fa_blocksparse_forward",
    "fa_blocksparse_backward", "fa_get_device_status", "fa_set_wait_limit_ns",
    "fa_debug_wait_timeout", "fa_debug_schedule", "fa_debug_mma_probe", "fa_forward_gqa",
    "fa_backward_gqa", "fa_debug_forward_config", "fa_forward_varlen", "fa_backward_varlen",
    "fa_forward_dropout", "fa_backward_dropout", "fa_backward_deterministic",
)

_HERE = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def library_path() -> str:
    from . import build as _build
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libfa_gb300.so (building it with nvcc when absent or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import build as _build
        if build_if_missing and not _build.is_fresh():
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError("libfa_gb300.so is missing: run "
                               "`python -m io_aware_exact_15_gb300.build`")
        lib = ctypes.CDLL(_build.LIB)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        U, UI = ctypes.c_ulonglong, ctypes.c_uint
        sig = {
            "fa_status_string": ([I], ctypes.c_char_p),
            "fa_forward": ([P, P, P, P, P, I, I, I, I, F, I, P], I),
            "fa_backward_workspace_size": ([I, I, I, I], Z),
            "fa_backward": ([P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, P, Z, P], I),
            "fa_backward_preprocess": ([P, P, I, I, I, I, P, Z, P], I),
            "fa_backward_main": ([P, P, P, P, P, P, P, I, I, I, I, F, I, P, Z, P], I),
            "fa_backward_dq_convert": ([P, I, I, I, I, F, P, Z, P], I),
            "fa_backward_noalloc": ([P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, P], I),
            "fa_blocksparse_workspace_size": ([I, I, I, I, I], Z),
            "fa_blocksparse_build_lists": ([P, I, I, P, Z, P], I),
            "fa_blocksparse_forward": ([P, P, P, P, P, I, I, I, I, F, I, P, I, P, Z, P], I),
            "fa_blocksparse_backward": ([P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, P, I, P, Z,
                                         P], I),
            "fa_get_device_status": ([P], I),
            "fa_set_wait_limit_ns": ([U], I),
            "fa_debug_wait_timeout": ([U, P], I),
            "fa_debug_schedule": ([I, I, P, I, P, Z, P, P, P, P, P], I),
            "fa_debug_mma_probe": ([P, P, P, I, I, P], I),
            "fa_forward_gqa": ([P, P, P, P, P, I, I, I, I, I, F, I, P], I),
            "fa_debug_forward_config": ([P, P, P, P, P, I, I, I, I, F, I, I, I, I, P], I),
            "fa_backward_gqa": ([P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, I, P, Z, P], I),
            "fa_forward_varlen": ([P, P, P, P, P, P, I, I, I, I, I, I, F, I, F, U, UI, P], I),
            "fa_backward_varlen": ([P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, I, F, U,
                                    UI, P, Z, P], I),
            "fa_forward_dropout": ([P, P, P, P, P, I, I, I, I, F, I, F, U, UI, P], I),
            "fa_backward_deterministic": ([P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, P, Z, P],
                                          I),
            "fa_backward_dropout": ([P, P, P, P, P, P, P, P, P, I, I, I, I, F, I, F, U, UI, P, Z,
                                     P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


# ------------------------------------------------------------------ marshalling
def _p(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


# ------------------------------------------------------------------ raw C-ABI calls
def fa_status_string(status: int) -> str:
    return status_string(status)


def fa_forward(q, k, v, o, lse, B, H, N, d, scale, causal, stream=None) -> int:
    return load().fa_forward(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, N, d, float(scale),
                             int(bool(causal)), _s(stream))


def fa_forward_gqa(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, stream=None) -> int:
    return load().fa_forward_gqa(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, Hkv, N, d,
                                 float(scale), int(bool(causal)), _s(stream))


def fa_backward_gqa(q, k, v, o, dO, lse, dq, dk, dv, B, H, Hkv, N, d, scale, causal, workspace,
                    workspace_bytes, stream=None) -> int:
    return load().fa_backward_gqa(_p(q), _p(k), _p(v), _p(o), _p(dO), _p(lse), _p(dq), _p(dk),
                                  _p(dv), B, H, Hkv, N, d, float(scale), int(bool(causal)),
                                  _p(workspace), int(workspace_bytes), _s(stream))


def fa_forward_varlen(q, k, v, o, lse, cu_seqlens, B, max_seqlen, total, H, Hkv, d, scale,
                      causal, p_drop, seed, offset, stream=None) -> int:
    return load().fa_forward_varlen(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(cu_seqlens), B,
                                    max_seqlen, total, H, Hkv, d, float(scale),
                                    int(bool(causal)), float(p_drop), int(seed), int(offset),
                                    _s(stream))


def fa_backward_varlen(q, k, v, o, dO, lse, dq, dk, dv, cu_seqlens, B, max_seqlen, total, H, Hkv,
                       d, scale, causal, p_drop, seed, offset, workspace, workspace_bytes,
                       stream=None) -> int:
    return load().fa_backward_varlen(_p(q), _p(k), _p(v), _p(o), _p(dO), _p(lse), _p(dq), _p(dk),
                                     _p(dv), _p(cu_seqlens), B, max_seqlen, total, H, Hkv, d,
                                     float(scale), int(bool(causal)), float(p_drop), int(seed),
                                     int(offset), _p(workspace), int(workspace_bytes), _s(stream))


def fa_forward_dropout(q, k, v, o, lse, B, H, N, d, scale, causal, p_drop, seed, offset,
                       stream=None) -> int:
    return load().fa_forward_dropout(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, N, d,
                                     float(scale), int(bool(causal)), float(p_drop), int(seed),
                                     int(offset), _s(stream))


def fa_backward_dropout(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, p_drop, seed,
                        offset, workspace, workspace_bytes, stream=None) -> int:
    return load().fa_backward_dropout(_p(q), _p(k), _p(v), _p(o), _p(dO), _p(lse), _p(dq),
                                      _p(dk), _p(dv), B, H, N, d, float(scale), int(bool(causal)),
                                      float(p_drop), int(seed), int(offset), _p(workspace),
                                      int(workspace_bytes), _s(stream))


def fa_backward_deterministic(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal,
                              workspace, workspace_bytes, stream=None) -> int:
    return load().fa_backward_deterministic(_p(q), _p(k), _p(v), _p(o), _p(dO), _p(lse), _p(dq),
                                            _p(dk), _p(dv), B, H, N, d, float(scale),
                                            int(bool(causal)), _p(workspace),
                                            int(workspace_bytes), _s(stream))


def fa_backward_workspace_size(B, H, N, d) -> int:
    return load().fa_backward_workspace_size(B, H, N, d)


def fa_backward(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, workspace,
                workspace_bytes, stream=None) -> int:
    return load().fa_backward(_p(q), _p(k), _p(v), _p(o), _p(dO), _p(lse), _p(dq), _p(dk), _p(dv),
                              B, H, N, d, float(scale), int(bool(causal)), _p(workspace),
                              int(workspace_bytes), _s(stream))


def fa_backward_preprocess(o, dO, B, H, N, d, workspace, workspace_bytes, stream=None) -> int:
    return load().fa_backward_preprocess(_p(o), _p(dO), B, H, N, d, _p(workspace),
                                         int(workspace_bytes), _s(stream))


def fa_backward_main(q, k, v, dO, lse, dk, dv, B, H, N, d, scale, causal, workspace,
                     workspace_bytes, stream=None) -> int:
    return load().fa_backward_main(_p(q), _p(k), _p(v), _p(dO), _p(lse), _p(dk), _p(dv), B, H, N,
                                   d, float(scale), int(bool(causal)), _p(workspace),
                                   int(workspace_bytes), _s(stream))


def fa_backward_dq_convert(dq, B, H, N, d, scale, workspace, workspace_bytes, stream=None) -> int:
    return load().fa_backward_dq_convert(_p(dq), B, H, N, d, float(scale), _p(workspace),
                                         int(workspace_bytes), _s(stream))


def fa_backward_noalloc(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal,
                        stream=None) -> int:
    """fa_backward with the library's fixed 32 MiB per-device scratch array
    instead of a caller workspace (for callers that cannot allocate)."""
    return load().fa_backward_noalloc(_p(q), _p(k), _p(v), _p(o), _p(dO), _p(lse), _p(dq), _p(dk),
                                      _p(dv), B, H, N, d, float(scale), int(bool(causal)),
                                      _s(stream))


def fa_blocksparse_workspace_size(B, H, N, d, mask_heads) -> int:
    return load().fa_blocksparse_workspace_size(B, H, N, d, mask_heads)


def fa_blocksparse_build_lists(block_mask, mask_heads, N, workspace, workspace_bytes,
                               stream=None) -> int:
    return load().fa_blocksparse_build_lists(_p(block_mask), mask_heads, N, _p(workspace),
                                             int(workspace_bytes), _s(stream))


def fa_blocksparse_forward(q, k, v, o, lse, B, H, N, d, scale, causal, block_mask, mask_heads,
                           workspace, workspace_bytes, stream=None) -> int:
    return load().fa_blocksparse_forward(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, N, d,
                                         float(scale), int(bool(causal)), _p(block_mask),
                                         mask_heads, _p(workspace), int(workspace_bytes),
                                         _s(stream))


def fa_blocksparse_backward(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, block_mask,
                            mask_heads, workspace, workspace_bytes, stream=None) -> int:
    return load().fa_blocksparse_backward(_p(q), _p(k), _p(v), _p(o), _p(dO), _p(lse), _p(dq),
                                          _p(dk), _p(dv), B, H, N, d, float(scale),
                                          int(bool(causal)), _p(block_mask), mask_heads,
                                          _p(workspace), int(workspace_bytes), _s(stream))


def fa_get_device_status(stream=None) -> int:
    return load().fa_get_device_status(_s(stream))


def fa_set_wait_limit_ns(ns: int) -> int:
    return load().fa_set_wait_limit_ns(int(ns))


def fa_debug_wait_timeout(limit_ns: int, stream=None) -> int:
    return load().fa_debug_wait_timeout(int(limit_ns), _s(stream))


def fa_debug_schedule(N, causal, block_mask, mask_heads, workspace, workspace_bytes, fwd_counts,
                      bwd_counts, fwd_lists, bwd_lists, stream=None) -> int:
    return load().fa_debug_schedule(N, int(bool(causal)), _p(block_mask), mask_heads,
                                    _p(workspace), int(workspace_bytes), _p(fwd_counts),
                                    _p(bwd_counts), _p(fwd_lists), _p(bwd_lists), _s(stream))


def fa_debug_forward_config(q, k, v, o, lse, B, H, N, d, scale, causal, rows_per_cta,
                            key_tile, kv_stages, stream=None) -> int:
    return load().fa_debug_forward_config(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, N, d,
                                          float(scale), int(bool(causal)), int(rows_per_cta),
                                          int(key_tile), int(kv_stages), _s(stream))


def fa_debug_mma_probe(a, b, c, mode, n, stream=None) -> int:
    return load().fa_debug_mma_probe(_p(a), _p(b), _p(c), int(mode), int(n), _s(stream))


# ------------------------------------------------------------------ allocating wrappers
def _check(status, what):
    if status != FA_OK:
        raise FaError(status, what)


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    return tuple(int(x) for x in q.shape)


def _varlen_shape(q, k, cu_seqlens, max_seqlen):
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("variable-length batches take [H, total, d] tensors")
    H, T, d = (int(x) for x in q.shape)
    B = int(cu_seqlens.numel()) - 1
    if B < 1:
        raise ValueError("cu_seqlens needs B + 1 >= 2 entries")
    if max_seqlen is None:  # one host read of the offsets
        cu = cu_seqlens.cpu()
        max_seqlen = int((cu[1:] - cu[:-1]).max()) if T > 0 else 0
    return B, H, int(k.shape[0]), T, d, int(max_seqlen)


def attention_forward(q, k, v, scale=None, causal=False, block_mask=None, workspace=None,
                      stream=None, cu_seqlens=None, max_seqlen=None, dropout_p=0.0, seed=0,
                      offset=0):
    """(o, lse) for bf16 CUDA tensors q [B, H, N, d] and k, v [B, Hkv, N, d]
    (Hkv = H, or a divisor of H for grouped heads).  With cu_seqlens (int32
    CUDA tensor [B+1]) the batch is packed: q [H, total, d], k, v
    [Hkv, total, d], lse [H, total].  dropout_p > 0: dropout on P with the
    Philox keep rule of (seed, offset); the backward must get the same."""
    import torch
    if cu_seqlens is not None:
        if block_mask is not None:
            raise ValueError("block masks apply to equal-length batches only")
        B, H, Hkv, T, d, ms = _varlen_shape(q, k, cu_seqlens, max_seqlen)
        scale = (1.0 / d ** 0.5) if scale is None else scale
        o = torch.empty_like(q)
        lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
        _check(fa_forward_varlen(q, k, v, o, lse, cu_seqlens, B, ms, T, H, Hkv, d, scale, causal,
                                 dropout_p, seed, offset, stream), "fa_forward_varlen")
        return o, lse
    B, H, N, d = _shape(q)
    Hkv = int(k.shape[1])
    scale = (1.0 / d ** 0.5) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if dropout_p:
        if block_mask is not None or Hkv != H:
            raise ValueError("dropout applies to dense Hkv = H or variable-length batches")
        _check(fa_forward_dropout(q, k, v, o, lse, B, H, N, d, scale, causal, dropout_p, seed,
                                  offset, stream), "fa_forward_dropout")
    elif block_mask is None:
        if Hkv == H:
            _check(fa_forward(q, k, v, o, lse, B, H, N, d, scale, causal, stream), "fa_forward")
        else:
            _check(fa_forward_gqa(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, stream),
                   "fa_forward_gqa")
    else:
        if Hkv != H:
            raise ValueError("block masks apply to Hkv = H only")
        mh = int(block_mask.shape[0])
        nbytes = fa_blocksparse_workspace_size(B, H, N, d, mh)
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        _check(fa_blocksparse_forward(q, k, v, o, lse, B, H, N, d, scale, causal, block_mask, mh,
                                      workspace, workspace.numel(), stream),
               "fa_blocksparse_forward")
    return o, lse


def attention_backward(q, k, v, o, dO, lse, scale=None, causal=False, block_mask=None,
                       workspace=None, stream=None, cu_seqlens=None, max_seqlen=None,
                       dropout_p=0.0, seed=0, offset=0):
    """(dq, dk, dv) of sum(O * dO); shapes and options as attention_forward."""
    import torch
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if cu_seqlens is not None:
        if block_mask is not None:
            raise ValueError("block masks apply to equal-length batches only")
        B, H, Hkv, T, d, ms = _varlen_shape(q, k, cu_seqlens, max_seqlen)
        scale = (1.0 / d ** 0.5) if scale is None else scale
        nbytes = fa_backward_workspace_size(1, H, max(T, 1), d)
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        _check(fa_backward_varlen(q, k, v, o, dO, lse, dq, dk, dv, cu_seqlens, B, ms, T, H, Hkv, d,
                                  scale, causal, dropout_p, seed, offset, workspace,
                                  workspace.numel(), stream), "fa_backward_varlen")
        return dq, dk, dv
    B, H, N, d = _shape(q)
    Hkv = int(k.shape[1])
    scale = (1.0 / d ** 0.5) if scale is None else scale
    if dropout_p:
        if block_mask is not None or Hkv != H:
            raise ValueError("dropout applies to dense Hkv = H or variable-length batches")
        nbytes = fa_backward_workspace_size(B, H, N, d)
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        _check(fa_backward_dropout(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal,
                                   dropout_p, seed, offset, workspace, workspace.numel(), stream),
               "fa_backward_dropout")
    elif block_mask is None:
        nbytes = fa_backward_workspace_size(B, H, N, d)
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        if Hkv == H:
            _check(fa_backward(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal,
                               workspace, workspace.numel(), stream), "fa_backward")
        else:
            _check(fa_backward_gqa(q, k, v, o, dO, lse, dq, dk, dv, B, H, Hkv, N, d, scale, causal,
                                   workspace, workspace.numel(), stream), "fa_backward_gqa")
    else:
        if Hkv != H:
            raise ValueError("block masks apply to Hkv = H only")
        mh = int(block_mask.shape[0])
        nbytes = fa_blocksparse_workspace_size(B, H, N, d, mh)
        if workspace is None:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
        _check(fa_blocksparse_backward(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal,
                                       block_mask, mh, workspace, workspace.numel(), stream),
               "fa_blocksparse_backward")
    return dq, dk, dv
