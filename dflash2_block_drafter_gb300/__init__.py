"""Python binding of libdflash2 (the GB300 library for the DFlash2 drafter's block-local tail).

Argument marshalling only: every step of the path runs in the library's CUDA kernels, called
through its C ABI (include/dflash2.h) with ctypes. PyTorch provides device memory and the
current stream. There is no CPU fallback: if the library is missing or no GPU is present the
calls raise.

The functions carry the C names. Tensors are torch tensors on the current CUDA device,
contiguous, dtype torch.bfloat16 or torch.float32 (activations/weights), float32 for base /
bias / scores, int32 for ids. Outputs are allocated here when not passed in.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "Dflash2Error", "library", "library_path", "dflash2_version", "dflash2_poll_error",
    "dflash2_conv_prepare_workspace_bytes", "dflash2_conv_prepare_launches", "dflash2_conv_finish_launches",
    "dflash2_conv_prepare", "dflash2_conv_finish",
    "dflash2_head_topk_workspace_bytes", "dflash2_head_topk", "dflash2_score_edges",
    "dflash2_select_path", "dflash2_selftest_bounded_wait", "dflash2_head_topk_noalloc", "dflash2_head_topk_vocab", "dflash2_score_edges_depths", "dflash2_select_path_depths",
    "dflash2_ragged_offsets", "dflash2_conv_finish_ragged", "dflash2_score_edges_ragged",
    "dflash2_conv_coefficients", "dflash2_proj", "dflash2_proj_conv_in", "dflash2_proj_conv_out",
    "dflash2_proj_workspace_bytes",
    "DTYPE_CODES",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "libdflash2.so")
_LIB = None

BF16, F32 = 0, 1
DTYPE_CODES = {torch.bfloat16: BF16, torch.float32: F32}
_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t

_SIGNATURES = {
    "dflash2_version": (_i, []),
    "dflash2_status_string": (ctypes.c_char_p, [_i]),
    "dflash2_last_error_message": (ctypes.c_char_p, []),
    "dflash2_poll_error": (_i, [_vp]),
    "dflash2_conv_prepare_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "dflash2_conv_prepare_launches": (_i, [_i, _i, _i, _i, _i, _i]),
    "dflash2_conv_finish_launches": (_i, [_i, _i, _i, _i, _i, _i]),
    "dflash2_conv_prepare": (_i, [_vp, _vp, _f, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dflash2_conv_finish": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _f, _vp, _i, _vp]),
    "dflash2_head_topk_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "dflash2_head_topk": (_i, [_vp, _i, _i, _vp, _i, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dflash2_score_edges": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp]),
    "dflash2_select_path": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp]),
    "dflash2_selftest_bounded_wait": (_i, [_i, _vp]),
    "dflash2_head_topk_noalloc": (_i, [_vp, _i, _i, _vp, _i, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "dflash2_score_edges_depths": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp]),
    "dflash2_select_path_depths": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp]),
    "dflash2_head_topk_vocab": (_i, [_vp, _i, _i, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _sz,
                                     _vp]),
    "dflash2_conv_finish_ragged": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _f, _vp, _i, _vp, _i,
                                        _vp]),
    "dflash2_score_edges_ragged": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp,
                                        _vp]),
    "dflash2_conv_coefficients": (_i, [_vp, _vp, _f, _vp, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dflash2_proj_workspace_bytes": (_sz, [_i, _i, _i]),
    "dflash2_proj": (_i, [_vp, _i, _i, _vp, _vp, _vp, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "dflash2_proj_conv_in": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "dflash2_proj_conv_out": (_i, [_vp, _i, _i, _vp, _vp, _vp, _i, _i, _vp, _vp, _i, _i, _vp, _i, _vp, _vp, _sz,
                                   _vp]),
}


class Dflash2Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


def library() -> ctypes.CDLL:
    """Load libdflash2.so (built in-tree by ``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"{library_path} is missing: build it with `python -c 'import __graft_entry__ as g; "
                               f"g.build()'` (needs nvcc); there is no CPU fallback")
        lib = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _check(rc: int):
    if rc != 0:
        lib = library()
        msg = lib.dflash2_last_error_message().decode(errors="replace")
        name = lib.dflash2_status_string(rc).decode()
        raise Dflash2Error(rc, f"{name}: {msg}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return _vp(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t, name, dtype=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return _vp(t.data_ptr())


def _code(t):
    try:
        return DTYPE_CODES[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}: use torch.bfloat16 or torch.float32") from None


def _head_shapes(h, w_head, w_proj, K, cand, unary, z, logits):
    """Shape checks of the head calls, before anything reaches the library: the kernels trust M, H,
    V and R, so an undersized output or a weight of the wrong width would be read or written out
    of bounds. Returns (M, H, V, R)."""
    if h.dim() != 2:
        raise ValueError(f"h must be [M, H], got shape {tuple(h.shape)}")
    M, H = h.shape
    if w_head.dim() != 2 or w_head.shape[1] != H:
        raise ValueError(f"w_head must be [V, {H}], got shape {tuple(w_head.shape)}")
    V = w_head.shape[0]
    R = 0
    if w_proj is not None:
        if w_proj.dim() != 2 or w_proj.shape[1] != H:
            raise ValueError(f"w_proj must be [R, {H}], got shape {tuple(w_proj.shape)}")
        R = w_proj.shape[0]
    for t, n, name in ((cand, M * K, "cand"), (unary, M * K, "unary"), (z, M * R, "z"), (logits, M * V, "logits")):
        if t is not None and t.numel() < n:
            raise ValueError(f"{name} holds {t.numel()} elements, fewer than the {n} the call writes")
    return M, H, V, R


def _workspace(nbytes, device, ws):
    if ws is None:
        ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    return ws


def dflash2_version() -> int:
    return library().dflash2_version()


def dflash2_poll_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word (0 = no error)."""
    return library().dflash2_poll_error(_stream(stream))


def dflash2_conv_prepare_workspace_bytes(B, G, H, group_size, dtype) -> int:
    return library().dflash2_conv_prepare_workspace_bytes(B, G, H, group_size, DTYPE_CODES[dtype])


def dflash2_conv_prepare_launches(B, G, H, group_size, dtype, with_norm) -> int:
    """Kernels one dflash2_conv_prepare call launches for this shape (-1: rejected shape)."""
    return library().dflash2_conv_prepare_launches(B, G, H, group_size, DTYPE_CODES[dtype], int(bool(with_norm)))


def dflash2_conv_finish_launches(B, G, H, group_size, dtype, with_next_norm) -> int:
    """Kernels one dflash2_conv_finish call launches for this shape (-1: rejected shape)."""
    return library().dflash2_conv_finish_launches(B, G, H, group_size, DTYPE_CODES[dtype], int(bool(with_next_norm)))


def dflash2_conv_prepare(x, norm_w, eps, w_kp, base, group_size, out=None, coef1=None, d_full=None, workspace=None,
                         stream=None, taps=2):
    """Pre-sublayer conv: returns (out [B,G,H], coef1 [B,G,2,groups]); see dflash2.h."""
    B, G, H = x.shape
    groups = H // group_size
    dt = x.dtype
    out = torch.empty_like(x) if out is None else out
    coef1 = torch.empty((B, G, 2, groups), dtype=dt, device=x.device) if coef1 is None else coef1
    nbytes = library().dflash2_conv_prepare_workspace_bytes(B, G, H, group_size, _code(x))
    workspace = _workspace(nbytes, x.device, workspace)
    _check(library().dflash2_conv_prepare(
        _dev(x, "x", dt), _dev(norm_w, "norm_w", dt, True), eps, _dev(w_kp, "w_kp", dt), _dev(base, "base", torch.float32),
        B, G, H, group_size, taps, _code(x), _dev(out, "out", dt), _dev(coef1, "coef1", dt),
        _dev(d_full, "d_full", torch.float32, True), _dev(workspace, "workspace"), workspace.numel(), _stream(stream)))
    return out, coef1


def dflash2_conv_finish(y, coef1, base, group_size, residual=None, out=None, next_norm_w=None, eps=1e-6,
                        next_n=None, next_row0=0, stream=None, taps=2):
    """Post-sublayer conv + residual add (+ optional next RMSNorm). Returns (out, next_n)."""
    B, G, H = y.shape
    dt = y.dtype
    out = torch.empty_like(y) if out is None else out
    if next_norm_w is not None and next_n is None:
        next_n = torch.empty((B, G - next_row0, H), dtype=dt, device=y.device)
    _check(library().dflash2_conv_finish(
        _dev(y, "y", dt), _dev(coef1, "coef1", dt), _dev(base, "base", torch.float32), B, G, H, group_size, taps,
        _code(y), _dev(residual, "residual", dt, True), _dev(out, "out", dt), _dev(next_norm_w, "next_norm_w", dt, True),
        eps, _dev(next_n, "next_n", dt, True), next_row0, _stream(stream)))
    return out, next_n


def dflash2_head_topk_workspace_bytes(M, H, V, K, R) -> int:
    return library().dflash2_head_topk_workspace_bytes(M, H, V, K, R)


def dflash2_head_topk(h, w_head, K, bias=None, w_proj=None, cand=None, unary=None, z=None, logits=None,
                      want_logits=False, workspace=None, stream=None):
    """Head GEMM + fused top-K (+ z). h: [M, H]. Returns (cand [M,K] int32, unary [M,K] f32, z [M,R] or None, logits or None)."""
    M, H, V, R = _head_shapes(h, w_head, w_proj, K, cand, unary, z, logits)
    dt = h.dtype
    dev = h.device
    cand = torch.empty((M, K), dtype=torch.int32, device=dev) if cand is None else cand
    unary = torch.empty((M, K), dtype=torch.float32, device=dev) if unary is None else unary
    if w_proj is not None and z is None:
        z = torch.empty((M, R), dtype=torch.float32, device=dev)
    if want_logits and logits is None:
        logits = torch.empty((M, V), dtype=torch.float32, device=dev)
    nbytes = library().dflash2_head_topk_workspace_bytes(M, H, V, K, R)
    workspace = _workspace(nbytes, dev, workspace)
    _check(library().dflash2_head_topk(
        _dev(h, "h", dt), M, H, _dev(w_head, "w_head", dt), V, _dev(bias, "bias", torch.float32, True),
        _dev(w_proj, "w_proj", dt, True), R, K, _code(h), _dev(cand, "cand", torch.int32),
        _dev(unary, "unary", torch.float32), _dev(z, "z", torch.float32, True),
        _dev(logits, "logits", torch.float32, True), _dev(workspace, "workspace"), workspace.numel(), _stream(stream)))
    return cand, unary, z, logits


def dflash2_head_topk_vocab(h, w_listed, vocab_ids, K, bias_listed=None, w_proj=None, cand=None, unary=None, z=None,
                            logits=None, want_logits=False, workspace=None, stream=None):
    """Head GEMM + fused top-K over a draft vocabulary: rows of w_listed are the listed tokens
    vocab_ids (int32). Returns (cand [M,K] token ids, unary, z or None, logits [M,V_listed] or None)."""
    M, H, V, R = _head_shapes(h, w_listed, w_proj, K, cand, unary, z, logits)
    if vocab_ids.numel() < V:
        raise ValueError(f"vocab_ids holds {vocab_ids.numel()} ids, fewer than the {V} listed rows")
    dt = h.dtype
    dev = h.device
    cand = torch.empty((M, K), dtype=torch.int32, device=dev) if cand is None else cand
    unary = torch.empty((M, K), dtype=torch.float32, device=dev) if unary is None else unary
    if w_proj is not None and z is None:
        z = torch.empty((M, R), dtype=torch.float32, device=dev)
    if want_logits and logits is None:
        logits = torch.empty((M, V), dtype=torch.float32, device=dev)
    nbytes = library().dflash2_head_topk_workspace_bytes(M, H, V, K, R)
    workspace = _workspace(nbytes, dev, workspace)
    _check(library().dflash2_head_topk_vocab(
        _dev(h, "h", dt), M, H, _dev(w_listed, "w_listed", dt), V, _dev(vocab_ids, "vocab_ids", torch.int32),
        _dev(bias_listed, "bias_listed", torch.float32, True), _dev(w_proj, "w_proj", dt, True), R, K, _code(h),
        _dev(cand, "cand", torch.int32), _dev(unary, "unary", torch.float32), _dev(z, "z", torch.float32, True),
        _dev(logits, "logits", torch.float32, True), _dev(workspace, "workspace"), workspace.numel(),
        _stream(stream)))
    return cand, unary, z, logits


def dflash2_score_edges(cand, unary, z, anchors, pred_book, succ_book, want_S=True, want_path=True, S=None, path=None,
                        stream=None):
    """Edge scores (+ fused greedy walk). cand/unary: [B,steps,K]; z: [B,steps,R]. Returns (S, path)."""
    B, steps, K = cand.shape
    R = z.shape[-1]
    V = pred_book.shape[0]
    dev = cand.device
    if want_S and S is None:
        S = torch.empty((B, steps, K, K), dtype=torch.float32, device=dev)
    if want_path and path is None:
        path = torch.empty((B, steps), dtype=torch.int32, device=dev)
    _check(library().dflash2_score_edges(
        _dev(cand, "cand", torch.int32), _dev(unary, "unary", torch.float32), _dev(z, "z", torch.float32),
        _dev(anchors, "anchors", torch.int32), _dev(pred_book, "pred_book", pred_book.dtype),
        _dev(succ_book, "succ_book", pred_book.dtype), B, steps, K, R, V, _code(pred_book),
        _dev(S, "S", torch.float32, True), _dev(path, "path", torch.int32, True), _stream(stream)))
    return S, path


def dflash2_select_path(S, cand, path=None, stream=None):
    """Greedy walk over S [B,steps,K,K]; returns path [B,steps] int32."""
    B, steps, K, _ = S.shape
    path = torch.empty((B, steps), dtype=torch.int32, device=S.device) if path is None else path
    _check(library().dflash2_select_path(_dev(S, "S", torch.float32), _dev(cand, "cand", torch.int32), B, steps, K,
                                         _dev(path, "path", torch.int32), _stream(stream)))
    return path


def dflash2_selftest_bounded_wait(limit_us: int, stream=None):
    _check(library().dflash2_selftest_bounded_wait(limit_us, _stream(stream)))


def dflash2_head_topk_noalloc(h, w_head, K, bias=None, w_proj=None, cand=None, unary=None, z=None, logits=None,
                              want_logits=False, stream=None):
    """dflash2_head_topk with its scratch in the library's fixed device array instead of a workspace.

    For callers that cannot allocate device memory while the head runs (a serving loop where an
    allocation would stall the device, or a host that only passes input and output buffers). Outputs not passed in are
    still allocated here by torch for convenience; pass them all to allocate nothing. Calls that
    overlap on the GPU share the array and race; keep them on one stream.
    """
    M, H, V, R = _head_shapes(h, w_head, w_proj, K, cand, unary, z, logits)
    dt = h.dtype
    dev = h.device
    cand = torch.empty((M, K), dtype=torch.int32, device=dev) if cand is None else cand
    unary = torch.empty((M, K), dtype=torch.float32, device=dev) if unary is None else unary
    if w_proj is not None and z is None:
        z = torch.empty((M, R), dtype=torch.float32, device=dev)
    if want_logits and logits is None:
        logits = torch.empty((M, V), dtype=torch.float32, device=dev)
    _check(library().dflash2_head_topk_noalloc(
        _dev(h, "h", dt), M, H, _dev(w_head, "w_head", dt), V, _dev(bias, "bias", torch.float32, True),
        _dev(w_proj, "w_proj", dt, True), R, K, _code(h), _dev(cand, "cand", torch.int32),
        _dev(unary, "unary", torch.float32), _dev(z, "z", torch.float32, True),
        _dev(logits, "logits", torch.float32, True), _stream(stream)))
    return cand, unary, z, logits


def dflash2_score_edges_depths(cand, unary, z, anchors, pred_book, succ_book, depths, want_S=True, S=None, path=None,
                               stream=None):
    """Edge scores + the greedy walk for a mixed-depth batch: block b walks depths[b] (int32) slots,
    later path entries are -1. Returns (S or None, path)."""
    B, steps, K = cand.shape
    R = z.shape[-1]
    V = pred_book.shape[0]
    dev = cand.device
    if want_S and S is None:
        S = torch.empty((B, steps, K, K), dtype=torch.float32, device=dev)
    path = torch.empty((B, steps), dtype=torch.int32, device=dev) if path is None else path
    _check(library().dflash2_score_edges_depths(
        _dev(cand, "cand", torch.int32), _dev(unary, "unary", torch.float32), _dev(z, "z", torch.float32),
        _dev(anchors, "anchors", torch.int32), _dev(pred_book, "pred_book", pred_book.dtype),
        _dev(succ_book, "succ_book", pred_book.dtype), _dev(depths, "depths", torch.int32), B, steps, K, R, V,
        _code(pred_book), _dev(S, "S", torch.float32, True), _dev(path, "path", torch.int32), _stream(stream)))
    return S, path


def dflash2_select_path_depths(S, cand, depths, path=None, stream=None):
    """Greedy walk over S for a mixed-depth batch; returns path [B, steps] with -1 padding."""
    B, steps, K, _ = S.shape
    path = torch.empty((B, steps), dtype=torch.int32, device=S.device) if path is None else path
    _check(library().dflash2_select_path_depths(_dev(S, "S", torch.float32), _dev(cand, "cand", torch.int32),
                                                _dev(depths, "depths", torch.int32), B, steps, K,
                                                _dev(path, "path", torch.int32), _stream(stream)))
    return path


def dflash2_ragged_offsets(depths, G, device="cuda"):
    """Row offsets of a ragged batch from the per-block requested depths (host ints): block b
    drafts d_b = min(G - 1, max(1, depths[b])) tokens (dflash2.ts blockColumns), so its head rows
    are [offsets[b], offsets[b + 1]). Returns (offsets int32 [B + 1] on `device`, m_rows). Host-side
    scheduling metadata: the row count sizes the head call."""
    d = [min(G - 1, max(1, int(x))) for x in depths]
    off = [0]
    for x in d:
        off.append(off[-1] + x)
    return torch.tensor(off, dtype=torch.int32, device=device), off[-1]


def dflash2_conv_finish_ragged(y, coef1, base, group_size, row_offsets, m_rows, next_norm_w, residual=None, out=None,
                               eps=1e-6, next_n=None, next_row0=1, stream=None, taps=2):
    """dflash2_conv_finish whose next norm is written only for each block's drafted rows, packed at
    row_offsets (next_n [m_rows, H]). Returns (out, next_n)."""
    B, G, H = y.shape
    dt = y.dtype
    if row_offsets.numel() != B + 1:
        raise ValueError(f"row_offsets holds {row_offsets.numel()} entries, expected B + 1 = {B + 1}")
    out = torch.empty_like(y) if out is None else out
    if next_n is None:
        next_n = torch.empty((m_rows, H), dtype=dt, device=y.device)
    if next_n.numel() < m_rows * H:
        raise ValueError(f"next_n holds {next_n.numel()} elements, fewer than m_rows * H = {m_rows * H}")
    _check(library().dflash2_conv_finish_ragged(
        _dev(y, "y", dt), _dev(coef1, "coef1", dt), _dev(base, "base", torch.float32), B, G, H, group_size, taps,
        _code(y), _dev(residual, "residual", dt, True), _dev(out, "out", dt), _dev(next_norm_w, "next_norm_w", dt),
        eps, _dev(next_n, "next_n", dt), next_row0, _dev(row_offsets, "row_offsets", torch.int32), m_rows,
        _stream(stream)))
    return out, next_n


def dflash2_score_edges_ragged(cand, unary, z, anchors, pred_book, succ_book, row_offsets, steps, want_S=True, S=None,
                               path=None, stream=None):
    """Edge scores + the greedy walk of a ragged batch: cand/unary [m_rows, K], z [m_rows, R], block b's
    slots at rows row_offsets[b] .. row_offsets[b + 1] - 1. Returns (S [m_rows, K, K] or None,
    path [B, steps] with -1 past each block's rows)."""
    m_rows, K = cand.shape
    R = z.shape[-1]
    V = pred_book.shape[0]
    B = row_offsets.numel() - 1
    dev = cand.device
    if unary.numel() < m_rows * K or z.numel() < m_rows * R:
        raise ValueError("unary and z must hold m_rows rows")
    if want_S and S is None:
        S = torch.empty((m_rows, K, K), dtype=torch.float32, device=dev)
    path = torch.empty((B, steps), dtype=torch.int32, device=dev) if path is None else path
    if path.numel() < B * steps or (S is not None and S.numel() < m_rows * K * K):
        raise ValueError("path must hold B * steps entries and S m_rows * K * K")
    _check(library().dflash2_score_edges_ragged(
        _dev(cand, "cand", torch.int32), _dev(unary, "unary", torch.float32), _dev(z, "z", torch.float32),
        _dev(anchors, "anchors", torch.int32), _dev(pred_book, "pred_book", pred_book.dtype),
        _dev(succ_book, "succ_book", pred_book.dtype), _dev(row_offsets, "row_offsets", torch.int32), B, steps, K, R,
        V, m_rows, _code(pred_book), _dev(S, "S", torch.float32, True), _dev(path, "path", torch.int32),
        _stream(stream)))
    return S, path


def _proj_weight(w, w_scales, w_biases, K):
    """(pointer args, wbits, N) of a projection weight: bf16 [N, K], or 4-bit words [N, K/8] (int32 or
    uint32 storage) with bf16 scales / biases [K/64, N] (group-major)."""
    if w_scales is None and w_biases is None:
        if w.dim() != 2 or w.shape[1] != K:
            raise ValueError(f"w must be [N, {K}] bf16, got shape {tuple(w.shape)}")
        return (_dev(w, "w", torch.bfloat16), None, None), 16, w.shape[0]
    if w_scales is None or w_biases is None:
        raise ValueError("4-bit weights need both w_scales and w_biases")
    if w.dim() != 2 or w.shape[1] * 8 != K or w.element_size() != 4:
        raise ValueError(f"packed 4-bit w must be [N, {K // 8}] 32-bit words, got {tuple(w.shape)} {w.dtype}")
    N = w.shape[0]
    for t, name in ((w_scales, "w_scales"), (w_biases, "w_biases")):
        if tuple(t.shape) != (K // 64, N):
            raise ValueError(f"{name} must be [{K // 64}, {N}] (group-major), got {tuple(t.shape)}")
    return (_dev(w, "w"), _dev(w_scales, "w_scales", torch.bfloat16), _dev(w_biases, "w_biases", torch.bfloat16)), 4, N


def dflash2_conv_coefficients(x, norm_w, eps, w_kp, group_size, n_out=None, d0=None, coef1=None, workspace=None,
                              stream=None, taps=2):
    """Prepare without the side-0 output: returns (n [B*G, H] (x itself when norm_w is None), d0
    [2, groups, B*G] fp32 (side 0's deltas, tap-and-group major), coef1 [B*G, 2, groups])."""
    B, G, H = x.shape
    groups = H // group_size
    dt = x.dtype
    if norm_w is not None and n_out is None:
        n_out = torch.empty((B * G, H), dtype=dt, device=x.device)
    d0 = torch.empty((2, groups, B * G), dtype=torch.float32, device=x.device) if d0 is None else d0
    coef1 = torch.empty((B * G, 2, groups), dtype=dt, device=x.device) if coef1 is None else coef1
    for t, n, name in ((d0, B * G * 2 * groups, "d0"), (coef1, B * G * 2 * groups, "coef1")):
        if t.numel() < n:
            raise ValueError(f"{name} holds {t.numel()} elements, fewer than {n}")
    nbytes = library().dflash2_conv_prepare_workspace_bytes(B, G, H, group_size, _code(x))
    workspace = _workspace(nbytes, x.device, workspace)
    _check(library().dflash2_conv_coefficients(
        _dev(x, "x", dt), _dev(norm_w, "norm_w", dt, True), eps, _dev(w_kp, "w_kp", dt), B, G, H, group_size, taps,
        _code(x), _dev(n_out, "n_out", dt, True), _dev(d0, "d0", torch.float32), _dev(coef1, "coef1", dt),
        _dev(workspace, "workspace"), workspace.numel(), _stream(stream)))
    return (n_out if norm_w is not None else x.view(B * G, H)), d0, coef1


def _proj_ws(M, N, K, dev, workspace):
    """(pointer, bytes) of the projection workspace (allocated here when not given; NULL, 0 when the
    shape needs none)."""
    need = library().dflash2_proj_workspace_bytes(M, N, K)
    if need == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if workspace.numel() < need:
        raise ValueError(f"workspace holds {workspace.numel()} bytes, fewer than the {need} needed")
    return _dev(workspace, "workspace"), workspace.numel()


def dflash2_proj_workspace_bytes(M, N, K) -> int:
    return library().dflash2_proj_workspace_bytes(M, N, K)


def _proj_out(out, M, N, dev):
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev) if out is None else out
    if out.numel() < M * N:
        raise ValueError(f"out holds {out.numel()} elements, fewer than M * N = {M * N}")
    return out


def dflash2_proj(a, w, w_scales=None, w_biases=None, out=None, workspace=None, stream=None):
    """out [M, N] = a [M, K] . W^T (bf16; W bf16 [N, K] or affine 4-bit with scales / biases)."""
    M, K = a.shape
    wp, wbits, N = _proj_weight(w, w_scales, w_biases, K)
    out = _proj_out(out, M, N, a.device)
    ws = _proj_ws(M, N, K, a.device, workspace)
    _check(library().dflash2_proj(_dev(a, "a", torch.bfloat16), M, K, *wp, wbits, N, BF16,
                                  _dev(out, "out", torch.bfloat16), *ws, _stream(stream)))
    return out


def dflash2_proj_conv_in(n, d0, base, G, group_size, w, w_scales=None, w_biases=None, out=None, workspace=None,
                         stream=None):
    """out = Conv_0(n) . W^T with the conv's side 0 computed inside the GEMM (n [M, K = H]; d0
    [2, K / 16, M] fp32 as dflash2_conv_coefficients returns it)."""
    M, K = n.shape
    wp, wbits, N = _proj_weight(w, w_scales, w_biases, K)
    if d0.numel() < M * 2 * (K // group_size) or base.numel() < 4 * K:
        raise ValueError("d0 must hold [M, 2, K / group_size] and base [2, 2, K]")
    out = _proj_out(out, M, N, n.device)
    ws = _proj_ws(M, N, K, n.device, workspace)
    _check(library().dflash2_proj_conv_in(
        _dev(n, "n", torch.bfloat16), _dev(d0, "d0", torch.float32), _dev(base, "base", torch.float32), G, group_size,
        M, K, *wp, wbits, N, BF16, _dev(out, "out", torch.bfloat16), *ws, _stream(stream)))
    return out


def dflash2_proj_conv_out(a, w, coef1, base, G, group_size, residual=None, w_scales=None, w_biases=None, out=None,
                          workspace=None, stream=None):
    """out = residual + Conv_1(a . W^T) with the conv's side 1 (and the residual add) in the GEMM's epilogue."""
    M, K = a.shape
    wp, wbits, N = _proj_weight(w, w_scales, w_biases, K)
    if coef1.numel() < M * 2 * (N // group_size) or base.numel() < 4 * N:
        raise ValueError("coef1 must hold [M, 2, N / group_size] and base [2, 2, N]")
    if residual is not None and residual.numel() < M * N:
        raise ValueError("residual must hold [M, N]")
    out = _proj_out(out, M, N, a.device)
    ws = _proj_ws(M, N, K, a.device, workspace)
    _check(library().dflash2_proj_conv_out(
        _dev(a, "a", torch.bfloat16), M, K, *wp, wbits, N, _dev(coef1, "coef1", torch.bfloat16),
        _dev(base, "base", torch.float32), G, group_size, _dev(residual, "residual", torch.bfloat16, True), BF16,
        _dev(out, "out", torch.bfloat16), *ws, _stream(stream)))
    return out
