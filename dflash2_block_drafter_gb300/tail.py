"""The block tail as a sequence of library calls, with every buffer allocated once.

``TailRunner`` holds the weights of one drafter tail on the device and preallocates all
activations and workspaces, so a pass is a fixed sequence of C-ABI launches on one stream (and
can be captured into a CUDA graph after a first eager pass). Per conv site (MAX
DFlash2TransformerBlock; dflash2.ts #block):

    a, coef1 = conv_prepare(n or x)            # side 0 (+ the first site's RMSNorm)
    (the sublayer: here its seeded output y)
    x = x + conv_finish(y, coef1)              # side 1 + residual, and the next site's RMSNorm

then h = final_norm(x[:, 1:]), head GEMM + top-K + z, edge scores and the greedy walk.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import numpy as np
import torch

from . import (dflash2_conv_finish, dflash2_conv_finish_launches, dflash2_conv_finish_ragged, dflash2_conv_prepare,
               dflash2_conv_prepare_launches, dflash2_conv_prepare_workspace_bytes, dflash2_head_topk,
               dflash2_head_topk_workspace_bytes, dflash2_score_edges, dflash2_score_edges_ragged)


def to_device(a: np.ndarray, device="cuda") -> torch.Tensor:
    """Upload a stored host tensor: uint16 arrays hold bf16 bits; float32 / int32 go as they are."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def to_pinned(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    return t.pin_memory()


@dataclass
class SiteWeights:
    w_kp: torch.Tensor
    base: torch.Tensor
    norm_w: torch.Tensor


class TailRunner:
    """One drafter tail (conv sites -> final norm -> selector) with preallocated buffers."""

    def __init__(self, wl, device="cuda", with_selector: bool = True):
        self.wl = wl
        self.device = device
        self.dtype = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
        B, G, H = wl.B, wl.G, wl.H
        self.sites: List[SiteWeights] = [SiteWeights(to_device(s.w_kp, device), to_device(s.base, device),
                                                     to_device(s.norm_w, device)) for s in wl.sites]
        self.with_selector = with_selector and wl.w_head is not None
        dt = self.dtype
        self.x = torch.empty((B, G, H), dtype=dt, device=device)
        self.a = torch.empty((B, G, H), dtype=dt, device=device)
        self.n = torch.empty((B, G, H), dtype=dt, device=device)
        self.coef1 = torch.empty((B, G, 2, H // wl.gs), dtype=dt, device=device)
        ws = dflash2_conv_prepare_workspace_bytes(B, G, H, wl.gs, dt)
        self.conv_ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=device)
        if self.with_selector:
            self.final_norm_w = to_device(wl.final_norm_w, device) if wl.final_norm_w is not None else None
            self.w_head = to_device(wl.w_head, device)
            self.bias = to_device(wl.bias, device) if wl.bias is not None else None
            self.w_proj = to_device(wl.w_proj, device)
            self.pred = to_device(wl.pred_book, device)
            self.succ = to_device(wl.succ_book, device)
            M = B * wl.steps
            self.h = torch.empty((B, wl.steps, H), dtype=dt, device=device)
            self.cand = torch.empty((M, wl.K), dtype=torch.int32, device=device)
            self.unary = torch.empty((M, wl.K), dtype=torch.float32, device=device)
            self.z = torch.empty((M, wl.R), dtype=torch.float32, device=device)
            self.S = torch.empty((B, wl.steps, wl.K, wl.K), dtype=torch.float32, device=device)
            self.path = torch.empty((B, wl.steps), dtype=torch.int32, device=device)
            hw = dflash2_head_topk_workspace_bytes(M, H, wl.V, wl.K, wl.R)
            self.head_ws = torch.empty(max(hw, 256), dtype=torch.uint8, device=device)

    # ------------------------------------------------------------------ passes
    def conv_chain(self, x0: torch.Tensor, ys: List[torch.Tensor], emit_h: bool, before_finish=None, ragged=None):
        """Every site in order, starting from x0 (left unchanged); returns the final residual stream (self.x).
        ``before_finish(i)``, if given, runs before site i's finish call is issued (full_from_host
        makes the compute stream wait there for y_i's copy). ``ragged`` = (row_offsets, m_rows): the
        final norm writes only each block's drafted rows, packed (h rows [0, m_rows))."""
        wl = self.wl
        nsites = len(self.sites)
        for i, s in enumerate(self.sites):
            if i == 0:
                dflash2_conv_prepare(x0, s.norm_w, wl.eps, s.w_kp, s.base, wl.gs, out=self.a, coef1=self.coef1,
                                     workspace=self.conv_ws)
            else:
                dflash2_conv_prepare(self.n, None, wl.eps, s.w_kp, s.base, wl.gs, out=self.a, coef1=self.coef1,
                                     workspace=self.conv_ws)
            residual = x0 if i == 0 else self.x
            if before_finish is not None:
                before_finish(i)
            if i + 1 < nsites:
                dflash2_conv_finish(ys[i], self.coef1, s.base, wl.gs, residual=residual, out=self.x,
                                    next_norm_w=self.sites[i + 1].norm_w, eps=wl.eps, next_n=self.n, next_row0=0)
            elif emit_h and ragged is not None:
                off, m_rows = ragged
                dflash2_conv_finish_ragged(ys[i], self.coef1, s.base, wl.gs, off, m_rows, self.final_norm_w,
                                           residual=residual, out=self.x, eps=wl.eps,
                                           next_n=self.h.view(-1, wl.H)[:m_rows], next_row0=1)
            elif emit_h:
                dflash2_conv_finish(ys[i], self.coef1, s.base, wl.gs, residual=residual, out=self.x,
                                    next_norm_w=self.final_norm_w, eps=wl.eps, next_n=self.h, next_row0=1)
            else:
                dflash2_conv_finish(ys[i], self.coef1, s.base, wl.gs, residual=residual, out=self.x)
        return self.x

    def launches_per_pass(self, conv: bool = True, selector: bool = True, emit_h: bool = True) -> int:
        """Library kernels one pass launches, as the library reports them per call: per site a
        prepare (the first with its RMSNorm) and a finish (with the next site's norm, or the final
        norm when h is emitted); then the head GEMM + top-K merge and the edge-score/walk kernel."""
        wl = self.wl
        n = 0
        ns = len(self.sites)
        if conv and ns:
            shape = (wl.B, wl.G, wl.H, wl.gs, self.dtype)
            n += dflash2_conv_prepare_launches(*shape, True) + (ns - 1) * dflash2_conv_prepare_launches(*shape, False)
            for i in range(ns):
                n += dflash2_conv_finish_launches(*shape, i + 1 < ns or emit_h)
        if selector and self.with_selector:
            n += 3
        return n

    def selector(self, h: torch.Tensor, anchors: torch.Tensor, want_S: bool = True):
        wl = self.wl
        M = h.shape[0] * h.shape[1]
        dflash2_head_topk(h.view(M, wl.H), self.w_head, wl.K, bias=self.bias, w_proj=self.w_proj, cand=self.cand,
                          unary=self.unary, z=self.z, workspace=self.head_ws)
        B = h.shape[0]
        dflash2_score_edges(self.cand.view(B, wl.steps, wl.K), self.unary.view(B, wl.steps, wl.K),
                            self.z.view(B, wl.steps, wl.R), anchors, self.pred, self.succ, want_S=want_S,
                            want_path=True, S=self.S if want_S else None, path=self.path)
        return self.path

    def full(self, x0: torch.Tensor, ys: List[torch.Tensor], anchors: torch.Tensor, want_S: bool = True):
        """The whole block tail; returns path [B, steps] int32 (device)."""
        self.conv_chain(x0, ys, emit_h=True)
        return self.selector(self.h, anchors, want_S=want_S)

    def full_ragged(self, x0: torch.Tensor, ys: List[torch.Tensor], anchors: torch.Tensor, row_offsets: torch.Tensor,
                    m_rows: int, want_S: bool = True):
        """The whole block tail of a ragged batch (``dflash2_ragged_offsets``): every conv site runs
        over the dense blocks, then only block b's drafted rows row_offsets[b] .. row_offsets[b + 1]
        - 1 go through the final norm, the head and the selector. cand, unary, z and S hold the packed
        rows [0, m_rows); returns path [B, steps] int32 (-1 past each block's rows)."""
        self.conv_chain(x0, ys, emit_h=True, ragged=(row_offsets, m_rows))
        return self.selector_ragged(anchors, row_offsets, m_rows, want_S=want_S)

    def selector_ragged(self, anchors: torch.Tensor, row_offsets: torch.Tensor, m_rows: int, want_S: bool = True):
        """Head + top-K + z over the packed rows h[0, m_rows), then the ragged edge scores and walk."""
        wl = self.wl
        need = dflash2_head_topk_workspace_bytes(m_rows, wl.H, wl.V, wl.K, wl.R)
        if need > self.head_ws.numel():
            self.head_ws = torch.empty(need, dtype=torch.uint8, device=self.device)
        h = self.h.view(-1, wl.H)[:m_rows]
        dflash2_head_topk(h, self.w_head, wl.K, bias=self.bias, w_proj=self.w_proj, cand=self.cand[:m_rows],
                          unary=self.unary[:m_rows], z=self.z[:m_rows], workspace=self.head_ws)
        S = self.S.view(-1, wl.K, wl.K)[:m_rows] if want_S else None
        dflash2_score_edges_ragged(self.cand[:m_rows], self.unary[:m_rows], self.z[:m_rows], anchors, self.pred,
                                   self.succ, row_offsets, wl.steps, want_S=want_S, S=S, path=self.path)
        return self.path

    def full_from_host(self, h_x0: torch.Tensor, h_ys: List[torch.Tensor], h_anchors: torch.Tensor,
                       x0: torch.Tensor, ys: List[torch.Tensor], anchors: torch.Tensor, want_S: bool = True,
                       ragged=None):
        """The whole block tail with its inputs in pinned host memory. Every input is copied into
        the given device buffers on a copy stream, one event per input; the compute stream waits
        for x0 before the first site, for y_i only before site i's finish and for the anchors
        before the selector, so the copies of later sites' inputs overlap the earlier sites. (Two
        or four copy streams were measured slower: concurrent host-to-device copies contend.) The
        pass can be captured with ``capture``: the copies become graph nodes on a forked branch
        whose events join it where each input is needed, and the host buffers are read at replay
        time (refresh them in place). ``ragged`` = (row_offsets, m_rows) runs ``full_ragged``'s
        selector instead. Returns path [B, steps] int32 (device)."""
        comp = torch.cuda.current_stream()
        if getattr(self, "_copy_stream", None) is None:
            self._copy_stream = torch.cuda.Stream(device=comp.device)
            self._ev_x0 = torch.cuda.Event()
            self._ev_y = [torch.cuda.Event() for _ in self.sites]
            self._ev_anchors = torch.cuda.Event()
        cs = self._copy_stream
        cs.wait_stream(comp)  # whatever still reads the device input buffers was queued before this
        with torch.cuda.stream(cs):
            x0.copy_(h_x0, non_blocking=True)
            self._ev_x0.record(cs)
            for i, (dst, src) in enumerate(zip(ys, h_ys)):
                dst.copy_(src, non_blocking=True)
                self._ev_y[i].record(cs)
            anchors.copy_(h_anchors, non_blocking=True)
            self._ev_anchors.record(cs)
        comp.wait_event(self._ev_x0)
        self.conv_chain(x0, ys, emit_h=True, before_finish=lambda i: comp.wait_event(self._ev_y[i]), ragged=ragged)
        comp.wait_event(self._ev_anchors)
        if ragged is not None:
            path = self.selector_ragged(anchors, *ragged, want_S=want_S)
        else:
            path = self.selector(self.h, anchors, want_S=want_S)
        if not torch.cuda.is_current_stream_capturing():
            for t in [x0, anchors] + list(ys):  # the copy stream wrote them: keep the allocator honest
                t.record_stream(cs)
        return path

    def pipeline_from_host(self, batches, sets, out_host, graphs=None, ragged=None):
        """Runs the tail over a sequence of batches in pinned host memory back to back, the way a
        serving loop does. Two device input sets alternate: batch i + 1's inputs are copied on
        the copy stream while batch i computes (a set is refilled only after the pass that read it
        has finished), and every batch's path is copied into its pinned host buffer right after
        its pass.

        batches: list of (h_x0, h_ys, h_anchors) pinned host tensors; sets: two (x0, ys, anchors)
        device buffer sets; out_host: one pinned [B, steps] int32 tensor per batch (a tensor may
        appear several times); graphs: optional two captured passes, ``graphs[k]`` over
        ``sets[k]`` (``capture(self.full, *sets[k])``); ragged = (row_offsets, m_rows) runs
        ``full_ragged`` instead of ``full``. Everything is enqueued on the current stream and the
        copy stream; the caller synchronizes."""
        comp = torch.cuda.current_stream()
        if getattr(self, "_copy_stream", None) is None:
            self._copy_stream = torch.cuda.Stream(device=comp.device)
        cs = self._copy_stream
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        freed = [None, None]  # after the last pass that read set k

        def issue(i):
            k = i % 2
            if freed[k] is not None:
                cs.wait_event(freed[k])
            else:
                cs.wait_stream(comp)
            h_x0, h_ys, h_anchors = batches[i]
            x0, ys, anchors = sets[k]
            with torch.cuda.stream(cs):
                x0.copy_(h_x0, non_blocking=True)
                for dst, src in zip(ys, h_ys):
                    dst.copy_(src, non_blocking=True)
                anchors.copy_(h_anchors, non_blocking=True)
                copied[k].record(cs)

        if batches:
            issue(0)
        for i in range(len(batches)):
            if i + 1 < len(batches):
                issue(i + 1)
            k = i % 2
            comp.wait_event(copied[k])
            if graphs is not None:
                graphs[k].replay()
            elif ragged is not None:
                self.full_ragged(*sets[k], *ragged)
            else:
                self.full(*sets[k])
            ev = torch.cuda.Event()
            ev.record(comp)
            freed[k] = ev
            out_host[i].copy_(self.path, non_blocking=True)

    def capture(self, fn, *args, **kwargs) -> "torch.cuda.CUDAGraph":
        """Record one pass of ``fn`` (e.g. ``self.full``) into a CUDA graph over the runner's fixed
        buffers; ``graph.replay()`` then re-launches every kernel of the pass with one call.

        The pass runs once eagerly first, so that every kernel's attributes are set outside the
        capture. Inputs are read from the tensors passed here at replay time: refresh them in place.
        """
        fn(*args, **kwargs)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                fn(*args, **kwargs)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        return graph
