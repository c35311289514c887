"""The allocation-free head entry point (dflash2_head_topk_noalloc) against dflash2_head_topk.

Callers that cannot allocate device memory while the head runs (a serving loop where an
allocation would stall the device, or a host that only passes input and output buffers) use this variant: its top-K
scratch is a fixed array inside the library rather than a caller workspace. Here both entry points
run through the C ABI on the same inputs, twice in a row with different shapes (the shared array
keeps the first call's contents), and must agree within the parity tolerance; every output buffer
is preallocated so the variant's calls allocate nothing. The file sorts last so that a run that
stops at the first failure has already run every other test.
"""
import numpy as np
import pytest

from synth import inputs as I
from tests.gpu_util import require_gpu
from tests.parity import assert_close_scaled

pytestmark = pytest.mark.gpu


def _both(torch, wl):
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    h = to_device(wl.h).reshape(-1, wl.H)
    w = to_device(wl.w_head)
    wp = to_device(wl.w_proj)
    bias = to_device(wl.bias) if wl.bias is not None else None
    M = h.shape[0]
    ref = d.dflash2_head_topk(h, w, wl.K, bias=bias, w_proj=wp)
    cand = torch.empty((M, wl.K), dtype=torch.int32, device="cuda")
    unary = torch.empty((M, wl.K), dtype=torch.float32, device="cuda")
    z = torch.empty((M, wl.R), dtype=torch.float32, device="cuda")
    got = d.dflash2_head_topk_noalloc(h, w, wl.K, bias=bias, w_proj=wp, cand=cand, unary=unary, z=z)
    assert d.dflash2_poll_error() == 0
    return ref, got


def test_noalloc_matches_workspace_entry_point_twice():
    torch = require_gpu()
    cases = [I.selector_case(301, B=20, G=16, H=512, V=5000, K=16, R=64, bias=True),   # 300 rows
             I.selector_case(302, B=1, G=16, H=256, V=3000, K=16, R=64)]               # 15 rows, after it
    for wl in cases:
        (rc, ru, rz, _), (gc, gu, gz, _) = _both(torch, wl)
        np.testing.assert_array_equal(gc.cpu().numpy(), rc.cpu().numpy())
        assert_close_scaled(gu.cpu().numpy(), ru.cpu().numpy(), what="unary")
        assert_close_scaled(gz.cpu().numpy(), rz.cpu().numpy(), what="z")


def test_noalloc_rejects_sizes_beyond_its_array():
    require_gpu()
    import ctypes
    import dflash2_block_drafter_gb300 as d
    lib = d.library()
    fake = ctypes.c_void_p(0x10000)
    # 2,000,000 rows need far more than the fixed 8 MiB of top-K scratch: rejected before any launch
    rc = lib.dflash2_head_topk_noalloc(fake, 2000000, 512, fake, 5000, None, None, 0, 16, 0, fake, fake, None, None,
                                       None)
    assert rc == -1
    assert b"allocation-free" in lib.dflash2_last_error_message()


def test_noalloc_replayed_from_a_cuda_graph():
    """The documented use: one warm call, then the call captured in a CUDA graph with every output
    preallocated, and the graph replayed after new inputs are copied into the captured buffers."""
    torch = require_gpu()
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    first = I.selector_case(303, B=8, G=16, H=512, V=4000, K=16, R=64, bias=True)
    second = I.selector_case(304, B=8, G=16, H=512, V=4000, K=16, R=64, bias=True)
    H, K, R = first.H, first.K, first.R
    h = to_device(first.h).reshape(-1, H).clone()
    w = to_device(first.w_head).clone()
    wp = to_device(first.w_proj).clone()
    bias = to_device(first.bias).clone()
    M = h.shape[0]
    cand = torch.empty((M, K), dtype=torch.int32, device="cuda")
    unary = torch.empty((M, K), dtype=torch.float32, device="cuda")
    z = torch.empty((M, R), dtype=torch.float32, device="cuda")
    d.dflash2_head_topk_noalloc(h, w, K, bias=bias, w_proj=wp, cand=cand, unary=unary, z=z)
    torch.cuda.synchronize()
    assert d.dflash2_poll_error() == 0
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        d.dflash2_head_topk_noalloc(h, w, K, bias=bias, w_proj=wp, cand=cand, unary=unary, z=z)
    h.copy_(to_device(second.h).reshape(-1, H))
    w.copy_(to_device(second.w_head))
    wp.copy_(to_device(second.w_proj))
    bias.copy_(to_device(second.bias))
    graph.replay()
    torch.cuda.synchronize()
    assert d.dflash2_poll_error() == 0
    rc, ru, rz, _ = d.dflash2_head_topk(h, w, K, bias=bias, w_proj=wp)
    np.testing.assert_array_equal(cand.cpu().numpy(), rc.cpu().numpy())
    assert_close_scaled(unary.cpu().numpy(), ru.cpu().numpy(), what="unary (graph replay)")
    assert_close_scaled(z.cpu().numpy(), rz.cpu().numpy(), what="z (graph replay)")
