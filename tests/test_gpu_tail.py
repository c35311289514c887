"""GPU parity of the whole block tail (conv chain -> final norm -> head + top-K + z -> S -> walk)."""
import numpy as np
import pytest

from oracle import dflash2_oracle as O
from synth import inputs as I
from tests.gpu_util import dev_f64, oracle_sites, require_gpu
from tests.parity import (REL_TOL, assert_close_scaled, path_parity, compare_topk, compare_walk, record,
                          scale_of)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


def _check_tail(run, wl, blocks, name, min_strict=0):
    """Compare the GPU tail with the oracle on the listed blocks (blocks never interact)."""
    blocks = list(blocks)
    ref = O.block_tail(I.to_f64(wl.x0)[blocks], oracle_sites(wl, blocks), I.to_f64(wl.final_norm_w), wl.eps, wl.gs,
                       I.f64_view(wl.w_head), wl.bias, I.to_f64(wl.w_proj), I.f64_view(wl.pred_book),
                       I.f64_view(wl.succ_book), wl.anchors[blocks], wl.K)
    h = dev_f64(run.h)[blocks]
    assert_close_scaled(h, ref["h"], what="h")
    steps, K, R = wl.steps, wl.K, wl.R
    cand = run.cand.view(wl.B, steps, K).cpu().numpy()[blocks]
    unary = run.unary.view(wl.B, steps, K).cpu().numpy()[blocks]
    z = run.z.view(wl.B, steps, R).cpu().numpy()[blocks]
    # top-K against the oracle's logits of the oracle's h (the chain's rounding is inside the tolerance)
    tol = REL_TOL * scale_of(ref["logits"])
    near = compare_topk(cand.reshape(-1, K), unary.reshape(-1, K), ref["logits"].reshape(-1, wl.V), K,
                        tol)
    assert_close_scaled(z, ref["z"], what="z")
    # the selector teacher-forced on the GPU's candidates (isolates it from head near-ties)
    ref_S = O.score_edges(cand, unary, z, wl.anchors[blocks], I.f64_view(wl.pred_book), I.f64_view(wl.succ_book))
    S = run.S.cpu().numpy()[blocks]
    assert_close_scaled(S, ref_S, what="S")
    ref_path, ref_pos = O.select_path(ref_S, cand)
    path = run.path.cpu().numpy()[blocks]
    walk_near, checked = compare_walk(path, ref_S, ref_pos, cand, REL_TOL * scale_of(ref_S))
    # end to end: the GPU's path against the oracle's own walk over the oracle's own candidates,
    # slot by slot while both the head row and the walk are decided
    e2e = path_parity(path, ref, wl.anchors[blocks], I.f64_view(wl.pred_book), I.f64_view(wl.succ_book), tol,
                      REL_TOL * scale_of(ref["S"]))
    e2e_near, e2e_checked = e2e["near_tie_blocks"], e2e["strict_slots"]
    assert e2e_checked >= min_strict, f"only {e2e_checked} slots of the end-to-end path were decided"
    # the same comparison at a tight tolerance (1e-3 of the scale), counted rather than asserted
    tight = path_parity(path, ref, wl.anchors[blocks], I.f64_view(wl.pred_book), I.f64_view(wl.succ_book),
                        1e-3 * scale_of(ref["logits"]), 1e-3 * scale_of(ref["S"]), strict=False)
    record(name, blocks=len(blocks), near_tie_rows=near, rows=len(blocks) * steps,
           walk_near_tie_blocks=walk_near, walk_strict_slots=checked,
           e2e_near_tie_blocks=e2e_near, e2e_strict_slots=e2e_checked,
           e2e_tight_strict_slots=tight["strict_slots"], e2e_tight_mismatches=tight["mismatches"])
    return ref


def test_tiny_full_tail_f32(torch):
    from dflash2_block_drafter_gb300.tail import TailRunner, to_device
    wl = I.make_config(0)
    run = TailRunner(wl)
    run.full(to_device(wl.x0), [to_device(s.y) for s in wl.sites], to_device(wl.anchors))
    import dflash2_block_drafter_gb300 as d
    assert d.dflash2_poll_error() == 0
    ref = _check_tail(run, wl, range(wl.B), "tail tiny f32 (B=1, G=8, H=256)")
    assert_close_scaled(dev_f64(run.x), ref["x"], rel=2e-3, what="x (f32)")


def test_full_tail_b64_sampled(torch):
    """The full tail at B=64 (drafter shape, Zipf bias); the oracle checks three sampled blocks."""
    from dflash2_block_drafter_gb300.tail import TailRunner, to_device
    wl = I.make_config(4)
    run = TailRunner(wl)
    run.full(to_device(wl.x0), [to_device(s.y) for s in wl.sites], to_device(wl.anchors))
    import dflash2_block_drafter_gb300 as d
    assert d.dflash2_poll_error() == 0
    _check_tail(run, wl, [0, 31, 63], "tail B=64 drafter shape (blocks 0, 31, 63)", min_strict=3)
    path = run.path.cpu().numpy()
    assert path.shape == (64, 15) and np.all((path >= 0) & (path < wl.V))


def test_graph_replay_matches_eager(torch):
    """The tail captured into a CUDA graph and replayed gives the eager pass's results exactly."""
    from dflash2_block_drafter_gb300.tail import TailRunner, to_device
    import dflash2_block_drafter_gb300 as d
    wl = I.make_config(0)
    run = TailRunner(wl)
    x0 = to_device(wl.x0)
    ys = [to_device(s.y) for s in wl.sites]
    anchors = to_device(wl.anchors)
    run.full(x0, ys, anchors)
    eager = (run.path.clone(), run.S.clone(), run.h.clone())
    graph = run.capture(run.full, x0, ys, anchors)
    run.path.zero_()
    run.S.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert d.dflash2_poll_error() == 0
    assert torch.equal(run.path, eager[0])
    assert torch.equal(run.S, eager[1])
    assert torch.equal(run.h, eager[2])


def test_full_from_host_matches_device_inputs(torch):
    """The pass that copies its inputs from pinned host memory on a copy stream (each site waiting
    only for its own sublayer output) gives exactly the results of the pass on device inputs,
    twice in a row (the second call's copies must not overtake the first call's readers)."""
    from dflash2_block_drafter_gb300.tail import TailRunner, to_device, to_pinned
    import dflash2_block_drafter_gb300 as d
    wl = I.make_config(0, B=4)
    run = TailRunner(wl)
    run.full(to_device(wl.x0), [to_device(s.y) for s in wl.sites], to_device(wl.anchors))
    want = (run.path.clone(), run.S.clone(), run.h.clone())
    x0 = torch.empty_like(run.x)
    ys = [torch.empty_like(run.x) for _ in wl.sites]
    anchors = torch.empty(wl.B, dtype=torch.int32, device="cuda")
    h_x0, h_ys, h_anchors = to_pinned(wl.x0), [to_pinned(s.y) for s in wl.sites], to_pinned(wl.anchors)
    for _ in range(2):
        run.path.zero_()
        run.S.zero_()
        run.full_from_host(h_x0, h_ys, h_anchors, x0, ys, anchors)
        torch.cuda.synchronize()
        assert d.dflash2_poll_error() == 0
        assert torch.equal(run.path, want[0])
        assert torch.equal(run.S, want[1])
        assert torch.equal(run.h, want[2])


def test_full_from_host_graph_replay(torch):
    """The host-input pass captured into one CUDA graph (copies as graph nodes on their own
    branch) gives the eager pass's results exactly, and reads the host buffers at replay time."""
    from dflash2_block_drafter_gb300.tail import TailRunner, to_device, to_pinned
    import dflash2_block_drafter_gb300 as d
    wl = I.make_config(0, B=4)
    run = TailRunner(wl)
    run.full(to_device(wl.x0), [to_device(s.y) for s in wl.sites], to_device(wl.anchors))
    want = (run.path.clone(), run.S.clone(), run.h.clone())
    x0 = torch.empty_like(run.x)
    ys = [torch.empty_like(run.x) for _ in wl.sites]
    anchors = torch.empty(wl.B, dtype=torch.int32, device="cuda")
    h_x0, h_ys, h_anchors = to_pinned(wl.x0), [to_pinned(s.y) for s in wl.sites], to_pinned(wl.anchors)
    real_y0 = h_ys[0].clone()
    h_ys[0].zero_()  # the capture pass sees other inputs than the replay
    graph = run.capture(run.full_from_host, h_x0, h_ys, h_anchors, x0, ys, anchors)
    h_ys[0].copy_(real_y0)
    run.path.zero_()
    run.S.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert d.dflash2_poll_error() == 0
    assert torch.equal(run.path, want[0])
    assert torch.equal(run.S, want[1])
    assert torch.equal(run.h, want[2])


def test_pipeline_from_host_matches_each_batch(torch):
    """Three host batches through the two-set pipeline (the third refills the first set after the
    first pass has read it): each batch's path equals the device-input pass on that batch, eager
    and with a captured pass per set."""
    from dflash2_block_drafter_gb300.tail import TailRunner, to_device
    import dflash2_block_drafter_gb300 as d
    wl = I.make_config(0, B=4)
    run = TailRunner(wl)
    base_x0 = to_device(wl.x0)
    base_ys = [to_device(s.y) for s in wl.sites]
    anchors = to_device(wl.anchors)
    batches, want = [], []
    for scale in (1.0, -1.0, 0.5):  # exact in bf16
        x0 = (base_x0.float() * scale).to(base_x0.dtype)
        ys = [(y.float() * scale).to(y.dtype) for y in base_ys]
        run.full(x0, ys, anchors)
        want.append(run.path.cpu().clone())
        batches.append((x0.cpu().pin_memory(), [y.cpu().pin_memory() for y in ys], anchors.cpu().pin_memory()))
    # both sets hold valid inputs before anything reads them (a capture runs its pass once)
    sets = [(base_x0.clone(), [y.clone() for y in base_ys], anchors.clone()) for _ in range(2)]
    for use_graphs in (False, True):
        graphs = [run.capture(run.full, *sets[k]) for k in range(2)] if use_graphs else None
        outs = [torch.full(tuple(run.path.shape), -7, dtype=torch.int32).pin_memory() for _ in batches]
        run.pipeline_from_host(batches, sets, outs, graphs)
        torch.cuda.synchronize()
        assert d.dflash2_poll_error() == 0
        for got, ref in zip(outs, want):
            assert torch.equal(got, ref)
