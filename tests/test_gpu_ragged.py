"""GPU parity of the ragged block tail (only the rows each block drafts go through the final norm,
the head and the selector; dflash2.ts blockColumns / #block) against the float64 oracle, and
against the dense tail's own rows."""
import numpy as np
import pytest

from oracle import dflash2_oracle as O
from synth import inputs as I
from tests.gpu_util import dev_f64, oracle_sites, require_gpu
from tests.parity import REL_TOL, assert_close_scaled, compare_topk, path_parity, record, scale_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


def _drafted(depths, G):
    return [min(G - 1, max(1, int(d))) for d in depths]


def _run_both(wl, depths):
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import TailRunner, to_device
    x0, ys, anchors = to_device(wl.x0), [to_device(s.y) for s in wl.sites], to_device(wl.anchors)
    run = TailRunner(wl)
    run.full(x0, ys, anchors)
    dense_h = run.h.clone()
    off, m = d.dflash2_ragged_offsets(depths, wl.G)
    run.full_ragged(x0, ys, anchors, off, m)
    assert d.dflash2_poll_error() == 0
    return run, dense_h, off.cpu().numpy(), m


def _check(run, wl, depths, blocks, name):
    """Ragged rows of the listed blocks against the oracle's ragged tail (blocks never interact)."""
    G, K, steps = wl.G, wl.K, wl.steps
    dr = _drafted(depths, G)
    off = np.concatenate([[0], np.cumsum(dr)])
    ref = O.block_tail_ragged(I.to_f64(wl.x0)[blocks], oracle_sites(wl, blocks), I.to_f64(wl.final_norm_w), wl.eps,
                              wl.gs, I.f64_view(wl.w_head), wl.bias, I.to_f64(wl.w_proj), I.f64_view(wl.pred_book),
                              I.f64_view(wl.succ_book), wl.anchors[blocks], K, [depths[b] for b in blocks])
    rows = np.concatenate([np.arange(off[b], off[b + 1]) for b in blocks])
    h = dev_f64(run.h.view(-1, wl.H))[rows]
    assert_close_scaled(h, ref["h"], what="ragged h")
    cand = run.cand.cpu().numpy()[rows]
    unary = run.unary.cpu().numpy()[rows]
    z = run.z.cpu().numpy()[rows]
    tol = REL_TOL * scale_of(ref["logits"])
    near = compare_topk(cand, unary, ref["logits"], K, tol)
    assert_close_scaled(z, ref["z"], what="ragged z")
    path = run.path.cpu().numpy()[blocks]
    S_gpu = run.S.view(-1, K, K).cpu().numpy()[rows]
    strict = e2e_near = 0
    for i, b in enumerate(blocks):
        lo, hi = ref["offsets"][i], ref["offsets"][i + 1]
        db = hi - lo
        # padding past the drafted rows, exactly
        assert (path[i, db:] == -1).all() and (path[i, :db] >= 0).all()
        # the selector teacher-forced on the GPU's own candidates
        rS = O.score_edges(cand[None, lo:hi], unary[None, lo:hi], z[None, lo:hi], wl.anchors[b:b + 1],
                           I.f64_view(wl.pred_book), I.f64_view(wl.succ_book))
        assert_close_scaled(S_gpu[None, lo:hi], rS, what=f"ragged S block {b}")
        gpath, _ = O.select_path(S_gpu[None, lo:hi].astype(np.float64), cand[None, lo:hi])
        np.testing.assert_array_equal(path[i, :db], gpath[0])
        # end to end against the oracle's own walk
        ref_b = dict(logits=ref["logits"][None, lo:hi], z=ref["z"][None, lo:hi], path=ref["path"][i:i + 1, :db],
                     cand=ref["cand"][None, lo:hi])
        pp = path_parity(path[i:i + 1, :db], ref_b, wl.anchors[b:b + 1], I.f64_view(wl.pred_book),
                         I.f64_view(wl.succ_book), tol, REL_TOL * scale_of(ref["S"]))
        strict += pp["strict_slots"]
        e2e_near += pp["near_tie_blocks"]
    record(name, blocks=len(blocks), rows=len(rows), near_tie_rows=near, e2e_near_tie_blocks=e2e_near,
           e2e_strict_slots=strict)


def test_ragged_tail_tiny_f32(torch):
    wl = I.make_config(0, B=5)
    depths = [1, 7, 3, 0, 9]          # G = 8: 0 drafts one token, 9 the block's seven
    run, dense_h, off, m = _run_both(wl, depths)
    assert m == 1 + 7 + 3 + 1 + 7
    dr = _drafted(depths, wl.G)
    for b in range(wl.B):   # the packed rows are the dense rows, bit for bit
        assert torch.equal(run.h.view(-1, wl.H)[off[b]:off[b + 1]], dense_h[b, :dr[b]])
    _check(run, wl, depths, list(range(wl.B)), "ragged tail tiny f32 (B=5)")


def test_ragged_tail_drafter_shape(torch):
    """B = 64 at the drafter's shape with seeded depths; the head runs over the drafted rows only."""
    wl = I.make_config(4)
    rng = np.random.default_rng(20261202)
    depths = rng.integers(1, wl.steps + 1, size=wl.B).tolist()
    depths[5], depths[9] = 0, 40
    run, dense_h, off, m = _run_both(wl, depths)
    dr = _drafted(depths, wl.G)
    assert m == sum(dr) < wl.B * wl.steps
    for b in range(wl.B):
        assert torch.equal(run.h.view(-1, wl.H)[off[b]:off[b + 1]], dense_h[b, :dr[b]])
    _check(run, wl, depths, [0, 5, 9, 63], "ragged tail B=64 drafter shape (blocks 0, 5, 9, 63)")


def test_ragged_tail_small_batch(torch):
    """B = 8 at the drafter's shape: the conv runs in the small-row kernels (prepare in one launch,
    finish + the final norm one CTA per row, which writes the drafted rows packed)."""
    wl = I.make_config(4, B=8)
    depths = [15, 1, 0, 7, 3, 20, 11, 2]
    run, dense_h, off, m = _run_both(wl, depths)
    dr = _drafted(depths, wl.G)
    assert m == sum(dr)
    for b in range(wl.B):
        assert torch.equal(run.h.view(-1, wl.H)[off[b]:off[b + 1]], dense_h[b, :dr[b]])
    _check(run, wl, depths, [0, 2, 5], "ragged tail B=8 drafter shape (blocks 0, 2, 5)")


def test_ragged_offsets_outside_their_rows_set_the_error_word(torch):
    """A block whose span holds no row, or reaches past m_rows, records DFLASH2_ERR_INVALID_ARG and is
    skipped (path -1); the other blocks are unaffected."""
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    rng = np.random.default_rng(3)
    V, K, R, steps = 700, 16, 64, 7
    m = 9
    cand = np.stack([rng.choice(V, size=K, replace=False) for _ in range(m)]).astype(np.int32)
    unary = -np.sort(-rng.standard_normal((m, K)).astype(np.float32), axis=-1)
    z = rng.standard_normal((m, R)).astype(np.float32)
    anchors = rng.integers(0, V, size=3).astype(np.int32)
    pred = I.normal(3, "pred", (V, R), 0.5)
    succ = I.normal(3, "succ", (V, R), 0.5)
    args = [to_device(a) for a in (cand, unary, z, anchors, pred, succ)]
    good = torch.tensor([0, 4, 4, 9], dtype=torch.int32, device="cuda")   # block 1 holds no row
    _, path = d.dflash2_score_edges_ragged(*args, good, steps)
    assert d.dflash2_poll_error() == -1
    p = path.cpu().numpy()
    assert (p[1] == -1).all() and (p[0, :4] >= 0).all() and (p[2, :5] >= 0).all()
    over = torch.tensor([0, 4, 6, 12], dtype=torch.int32, device="cuda")  # block 2 reaches past m_rows = 9
    _, path = d.dflash2_score_edges_ragged(*args, over, steps)
    assert d.dflash2_poll_error() == -1
    assert (path.cpu().numpy()[2] == -1).all()
