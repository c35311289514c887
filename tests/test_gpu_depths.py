"""GPU parity of the mixed-depth walk (blocks of one batch drafting different numbers of tokens)
against the float64 oracle: block b walks its first min(steps, max(1, depths[b])) slots (dflash2.ts
blockColumns), the rest of its path is -1."""
import numpy as np
import pytest

from oracle import dflash2_oracle as O
from synth import inputs as I
from tests.gpu_util import require_gpu
from tests.parity import REL_TOL, assert_close_scaled, compare_walk, scale_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


def _case(seed, B, steps, K, R, V, dtype="bf16"):
    rng = np.random.default_rng(seed)
    cand = np.stack([np.stack([rng.choice(V, size=K, replace=False) for _ in range(steps)]) for _ in range(B)])
    cand = cand.astype(np.int32)
    unary = np.sort(rng.standard_normal((B, steps, K)).astype(np.float32), axis=-1)[..., ::-1].copy()
    z = rng.standard_normal((B, steps, R)).astype(np.float32)
    anchors = rng.integers(0, V, size=B).astype(np.int32)
    pred = I.normal(seed, "pred", (V, R), 0.5, dtype=dtype)
    succ = I.normal(seed, "succ", (V, R), 0.5, dtype=dtype)
    depths = rng.integers(1, steps + 1, size=B).astype(np.int32)
    depths[0] = steps          # one full-depth block
    if B > 1:
        depths[1] = 0          # one asked for nothing: it drafts one token (blockColumns)
    if B > 2:
        depths[2] = steps + 5  # one asked for more than the block holds: it drafts `steps`
    return cand, unary, z, anchors, pred, succ, depths


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,steps,K,R,V", [(64, 15, 16, 64, 248320), (5, 4, 3, 8, 50), (37, 31, 32, 128, 1000)])
def test_mixed_depth_walk(torch, dtype, B, steps, K, R, V):
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    cand, unary, z, anchors, pred, succ, depths = _case(B * 7 + K, B, steps, K, R, V, dtype)
    S, path = d.dflash2_score_edges_depths(to_device(cand), to_device(unary), to_device(z), to_device(anchors),
                                           to_device(pred), to_device(succ), to_device(depths))
    assert d.dflash2_poll_error() == 0
    S = S.cpu().numpy()
    path = path.cpu().numpy()
    rS = O.score_edges(cand, unary, z, anchors, I.to_f64(pred), I.to_f64(succ))
    assert_close_scaled(S, rS, what="S")       # S covers every slot whatever the depths
    rpath, rpos = O.select_path_depths(rS, cand, depths)
    # padding is exact
    np.testing.assert_array_equal(path < 0, rpath < 0)
    assert (path[rpath < 0] == -1).all()
    # the walked prefix: exact over the GPU's own S, near-tie aware against the oracle's S
    gpath, _ = O.select_path_depths(S.astype(np.float64), cand, depths)
    np.testing.assert_array_equal(path, gpath)
    full_path, full_pos = O.select_path(rS, cand)
    tol = REL_TOL * scale_of(rS)
    mask = rpath >= 0
    compare_walk(np.where(mask, path, full_path), rS, full_pos, cand, tol)
    # the standalone walk agrees with the fused one
    p2 = d.dflash2_select_path_depths(to_device(S), to_device(cand), to_device(depths)).cpu().numpy()
    np.testing.assert_array_equal(p2, path)


def test_full_depths_equal_the_plain_walk(torch):
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    cand, unary, z, anchors, pred, succ, _ = _case(5, 16, 15, 16, 64, 5000)
    args = [to_device(a) for a in (cand, unary, z, anchors, pred, succ)]
    S0, p0 = d.dflash2_score_edges(*args)
    S1, p1 = d.dflash2_score_edges_depths(*args, to_device(np.full(16, 15, np.int32)))
    np.testing.assert_array_equal(S1.cpu().numpy(), S0.cpu().numpy())
    np.testing.assert_array_equal(p1.cpu().numpy(), p0.cpu().numpy())


def test_depths_clamp_like_block_columns(torch):
    """Depths outside [1, steps] draft min(steps, max(1, depth)) tokens and set no error."""
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    cand, unary, z, anchors, pred, succ, _ = _case(6, 4, 7, 8, 16, 500)
    depths = np.array([7, 9, -2, 0], np.int32)
    args = [to_device(a) for a in (cand, unary, z, anchors, pred, succ)]
    S, path = d.dflash2_score_edges_depths(*args, to_device(depths))
    assert d.dflash2_poll_error() == 0
    path = path.cpu().numpy()
    _, full = d.dflash2_score_edges(*args)
    full = full.cpu().numpy()
    np.testing.assert_array_equal(path[0], full[0])
    np.testing.assert_array_equal(path[1], full[1])        # 9 -> the 7 slots
    for b in (2, 3):                                        # -2 and 0 -> one token
        assert path[b, 0] == full[b, 0] and (path[b, 1:] == -1).all()
    p2 = d.dflash2_select_path_depths(S, args[0], to_device(depths)).cpu().numpy()
    np.testing.assert_array_equal(p2, path)
