"""GPU parity of score_edges and the greedy walk against the float64 oracle."""
import numpy as np
import pytest

from oracle import dflash2_oracle as O
from synth import inputs as I
from tests.gpu_util import require_gpu
from tests.parity import REL_TOL, assert_close_scaled, compare_walk, record, scale_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


def _case(seed, B, steps, K, R, V, dtype="bf16", book_std=0.5):
    rng = np.random.default_rng(seed)
    cand = rng.integers(0, V, size=(B, steps, K))
    for idx in np.ndindex(B, steps):   # distinct ids within a slot (a top-K list never repeats one)
        if len(set(cand[idx].tolist())) < K:
            cand[idx] = rng.choice(V, size=K, replace=False)
    cand = cand.astype(np.int32)
    unary = np.sort(rng.standard_normal((B, steps, K)).astype(np.float32), axis=-1)[..., ::-1].copy()
    z = rng.standard_normal((B, steps, R)).astype(np.float32)
    anchors = rng.integers(0, V, size=B).astype(np.int32)
    pred = I.normal(seed, "pred", (V, R), book_std, dtype=dtype)
    succ = I.normal(seed, "succ", (V, R), book_std, dtype=dtype)
    return cand, unary, z, anchors, pred, succ


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,steps,K,R,V", [(1, 15, 16, 64, 5000), (33, 15, 16, 64, 248320), (7, 7, 16, 16, 4096),
                                           (5, 4, 3, 8, 50), (3, 31, 32, 128, 1000),
                                           (4, 15, 16, 128, 3000),   # K = 16 tiles with R = 128
                                           (200, 15, 16, 64, 9000),   # more blocks than SMs
                                           (700, 15, 16, 64, 248320),  # two warps per block, pipelined
                                           (3, 63, 16, 32, 2000)])     # the longest block
def test_score_edges_and_walk(torch, dtype, B, steps, K, R, V):
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    cand, unary, z, anchors, pred, succ = _case(B * 100 + K, B, steps, K, R, V, dtype)
    S, path = d.dflash2_score_edges(to_device(cand), to_device(unary), to_device(z), to_device(anchors),
                                    to_device(pred), to_device(succ))
    assert d.dflash2_poll_error() == 0
    S = S.cpu().numpy()
    path = path.cpu().numpy()
    rS = O.score_edges(cand, unary, z, anchors, I.to_f64(pred), I.to_f64(succ))
    assert_close_scaled(S, rS, what="S")
    assert_close_scaled(S, rS, rel=1e-5, what="S (fp32 bound)")
    rpath, rpos = O.select_path(rS, cand)
    tol = REL_TOL * scale_of(rS)
    near, checked = compare_walk(path, rS, rpos, cand, tol)
    # the walk over the GPU's own S is exact (same fp32 values, same tie rule)
    gpath, _ = O.select_path(S.astype(np.float64), cand)
    np.testing.assert_array_equal(path, gpath)
    # the standalone walk agrees with the fused one
    p2 = d.dflash2_select_path(to_device(S), to_device(cand)).cpu().numpy()
    np.testing.assert_array_equal(p2, path)
    record(f"score_edges {dtype} B={B} steps={steps} K={K} R={R} V={V}", near_tie_blocks=near, strict_slots=checked)


def test_zero_codebooks_walk_is_top1(torch):
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    cand, unary, z, anchors, pred, succ = _case(9, 8, 15, 16, 64, 3000)
    zero = np.zeros_like(pred)
    S, path = d.dflash2_score_edges(to_device(cand), to_device(unary), to_device(z), to_device(anchors),
                                    to_device(zero), to_device(zero))
    np.testing.assert_array_equal(path.cpu().numpy(), cand[:, :, 0])
    np.testing.assert_array_equal(S.cpu().numpy(), np.broadcast_to(unary[:, :, None, :], S.shape))


def test_slot0_rows_identical(torch):
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    cand, unary, z, anchors, pred, succ = _case(10, 4, 15, 16, 64, 3000)
    S, _ = d.dflash2_score_edges(to_device(cand), to_device(unary), to_device(z), to_device(anchors),
                                 to_device(pred), to_device(succ), want_path=False)
    S = S.cpu().numpy()
    for p in range(1, 16):
        np.testing.assert_array_equal(S[:, 0, p], S[:, 0, 0])


def test_bad_index_sets_error_word(torch):
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    cand, unary, z, anchors, pred, succ = _case(12, 2, 5, 4, 16, 100)
    cand[1, 2, 3] = 100      # == V: out of range
    d.dflash2_score_edges(to_device(cand), to_device(unary), to_device(z), to_device(anchors), to_device(pred),
                          to_device(succ))
    assert d.dflash2_poll_error() == -6
    assert d.dflash2_poll_error() == 0   # cleared


@pytest.mark.parametrize("dtype,R", [("bf16", 64), ("f32", 16)])
def test_bad_index_sets_error_word_k16(torch, dtype, R):
    """The K = 16 kernel: an id outside [0, V) in a successor and in a predecessor position sets
    DFLASH2_ERR_BAD_INDEX and reads as a zero row (its edge term is 0: S equals unary there)."""
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    cand, unary, z, anchors, pred, succ = _case(13, 3, 6, 16, R, 500, dtype)
    cand[1, 2, 5] = 500       # == V
    cand[2, 0, 7] = -1        # a predecessor of slot 1
    S, _ = d.dflash2_score_edges(to_device(cand), to_device(unary), to_device(z), to_device(anchors),
                                 to_device(pred), to_device(succ))
    assert d.dflash2_poll_error() == -6
    assert d.dflash2_poll_error() == 0
    S = S.cpu().numpy()
    np.testing.assert_array_equal(S[1, 2, :, 5], np.full(16, unary[1, 2, 5], np.float32))
    np.testing.assert_array_equal(S[2, 1, 7, :], unary[2, 1, :])


def test_misaligned_unary_and_S_take_the_scalar_path(torch):
    """unary and S 4 bytes off a 16-byte boundary: the edge-score kernel must not use its float4
    tiles there, and gives the same scores and walk as with aligned buffers."""
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    cand, unary, z, anchors, pred, succ = _case(31, 6, 15, 16, 64, 4000)
    args = [to_device(cand), None, to_device(z), to_device(anchors), to_device(pred), to_device(succ)]
    S0, p0 = d.dflash2_score_edges(args[0], to_device(unary), *args[2:])
    flat_u = torch.empty(unary.size + 1, dtype=torch.float32, device="cuda")
    u_off = flat_u[1:].view(unary.shape)
    u_off.copy_(to_device(unary))
    flat_s = torch.empty(S0.numel() + 1, dtype=torch.float32, device="cuda")
    s_off = flat_s[1:].view(S0.shape)
    S1, p1 = d.dflash2_score_edges(args[0], u_off, *args[2:], S=s_off)
    assert d.dflash2_poll_error() == 0
    assert torch.equal(S1, S0)
    assert torch.equal(p1, p0)
