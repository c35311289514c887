"""GPU parity of the head over a draft vocabulary (dflash2_head_topk_vocab) against the oracle."""
import numpy as np
import pytest

from oracle import dflash2_oracle as O
from synth import inputs as I
from tests.gpu_util import dev_f64, require_gpu
from tests.parity import REL_TOL, assert_close_scaled, compare_topk, compare_walk, record, scale_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


def _listed_run(wl, S, want_logits=False):
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    h = to_device(wl.h).reshape(-1, wl.H)
    w = to_device(wl.w_head)
    ids = to_device(S)
    w_listed = w.index_select(0, ids.long()).contiguous()
    bias = to_device(wl.bias).index_select(0, ids.long()).contiguous() if wl.bias is not None else None
    cand, unary, z, logits = d.dflash2_head_topk_vocab(h, w_listed, ids, wl.K, bias_listed=bias,
                                                       w_proj=to_device(wl.w_proj), want_logits=want_logits)
    assert d.dflash2_poll_error() == 0
    return cand.cpu().numpy(), unary.cpu().numpy(), dev_f64(z), (dev_f64(logits) if want_logits else None)


@pytest.mark.parametrize("B,V,n_listed,bias", [(6, 6000, 1500, True), (1, 5000, 777, False)])
def test_listed_head_parity(torch, B, V, n_listed, bias):
    wl = I.selector_case(500 + B, B=B, G=16, H=512, V=V, K=16, R=64, bias=bias)
    S = I.draft_vocabulary(500 + B, V, n_listed)
    cand, unary, z, logits = _listed_run(wl, S, want_logits=True)
    h = I.to_f64(wl.h).reshape(-1, wl.H)
    Wl = I.to_f64(wl.w_head)[S]
    ref = O.head_logits(h, Wl, wl.bias[S] if wl.bias is not None else None)
    assert_close_scaled(logits, ref, what="listed logits")
    # the ids the GPU returns are token ids: map them back to listed columns for the comparison
    col_of = {int(t): i for i, t in enumerate(S)}
    cols = np.vectorize(col_of.__getitem__)(cand)
    near = compare_topk(cols, unary, ref, wl.K, REL_TOL * scale_of(ref))
    bound = (wl.H * 2.0 ** -24) * float(np.max(np.abs(h) @ np.abs(Wl).T))
    tight = compare_topk(cols, unary, ref, wl.K, bound)
    ref_cols, _ = O.top_k(ref, wl.K)
    ref_ids = O.listed_candidates(ref_cols, S)
    decided = O.kth_margin(ref, wl.K) > 4 * bound
    for r in np.where(decided)[0]:
        assert set(cand[r].tolist()) == set(ref_ids[r].tolist())
    record(f"listed head M={h.shape[0]} V_listed={len(S)}", near_tie_rows=near, near_tie_rows_arith_bound=tight,
           rows=h.shape[0])


def test_identity_vocabulary_equals_full_head(torch):
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    wl = I.selector_case(77, B=5, G=16, H=256, V=3000, K=16, R=64, bias=True)
    h = to_device(wl.h).reshape(-1, wl.H)
    w = to_device(wl.w_head)
    ids = torch.arange(wl.V, dtype=torch.int32, device="cuda")
    a = d.dflash2_head_topk(h, w, 16, bias=to_device(wl.bias), w_proj=to_device(wl.w_proj))
    b = d.dflash2_head_topk_vocab(h, w, ids, 16, bias_listed=to_device(wl.bias), w_proj=to_device(wl.w_proj))
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x, y)


def test_listed_head_drafter_shape_feeds_the_walk(torch):
    """V = 248320 head restricted to a 32768-token draft vocabulary; the mapped token ids drive the
    codebook gathers of the selector (teacher-forced walk against the oracle)."""
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    wl = I.make_config(3, B=4)
    S = I.draft_vocabulary(3, wl.V, 32768)
    cand, unary, z, _ = _listed_run(wl, S)
    assert np.all(np.isin(cand, S))
    h = I.to_f64(wl.h).reshape(-1, wl.H)
    ref = O.head_logits(h, I.to_f64(wl.w_head[S]), wl.bias[S])
    col_of = {int(t): i for i, t in enumerate(S)}
    cols = np.vectorize(col_of.__getitem__)(cand)
    compare_topk(cols, unary, ref, wl.K, REL_TOL * scale_of(ref))
    B, steps, K = wl.B, wl.steps, wl.K
    S_gpu, path = d.dflash2_score_edges(to_device(cand.reshape(B, steps, K)), to_device(unary.reshape(B, steps, K)),
                                        to_device(z.reshape(B, steps, wl.R).astype(np.float32)),
                                        to_device(wl.anchors), to_device(wl.pred_book), to_device(wl.succ_book))
    assert d.dflash2_poll_error() == 0
    rS = O.score_edges(cand.reshape(B, steps, K), unary.reshape(B, steps, K), z.reshape(B, steps, wl.R), wl.anchors,
                       I.f64_view(wl.pred_book), I.f64_view(wl.succ_book))
    assert_close_scaled(S_gpu.cpu().numpy(), rS, what="S over listed candidates")
    rpath, rpos = O.select_path(rS, cand.reshape(B, steps, K))
    compare_walk(path.cpu().numpy(), rS, rpos, cand.reshape(B, steps, K), REL_TOL * scale_of(rS))
    assert np.all(np.isin(path.cpu().numpy(), S))
