"""GPU parity of the head GEMM with fused top-K and hidden_projection against the float64 oracle."""
import numpy as np
import pytest

from oracle import dflash2_oracle as O
from synth import inputs as I
from tests.gpu_util import dev_f64, require_gpu
from tests.parity import REL_TOL, assert_close_scaled, compare_topk, record, scale_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


def _arith_bound(abs_products, H, dtype):
    """max over entries of c * sum_k |h_k w_k|, c = H * 2^-24 (+ 2^-10 for tf32 operands)."""
    c = H * 2.0 ** -24 + (2.0 ** -10 if dtype == "f32" else 0.0)
    return c * float(np.max(abs_products))


def _run(wl, want_logits=False, K=None):
    import dflash2_block_drafter_gb300 as d
    from dflash2_block_drafter_gb300.tail import to_device
    K = wl.K if K is None else K
    h = to_device(wl.h).reshape(-1, wl.H)
    bias = to_device(wl.bias) if wl.bias is not None else None
    cand, unary, z, logits = d.dflash2_head_topk(h, to_device(wl.w_head), K, bias=bias, w_proj=to_device(wl.w_proj),
                                                 want_logits=want_logits)
    assert d.dflash2_poll_error() == 0
    return cand.cpu().numpy(), unary.cpu().numpy(), dev_f64(z), (dev_f64(logits) if want_logits else None)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,G,H,V,R,bias", [
    (1, 16, 512, 4096, 64, False),     # one M tile, 64 chunks
    (20, 16, 512, 5000, 64, True),     # 300 rows (2 x 256-row groups, ragged), ragged vocab tail
    (9, 8, 256, 1234, 16, False),      # 63 rows, R = 16 (partial extra chunk)
])
def test_head_topk_parity(torch, dtype, B, G, H, V, R, bias):
    wl = I.selector_case(11 + B + V, B=B, G=G, H=H, V=V, K=16, R=R, dtype=dtype, bias=bias)
    _check_head(wl, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("M,V,R", [
    (129, 3001, 128),   # one row past a 128-row tile; vocabulary ends inside a 128-column unit
    (257, 1000, 192),   # one row past a 256-row group; fewer column units than CTA pairs; 1.5 units of z
    (513, 9000, 16),    # ragged third group; z narrower than a chunk
    (1024, 2500, 64),   # four full groups; units not a multiple of the column ranges
    (128, 4096, 64),    # the largest single-CTA head
    (256, 4096, 64),    # exactly one CTA-pair row group
])
def test_head_topk_row_and_column_edges(torch, dtype, M, V, R):
    """Row counts just past the 128- and 256-row boundaries of the head's tiles (some CTAs hold a
    single valid row or none), ragged vocabularies and hidden_projection widths."""
    wl = I.selector_case(40 + M, B=M, G=2, H=256, V=V, K=16, R=R, dtype=dtype, bias=True)
    _check_head(wl, dtype)


def _check_head(wl, dtype):
    H = wl.H
    cand, unary, z, logits = _run(wl, want_logits=True)
    h = I.to_f64(wl.h).reshape(-1, H)
    W = I.to_f64(wl.w_head)
    ref = O.head_logits(h, W, wl.bias)
    tol = REL_TOL * scale_of(ref)
    assert_close_scaled(logits, ref, what="logits")
    assert_close_scaled(z, O.hidden_projection(h, I.to_f64(wl.w_proj)), what="z")
    near = compare_topk(cand, unary, ref, wl.K, tol)
    # The stated margin is loose. The arithmetic gives a much tighter bound: bf16 products are exact
    # in fp32 and a K-term fp32 sum errs by at most K * 2^-24 * sum|h w|; tf32 (f32 storage) adds a
    # relative 2^-10 per product. Every logit must sit inside that bound, and every row whose
    # K-th/(K+1)-th gap exceeds 4x the bound must give exactly the oracle's ids.
    bound = _arith_bound(np.abs(h) @ np.abs(W).T, H, dtype)
    assert np.max(np.abs(logits - ref)) <= bound, "logits outside the fp32-accumulation bound"
    tight = compare_topk(cand, unary, ref, wl.K, bound)
    record(f"head {dtype} M={h.shape[0]} V={wl.V}", near_tie_rows=near, near_tie_rows_arith_bound=tight,
           rows=h.shape[0])
    # the unary values equal the logits the same kernel reported (no second rounding)
    np.testing.assert_array_equal(unary, np.take_along_axis(logits, cand.astype(np.int64), axis=1).astype(np.float32))


def test_zero_head_tie_rule(torch):
    import dflash2_block_drafter_gb300 as d
    H, V, M = 256, 3000, 40
    h = torch.randn(M, H, device="cuda").to(torch.bfloat16)
    w = torch.zeros(V, H, dtype=torch.bfloat16, device="cuda")
    cand, unary, _, _ = d.dflash2_head_topk(h, w, 16)
    assert torch.equal(cand.cpu(), torch.arange(16, dtype=torch.int32).repeat(M, 1))
    assert torch.count_nonzero(unary) == 0


def test_k1_is_argmax(torch):
    wl = I.selector_case(21, B=4, G=16, H=512, V=7000, K=16, R=64)
    cand, unary, _, logits = _run(wl, want_logits=True, K=1)
    np.testing.assert_array_equal(cand[:, 0], np.argmax(logits, axis=1))


@pytest.mark.parametrize("cfg,rows", [(2, None), (3, [0, 1, 77, 200, 479])])
def test_head_topk_drafter_shape(torch, cfg, rows):
    """V = 248320, H = 5120: every row at B=1, sampled rows at B=32 (Zipf bias)."""
    wl = I.make_config(cfg)
    cand, unary, z, _ = _run(wl)
    h = I.to_f64(wl.h).reshape(-1, wl.H)
    sel = np.arange(h.shape[0]) if rows is None else np.array(rows)
    W = I.f64_view(wl.w_head)
    ref = O.head_logits(h[sel], W, wl.bias)
    tol = REL_TOL * scale_of(ref)
    near = compare_topk(cand[sel], unary[sel], ref, wl.K, tol)
    # arithmetic bound (see test_head_topk_parity), sum |h w| taken slab by slab
    mx = 0.0
    for v0 in range(0, wl.V, 16384):
        mx = max(mx, float(np.max(np.abs(h[sel]) @ np.abs(W[v0:v0 + 16384]).T)))
    bound = _arith_bound(np.array([mx]), wl.H, "bf16")
    tight = compare_topk(cand[sel], unary[sel], ref, wl.K, bound)
    record(f"head drafter shape config {cfg}", near_tie_rows=near, near_tie_rows_arith_bound=tight, rows=len(sel))
    assert_close_scaled(z[sel], O.hidden_projection(h[sel], I.to_f64(wl.w_proj)), what="z")
