"""GPU parity of the sublayer projections around a conv site (tcgen05 GEMM with the conv fused into
its operand producer or its epilogue, bf16 or affine 4-bit weights) against the float64 oracle."""
import numpy as np
import pytest

from oracle import dflash2_oracle as O
from synth import inputs as I
from tests.parity import REL_TOL, assert_close_scaled, record

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    from tests.gpu_util import require_gpu
    return require_gpu()


def _dev(a):
    from dflash2_block_drafter_gb300.tail import to_device
    return to_device(a)


def _u32(packed):
    import torch
    return torch.from_numpy(packed.view(np.int32)).cuda()


def _gm(t):
    """Scales / biases [N, K/64] -> the library's group-major [K/64, N]."""
    return _dev(np.ascontiguousarray(t.T))


def _bound(a64, W64):
    """fp32 accumulation over K of exact bf16 products, then one bf16 rounding of the output."""
    K = a64.shape[-1]
    s = np.abs(a64) @ np.abs(W64).T
    return K * 2.0 ** -24 * s + 2.0 ** -8 * np.abs(a64 @ W64.T)


def _conv_case(seed, B, G, H, gs):
    n = I.normal(seed, "n", (B * G, H), 1.0)
    d = I.normal(seed, "d", (B * G, 2, 2, H // gs), 0.2, dtype="f32")
    base = np.zeros((2, 2, H), np.float32)
    base[:, 0] = 1.0
    base += I.normal(seed, "base", (2, 2, H), 0.1, dtype="f32")
    return n, d, base


# 1024 x 1024 x 5120 and 2048 x 256 x 4096: stream-K shares over CTA pairs (256-row tiles, pieces
# that straddle tiles and hand their partial sums to the tile's owner); 600 x 512 x 4096: the last
# pair tile has 88 rows, so its second CTA holds no row at all; 1000 x 320 x 2536: a ragged column
# tile (N % 256 = 232) and a ragged row tile under stream-K
@pytest.mark.parametrize("M,K,N", [(16, 256, 256), (300, 512, 264), (1024, 5120, 512), (129, 128, 1000),
                                   (2048, 256, 4096), (1024, 1024, 5120), (600, 512, 4096), (1000, 320, 2536)])
def test_proj_bf16(torch, M, K, N):
    import dflash2_block_drafter_gb300 as d
    a = I.normal(M, "a", (M, K), 1.0)
    W = I.normal(M, "W", (N, K), K ** -0.5)
    y = d.dflash2_proj(_dev(a), _dev(W))
    assert d.dflash2_poll_error() == 0
    got = y.float().cpu().numpy().astype(np.float64)
    ref = O.projection(I.to_f64(a), I.to_f64(W))
    assert_close_scaled(got, ref, what="projection")
    assert np.all(np.abs(got - ref) <= _bound(I.to_f64(a), I.to_f64(W))), "outside the fp32-accumulation bound"


# 1024 rows: the 4-bit weight is dequantised once into the workspace and the bf16 path runs on it
@pytest.mark.parametrize("M,K,N,same_plan", [(48, 256, 128, True), (272, 5120, 520, True), (1024, 512, 5120, True),
                                             (320, 512, 6656, False)])
def test_proj_w4_exact_codes_equal_the_bf16_weight(torch, M, K, N, same_plan):
    """4-bit weights whose scale * q + bias are bf16 values: the dequantised operand is exact, so the
    W4 GEMM equals the bf16 GEMM on that weight bit for bit where both run the same tiles and K
    splits (same accumulation order). At 320 rows the bf16 weight runs in CTA pairs and the 4-bit
    one on single CTAs, whose stream-K shares split K at other k-blocks: there both hold the
    fp32-accumulation bound against the exact product instead."""
    import dflash2_block_drafter_gb300 as d
    q = I.affine4_weight(M + N, "w4", N, K, exact=True)
    W = O.affine_dequantize(q.q, I.to_f64(q.scales), I.to_f64(q.biases))
    W_bf16 = I.round_to_bf16_bits(W.astype(np.float32))
    assert np.array_equal(I.to_f64(W_bf16), W)       # exactly representable
    a_host = I.normal(M, "a", (M, K), 1.0)
    a = _dev(a_host)
    y4 = d.dflash2_proj(a, _u32(q.packed), w_scales=_gm(q.scales), w_biases=_gm(q.biases))
    y16 = d.dflash2_proj(a, _dev(W_bf16))
    assert d.dflash2_poll_error() == 0
    if same_plan:
        assert torch.equal(y4, y16)
    else:
        ref = O.projection(I.to_f64(a_host), W)
        bound = _bound(I.to_f64(a_host), W)
        for y in (y4, y16):
            assert np.all(np.abs(y.float().cpu().numpy().astype(np.float64) - ref) <= bound)


@pytest.mark.parametrize("M,K,N", [(200, 1024, 384), (1000, 512, 4864)])  # split K; stream-K shares on single CTAs
def test_proj_w4_parity(torch, M, K, N):
    import dflash2_block_drafter_gb300 as d
    q = I.affine4_weight(7, "w4", N, K)
    a = I.normal(7, "a", (M, K), 1.0)
    y = d.dflash2_proj(_dev(a), _u32(q.packed), w_scales=_gm(q.scales), w_biases=_gm(q.biases))
    assert d.dflash2_poll_error() == 0
    W = O.affine_dequantize(q.q, I.to_f64(q.scales), I.to_f64(q.biases))
    ref = O.projection(I.to_f64(a), W)
    got = y.float().cpu().numpy().astype(np.float64)
    assert_close_scaled(got, ref, what="W4 projection")
    # the weight is rounded to bf16 once (relative 2^-9) before exact products and fp32 sums
    assert np.all(np.abs(got - ref) <= _bound(I.to_f64(a), W) + 2.0 ** -9 * np.abs(I.to_f64(a)) @ np.abs(W).T)


# 960 and 1024 rows: side 0 applied to the rows once, then the plain projection (CTA pairs, stream-K)
@pytest.mark.parametrize("B,G,H,gs,N", [(2, 16, 256, 16, 256), (9, 16, 5120, 16, 512), (5, 8, 512, 16, 136),
                                        (64, 16, 1024, 16, 4864), (60, 16, 512, 16, 4864), (60, 16, 512, 16, 5120)])
def test_proj_conv_in(torch, B, G, H, gs, N):
    import dflash2_block_drafter_gb300 as d
    n, D, base = _conv_case(B * G, B, G, H, gs)
    W = I.normal(B, "W", (N, H), H ** -0.5)
    d0 = np.ascontiguousarray(D[:, 0].transpose(1, 2, 0))  # side 0's deltas [tap, group, M]
    y = d.dflash2_proj_conv_in(_dev(n), _dev(d0), _dev(base), G, gs, _dev(W))
    assert d.dflash2_poll_error() == 0
    ref = O.sublayer_in(I.to_f64(n).reshape(B, G, H), D.reshape(B, G, 2, 2, -1)[:, :, 0].astype(np.float64),
                        base.astype(np.float64), gs, I.to_f64(W)).reshape(B * G, N)
    rel = assert_close_scaled(y.float().cpu().numpy(), ref, what="conv side 0 + projection")
    record(f"proj conv-in B={B} G={G} H={H} N={N}", max_rel_err=f"{rel:.2e}")
    # identity coefficients: the fused operand is n itself, so the result is the plain GEMM's exactly
    ident = np.zeros((2, 2, H), np.float32)
    ident[0, 0] = 1.0
    y_id = d.dflash2_proj_conv_in(_dev(n), _dev(np.zeros_like(d0)), _dev(ident), G, gs, _dev(W))
    assert torch.equal(y_id, d.dflash2_proj(_dev(n), _dev(W)))


# 1024 and 640 rows: the projection into the workspace, then the finish pass applies side 1 (+ residual)
@pytest.mark.parametrize("B,G,K,H,gs,res", [(2, 16, 256, 256, 16, True), (9, 16, 512, 5120, 16, True),
                                            (12, 8, 128, 96, 8, False), (64, 16, 256, 5120, 16, True),
                                            (40, 16, 512, 1056, 32, False)])
def test_proj_conv_out(torch, B, G, K, H, gs, res):
    import dflash2_block_drafter_gb300 as d
    M = B * G
    a = I.normal(M, "a", (M, K), 1.0)
    W = I.normal(M, "W", (H, K), K ** -0.5)
    d1 = I.normal(M, "d1", (M, 2, H // gs), 0.2)          # bf16 side-1 deltas, as prepare stores them
    base = np.zeros((2, 2, H), np.float32)
    base[:, 0] = 1.0
    base += I.normal(M, "base", (2, 2, H), 0.1, dtype="f32")
    residual = I.normal(M, "res", (M, H), 1.0) if res else None
    out = d.dflash2_proj_conv_out(_dev(a), _dev(W), _dev(d1), _dev(base), G, gs,
                                  residual=_dev(residual) if res else None)
    assert d.dflash2_poll_error() == 0
    ref = O.sublayer_out(I.to_f64(a).reshape(B, G, K), I.to_f64(W), I.to_f64(d1).reshape(B, G, 2, -1),
                         base.astype(np.float64), gs,
                         residual=I.to_f64(residual).reshape(B, G, H) if res else None).reshape(M, H)
    rel = assert_close_scaled(out.float().cpu().numpy(), ref, what="projection + conv side 1 + residual")
    record(f"proj conv-out B={B} G={G} K={K} H={H}", max_rel_err=f"{rel:.2e}")


def test_proj_conv_out_matches_finish_on_an_identity_weight(torch):
    """With W = I the GEMM returns a exactly, so the fused epilogue must agree with
    dflash2_conv_finish on the same rows to one bf16 rounding."""
    import dflash2_block_drafter_gb300 as d
    B, G, H, gs = 4, 16, 256, 16
    M = B * G
    a = I.normal(3, "a", (M, H), 1.0)
    d1 = I.normal(3, "d1", (M, 2, H // gs), 0.2)
    base = np.zeros((2, 2, H), np.float32)
    base[:, 0] = 1.0
    base += I.normal(3, "base", (2, 2, H), 0.1, dtype="f32")
    residual = I.normal(3, "res", (M, H), 1.0)
    eye = I.round_to_bf16_bits(np.eye(H, dtype=np.float32))
    fused = d.dflash2_proj_conv_out(_dev(a), _dev(eye), _dev(d1), _dev(base), G, gs, residual=_dev(residual))
    plain, _ = d.dflash2_conv_finish(_dev(a).view(B, G, H), _dev(d1).view(B, G, 2, H // gs), _dev(base), gs,
                                     residual=_dev(residual).view(B, G, H))
    assert d.dflash2_poll_error() == 0
    f = fused.float().cpu().numpy()
    p = plain.float().cpu().numpy().reshape(M, H)
    assert np.all(np.abs(f - p) <= 2.0 ** -7 * np.maximum(np.abs(f), np.abs(p)) + 1e-6)


def test_fused_site_equals_the_unfused_sequence(torch):
    """One conv site around stand-in projections at the drafter's width, both ways: prepare ->
    projection, projection -> finish (four launches with the conv's output and input in memory)
    against coefficients -> fused input projection, fused output projection."""
    import dflash2_block_drafter_gb300 as d
    B, G, H, gs, N = 8, 16, 5120, 16, 1024
    M = B * G
    site = I.conv_site(11, "site", B, G, H, gs, "bf16")
    x = _dev(I.normal(11, "x", (B, G, H), 1.0))
    w_in = _dev(I.normal(11, "w_in", (N, H), H ** -0.5))
    w_out = _dev(I.normal(11, "w_out", (H, N), N ** -0.5))
    w_kp, base, norm_w = _dev(site.w_kp), _dev(site.base), _dev(site.norm_w)
    # unfused
    a, coef1 = d.dflash2_conv_prepare(x, norm_w, 1e-6, w_kp, base, gs)
    u = d.dflash2_proj(a.view(M, H), w_in)
    ref_out, _ = d.dflash2_conv_finish(d.dflash2_proj(u, w_out).view(B, G, H), coef1, base, gs, residual=x)
    # fused
    n, d0, c1 = d.dflash2_conv_coefficients(x, norm_w, 1e-6, w_kp, gs)
    u2 = d.dflash2_proj_conv_in(n, d0, base, G, gs, w_in)
    out = d.dflash2_proj_conv_out(u2, w_out, c1, base, G, gs, residual=x.view(M, H))
    assert d.dflash2_poll_error() == 0
    assert torch.equal(c1.view(-1), coef1.view(-1))
    assert_close_scaled(u2.float().cpu().numpy(), u.float().cpu().numpy(), rel=1e-2, what="input projection")
    assert_close_scaled(out.float().cpu().numpy(), ref_out.view(M, H).float().cpu().numpy(), rel=1e-2,
                        what="site output")


@pytest.mark.parametrize("B", [4, 40])  # 64 rows, and 640 rows (the weight dequantised once first)
def test_proj_w4_with_both_conv_fusions(torch, B):
    import dflash2_block_drafter_gb300 as d
    G, H, gs, N = 16, 512, 16, 256
    M = B * G
    n, D, base = _conv_case(5, B, G, H, gs)
    q_in = I.affine4_weight(5, "w_in", N, H)
    q_out = I.affine4_weight(5, "w_out", H, N)
    d0 = np.ascontiguousarray(D[:, 0].transpose(1, 2, 0))
    d1 = I.round_to_bf16_bits(np.ascontiguousarray(D[:, 1]))
    u = d.dflash2_proj_conv_in(_dev(n), _dev(d0), _dev(base), G, gs, _u32(q_in.packed), w_scales=_gm(q_in.scales),
                               w_biases=_gm(q_in.biases))
    out = d.dflash2_proj_conv_out(u, _u32(q_out.packed), _dev(d1), _dev(base), G, gs, w_scales=_gm(q_out.scales),
                                  w_biases=_gm(q_out.biases))
    assert d.dflash2_poll_error() == 0
    W_in = O.affine_dequantize(q_in.q, I.to_f64(q_in.scales), I.to_f64(q_in.biases))
    W_out = O.affine_dequantize(q_out.q, I.to_f64(q_out.scales), I.to_f64(q_out.biases))
    u_ref = O.sublayer_in(I.to_f64(n).reshape(B, G, H), D.reshape(B, G, 2, 2, -1)[:, :, 0].astype(np.float64),
                          base.astype(np.float64), gs, W_in)
    assert_close_scaled(u.float().cpu().numpy(), u_ref.reshape(M, N), what="W4 conv-in")
    # the output side on the GPU's own (bf16) u, as the next GEMM sees it
    out_ref = O.sublayer_out(u.float().cpu().numpy().astype(np.float64).reshape(B, G, N), W_out,
                             I.to_f64(d1).reshape(B, G, 2, -1), base.astype(np.float64), gs)
    assert_close_scaled(out.float().cpu().numpy(), out_ref.reshape(M, H), what="W4 conv-out")


@pytest.mark.parametrize("M,K,N", [(1, 64, 8), (5, 320, 136), (128, 5120, 256), (16, 5120, 5120)])
def test_proj_small_rows_bf16_and_w4(torch, M, K, N):
    """The small-row kernel at its edges: one row (15 zero-filled MMA columns), a K of five
    k-blocks (a partial 4-bit stage), a weight-row count that is not a multiple of the 128-row tile,
    the full 128 rows, and the drafter's width. bf16 within the fp32-accumulation bound; 4-bit
    against the dequantised weight; exact codes equal the bf16 weight bit for bit."""
    import dflash2_block_drafter_gb300 as d
    a = I.normal(M + K, "a", (M, K), 1.0)
    W = I.normal(M + K, "W", (N, K), K ** -0.5)
    y = d.dflash2_proj(_dev(a), _dev(W))
    assert d.dflash2_poll_error() == 0
    got = y.float().cpu().numpy().astype(np.float64)
    ref = O.projection(I.to_f64(a), I.to_f64(W))
    assert np.all(np.abs(got - ref) <= _bound(I.to_f64(a), I.to_f64(W))), "outside the fp32-accumulation bound"
    q = I.affine4_weight(M + N, "w4", N, K)
    y4 = d.dflash2_proj(_dev(a), _u32(q.packed), w_scales=_gm(q.scales), w_biases=_gm(q.biases))
    assert d.dflash2_poll_error() == 0
    W4 = O.affine_dequantize(q.q, I.to_f64(q.scales), I.to_f64(q.biases))
    got4 = y4.float().cpu().numpy().astype(np.float64)
    ref4 = O.projection(I.to_f64(a), W4)
    assert np.all(np.abs(got4 - ref4) <= _bound(I.to_f64(a), W4) + 2.0 ** -9 * np.abs(I.to_f64(a)) @ np.abs(W4).T)
    qe = I.affine4_weight(M + N + 1, "w4e", N, K, exact=True)
    We = I.round_to_bf16_bits(O.affine_dequantize(qe.q, I.to_f64(qe.scales), I.to_f64(qe.biases)).astype(np.float32))
    ye = d.dflash2_proj(_dev(a), _u32(qe.packed), w_scales=_gm(qe.scales), w_biases=_gm(qe.biases))
    assert torch.equal(ye, d.dflash2_proj(_dev(a), _dev(We)))
    assert d.dflash2_poll_error() == 0


def test_stream_k_hand_off_repeats_in_a_graph(torch):
    """Stream-K shares hand partial tiles to the tile owners through flags that the owners reset:
    the same projections launched back to back and replayed from a CUDA graph give the same bits
    every time (the plain projection on CTA pairs and the 4-bit one on single CTAs)."""
    import dflash2_block_drafter_gb300 as d
    M, K, N = 1000, 512, 4096
    a = _dev(I.normal(11, "a", (M, K), 1.0))
    W = _dev(I.normal(11, "W", (N, K), K ** -0.5))
    q = I.affine4_weight(11, "w4", N, K)
    codes, sc, bi = _u32(q.packed), _gm(q.scales), _gm(q.biases)
    out16 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out4 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(d.library().dflash2_proj_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    d.dflash2_proj(a, W, out=out16, workspace=ws)
    d.dflash2_proj(a, codes, w_scales=sc, w_biases=bi, out=out4, workspace=ws)
    torch.cuda.synchronize()
    assert d.dflash2_poll_error() == 0
    ref16, ref4 = out16.clone(), out4.clone()
    for _ in range(3):
        d.dflash2_proj(a, W, out=out16, workspace=ws)
        d.dflash2_proj(a, codes, w_scales=sc, w_biases=bi, out=out4, workspace=ws)
    torch.cuda.synchronize()
    assert d.dflash2_poll_error() == 0
    assert torch.equal(out16, ref16) and torch.equal(out4, ref4)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        d.dflash2_proj(a, W, out=out16, workspace=ws)
        d.dflash2_proj(a, codes, w_scales=sc, w_biases=bi, out=out4, workspace=ws)
    for _ in range(3):
        out16.zero_()
        out4.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert d.dflash2_poll_error() == 0
        assert torch.equal(out16, ref16) and torch.equal(out4, ref4)
