"""GPU parity of the two-tap dynamic grouped conv (prepare / finish) against the float64 oracle."""
import numpy as np
import pytest

from oracle import dflash2_oracle as O
from synth import inputs as I
from tests.gpu_util import dev_f64, oracle_sites, require_gpu
from tests.parity import REL_TOL, assert_close_scaled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return require_gpu()


def _dev(torch, a):
    from dflash2_block_drafter_gb300.tail import to_device
    return to_device(a)


def _site_dev(torch, s):
    return _dev(torch, s.w_kp), _dev(torch, s.base), _dev(torch, s.norm_w)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,G,H,gs", [
    (1, 8, 256, 16), (3, 16, 512, 16), (5, 7, 320, 16), (2, 16, 1024, 32),
    # above 128 rows kernel_projection runs on CTA pairs: a ragged second row group (144 rows),
    # G = 64 (320 rows), and 260 rows with 48 groups (N = 192: half a column unit past the end)
    (9, 16, 512, 16), (5, 64, 256, 16), (20, 13, 384, 8),
    # the streamed / fused passes at their limits: G = 2 (smallest), G = 32 (largest fused
    # finish), G = 33 (falls back to the side-1 pass and a separate norm), group 64 (the
    # coefficient tiles are too narrow for TMA: per-thread passes)
    (4, 2, 512, 16), (3, 32, 512, 16), (2, 33, 512, 16), (2, 16, 512, 64),
    # CTA pairs: 320 columns (two and a half units) over 160 rows, and two row groups with
    # group 32 where the second group's peer CTA has no rows
    (10, 16, 1280, 16), (10, 30, 1024, 32)])
def test_prepare_finish_parity(torch, dtype, B, G, H, gs):
    import dflash2_block_drafter_gb300 as d
    wl = I.conv_case(100 + B * G + H, B, G, H, gs, dtype=dtype)
    s = wl.sites[0]
    x = _dev(torch, wl.x0)
    w_kp, base, norm_w = _site_dev(torch, s)
    groups = H // gs
    d_full = torch.empty((B, G, 2, 2, groups), dtype=torch.float32, device="cuda")
    a, coef1 = d.dflash2_conv_prepare(x, norm_w, wl.eps, w_kp, base, gs, d_full=d_full)
    nxt = torch.empty((B, G, H), dtype=x.dtype, device="cuda")
    out, _ = d.dflash2_conv_finish(_dev(torch, s.y), coef1, base, gs, residual=x, next_norm_w=norm_w, eps=wl.eps,
                                   next_n=nxt)
    assert d.dflash2_poll_error() == 0
    os_ = oracle_sites(wl)[0]
    ra, rd1, rn = O.conv_prepare(I.to_f64(wl.x0), os_.norm_w, wl.eps, os_.w_kp, os_.base, gs)
    rD = O.kernel_projection(rn, os_.w_kp)
    rx = O.conv_finish(os_.y, rd1, os_.base, gs, residual=I.to_f64(wl.x0))
    assert_close_scaled(dev_f64(d_full), rD, what="D")
    assert_close_scaled(dev_f64(a), ra, what="prepare out")
    assert_close_scaled(dev_f64(coef1), rd1, what="coef1")
    assert_close_scaled(dev_f64(out), rx, what="finish out")
    assert_close_scaled(dev_f64(nxt), O.rms_norm(rx, os_.norm_w, wl.eps), what="next norm")
    # the stated bound is loose for a single site: hold the fp32 path to a much tighter one
    if dtype == "f32":
        assert_close_scaled(dev_f64(out), rx, rel=2e-3, what="finish out (f32)")


@pytest.mark.parametrize("B", [4, 12])  # 64 rows (single-CTA GEMM) and 192 rows (CTA pairs)
def test_identity_and_shift_bit_exact(torch, B):
    import dflash2_block_drafter_gb300 as d
    G, H, gs = 16, 512, 16
    wl = I.conv_case(3, B, G, H, gs)
    x = _dev(torch, wl.x0)
    w0 = torch.zeros((4 * H // gs, H), dtype=torch.bfloat16, device="cuda")
    ident = torch.zeros((2, 2, H), dtype=torch.float32, device="cuda")
    ident[:, 0] = 1.0
    a, coef1 = d.dflash2_conv_prepare(x, None, 1e-6, w0, ident, gs)
    assert torch.equal(a, x)
    assert torch.count_nonzero(coef1.float()) == 0
    y = _dev(torch, wl.sites[0].y)
    out, _ = d.dflash2_conv_finish(y, coef1, ident, gs)
    assert torch.equal(out, y)
    shift = torch.zeros((2, 2, H), dtype=torch.float32, device="cuda")
    shift[:, 1] = 1.0
    a, coef1 = d.dflash2_conv_prepare(x, None, 1e-6, w0, shift, gs)
    assert torch.count_nonzero(a[:, 0].float()) == 0
    assert torch.equal(a[:, 1:], x[:, :-1])
    out, _ = d.dflash2_conv_finish(y, coef1, shift, gs)
    assert torch.equal(out[:, 1:], y[:, :-1])
    assert torch.count_nonzero(out[:, 0].float()) == 0


def test_block_isolation_on_gpu(torch):
    import dflash2_block_drafter_gb300 as d
    B, G, H, gs = 6, 16, 512, 16
    wl = I.conv_case(5, B, G, H, gs)
    s = wl.sites[0]
    w_kp, base, norm_w = _site_dev(torch, s)
    x = _dev(torch, wl.x0)
    y = _dev(torch, s.y)
    a1, c1 = d.dflash2_conv_prepare(x, norm_w, wl.eps, w_kp, base, gs)
    o1, _ = d.dflash2_conv_finish(y, c1, base, gs, residual=x)
    x2, y2 = x.clone(), y.clone()
    x2[3] = -x2[3] * 2
    y2[3] = y2[3] + 1
    a2, c2 = d.dflash2_conv_prepare(x2, norm_w, wl.eps, w_kp, base, gs)
    o2, _ = d.dflash2_conv_finish(y2, c2, base, gs, residual=x2)
    keep = [0, 1, 2, 4, 5]
    assert torch.equal(a1[keep], a2[keep])
    assert torch.equal(o1[keep], o2[keep])
    assert not torch.equal(a1[3], a2[3])


@pytest.mark.parametrize("B,G", [(64, 16), (60, 15), (17, 16)])
def test_prepare_drafter_shape_every_row(torch, B, G):
    """kernel_projection + side 0 at H=5120 over every row: 1024 rows (four pair row groups, K
    split in two), 900 rows (a ragged last row group, blocks of 15 straddling the 256-row groups)
    and 272 rows."""
    import dflash2_block_drafter_gb300 as d
    H, gs = 5120, 16
    wl = I.conv_case(7 + B, B, G, H, gs)
    s = wl.sites[0]
    x = _dev(torch, wl.x0)
    w_kp, base, norm_w = _site_dev(torch, s)
    d_full = torch.empty((B, G, 2, 2, H // gs), dtype=torch.float32, device="cuda")
    a, coef1 = d.dflash2_conv_prepare(x, norm_w, wl.eps, w_kp, base, gs, d_full=d_full)
    assert d.dflash2_poll_error() == 0
    os_ = oracle_sites(wl)[0]
    ra, rd1, rn = O.conv_prepare(I.to_f64(wl.x0), os_.norm_w, wl.eps, os_.w_kp, os_.base, gs)
    assert_close_scaled(dev_f64(d_full), O.kernel_projection(rn, os_.w_kp), what="D")
    assert_close_scaled(dev_f64(a), ra, what="prepare out")
    assert_close_scaled(dev_f64(coef1), rd1, what="coef1")
    # the coefficients-only entry computes the same D in the same order
    _, d0, c1b = d.dflash2_conv_coefficients(x, norm_w, wl.eps, w_kp, gs)
    assert d.dflash2_poll_error() == 0
    assert torch.equal(c1b.reshape(-1), coef1.reshape(-1))
    assert torch.equal(d0.permute(2, 0, 1).reshape(B, G, 2, H // gs), d_full[:, :, 0])


@pytest.mark.parametrize("B", [1, 8])
def test_conv_chain_drafter_shape(torch, B):
    """The ten-site chain at H=5120, G=16, group 16, compared over every block."""
    from dflash2_block_drafter_gb300.tail import TailRunner, to_device
    wl = I.make_config(1, B=B)
    run = TailRunner(wl)
    x = run.conv_chain(to_device(wl.x0), [to_device(s.y) for s in wl.sites], emit_h=False)
    got = dev_f64(x)
    import dflash2_block_drafter_gb300 as d
    assert d.dflash2_poll_error() == 0
    ref, _ = O.conv_chain(I.to_f64(wl.x0), oracle_sites(wl), wl.eps, wl.gs)
    assert_close_scaled(got, ref, what=f"chain B={B}")


def test_conv_chain_b64_sampled_blocks(torch):
    """B=64 at drafter shape; blocks never interact, so the oracle runs on three sampled blocks."""
    from dflash2_block_drafter_gb300.tail import TailRunner, to_device
    wl = I.make_config(1, B=64)
    run = TailRunner(wl)
    x = run.conv_chain(to_device(wl.x0), [to_device(s.y) for s in wl.sites], emit_h=False)
    got = dev_f64(x)
    blocks = [0, 37, 63]
    ref, _ = O.conv_chain(I.to_f64(wl.x0)[blocks], oracle_sites(wl, blocks), wl.eps, wl.gs)
    assert_close_scaled(got[blocks], ref, what="chain B=64 (sampled)")
    assert np.all(np.isfinite(got))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("B,G,H,gs", [(1, 16, 5120, 16), (3, 7, 320, 16), (8, 16, 1024, 32), (9, 16, 512, 16)])
def test_conv_coefficients_parity(torch, dtype, B, G, H, gs):
    """Prepare without the side-0 output: side 0's deltas [tap][group][row] (fp32) and side 1's
    [row][tap][group] against the oracle's kernel_projection of the normed rows, and the normed
    rows themselves. Up to 128 bf16 rows this is the small-row kernel's coefficients-only mode,
    else the split-K GEMM and its reduce pass."""
    import dflash2_block_drafter_gb300 as d
    wl = I.conv_case(300 + B * G + H, B, G, H, gs, dtype=dtype)
    s = wl.sites[0]
    x = _dev(torch, wl.x0)
    w_kp, base, norm_w = _site_dev(torch, s)
    n, d0, c1 = d.dflash2_conv_coefficients(x, norm_w, wl.eps, w_kp, gs)
    assert d.dflash2_poll_error() == 0
    os_ = oracle_sites(wl)[0]
    _, _, rn = O.conv_prepare(I.to_f64(wl.x0), os_.norm_w, wl.eps, os_.w_kp, os_.base, gs)
    rD = O.kernel_projection(rn, os_.w_kp).reshape(B * G, 2, 2, H // gs)
    assert_close_scaled(dev_f64(n).reshape(B, G, H), rn, what="normed rows")
    assert_close_scaled(dev_f64(d0), np.ascontiguousarray(rD[:, 0].transpose(1, 2, 0)), what="side-0 deltas")
    assert_close_scaled(dev_f64(c1), rD[:, 1], what="side-1 deltas")
    # the same deltas prepare computes, bit for bit (one kernel_projection per shape)
    _, coef1 = d.dflash2_conv_prepare(x, norm_w, wl.eps, w_kp, base, gs)
    assert torch.equal(coef1.reshape(-1), c1.reshape(-1))
