"""Host-side checks of the C ABI that need no GPU: the library builds and loads, exports every
symbol include/dflash2.h declares, and rejects bad arguments before launching anything."""
import ctypes
import os
import re
import subprocess

import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "dflash2.h")


@pytest.fixture(scope="module")
def lib():
    from dflash2_block_drafter_gb300 import _build
    import dflash2_block_drafter_gb300 as pkg
    _build.build()
    return pkg.library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DFLASH2_API\s+[\w\s\*]+?\b(dflash2_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("dflash2_conv_prepare", "dflash2_conv_finish", "dflash2_head_topk", "dflash2_score_edges",
                     "dflash2_select_path"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from dflash2_block_drafter_gb300 import library_path
    out = subprocess.run(["nm", "-D", "--defined-only", library_path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(dflash2_\w+)", out))
    for name in declared_symbols():
        assert name in exported, f"{name} declared in dflash2.h but not exported"
        assert hasattr(lib, name)
    # nothing else leaks out of the library's namespace
    assert all(n.startswith("dflash2_") for n in exported)


def test_status_strings_and_version(lib):
    assert lib.dflash2_version() == 100
    assert lib.dflash2_status_string(0) == b"DFLASH2_OK"
    assert lib.dflash2_status_string(-1) == b"DFLASH2_ERR_INVALID_ARG"
    assert lib.dflash2_status_string(-5) == b"DFLASH2_ERR_TIMEOUT"
    assert lib.dflash2_status_string(12345) == b"DFLASH2_ERR_UNKNOWN"


FAKE = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced: validation fails first
FAKE_MIS = ctypes.c_void_p(0x10008)  # misaligned


def _prep(lib, **kw):
    a = dict(x=FAKE, norm_w=None, eps=1e-6, w_kp=FAKE, base=FAKE, B=1, G=16, H=5120, gs=16, taps=2, dtype=0,
             out=FAKE, coef1=FAKE, d_full=None, ws=FAKE, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.dflash2_conv_prepare(a["x"], a["norm_w"], a["eps"], a["w_kp"], a["base"], a["B"], a["G"], a["H"],
                                    a["gs"], a["taps"], a["dtype"], a["out"], a["coef1"], a["d_full"], a["ws"],
                                    a["ws_bytes"], a["stream"])


def test_conv_prepare_rejects_bad_arguments(lib):
    assert _prep(lib, taps=3) == -2                      # two-tap only
    assert _prep(lib, G=1) == -1                         # no zero-draft-row blocks
    assert _prep(lib, G=65) == -1
    assert _prep(lib, H=5000) == -1                      # H % 64
    assert _prep(lib, gs=12) == -1                       # group size % 8
    assert _prep(lib, gs=24, H=5120) == -1               # H % group size
    assert _prep(lib, B=0) == -1
    assert _prep(lib, dtype=7) == -1
    assert _prep(lib, x=None) == -1
    assert _prep(lib, x=FAKE_MIS) == -1
    assert _prep(lib, ws=ctypes.c_void_p(0x10010)) == -1  # workspace not 256-aligned
    assert _prep(lib, ws_bytes=16) == -4                  # workspace too small
    assert b"workspace" in lib.dflash2_last_error_message()


def test_conv_finish_rejects_bad_arguments(lib):
    f = lib.dflash2_conv_finish
    assert f(FAKE, FAKE, FAKE, 1, 16, 5120, 16, 2, 0, None, FAKE, FAKE, 1e-6, None, 0, None) == -1  # half a norm pair
    assert f(FAKE, FAKE, FAKE, 1, 16, 5120, 16, 2, 0, None, FAKE, FAKE, 1e-6, FAKE, 16, None) == -1  # next_row0 >= G
    assert f(FAKE, FAKE, FAKE, 1, 16, 5120, 16, 3, 0, None, FAKE, None, 1e-6, None, 0, None) == -2
    assert f(None, FAKE, FAKE, 1, 16, 5120, 16, 2, 0, None, FAKE, None, 1e-6, None, 0, None) == -1
    assert f(FAKE, FAKE, FAKE, 1, 16, 5120, 16, 2, 0, FAKE_MIS, FAKE, None, 1e-6, None, 0, None) == -1


def test_head_topk_rejects_bad_arguments(lib):
    f = lib.dflash2_head_topk
    ok = dict(h=FAKE, M=15, H=5120, w=FAKE, V=248320, bias=None, wp=FAKE, R=64, K=16, dt=0, cand=FAKE, unary=FAKE,
              z=FAKE, logits=None, ws=FAKE, wsb=0, st=None)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(a["h"], a["M"], a["H"], a["w"], a["V"], a["bias"], a["wp"], a["R"], a["K"], a["dt"], a["cand"],
                 a["unary"], a["z"], a["logits"], a["ws"], a["wsb"], a["st"])
    assert call(K=17) == -1
    assert call(K=0) == -1
    assert call(V=8) == -1        # K > V
    assert call(M=0) == -1
    assert call(H=100) == -1
    assert call(R=24) == -1       # R % 16
    assert call(z=None) == -1     # w_proj without z
    assert call(h=FAKE_MIS) == -1
    assert call() == -4           # workspace too small
    assert lib.dflash2_head_topk_workspace_bytes(15, 5120, 248320, 16, 64) > 0


def test_score_edges_and_walk_reject_bad_arguments(lib):
    f = lib.dflash2_score_edges
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 15, 16, 64, 1000, 0, None, None, None) == -1  # no output
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 15, 33, 64, 1000, 0, FAKE, None, None) == -1  # K > 32
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, 16, 64, 1000, 0, FAKE, None, None) == -1  # steps > 63
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 15, 16, 60, 1000, 0, FAKE, None, None) == -1  # R % 8
    assert f(FAKE, FAKE, FAKE_MIS, FAKE, FAKE, FAKE, 1, 15, 16, 64, 1000, 0, FAKE, None, None) == -1
    g = lib.dflash2_select_path
    assert g(FAKE, FAKE, 1, 15, 0, FAKE, None) == -1
    assert g(None, FAKE, 1, 15, 16, FAKE, None) == -1
    assert lib.dflash2_selftest_bounded_wait(0, None) == -1
    assert lib.dflash2_selftest_bounded_wait(2000000, None) == -1


def test_binding_requires_cuda_tensors(lib):
    import torch
    import dflash2_block_drafter_gb300 as d
    x = torch.zeros(1, 16, 64, dtype=torch.bfloat16)
    with pytest.raises((ValueError, RuntimeError)):
        d.dflash2_conv_finish(x, torch.zeros(1, 16, 2, 4, dtype=torch.bfloat16), torch.zeros(2, 2, 64), 16)


def test_head_topk_vocab_rejects_bad_arguments(lib):
    f = lib.dflash2_head_topk_vocab
    #          h    M   H     w    V     ids   bias  wp    R   K   dt cand  un    z     lg    ws   wsb st
    assert f(FAKE, 15, 5120, FAKE, 1000, None, None, FAKE, 64, 16, 0, FAKE, FAKE, FAKE, None, FAKE, 0, None) == -1
    assert f(FAKE, 15, 5120, FAKE, 8, FAKE, None, FAKE, 64, 16, 0, FAKE, FAKE, FAKE, None, FAKE, 0, None) == -1
    assert f(FAKE, 15, 5120, FAKE, 1000, FAKE, None, FAKE, 64, 16, 0, FAKE, FAKE, FAKE, None, FAKE, 0, None) == -4


def test_mixed_depth_walk_rejects_bad_arguments(lib):
    f = lib.dflash2_score_edges_depths
    #        cand  un    z     anch  pred  succ  depths B  st  K   R   V     dt S     path  stream
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 15, 16, 64, 1000, 0, None, FAKE, None) == -1  # no depths
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 15, 16, 64, 1000, 0, FAKE, None, None) == -1  # no path
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, 16, 64, 1000, 0, None, FAKE, None) == -1  # steps > 63
    assert b"depths" in lib.dflash2_last_error_message() or b"steps" in lib.dflash2_last_error_message()
    g = lib.dflash2_select_path_depths
    assert g(FAKE, FAKE, None, 1, 15, 16, FAKE, None) == -1
    assert g(FAKE, FAKE, FAKE, 1, 15, 33, FAKE, None) == -1


def test_launch_count_queries(lib):
    bf16, f32 = 0, 1
    # drafter shape: prepare = kernel_projection + side-0 pass (+ the first site's norm)
    assert lib.dflash2_conv_prepare_launches(64, 16, 5120, 16, bf16, 0) == 2
    assert lib.dflash2_conv_prepare_launches(64, 16, 5120, 16, bf16, 1) == 3
    # finish with the next norm is one fused kernel where its tiles fit
    assert lib.dflash2_conv_finish_launches(64, 16, 5120, 16, bf16, 1) == 1
    assert lib.dflash2_conv_finish_launches(64, 16, 5120, 16, bf16, 0) == 1
    # up to 128 bf16 rows: kernel_projection and the side-0 pass in one kernel
    assert lib.dflash2_conv_prepare_launches(1, 16, 5120, 16, bf16, 0) == 1
    assert lib.dflash2_conv_prepare_launches(8, 16, 5120, 16, bf16, 1) == 2
    assert lib.dflash2_conv_prepare_launches(9, 16, 5120, 16, bf16, 0) == 2
    assert lib.dflash2_conv_prepare_launches(1, 16, 5120, 16, f32, 0) == 2
    # up to 256 rows: finish and the next norm in one row-per-CTA kernel, whatever H and G
    assert lib.dflash2_conv_finish_launches(5, 7, 320, 16, bf16, 1) == 1
    assert lib.dflash2_conv_finish_launches(16, 16, 5120, 16, bf16, 1) == 1
    # above that, H not a multiple of 256 channels or G above 32 rows per block: a side-1 pass and
    # a separate norm
    assert lib.dflash2_conv_finish_launches(5, 64, 256, 16, f32, 1) == 2
    assert lib.dflash2_conv_finish_launches(64, 7, 320, 16, bf16, 1) == 2
    assert lib.dflash2_conv_prepare_launches(1, 16, 5000, 16, bf16, 0) == -1  # H % 64: rejected
    assert lib.dflash2_conv_finish_launches(1, 65, 5120, 16, bf16, 1) == -1   # G > 64: rejected


@pytest.mark.parametrize("entry", ["dflash2_head_topk", "dflash2_head_topk_noalloc", "dflash2_head_topk_vocab"])
def test_head_bindings_reject_mismatched_shapes_before_the_library(entry):
    """The bindings check sizes before any pointer reaches the library: an undersized output or a
    weight of the wrong width would make the head kernels read or write out of bounds."""
    import torch
    import dflash2_block_drafter_gb300 as d
    fn = getattr(d, entry)
    M, H, V, R, K = 6, 64, 100, 16, 4
    h = torch.zeros(M, H)
    good = dict(w=torch.zeros(V, H), w_proj=torch.zeros(R, H))
    extra = (torch.arange(V, dtype=torch.int32),) if entry.endswith("vocab") else ()

    def call(w=good["w"], **kw):
        kw.setdefault("w_proj", good["w_proj"])
        return fn(h, w, *extra, K, **kw)
    bad = [dict(w=torch.zeros(V, H + 64)),                       # head width != H
           dict(w_proj=torch.zeros(R, H - 8)),                   # projection width != H
           dict(cand=torch.zeros(M * K - 1, dtype=torch.int32)),  # undersized outputs
           dict(unary=torch.zeros(M, K - 1)),
           dict(z=torch.zeros(M, R - 1)),
           dict(logits=torch.zeros(M, V - 1))]
    for kw in bad:
        with pytest.raises(ValueError):
            call(**kw)
    if extra:
        with pytest.raises(ValueError):
            fn(h, good["w"], extra[0][:V - 1], K, w_proj=good["w_proj"])


def test_ragged_entry_points_reject_bad_arguments(lib):
    f = lib.dflash2_conv_finish_ragged
    #        y     coef  base  B   G   H     gs  taps dt resid out   nw    eps   nn    row0 off   m   stream
    assert f(FAKE, FAKE, FAKE, 4, 16, 5120, 16, 2, 0, None, FAKE, FAKE, 1e-6, FAKE, 1, None, 30, None) == -1  # offsets
    assert f(FAKE, FAKE, FAKE, 4, 16, 5120, 16, 2, 0, None, FAKE, None, 1e-6, FAKE, 1, FAKE, 30, None) == -1  # no norm
    assert f(FAKE, FAKE, FAKE, 4, 16, 5120, 16, 2, 0, None, FAKE, FAKE, 1e-6, FAKE, 1, FAKE, 0, None) == -1   # m_rows
    assert f(FAKE, FAKE, FAKE, 4, 16, 5120, 16, 3, 0, None, FAKE, FAKE, 1e-6, FAKE, 1, FAKE, 30, None) == -2  # taps
    g = lib.dflash2_score_edges_ragged
    #        cand  un    z     anch  pred  succ  off   B  st  K   R   V     m   dt S     path  stream
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 4, 15, 16, 64, 1000, 30, 0, None, FAKE, None) == -1  # offsets
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 15, 8, 64, 1000, 30, 0, None, FAKE, None) == -1   # K != 16
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 15, 16, 64, 1000, 30, 1, None, FAKE, None) == -1  # f32 R=64
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 15, 16, 64, 1000, 30, 0, None, None, None) == -1  # no path
    assert b"path" in lib.dflash2_last_error_message() or b"NULL" in lib.dflash2_last_error_message()


def test_projection_workspace_query(lib):
    """Up to 128 rows the projections reduce their K splits in shared memory and need no
    workspace; a few more rows than one 128-row tile split K through the workspace instead, and
    with at least half as many 256-column tiles as SMs the stream-K shares need one 128 x 256 fp32
    partial tile per CTA; above 384 rows the query also counts the bf16 copy of a 4-bit weight and the
    side-0 conv of the rows (the query is host-only and needs no device: 148 SMs are assumed)."""
    lib.dflash2_proj_workspace_bytes.restype = ctypes.c_size_t
    assert lib.dflash2_proj_workspace_bytes(1, 5120, 5120) == 0
    assert lib.dflash2_proj_workspace_bytes(128, 5120, 5120) == 0
    assert lib.dflash2_proj_workspace_bytes(129, 5120, 5120) == 3 * 129 * 5120 * 4  # 40 tiles: 3 K ranges
    # 1024 rows: the stream-K slots, then room to dequantise a 4-bit weight once (5120 x 5120 bf16) and
    # for the rows' side-0 conv or the projection before side 1 (1024 x 5120 bf16)
    assert lib.dflash2_proj_workspace_bytes(1024, 5120, 5120) == 148 * 128 * 256 * 4 + 5120 * 5120 * 2 + 1024 * 5120 * 2
