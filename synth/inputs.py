"""Seeded synthetic inputs for the DFlash2 block-local tail.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's callers. It draws random tensors, rounds them to their storage dtype
and decodes storage back to float64; it holds none of the method's arithmetic.

Storage convention
------------------
* ``"bf16"`` tensors are ``numpy.uint16`` arrays holding bfloat16 bit patterns
  (round-to-nearest-even from a float32 draw). The GPU path views them as
  ``torch.bfloat16``; the oracle decodes them to float64 with :func:`to_f64`.
* ``"f32"`` tensors are ``numpy.float32`` arrays.
* ``base`` kernels are always float32 (the drafter upcasts them to f32 at load,
  dflash2.ts ``#baseKernel``); ``bias`` is float32; ids are int32.

Recipe (seed ``20261202 + config``; every tensor has its own stream derived
from the config seed and the tensor's name, so tensors never shift one another):

=====  =====================================================================
cfg    contents
=====  =====================================================================
0      tiny full tail in f32: B=1, G=8, H=256, group 16, one conv site
       (kernel_projection [64,256] ~N(0,1/16), base tap0=1+N(0,0.1),
       tap1=N(0,0.1)), x and y ~N(0,1); head [4096,256] ~N(0,1/16), K=16,
       R=16, hidden_projection [16,256] ~N(0,1/16), codebooks [4096,16]
       ~N(0,0.5), anchor uniform in [0,4096)
1      conv chain at drafter shape, bf16: H=5120, G=16, group 16, 10 sites
       (5 layers x attention/MLP), kernel_projection [1280,5120]
       ~N(0,1/sqrt(5120)), base as cfg 0, gain-1 norms, x0 and the 10
       sublayer stand-ins y ~N(0,1); B in {1, 8, 64}
2      selector at B=1, bf16: h [1,15,5120] ~N(0,1); head [248320,5120]
       ~N(0,1/sqrt(5120)); hidden_projection [64,5120] ~N(0,1/sqrt(5120));
       codebooks [248320,64] ~N(0,0.3); K=16; anchor uniform in [0,V)
3      as 2 with B=32 and a log-Zipf bias  bias[v] = -1.1*ln(v+1)
4      cfg-1 chain at B=64 -> final norm (gain 1) -> cfg-3 selector
=====  =====================================================================

"N(0, s)" means standard deviation s.
"""
from __future__ import annotations

import math
import os
import zlib
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

SEED_BASE = 20261202
EPS = 1e-6

# drafter shape
H_DRAFTER = 5120
G_DRAFTER = 16
GS_DRAFTER = 16
V_DRAFTER = 248320
R_DRAFTER = 64
K_DRAFTER = 16
LAYERS_DRAFTER = 5


# --------------------------------------------------------------------------- storage helpers

def round_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_f64(a, dtype: Optional[str] = None) -> np.ndarray:
    """Decode a stored tensor to float64 (bf16 bits are recognised by dtype uint16)."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)


class Bf16Rows:
    """A read-only [rows, cols] view of bf16 bits whose row slices decode to float64.

    Lets a caller hand a multi-GB bf16 matrix to code that reads it slab by slab
    (``w[v0:v1]``) without ever holding a float64 copy of the whole matrix.
    """

    def __init__(self, bits: np.ndarray):
        assert bits.dtype == np.uint16 and bits.ndim == 2
        self.bits = bits
        self.shape = bits.shape

    def __len__(self):
        return self.shape[0]

    def __getitem__(self, idx):
        return bf16_bits_to_f32(self.bits[idx]).astype(np.float64)


def f64_view(a):
    """A row-sliceable float64 view of a stored tensor (lazy for big bf16 matrices)."""
    a = np.asarray(a)
    if a.dtype == np.uint16 and a.ndim == 2 and a.size > (1 << 24):
        return Bf16Rows(a)
    return to_f64(a)


# --------------------------------------------------------------------------- seeded draws

def _seed_for(config_seed: int, name: str) -> np.random.SeedSequence:
    return np.random.SeedSequence([config_seed, zlib.crc32(name.encode())])


def _store(f32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_to_bf16_bits(f32)
    if dtype == "f32":
        return np.ascontiguousarray(f32, dtype=np.float32)
    raise ValueError(dtype)


def normal(config_seed: int, name: str, shape, std: float, mean: float = 0.0,
           dtype: str = "bf16", slab_rows: int = 8192) -> np.ndarray:
    """N(mean, std) draw of ``shape``, stored as ``dtype``.

    Large matrices are drawn in row slabs, each slab from its own child stream,
    on a thread pool (the result does not depend on the thread count).
    """
    shape = tuple(int(s) for s in shape)
    ss = _seed_for(config_seed, name)
    rows = shape[0] if shape else 1
    inner = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    if rows * inner <= (1 << 22) or len(shape) < 2:
        g = np.random.Generator(np.random.PCG64(ss))
        f = g.standard_normal(shape, dtype=np.float32)
        if std != 1.0:
            f *= np.float32(std)
        if mean != 0.0:
            f += np.float32(mean)
        return _store(f, dtype)
    n_slabs = (rows + slab_rows - 1) // slab_rows
    children = ss.spawn(n_slabs)
    out = np.empty(shape, dtype=np.uint16 if dtype == "bf16" else np.float32)

    def work(i):
        r0, r1 = i * slab_rows, min(rows, (i + 1) * slab_rows)
        g = np.random.Generator(np.random.PCG64(children[i]))
        f = g.standard_normal((r1 - r0,) + shape[1:], dtype=np.float32)
        if std != 1.0:
            f *= np.float32(std)
        if mean != 0.0:
            f += np.float32(mean)
        out[r0:r1] = _store(f, dtype)

    workers = min(n_slabs, max(1, (os.cpu_count() or 1)))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(work, range(n_slabs)))
    return out


def uniform_ids(config_seed: int, name: str, n: int, high: int) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(_seed_for(config_seed, name)))
    return g.integers(0, high, size=n, dtype=np.int64).astype(np.int32)


def draft_vocabulary(config_seed: int, V: int, n: int) -> np.ndarray:
    """A seeded draft vocabulary: n distinct token ids in [0, V), ascending (int32)."""
    g = np.random.Generator(np.random.PCG64(_seed_for(config_seed, "draft_vocabulary")))
    return np.sort(g.choice(V, size=n, replace=False)).astype(np.int32)


def ones(shape, dtype: str) -> np.ndarray:
    return _store(np.ones(shape, dtype=np.float32), dtype)


def zipf_bias(V: int, s: float = 1.1) -> np.ndarray:
    """Log-Zipf logit bias over vocabulary id: bias[v] = -s * ln(v + 1) (float32)."""
    return (-s * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)


def pack_int4(q: np.ndarray) -> np.ndarray:
    """Storage of 4-bit codes q [N, K] (values 0..15): [N, K/8] uint32 words, code k in bits
    4 (k % 8) .. 4 (k % 8) + 3 of word k / 8."""
    q = np.asarray(q, dtype=np.uint32)
    N, K = q.shape
    w = np.zeros((N, K // 8), dtype=np.uint32)
    for j in range(8):
        w |= q[:, j::8] << np.uint32(4 * j)
    return w


def unpack_int4(w: np.ndarray, K: int) -> np.ndarray:
    """The codes [N, K] (uint8) held by pack_int4's words."""
    w = np.asarray(w, dtype=np.uint32)
    q = np.empty((w.shape[0], K), dtype=np.uint8)
    for j in range(8):
        q[:, j::8] = (w >> np.uint32(4 * j)) & np.uint32(15)
    return q


@dataclass
class Affine4:
    """A seeded affine 4-bit weight [N, K] in groups of 64 along K: codes q, packed words, and
    bf16 scales / biases [N, K/64] (bf16 bit patterns)."""
    q: np.ndarray
    packed: np.ndarray
    scales: np.ndarray
    biases: np.ndarray


def affine4_weight(config_seed: int, name: str, N: int, K: int, exact: bool = False) -> Affine4:
    """Uniform codes in [0, 15]. exact=False: scales ~ U(0.5, 1.5) / 64 and biases ~ N(0, 1/128).
    exact=True: scales in {1/4, 1/8, 1/16} and biases in {-8..8} / 64, so that every
    scale * q + bias (|.| < 4, a multiple of 1/64) is exactly a bf16 value."""
    g = np.random.Generator(np.random.PCG64(_seed_for(config_seed, name)))
    q = g.integers(0, 16, size=(N, K), dtype=np.int64).astype(np.uint8)
    G = K // 64
    if exact:
        sc = np.float32(2.0) ** -g.integers(2, 5, size=(N, G)).astype(np.float32)
        bi = g.integers(-8, 9, size=(N, G)).astype(np.float32) / np.float32(64.0)
    else:
        sc = g.uniform(0.5, 1.5, size=(N, G)).astype(np.float32) / np.float32(64.0)
        bi = g.standard_normal((N, G)).astype(np.float32) / np.float32(128.0)
    return Affine4(q=q, packed=pack_int4(q), scales=round_to_bf16_bits(sc), biases=round_to_bf16_bits(bi))


# --------------------------------------------------------------------------- workloads

@dataclass
class ConvSite:
    """One sublayer's convolution weights plus the seeded stand-in for the sublayer."""
    w_kp: np.ndarray          # [2*2*H/gs, H] (out, in) storage dtype
    base: np.ndarray          # [2, 2, H] float32  (side, tap, channel)
    norm_w: np.ndarray        # [H] storage dtype (RMSNorm gain, all ones here)
    y: np.ndarray             # [B, G, H] storage dtype (the sublayer's output)


@dataclass
class Workload:
    name: str
    dtype: str                # "bf16" | "f32"
    B: int
    G: int
    H: int
    gs: int
    eps: float = EPS
    x0: Optional[np.ndarray] = None            # [B, G, H]
    sites: list = field(default_factory=list)  # list[ConvSite]
    final_norm_w: Optional[np.ndarray] = None  # [H]
    V: int = 0
    K: int = 0
    R: int = 0
    w_head: Optional[np.ndarray] = None        # [V, H]
    bias: Optional[np.ndarray] = None          # [V] float32
    w_proj: Optional[np.ndarray] = None        # [R, H]
    pred_book: Optional[np.ndarray] = None     # [V, R]
    succ_book: Optional[np.ndarray] = None     # [V, R]
    anchors: Optional[np.ndarray] = None       # [B] int32
    h: Optional[np.ndarray] = None             # [B, G-1, H]  (selector-only workloads)

    @property
    def steps(self) -> int:
        return self.G - 1

    @property
    def groups(self) -> int:
        return self.H // self.gs


def conv_site(seed: int, tag: str, B: int, G: int, H: int, gs: int, dtype: str) -> ConvSite:
    groups = H // gs
    w_kp = normal(seed, f"{tag}.kernel_projection", (4 * groups, H), 1.0 / math.sqrt(H), dtype=dtype)
    base = np.empty((2, 2, H), dtype=np.float32)
    for side in range(2):
        base[side, 0] = normal(seed, f"{tag}.base.side{side}.tap0", (H,), 0.1, mean=1.0, dtype="f32")
        base[side, 1] = normal(seed, f"{tag}.base.side{side}.tap1", (H,), 0.1, dtype="f32")
    return ConvSite(w_kp=w_kp, base=base, norm_w=ones((H,), dtype),
                    y=normal(seed, f"{tag}.sublayer_out", (B, G, H), 1.0, dtype=dtype))


def _selector_weights(wl: Workload, seed: int, head_std: float, book_std: float):
    wl.w_head = normal(seed, "head", (wl.V, wl.H), head_std, dtype=wl.dtype)
    wl.w_proj = normal(seed, "hidden_projection", (wl.R, wl.H), head_std, dtype=wl.dtype)
    wl.pred_book = normal(seed, "predecessor_codebook", (wl.V, wl.R), book_std, dtype=wl.dtype)
    wl.succ_book = normal(seed, "successor_codebook", (wl.V, wl.R), book_std, dtype=wl.dtype)
    wl.anchors = uniform_ids(seed, "anchors", wl.B, wl.V)


def make_config(index: int, B: Optional[int] = None, with_selector_weights: bool = True) -> Workload:
    """The five seeded workloads (see the module docstring)."""
    seed = SEED_BASE + index
    if index == 0:
        B = 1 if B is None else B
        wl = Workload("tiny-full-tail-f32", "f32", B=B, G=8, H=256, gs=16, V=4096, K=16, R=16)
        wl.x0 = normal(seed, "x0", (B, wl.G, wl.H), 1.0, dtype="f32")
        wl.sites = [conv_site(seed, "site0", B, wl.G, wl.H, wl.gs, "f32")]
        wl.final_norm_w = ones((wl.H,), "f32")
        _selector_weights(wl, seed, 1.0 / math.sqrt(wl.H), 0.5)
        return wl
    if index == 1:
        B = 1 if B is None else B
        wl = Workload(f"conv-chain-B{B}", "bf16", B=B, G=G_DRAFTER, H=H_DRAFTER, gs=GS_DRAFTER)
        wl.x0 = normal(seed, "x0", (B, wl.G, wl.H), 1.0)
        wl.sites = [conv_site(seed, f"layer{l}.{s}", B, wl.G, wl.H, wl.gs, "bf16")
                    for l in range(LAYERS_DRAFTER) for s in ("attention_conv", "mlp_conv")]
        return wl
    if index in (2, 3):
        B = (1 if index == 2 else 32) if B is None else B
        wl = Workload(f"selector-B{B}", "bf16", B=B, G=G_DRAFTER, H=H_DRAFTER, gs=GS_DRAFTER,
                      V=V_DRAFTER, K=K_DRAFTER, R=R_DRAFTER)
        wl.h = normal(seed, "h", (B, wl.steps, wl.H), 1.0)
        if with_selector_weights:
            _selector_weights(wl, seed, 1.0 / math.sqrt(wl.H), 0.3)
        else:
            wl.anchors = uniform_ids(seed, "anchors", wl.B, wl.V)
        if index == 3:
            wl.bias = zipf_bias(wl.V)
        return wl
    if index == 4:
        B = 64 if B is None else B
        wl = Workload(f"full-tail-B{B}", "bf16", B=B, G=G_DRAFTER, H=H_DRAFTER, gs=GS_DRAFTER)
        wl.x0 = normal(seed, "x0", (B, wl.G, wl.H), 1.0)
        wl.sites = [conv_site(seed, f"layer{l}.{s}", B, wl.G, wl.H, wl.gs, "bf16")
                    for l in range(LAYERS_DRAFTER) for s in ("attention_conv", "mlp_conv")]
        wl.final_norm_w = ones((wl.H,), "bf16")
        wl.V, wl.K, wl.R = V_DRAFTER, K_DRAFTER, R_DRAFTER
        if with_selector_weights:
            _selector_weights(wl, seed, 1.0 / math.sqrt(wl.H), 0.3)
        else:
            wl.anchors = uniform_ids(seed, "anchors", wl.B, wl.V)
        wl.bias = zipf_bias(wl.V)
        return wl
    raise ValueError(f"no config {index}")


# --------------------------------------------------------------------------- small cases for tests

def conv_case(seed: int, B: int, G: int, H: int, gs: int, dtype: str = "bf16", n_sites: int = 1,
              kp_std: Optional[float] = None) -> Workload:
    """A conv-only workload of arbitrary shape (parity tests)."""
    wl = Workload(f"conv-B{B}-G{G}-H{H}", dtype, B=B, G=G, H=H, gs=gs)
    wl.x0 = normal(seed, "x0", (B, G, H), 1.0, dtype=dtype)
    wl.sites = [conv_site(seed, f"site{i}", B, G, H, gs, dtype) for i in range(n_sites)]
    if kp_std is not None:
        for i, s in enumerate(wl.sites):
            s.w_kp = normal(seed, f"site{i}.kernel_projection.custom", s.w_kp.shape, kp_std, dtype=dtype)
    wl.final_norm_w = ones((H,), dtype)
    return wl


def selector_case(seed: int, B: int, G: int, H: int, V: int, K: int, R: int, dtype: str = "bf16",
                  book_std: float = 0.3, bias: bool = False, h_std: float = 1.0) -> Workload:
    """A selector-only workload of arbitrary shape (parity tests)."""
    wl = Workload(f"selector-B{B}-V{V}", dtype, B=B, G=G, H=H, gs=16, V=V, K=K, R=R)
    wl.h = normal(seed, "h", (B, G - 1, H), h_std, dtype=dtype)
    _selector_weights(wl, seed, 1.0 / math.sqrt(H), book_std)
    if bias:
        wl.bias = zipf_bias(V)
    return wl
