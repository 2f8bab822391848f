"""Seeded synthetic workloads shared by the oracle-side tests and the CUDA-side
tests and bench.

This module holds no arithmetic of the method itself (no norm, no rotary
angle, no softmax): only

* a counter-based splitmix64 stream (the published SplitMix64 finaliser of
  Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
  OOPSLA 2014), turned into uniforms and Box-Muller normals in fp64;
* round-to-nearest-even conversion of those numbers to bf16 bit patterns, so
  both sides consume the *same* bf16 values;
* the five packed-sequence workloads as lists of documents made of 3D grid
  spans (extents, starts, steps).  The spans are descriptions, not positions:
  each side turns them into positions with its own code.

The workload shapes follow the pages: the 864x480x124-frame six-reference
Ref2VA render with S = 20,423 tokens ("h3-spark" model card, "Measured on one
DGX Spark"), the 960x544x124-frame benchmark (H3 Blackwell Runtime README,
"Benchmark Contract"), and the per-document cu_seqlens packing of the
"feat(minimax-h3)" pull request (vllm.cpp PR #26, description: packed varlen
non-causal attention).  Activations are N(0, 1) stand-ins: the real
activation statistics and the benchmark JSON are not available.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_M64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15

# stream ids: one independent counter stream per drawn quantity
STREAM_Q, STREAM_K, STREAM_V = 1, 2, 3
STREAM_GAIN_Q, STREAM_GAIN_K = 4, 5
STREAM_K_CHANNEL_SCALE = 6
STREAM_DOC_LENGTHS = 7
STREAM_PERTURB = 8


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output finaliser on a uint64 array (wrapping arithmetic)."""
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= np.uint64(0xBF58476D1CE4E5B9)
    z ^= z >> np.uint64(27)
    z *= np.uint64(0x94D049BB133111EB)
    z ^= z >> np.uint64(31)
    return z


def _mix64_int(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    """64-bit key of one named stream under one seed."""
    return _mix64_int((seed * 0x1000193 + stream) * _GOLDEN)


def raw_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Counter-based splitmix64: element i is mix(key + (start+i+1)*golden)."""
    key = np.uint64(stream_key(seed, stream))
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = key + idx * np.uint64(_GOLDEN)
    return _mix64(z)


def uniform01(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    """Uniforms in the open interval (0, 1) from the top 53 bits."""
    z = raw_u64(seed, stream, start, count)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def normal(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    """Standard normals (Box-Muller, both branches) in fp64.

    Pair p uses uniforms 2p and 2p+1; element 2p is the cosine branch and
    2p+1 the sine branch.  ``start`` must be even.
    """
    assert start % 2 == 0
    npairs = (count + 1) // 2
    u = uniform01(seed, stream, 2 * npairs, start)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    ang = 2.0 * math.pi * u2
    out = np.empty(2 * npairs, dtype=np.float64)
    out[0::2] = r * np.cos(ang)
    out[1::2] = r * np.sin(ang)
    return out[:count]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits.

    NaN is not produced by the generators and is not handled specially.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = b + np.uint32(0x7FFF) + lsb
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def normal_bf16_bits(seed: int, stream: int, count: int, chunk: int = 1 << 24) -> np.ndarray:
    """count N(0,1) values rounded fp64 -> fp32 -> bf16, as uint16 bits."""
    out = np.empty(count, dtype=np.uint16)
    for s in range(0, count, chunk):
        n = min(chunk, count - s)
        out[s:s + n] = f32_to_bf16_bits(normal(seed, stream, n, start=s).astype(np.float32))
    return out


# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Span:
    """A grid of n_t x n_h x n_w tokens (t-major, w fastest); the position of
    token (i_t, i_h, i_w) on axis a is i_a * step[a] + start[a]."""
    n_t: int
    n_h: int
    n_w: int
    start: tuple = (0.0, 0.0, 0.0)
    step: tuple = (1.0, 1.0, 1.0)

    @property
    def ntok(self) -> int:
        return self.n_t * self.n_h * self.n_w


def grid(n_t, n_h, n_w, t0=0.0) -> Span:
    return Span(n_t, n_h, n_w, (float(t0), 0.0, 0.0), (1.0, 1.0, 1.0))


def run1d(n) -> Span:
    """A 1D run: positions t = 0..n-1 with h = w = 0."""
    return Span(n, 1, 1, (0.0, 0.0, 0.0), (1.0, 0.0, 0.0))


@dataclass
class Workload:
    name: str
    seed: int
    num_heads: int
    docs: list            # list of documents, each a list of Span
    head_dim: int = 128
    rope_base: float = 10000.0
    rope_dims: int = 96
    eps: float = 1e-6
    k_channel_outliers: bool = False
    notes: str = ""
    doc_lengths: list = field(default_factory=list)

    def __post_init__(self):
        self.doc_lengths = [sum(s.ntok for s in d) for d in self.docs]

    @property
    def S(self) -> int:
        return sum(self.doc_lengths)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def flops(self) -> int:
        """Algorithmic FLOPs of one forward: QK^T and PV inside each document."""
        return 4 * self.head_dim * self.num_heads * sum(L * L for L in self.doc_lengths)


def config5_doc_lengths(seed: int, n_docs: int = 16, total: int = 32768,
                        lo: float = 512.0, hi: float = 4096.0, unit: int = 8) -> list:
    """Seeded document lengths: u_i ~ U[lo, hi], rescaled to sum to ``total``,
    floored to multiples of ``unit``; the leftover units go to the largest
    fractional remainders (ties to the lower index)."""
    u = lo + (hi - lo) * uniform01(seed, STREAM_DOC_LENGTHS, n_docs)
    raw = u * (total / u.sum()) / unit
    base = np.floor(raw).astype(np.int64)
    left = total // unit - int(base.sum())
    frac = raw - base
    order = sorted(range(n_docs), key=lambda i: (-frac[i], i))
    for i in order[:left]:
        base[i] += 1
    lens = [int(b) * unit for b in base]
    assert sum(lens) == total and min(lens) >= unit
    return lens


def config5_doc(length: int) -> list:
    """t = 4 grid with h x w near-square, remainder as a 1D tail."""
    m = length // 4
    h = math.isqrt(m)
    w = m // h
    spans = [grid(4, h, w)]
    tail = length - 4 * h * w
    if tail:
        spans.append(run1d(tail))
    return spans


def config(n: int) -> Workload:
    """The five packed-attention workloads (1-based, as named in the docs)."""
    seed = 1000 + n
    if n == 1:
        return Workload("tiny-2doc-S144", seed, 2, [[grid(2, 4, 8)], [grid(1, 8, 10)]],
                        notes="grids (2,4,8) and (1,8,10); cu_seqlens [0,64,144]")
    if n == 2:
        return Workload("video-1doc-S4096", seed, 21, [[grid(8, 16, 32)]])
    if n == 3:
        doc = [grid(32, 15, 27)] + [grid(1, 15, 27, t0=-(i + 1)) for i in range(6)] + [run1d(5033)]
        return Workload("ref2va-1doc-S20423", seed, 21, [doc], k_channel_outliers=True,
                        notes="video 32x15x27 + 6 refs 1x15x27 at t=-1..-6 + audio 5033 (1D)")
    if n == 4:
        return Workload("960x544x124-2doc-S21353", seed, 21, [[grid(32, 17, 30)], [run1d(5033)]])
    if n == 5:
        lens = config5_doc_lengths(seed)
        return Workload("varlen-16doc-S32768", seed, 21, [config5_doc(L) for L in lens])
    raise ValueError(n)


@dataclass
class Tensors:
    """bf16 bit patterns [S, H, 128] and fp32 gains [128]."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    gain_q: np.ndarray
    gain_k: np.ndarray


def make_tensors(w: Workload, seed: int | None = None) -> Tensors:
    seed = w.seed if seed is None else seed
    S, H, D = w.S, w.num_heads, w.head_dim
    n = S * H * D
    q = normal_bf16_bits(seed, STREAM_Q, n).reshape(S, H, D)
    v = normal_bf16_bits(seed, STREAM_V, n).reshape(S, H, D)
    if w.k_channel_outliers:
        # per (head, dim) column scale ~ LogNormal(0, 0.5), applied before rounding
        cs = np.exp(0.5 * normal(seed, STREAM_K_CHANNEL_SCALE, H * D)).reshape(H, D)
        k = np.empty(n, dtype=np.uint16)
        chunk = (1 << 24) // (H * D) * (H * D)
        for s in range(0, n, chunk):
            m = min(chunk, n - s)
            x = normal(seed, STREAM_K, m, start=s).reshape(-1, H, D) * cs
            k[s:s + m] = f32_to_bf16_bits(x.astype(np.float32)).ravel()
        k = k.reshape(S, H, D)
    else:
        k = normal_bf16_bits(seed, STREAM_K, n).reshape(S, H, D)
    gq = (1.0 + 0.1 * normal(seed, STREAM_GAIN_Q, D)).astype(np.float32)
    gk = (1.0 + 0.1 * normal(seed, STREAM_GAIN_K, D)).astype(np.float32)
    return Tensors(q, k, v, gq, gk)


def spans_to_tuples(docs) -> list:
    """[[(n_t, n_h, n_w, start(3), step(3)), ...], ...] plain tuples."""
    return [[(s.n_t, s.n_h, s.n_w, tuple(s.start), tuple(s.step)) for s in d] for d in docs]
