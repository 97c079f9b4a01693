"""Seeded synthetic inputs for the RMSNorm family.

This module holds only random-number generation and storage-type casts; none
of the normalisation arithmetic lives here.  It is the one piece shared by the
tests, the benchmark and the package smoke check: the same seed gives the same
storage bits on both sides of every comparison.

Recipe (seed s):

* Each [T, H] input stream is drawn in blocks of CHUNK_ROWS rows; block b of
  stream k comes from its own ``numpy.random.Generator(PCG64(SeedSequence(
  [s, k, b])))``, so any row range can be generated on its own and blocks are
  drawn in parallel threads.  Streams: plain k=0 is x; fused k=0 is x, k=1 the
  residual; reduce k=0..R-1 are the partials, k=R the residual.
* Normal draws use the Box-Muller transform on binary32 uniforms: u1, u2 in
  [0, 1), r = sqrt(-2 log(1 - u1)) (1 - u1 is exact in binary32),
  z0 = r cos(2 pi u2), z1 = r sin(2 pi u2), interleaved z0, z1 along the row
  block.
* gamma ~ U(0.5, 1.5) from SeedSequence([s, GAMMA_KEY]).
* Values are formed in binary32 and cast to the storage type with
  round-to-nearest-even (numpy for f16, torch for bf16).
* Scaled-token workload: every row t of both x and residual is multiplied by
  s_t = 10 ** U(-3, 3) (SeedSequence([s, SCALE_KEY]), T draws); ceil(H / 100)
  channels, the first ones of a permutation drawn from
  SeedSequence([s, OUTLIER_KEY]), are multiplied by 100 in x and residual.
* Reduce partials are N(0, partial_std^2); x and residual are N(0, 1).
* A binary32 residual (``rdtype="f32"``) keeps the binary32 draws of its
  stream without rounding to the inputs' type.
* GEMM-producer workloads (``GemmWorkload``): A [T, K] ~ N(0, 1) (stream 0,
  blocks of CHUNK_ROWS rows), W [H, K] ~ N(0, 1 / K) (stream 1), residual
  [T, H] ~ N(0, 1) (stream 2), gamma as above; so P = A W^T ~ N(0, 1).

Arrays hold raw storage bits: ``np.float32`` for f32, ``np.uint16`` for f16 and
bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

STORAGE = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16}
ELEM_SIZE = {"f32": 4, "f16": 2, "bf16": 2}


@dataclass(frozen=True)
class Workload:
    """One problem instance of the RMSNorm family.

    op      'rms_norm' | 'fused_add_rms_norm' | 'reduce_add_rms_norm'
    R       number of partial buffers (reduce only; 1 for fused, 0 for plain)
    scaled  per-row log-uniform scale and x100 outlier channels
    """
    name: str
    op: str
    dtype: str
    T: int
    H: int
    eps: float
    R: int = 0
    seed: int = 0
    partial_std: float = 1.0
    scaled: bool = False
    rdtype: str = ""   # residual storage type ("": the inputs' type)
    ld: int = 0        # row stride of x / partials, residual and y (0: H)
    qfmt: str = ""     # 8-bit output: "e4m3" | "e5m2" ("": y in the inputs' type)
    qmode: str = ""    # 8-bit output scale: "tensor" (given) | "row" (computed per row)
    qscale: float = 1.0  # the per-tensor scale
    note: str = field(default="", compare=False)

    @property
    def res_dtype(self) -> str:
        return self.rdtype or self.dtype

    @property
    def row_stride(self) -> int:
        return self.ld or self.H

    @property
    def n_inputs(self) -> int:
        """Input streams read per element (x or partials, plus residual)."""
        return {"rms_norm": 1, "fused_add_rms_norm": 2}.get(self.op, self.R + 1)

    @property
    def n_outputs(self) -> int:
        """Output streams written per element (y, plus residual)."""
        return 1 if self.op == "rms_norm" else 2

    def algorithmic_bytes(self) -> int:
        """Bytes the operation must move at minimum: every input element read
        once, every output element written once, gamma read once (the
        residual counted in its own storage type; an 8-bit y as one byte per
        element plus its scales)."""
        s = ELEM_SIZE[self.dtype]
        ys = 1 if self.qfmt else s
        scales = (4 * self.T if self.qmode == "row" else 4) if self.qfmt else 0
        if self.op == "rms_norm":
            return self.T * self.H * (s + ys) + s * self.H + scales
        rs = ELEM_SIZE[self.res_dtype]
        n_x = self.n_inputs - 1  # partials (or x)
        return self.T * self.H * (s * n_x + rs * 2 + ys) + s * self.H + scales


# The five benchmark configurations of the method (the token sweep is five
# shapes of one configuration).
CONFIGS = [
    Workload("plain_f32_T512_H2048", "rms_norm", "f32", 512, 2048, 1e-6),
    Workload("plain_f16_T512_H1592", "rms_norm", "f16", 512, 1592, 1e-5),
    Workload("fused_bf16_T4096_H4096", "fused_add_rms_norm", "bf16", 4096, 4096, 1e-6, R=1),
    Workload("reduce8_bf16_T8192_H8192", "reduce_add_rms_norm", "bf16", 8192, 8192, 1e-6, R=8,
             partial_std=math.sqrt(1.0 / 8.0)),
    Workload("fused_scaled_bf16_T1_H5120", "fused_add_rms_norm", "bf16", 1, 5120, 1e-6, R=1,
             scaled=True),
    Workload("fused_scaled_bf16_T16_H5120", "fused_add_rms_norm", "bf16", 16, 5120, 1e-6, R=1,
             scaled=True),
    Workload("fused_scaled_bf16_T128_H5120", "fused_add_rms_norm", "bf16", 128, 5120, 1e-6, R=1,
             scaled=True),
    Workload("fused_scaled_bf16_T32768_H5120", "fused_add_rms_norm", "bf16", 32768, 5120, 1e-6,
             R=1, scaled=True),
    Workload("fused_scaled_bf16_T64_H16384", "fused_add_rms_norm", "bf16", 64, 16384, 1e-6, R=1,
             scaled=True),
]
# The widened rows: a row-strided plain norm (the first H = 512 of 576
# columns, as a latent slice inside a wider projection output), a fused
# norm with a binary32 residual stream and bf16 inputs / output, and the fused
# norm with an e4m3 output under a per-row (dynamic) or a per-tensor (static)
# scale.
EXTENDED = [
    Workload("plain_strided_bf16_T32768_H512_ld576", "rms_norm", "bf16", 32768, 512, 1e-6,
             ld=576),
    Workload("fused_r32_bf16_T32768_H5120", "fused_add_rms_norm", "bf16", 32768, 5120, 1e-6,
             R=1, rdtype="f32"),
    Workload("fused_e4m3row_bf16_T32768_H5120", "fused_add_rms_norm", "bf16", 32768, 5120, 1e-6,
             R=1, qfmt="e4m3", qmode="row"),
    Workload("fused_e4m3_bf16_T32768_H5120", "fused_add_rms_norm", "bf16", 32768, 5120, 1e-6,
             R=1, qfmt="e4m3", qmode="tensor", qscale=0.02),
]
BY_NAME = {w.name: w for w in CONFIGS + EXTENDED}


@dataclass(frozen=True)
class GemmWorkload:
    """The fused form whose partial is a matrix product: A [T, K] times a
    linear layer's weight W [H, K] (transposed), plus the residual, RMSNorm."""
    name: str
    dtype: str
    T: int
    H: int
    K: int
    eps: float
    seed: int = 0

    def flops(self) -> int:
        return 2 * self.T * self.H * self.K

    def algorithmic_bytes(self) -> int:
        """A and W read once, the residual read and written, y written, gamma."""
        s = ELEM_SIZE[self.dtype]
        return s * (self.T * self.K + self.H * self.K + 3 * self.T * self.H + self.H)


# The GEMM-producer workload: the fused form's [4096, 4096] shape (C3) with
# its partial produced by a 4096 x 4096 projection.
GEMM_CONFIGS = [GemmWorkload("gemm_fused_bf16_T4096_K4096_H4096", "bf16", 4096, 4096, 4096, 1e-6)]

# Wider GEMM-producer shapes, timed beside it: twice the tokens, and a
# [16384 tokens, 5120] projection (C5's row length).
GEMM_WIDER = [GemmWorkload("gemm_fused_bf16_T8192_K4096_H4096", "bf16", 8192, 4096, 4096, 1e-6),
              GemmWorkload("gemm_fused_bf16_T16384_K5120_H5120", "bf16", 16384, 5120, 5120, 1e-6)]


def generate_gemm(w: GemmWorkload, rows: tuple[int, int] | None = None) -> dict:
    """Inputs of a GEMM workload as storage bits: 'a' [T', K], 'w' [H, K],
    'residual' [T', H], 'gamma' [H]; ``rows`` as for ``generate``."""
    T, H, K = w.T, w.H, w.K
    a, b = (0, T) if rows is None else rows
    if not 0 <= a <= b <= T:
        raise ValueError(f"rows {rows} outside 0..{T}")

    def draw(stream, nrows, ncols, lo, hi, scale):
        out = np.empty((hi - lo, ncols), STORAGE[w.dtype])

        def block(c):
            r0, r1 = c * CHUNK_ROWS, min((c + 1) * CHUNK_ROWS, nrows)
            z = _normal_f32(_rng(w.seed, stream, c), (r1 - r0) * ncols).reshape(r1 - r0, ncols)
            l2, h2 = max(r0, lo), min(r1, hi)
            z = z[l2 - r0:h2 - r0]
            if scale != 1.0:
                z = z * np.float32(scale)
            out[l2 - lo:h2 - lo] = to_storage(z, w.dtype)

        if hi > lo:
            with _pool() as ex:
                list(ex.map(block, range(lo // CHUNK_ROWS, (hi + CHUNK_ROWS - 1) // CHUNK_ROWS)))
        return out

    g = _rng(w.seed, GAMMA_KEY).uniform(0.5, 1.5, size=H).astype(np.float32)
    return {"a": draw(0, T, K, a, b, 1.0), "w": draw(1, H, K, 0, H, 1.0 / math.sqrt(K)),
            "residual": draw(2, T, H, a, b, 1.0), "gamma": to_storage(g, w.dtype)}


def workload(op: str, dtype: str, T: int, H: int, *, R: int | None = None, eps: float = 1e-6,
             seed: int = 0, scaled: bool = False, partial_std: float = 1.0, rdtype: str = "",
             ld: int = 0) -> Workload:
    """An ad-hoc problem (edge-shape grids in the tests)."""
    if R is None:
        R = {"rms_norm": 0, "fused_add_rms_norm": 1}.get(op, 2)
    name = f"{op}_{dtype}_T{T}_H{H}_R{R}" + (f"_r{rdtype}" if rdtype else "") + \
        (f"_ld{ld}" if ld else "")
    return Workload(name, op, dtype, T, H, eps, R=R, seed=seed, partial_std=partial_std,
                    scaled=scaled, rdtype=rdtype, ld=ld)


CHUNK_ROWS = 256
GAMMA_KEY, SCALE_KEY, OUTLIER_KEY = 1 << 20, (1 << 20) + 1, (1 << 20) + 2


def _rng(*key) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def _normal_f32(rng: np.random.Generator, n: int) -> np.ndarray:
    m = (n + 1) // 2
    u1 = rng.random(m, dtype=np.float32)
    u2 = rng.random(m, dtype=np.float32)
    r = np.sqrt(np.float32(-2.0) * np.log(np.float32(1.0) - u1))
    th = np.float32(2.0 * np.pi) * u2
    z = np.empty(2 * m, np.float32)
    z[0::2] = r * np.cos(th)
    z[1::2] = r * np.sin(th)
    return z[:n]


def to_storage(v: np.ndarray, dtype: str) -> np.ndarray:
    """binary32 values -> storage bits (round to nearest even)."""
    v = np.ascontiguousarray(v, np.float32)
    if dtype == "f32":
        return v
    if dtype == "f16":
        return v.astype(np.float16).view(np.uint16)
    import torch
    return torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def from_storage(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Storage bits -> binary32 values (exact widening)."""
    if dtype == "f32":
        return np.asarray(bits, np.float32)
    if dtype == "f16":
        return np.asarray(bits, np.uint16).view(np.float16).astype(np.float32)
    u = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


def _pool():
    import concurrent.futures as cf
    import os
    return cf.ThreadPoolExecutor(max_workers=min(32, os.cpu_count() or 1))


def generate(w: Workload, rows: tuple[int, int] | None = None) -> dict:
    """Inputs of ``w`` as storage bits: keys 'x' (plain, fused), 'partials'
    (reduce, shape [R, T', H]), 'residual' (fused, reduce) and 'gamma'.

    ``rows=(a, b)`` generates only rows a..b-1 (T' = b - a); the bits equal
    those rows of the full problem."""
    T, H = w.T, w.H
    a, b = (0, T) if rows is None else rows
    if not 0 <= a <= b <= T:
        raise ValueError(f"rows {rows} outside 0..{T}")
    n = b - a
    if w.op == "reduce_add_rms_norm":
        nstreams, names = w.R + 1, None
    elif w.op == "fused_add_rms_norm":
        nstreams, names = 2, ("x", "residual")
    else:
        nstreams, names = 1, ("x",)
    row_scale = col_scale = None
    if w.scaled:
        row_scale = np.power(10.0, _rng(w.seed, SCALE_KEY).uniform(-3.0, 3.0, size=T)).astype(
            np.float32)
        col_scale = np.ones(H, np.float32)
        col_scale[_rng(w.seed, OUTLIER_KEY).permutation(H)[:math.ceil(H / 100)]] = 100.0
    std = np.float32(w.partial_std)
    out_arr = np.empty((nstreams, n, H), STORAGE[w.dtype])

    def block(job):
        k, c = job
        r0, r1 = c * CHUNK_ROWS, min((c + 1) * CHUNK_ROWS, T)
        z = _normal_f32(_rng(w.seed, k, c), (r1 - r0) * H).reshape(r1 - r0, H)
        lo, hi = max(r0, a), min(r1, b)
        z = z[lo - r0:hi - r0]
        if w.op == "reduce_add_rms_norm" and k < w.R and w.partial_std != 1.0:
            z = z * std
        if row_scale is not None:
            z = z * row_scale[lo:hi, None] * col_scale[None, :]
        out_arr[k, lo - a:hi - a] = to_storage(z, w.dtype)

    jobs = [(k, c) for k in range(nstreams)
            for c in range(a // CHUNK_ROWS, (b + CHUNK_ROWS - 1) // CHUNK_ROWS)]
    if n > 0:
        with _pool() as ex:
            list(ex.map(block, jobs))
    out = {}
    if names is None:
        out["partials"] = out_arr[:w.R]
        out["residual"] = out_arr[w.R]
    else:
        for k, name in enumerate(names):
            out[name] = out_arr[k]
    if w.op != "rms_norm" and w.res_dtype != w.dtype:
        # the residual keeps its binary32 draws (stream R of the same blocks)
        k_res = w.R if w.op == "reduce_add_rms_norm" else 1
        res32 = np.empty((n, H), np.float32)

        def rblock(c):
            r0, r1 = c * CHUNK_ROWS, min((c + 1) * CHUNK_ROWS, T)
            z = _normal_f32(_rng(w.seed, k_res, c), (r1 - r0) * H).reshape(r1 - r0, H)
            lo, hi = max(r0, a), min(r1, b)
            z = z[lo - r0:hi - r0]
            if row_scale is not None:
                z = z * row_scale[lo:hi, None] * col_scale[None, :]
            res32[lo - a:hi - a] = z

        if n > 0:
            with _pool() as ex:
                list(ex.map(rblock, range(a // CHUNK_ROWS, (b + CHUNK_ROWS - 1) // CHUNK_ROWS)))
        out["residual"] = to_storage(res32, w.res_dtype)
    g = _rng(w.seed, GAMMA_KEY).uniform(0.5, 1.5, size=H).astype(np.float32)
    out["gamma"] = to_storage(g, w.dtype)
    return out
