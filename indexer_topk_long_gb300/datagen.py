"""Seeded synthetic inputs for the indexer top-k path.

This module only *generates inputs*. It holds none of the method's arithmetic
(no scoring, binning, thresholding or selection), so both the CUDA path and the
CPU oracle may consume what it returns.

Workload shapes follow the LiteTopK summaries (gist.science, "Resultados
Experimentales" / "Experimental Results"): 8192-token prefill chunks at 128K,
256K and 1M context with k = 2048, plus a high-dimensional vector-retrieval
workload. The datasets the pages use (GLM-5.2 long-context traces, MSMARCO) are
not available, so the generators below synthesise data with the property the
method relies on (scores concentrated in a narrow range with a long tail, the
"curse of dimensionality" of the pages' Methodology section).

Key/query recipe (indexer workloads):
  * keys  k[s] ~ N(0, 1)^d; a seeded 1% of positions ("hot" keys) get
    +3 * u_g, where u_g is a random unit vector of the 8192-key segment g that
    contains s;
  * queries q[t, h] ~ N(0, 1)/sqrt(d) + 1.5 * u_g for the segment g holding the
    query's position; the noise is independent per head, u_g is shared;
  * w[t, h] ~ U(0, 1) / 8;
  * integer mode: q, k rounded to integers in [-3, 3], w = 2^-e, e ~ U{1..4},
    so that fp32 accumulation in any order is exact.
Keys are generated per 8192-key segment from a stream keyed on (seed, segment),
so the key cache of a shorter context is a prefix of a longer one and two
consecutive chunks see the same keys.

Rounding to the device formats:
  * bf16: round-to-nearest-even of the fp32 value (bit manipulation below);
  * fp8 e4m3 (OCP 8-bit float, 4 exponent bits, bias 7, 3 mantissa bits,
    max finite 448, no infinities): per-token scale = amax / 448, value / scale
    rounded to the nearest representable e4m3 value, ties to even code.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

SEGMENT = 8192            # keys per topic segment
DEFAULT_SEED = 20260715

# ---------------------------------------------------------------------------
# Named workloads (positions are the absolute positions of the chunk's queries)
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class Workload:
    name: str
    T: int                 # queries in the chunk
    first_pos: int         # absolute position of query 0
    S: int                 # keys in the cache (= last position + 1)
    H: int = 64
    d: int = 128
    k: int = 2048
    sample_size: int = 6144

    @property
    def positions(self) -> np.ndarray:
        return np.arange(self.first_pos, self.first_pos + self.T, dtype=np.int32)

    @property
    def visible_pairs(self) -> int:
        p = self.positions.astype(np.int64)
        return int(np.minimum(p + 1, self.S).sum())


WORKLOADS = {
    "tiny": Workload("tiny", T=32, first_pos=8160, S=8192),
    "128k_chunk1": Workload("128k_chunk1", T=8192, first_pos=114688, S=122880),
    "128k_chunk2": Workload("128k_chunk2", T=8192, first_pos=122880, S=131072),
    "256k_prev": Workload("256k_prev", T=8192, first_pos=245760, S=253952),
    "256k": Workload("256k", T=8192, first_pos=253952, S=262144),
    "1m_prev": Workload("1m_prev", T=8192, first_pos=1032192, S=1040384),
    "1m": Workload("1m", T=8192, first_pos=1040384, S=1048576),
}


# ---------------------------------------------------------------------------
# Rounding helpers (input formats, not method arithmetic)
# ---------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def _e4m3_positive_table() -> np.ndarray:
    """Values of codes 0x00..0x7E (all non-negative finite e4m3 numbers)."""
    vals = np.empty(0x7F, dtype=np.float64)
    for code in range(0x7F):
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0:
            vals[code] = (m / 8.0) * 2.0 ** (1 - 7)
        else:
            vals[code] = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_E4M3_POS = _e4m3_positive_table()


def _e4m3_codes_block(x: np.ndarray) -> np.ndarray:
    """e4m3 codes of one block (float64 values, |x| <= 448 after saturation).

    Normal range: the binary64 significand is rounded to 3 bits, ties to even
    (adding 2^48 - 1 plus the kept LSB, then dropping 49 bits; a carry moves
    into the exponent field), and the exponent is re-biased from 1023 to 7.
    Below 2^-6 the e4m3 quantum is 2^-9, so the code is round-half-even of
    |x| * 512.  Ties to the even value are ties to the even code."""
    a = np.minimum(np.abs(x), 448.0)
    b = a.view(np.uint64)
    rb = (b + (np.uint64((1 << 48) - 1) + ((b >> np.uint64(49)) & np.uint64(1)))) >> np.uint64(49)
    code = rb.astype(np.int64) - ((1023 - 7) << 3)
    sub = a < 2.0 ** -6
    code = np.where(sub, np.rint(a * 512.0).astype(np.int64), code).astype(np.uint8)
    sign = (x < 0) & (code != 0)
    return code | (sign.astype(np.uint8) << np.uint8(7))


def _blocks(n: int, block: int):
    return [(i, min(n, i + block)) for i in range(0, n, block)]


def _threads() -> int:
    import os
    return max(1, min(16, os.cpu_count() or 1))


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    """float -> e4m3 codes (uint8), nearest value, ties to the even code.

    Magnitudes above 448 saturate to 448 (the generator never produces them,
    since values are pre-divided by amax / 448).  Large arrays are encoded in
    blocks on a thread pool (numpy releases the GIL)."""
    flat = np.asarray(x, dtype=np.float64).reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    parts = _blocks(flat.size, 1 << 22)
    if len(parts) <= 1:
        out[:] = _e4m3_codes_block(flat)
    else:
        from concurrent.futures import ThreadPoolExecutor

        def run(ab):
            out[ab[0]:ab[1]] = _e4m3_codes_block(flat[ab[0]:ab[1]])
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(run, parts))
    return out.reshape(np.shape(x))


def fp8_quantize_rows(x: np.ndarray):
    """Per-row (per-token) e4m3 quantisation: returns (codes, scale fp32)."""
    x = np.asarray(x, dtype=np.float32)
    rows = x.reshape(x.shape[0], -1)
    n, m = rows.shape
    codes = np.empty((n, m), dtype=np.uint8)
    scale = np.empty(n, dtype=np.float32)

    def run(ab):
        r = rows[ab[0]:ab[1]]
        amax = np.abs(r).max(axis=1).astype(np.float32) if m else np.zeros(len(r), np.float32)
        sc = (np.maximum(amax, np.float32(1e-12)) / np.float32(448.0)).astype(np.float32)
        scale[ab[0]:ab[1]] = sc
        codes[ab[0]:ab[1]] = _e4m3_codes_block(r.astype(np.float64) / sc[:, None].astype(np.float64))
    parts = _blocks(n, max(1, (1 << 21) // max(m, 1)))
    if len(parts) <= 1:
        for ab in parts:
            run(ab)
    else:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(run, parts))
    return codes.reshape(x.shape), scale


# ---------------------------------------------------------------------------
# Random streams
# ---------------------------------------------------------------------------

def _rng(seed: int, *tags: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *tags])))


_TAG_KEYS, _TAG_TOPIC, _TAG_QUERY, _TAG_W, _TAG_HOT = 1, 2, 3, 4, 5


def topic_vector(seed: int, segment: int, d: int) -> np.ndarray:
    u = _rng(seed, _TAG_TOPIC, segment).standard_normal(d)
    return (u / np.linalg.norm(u)).astype(np.float32)


def keys_fp32(S: int, d: int = 128, seed: int = DEFAULT_SEED, hot_frac: float = 0.01) -> np.ndarray:
    """k[s] ~ N(0,1)^d with 1% hot positions pushed along the segment topic."""
    out = np.empty((S, d), dtype=np.float32)
    for g in range((S + SEGMENT - 1) // SEGMENT):
        a, b = g * SEGMENT, min(S, (g + 1) * SEGMENT)
        full = _rng(seed, _TAG_KEYS, g).standard_normal((SEGMENT, d), dtype=np.float32)
        hot = _rng(seed, _TAG_HOT, g).random(SEGMENT) < hot_frac
        full[hot] += 3.0 * topic_vector(seed, g, d)
        out[a:b] = full[: b - a]
    return out


def queries_fp32(positions: np.ndarray, H: int = 64, d: int = 128, seed: int = DEFAULT_SEED) -> np.ndarray:
    """q[t,h] ~ N(0,1)/sqrt(d) + 1.5 * u(segment of pos[t])."""
    positions = np.asarray(positions, dtype=np.int64)
    T = positions.shape[0]
    rng = _rng(seed, _TAG_QUERY, int(positions[0]) if T else 0, T)
    q = rng.standard_normal((T, H, d), dtype=np.float32) / np.float32(np.sqrt(d))
    segs = positions // SEGMENT
    for g in np.unique(segs):
        q[segs == g] += 1.5 * topic_vector(seed, int(g), d)[None, None, :]
    return q


def weights_fp32(T: int, H: int = 64, seed: int = DEFAULT_SEED, first_pos: int = 0) -> np.ndarray:
    rng = _rng(seed, _TAG_W, first_pos, T)
    return (rng.random((T, H), dtype=np.float32) / np.float32(8.0)).astype(np.float32)


def integer_mode(q: np.ndarray, k: np.ndarray, T: int, H: int, seed: int, first_pos: int):
    """Small-integer q, k in [-3, 3] and power-of-two w (exact fp32 sums)."""
    d = q.shape[-1]
    qi = np.clip(np.rint(q * np.float32(np.sqrt(d))), -3, 3).astype(np.float32)
    ki = np.clip(np.rint(k), -3, 3).astype(np.float32)
    e = _rng(seed, _TAG_W, first_pos, T, 7).integers(1, 5, size=(T, H))
    wi = np.ldexp(np.ones((T, H), dtype=np.float32), -e).astype(np.float32)
    return qi, ki, wi


@dataclass
class IndexerInputs:
    """One chunk's inputs. Device formats are bit patterns plus fp32 scales."""
    dtype: str                    # "bf16" or "fp8"
    q: np.ndarray                 # bf16: uint16 [T,H,d]; fp8: uint8 [T,H,d]
    k: np.ndarray                 # bf16: uint16 [S,d];   fp8: uint8 [S,d]
    w: np.ndarray                 # fp32 [T,H]
    positions: np.ndarray         # int32 [T]
    q_scale: np.ndarray | None = None   # fp32 [T]   (fp8 only)
    k_scale: np.ndarray | None = None   # fp32 [S]   (fp8 only)

    @property
    def T(self) -> int:
        return self.q.shape[0]

    @property
    def S(self) -> int:
        return self.k.shape[0]


def make_indexer_inputs(T: int, first_pos: int, S: int, H: int = 64, d: int = 128,
                        seed: int = DEFAULT_SEED, dtype: str = "bf16",
                        integer: bool = False, positions: np.ndarray | None = None,
                        keys: np.ndarray | None = None) -> IndexerInputs:
    """Inputs of one chunk. ``keys`` may pass a pre-generated fp32 key cache."""
    if positions is None:
        positions = np.arange(first_pos, first_pos + T, dtype=np.int32)
    positions = np.asarray(positions, dtype=np.int32)
    kf = keys_fp32(S, d, seed) if keys is None else keys[:S]
    qf = queries_fp32(positions, H, d, seed)
    wf = weights_fp32(T, H, seed, first_pos)
    if integer:
        qf, kf, wf = integer_mode(qf, kf, T, H, seed, first_pos)
    if dtype == "bf16":
        return IndexerInputs("bf16", bf16_bits(qf), bf16_bits(kf), wf, positions)
    if dtype == "fp8":
        q8, qs = fp8_quantize_rows(qf)
        k8, ks = fp8_quantize_rows(kf)
        return IndexerInputs("fp8", q8, k8, wf, positions, qs, ks)
    raise ValueError(f"unknown dtype {dtype}")


def workload_inputs(name: str, seed: int = DEFAULT_SEED, dtype: str = "bf16",
                    integer: bool = False, keys: np.ndarray | None = None) -> IndexerInputs:
    wl = WORKLOADS[name]
    return make_indexer_inputs(wl.T, wl.first_pos, wl.S, wl.H, wl.d, seed, dtype, integer,
                               keys=keys)


# ---------------------------------------------------------------------------
# Vector retrieval workload (H = 1, plain inner product, no causal mask)
# ---------------------------------------------------------------------------

def retrieval_corpus_block(row0: int, rows: int, d: int = 768, n_centroids: int = 4096,
                           seed: int = DEFAULT_SEED, block: int = 65536) -> np.ndarray:
    """Rows [row0, row0+rows) of the clustered corpus: 0.3*centroid + N(0,1).

    Generated per ``block`` rows from a stream keyed on the block index, so any
    slice is reproducible on its own.
    """
    cents = _rng(seed, 11).standard_normal((n_centroids, d), dtype=np.float32)
    out = np.empty((rows, d), dtype=np.float32)
    r = row0
    while r < row0 + rows:
        blk = r // block
        b0 = blk * block
        rng = _rng(seed, 12, blk)
        assign = rng.integers(0, n_centroids, size=block)
        noise = rng.standard_normal((block, d), dtype=np.float32)
        hi = min(row0 + rows, b0 + block)
        sl = slice(r - b0, hi - b0)
        out[r - row0: hi - row0] = np.float32(0.3) * cents[assign[sl]] + noise[sl]
        r = hi
    return out


def retrieval_queries(n: int = 1024, d: int = 768, n_centroids: int = 4096,
                      seed: int = DEFAULT_SEED) -> np.ndarray:
    cents = _rng(seed, 11).standard_normal((n_centroids, d), dtype=np.float32)
    rng = _rng(seed, 13)
    pick = rng.integers(0, n_centroids, size=n)
    return (np.float32(0.3) * cents[pick] + rng.standard_normal((n, d), dtype=np.float32)).astype(np.float32)


def retrieval_inputs_torch(n_corpus: int = 8388608, n_queries: int = 1024, d: int = 768,
                           n_centroids: int = 4096, seed: int = DEFAULT_SEED, device="cuda"):
    """The retrieval workload generated on a device with a seeded torch
    generator (a 12.9 GB corpus is impractical to draw with numpy): corpus rows
    0.3 * centroid + N(0, 1) over random centroids, queries 0.3 * c + N(0, 1)
    near random centroids, both rounded to bf16.  Returns (queries, corpus) as
    bf16 tensors on ``device``; copy them to the host to feed the oracle."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    cents = torch.randn((n_centroids, d), generator=g, device=device)
    corpus = torch.empty((n_corpus, d), dtype=torch.bfloat16, device=device)
    step = 1 << 20
    for r0 in range(0, n_corpus, step):
        r1 = min(n_corpus, r0 + step)
        a = torch.randint(0, n_centroids, (r1 - r0,), generator=g, device=device)
        x = torch.randn((r1 - r0, d), generator=g, device=device)
        corpus[r0:r1] = (0.3 * cents[a] + x).to(torch.bfloat16)
    pick = torch.randint(0, n_centroids, (n_queries,), generator=g, device=device)
    queries = (0.3 * cents[pick] + torch.randn((n_queries, d), generator=g, device=device)).to(torch.bfloat16)
    return queries, corpus
