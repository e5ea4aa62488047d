"""CPU oracle for the exact indexer top-k (test infrastructure only).

This module is a checker, not part of the product: only ``tests/``, the smoke
check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import
it. It shares no code with the CUDA path and imports nothing from it.

What it computes (the plain definition, not the algorithm):

  LiteTopK ("LiteTopK: Exploiting the Curse of Dimensionality for a Fused
  Indexer-TopK Kernel in Long-Context Sparse Attention", gist.science technical
  summary, "Declaración del Problema" / Problem Statement) states the
  Indexer-TopK problem: compute a relevance score for every candidate token of
  each query and return the top-k candidates.  Its "Contribuciones Clave"
  section and the arXiv abstract state that the fused kernel keeps *exact*
  top-k.  Because the method is exact, the oracle is the definition itself:

  1. score   I[t, s] = sum_h w[t, h] * max(0, sum_i q[t, h, i] * k[s, i])
     -- the DeepSeek Sparse Attention indexer score that the Problem Statement
     refers to; the pages name it I_{t,s} in the bin map of Methodology step 2.
     Only keys visible to the query are scored: s <= pos[t] (causal).
     Retrieval variant (the abstract's vector-retrieval use): H = 1, w = 1, no
     ReLU and no mask, i.e. a plain inner product.
  2. order the visible keys by (score descending, key index ascending);
  3. return the first min(k, V_t) (index, fp32 score) pairs, padded with
     (-1, -inf) up to k.

Inputs arrive as the device bit patterns (bf16 as uint16, fp8 e4m3 as uint8
codes with fp32 per-token scales) and are widened *exactly* to float64 here;
all arithmetic is float64.  The sample, bins, thresholds and candidate lists of
the method do not appear: they change the speed of the method, never its
result.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Exact widening of the device formats
# ---------------------------------------------------------------------------


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64.

    bf16 is the upper half of an IEEE-754 binary32: the value is the binary32
    whose high 16 bits are ``bits`` and whose low 16 bits are zero.
    """
    b32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b32.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP fp8 E4M3 codes -> float64, from the format's definition.

    Layout: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.  Exponent
    field 0 encodes subnormals m/8 * 2^(1-7); otherwise (1 + m/8) * 2^(e-7).
    E4M3 has no infinities; S.1111.111 is NaN.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    out = sign * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


def widen_queries(inputs) -> tuple[np.ndarray, np.ndarray]:
    """(q [T,H,d], w [T,H]) in float64 from an input bundle.

    bf16: q is the widened bf16 value.  fp8 e4m3 with per-token scales: the
    value of query t is code(q[t,h,i]) * q_scale[t] -- one fp32 scale per
    query token, shared by all its heads and dimensions.  w is fp32 in both
    formats and is never scaled.
    """
    w = np.asarray(inputs.w, dtype=np.float32).astype(np.float64)
    if inputs.dtype == "bf16":
        return bf16_to_f64(inputs.q), w
    if inputs.dtype == "fp8":
        qs = np.asarray(inputs.q_scale, np.float32).astype(np.float64)
        return e4m3_to_f64(inputs.q) * qs[:, None, None], w
    raise ValueError(inputs.dtype)


def widen_keys(inputs) -> np.ndarray:
    """k [S,d] in float64 from an input bundle.

    bf16: the widened bf16 value.  fp8 e4m3: code(k[s,i]) * k_scale[s], one
    fp32 scale per key token.
    """
    if inputs.dtype == "bf16":
        return bf16_to_f64(inputs.k)
    if inputs.dtype == "fp8":
        ks = np.asarray(inputs.k_scale, np.float32).astype(np.float64)
        return e4m3_to_f64(inputs.k) * ks[:, None]
    raise ValueError(inputs.dtype)


# ---------------------------------------------------------------------------
# Step 1: scores
# ---------------------------------------------------------------------------


def scores_one_query(q_t: np.ndarray, w_t: np.ndarray, keys: np.ndarray, relu: bool = True) -> np.ndarray:
    """I[s] = sum_h w[h] * max(0, q[h] . k[s]) for every row of ``keys`` (fp64).

    q_t: [H, d], w_t: [H], keys: [V, d].  The matmul is a library primitive;
    ReLU and the weighted head sum follow the formula term by term.
    """
    dots = keys @ q_t.T                       # [V, H]: q[h] . k[s]
    if relu:
        dots = np.maximum(dots, 0.0)
    return dots @ w_t                         # sum over heads, weighted


def visible_count(pos: int, S: int, causal: bool) -> int:
    """Number of keys a query at position ``pos`` may see (keys s <= pos)."""
    return min(int(pos) + 1, S) if causal else S


# ---------------------------------------------------------------------------
# Steps 2-3: exact ordering and the top-k
# ---------------------------------------------------------------------------


def exact_topk_row(scores: np.ndarray, k: int) -> tuple[np.ndarray, np.ndarray]:
    """Top-k of one row by (score desc, index asc); pads with (-1, -inf)."""
    V = scores.shape[0]
    order = np.lexsort((np.arange(V), -scores))   # primary: -score, secondary: index
    n = min(k, V)
    idx = np.full(k, -1, dtype=np.int32)
    val = np.full(k, -np.inf, dtype=np.float32)
    idx[:n] = order[:n]
    val[:n] = scores[order[:n]].astype(np.float32)
    return idx, val


def indexer_topk(inputs, k: int, causal: bool = True, relu: bool = True,
                 queries=None, keys64: np.ndarray | None = None):
    """Exact top-k for the chosen queries (all by default).

    Returns (idx int32 [n, k], score fp32 [n, k]).  ``keys64`` may pass the
    already-widened key matrix to avoid re-widening it for large contexts.
    """
    q, w = widen_queries(inputs)
    kk = widen_keys(inputs) if keys64 is None else keys64
    T = q.shape[0]
    S = kk.shape[0]
    sel = range(T) if queries is None else list(queries)
    out_idx = np.full((len(sel), k), -1, dtype=np.int32)
    out_val = np.full((len(sel), k), -np.inf, dtype=np.float32)
    for r, t in enumerate(sel):
        V = visible_count(inputs.positions[t], S, causal)
        if V <= 0:
            continue
        I = scores_one_query(q[t], w[t], kk[:V], relu)
        out_idx[r], out_val[r] = exact_topk_row(I, k)
    return out_idx, out_val


def full_scores(inputs, t: int, causal: bool = True, relu: bool = True,
                keys64: np.ndarray | None = None) -> np.ndarray:
    """All visible scores of query t in fp64 (used by tolerance checks)."""
    q, w = widen_queries(inputs)
    kk = widen_keys(inputs) if keys64 is None else keys64
    V = visible_count(inputs.positions[t], kk.shape[0], causal)
    return scores_one_query(q[t], w[t], kk[:V], relu)


# ---------------------------------------------------------------------------
# Retrieval variant: H = 1, w = 1, no ReLU, no mask
# ---------------------------------------------------------------------------


def retrieval_scores(queries_bits: np.ndarray, corpus_bits: np.ndarray,
                     rows=None, block: int = 1 << 18) -> np.ndarray:
    """fp64 inner products q . c of the chosen queries with every corpus row.

    The corpus is widened block by block so that large corpora fit in memory.
    """
    qs = bf16_to_f64(queries_bits)
    sel = range(qs.shape[0]) if rows is None else list(rows)
    qsel = qs[list(sel)]
    N = corpus_bits.shape[0]
    scores = np.empty((qsel.shape[0], N), dtype=np.float64)
    for b0 in range(0, N, block):
        blk = bf16_to_f64(corpus_bits[b0:b0 + block])
        scores[:, b0:b0 + blk.shape[0]] = qsel @ blk.T
    return scores


def retrieval_topk(queries_bits: np.ndarray, corpus_bits: np.ndarray, k: int,
                   rows=None, block: int = 1 << 18):
    """Exact top-k inner-product retrieval over a bf16 corpus (fp64 scores)."""
    scores = retrieval_scores(queries_bits, corpus_bits, rows=rows, block=block)
    out_idx = np.full((scores.shape[0], k), -1, dtype=np.int32)
    out_val = np.full((scores.shape[0], k), -np.inf, dtype=np.float32)
    for r in range(scores.shape[0]):
        out_idx[r], out_val[r] = exact_topk_row(scores[r], k)
    return out_idx, out_val
