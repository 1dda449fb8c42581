"""CPU oracle for dynamic sparse attention (indexer -> top-k -> sparse GQA attention).

TEST INFRASTRUCTURE ONLY. This module exists so that the tests, the smoke check
and the benchmark's CPU-baseline leg can check the CUDA library against a
plain, slow, obviously correct float64 restatement of what the method
computes. The library never imports, links or calls it, and it shares no code
with the library: it takes numpy arrays and returns numpy arrays.

Sources (public pull-request pages of ONNX Runtime's CUDA contrib ops):

* "[CUDA] Support FP16 KV cache and FP16 query/key in DynamicSparseAttention<
  BFloat16> and FP32 rotary cache / FP16 output in RMSNormRotary" (PR #33997),
  Description item 2: the op attends over a *selected* subset of the K/V cache
  (prefill and grouped GQA decode), with BF16/FP16 query and BF16/FP16 cache.
* "[CUDA] Optimize Qwen3.8-Flash-Next DSA, Indexer, HC, and QMoE kernels for
  SM12x and 256K context" (PR #33802), Summary items 1-2: the indexer scores
  every cached index key ("present_key_state") for each query token over 16
  index heads, in 2,048-key chunks, and a radix top-k (per-chunk partial
  histograms + one final merge-and-emit) picks the keys; INT8 KV cache with a
  value scale.
* Follow-up PR #33847 "... a large-value-scale accumulator", Description and
  Changes table: the online-softmax rescale must not lose earlier tiles when
  the running maximum rises by ~88 nats; worked example 2^120*e^-88/(1+e^-88).

The pages print no formula. The readings taken here (each also listed in the
design notes):

R1  positions: the cache holds T rows and the S new query tokens are its last
    S rows; query s sits at T-S+s and sees keys 0..T-S+s.
R2  indexer score (the form fixed for this library):
        score[t] = sum_h w[h] * max(0, qI[h] . kI[t])
    one index key per token shared by all index heads; no 1/sqrt(d) factor.
R3  top-k: k_eff = min(k, n) keys with the highest score; equal scores go to
    the lower index; emitted in ascending index order, padded with -1.
    -0.0 compares equal to +0.0.
R4  attention: head h uses KV head g = h // (Hq/Hkv) (consecutive grouping);
    logits = scale * q_h . K^[t,g] with scale = 1/sqrt(head_dim) unless given;
    exact softmax over the selected keys; out_h = sum_t p_t V^[t,g].
R5  INT8 cache: K^[t,g,:] = code[t,g,:] * k_scale[t,g] (same for V).
R11 cache append (the step before the indexer): the S new tokens of a
    sequence are written to cache rows T-S .. T-1 (R1). An INT8 cache stores,
    per token and KV head, scale = absmax/127 and code = clamp(rint(x /
    scale), -127, 127) with ties to even (scale 0 and codes 0 for an all-zero
    row). The codes are integers decided by floating point, so they are
    computed in fp32 (the kernel's precision): absmax and x are exact fp32
    values, scale and x / scale are IEEE fp32 divisions. A 16-bit cache of
    the other 16-bit type takes the value rounded to nearest even.
R12 paged caches (PR #33802's page, the companion 256K change: a pool of
    block_size-token blocks and a per-sequence block table): token t of
    sequence b is pool row table[b, t // block_size] * block_size
    + t % block_size; every result is the dense one on the gathered caches.
R13 RMSNorm + rotary embedding (PR #33997 Description item 1, the exact FP32
    RMSNormRotary): each head vector x (head_dim D) of a token at position p
    becomes y = x * gamma / sqrt(mean(x^2) + eps), then its first r dims are
    rotated in pairs (i, i + r/2), i < r/2, by the cache's angle for p:
    out_i = y_i cos[p,i] - y_{i+r/2} sin[p,i],
    out_{i+r/2} = y_{i+r/2} cos[p,i] + y_i sin[p,i]; dims r..D-1 stay y.
    Computed here exactly (float64); the library computes in fp32 and rounds
    once to the output type.
R14 floating auxiliary K/V (PR #33997: the op takes the step's own key and
    value as inputs beside the caches; its review notes that grouped attention
    can overflow BF16 auxiliary values when converting them to an FP16 cache's
    type, and the fix keeps floating auxiliary K/V with FP16 main caches): the
    S new tokens' K and V may be given as separate tensors k_aux, v_aux
    [B, S, Hkv, D] in the query's floating type. A selected key t of
    sequence b with t >= T_b - S (a new token, R1) then reads
    k_aux[b, t - (T_b - S)] and v_aux[...] at their own values -- never
    converted to the cache's type -- and every other selected key reads the
    cache. The indexer and the selection are unchanged.

Parity pins for every function live in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# positions (R1)
# ---------------------------------------------------------------------------
def visible_len(T: int, S: int, s: int) -> int:
    """Number of keys visible to query s of a sequence whose cache holds T rows
    with the S new tokens as its last rows: positions 0 .. T-S+s (R1)."""
    n = T - S + s + 1
    if n < 1:
        raise ValueError("query position precedes the cache start")
    return n


# ---------------------------------------------------------------------------
# indexer (R2) -- PR #33802 Summary item 2, PackedSparseAttentionIndexer
# ---------------------------------------------------------------------------
def index_scores_row(qI_s: np.ndarray, w_s: np.ndarray, kI_b: np.ndarray,
                     n: int) -> np.ndarray:
    """Scores of keys 0..n-1 for one query token.

    qI_s [HI, DI], w_s [HI], kI_b [cap, DI] (float64 copies of the stored
    values). Returns float64 [n]: sum_h w[h] * max(0, qI[h] . kI[t]).
    """
    dots = kI_b[:n] @ qI_s.T                      # [n, HI]: qI_h . kI_t
    return np.maximum(dots, 0.0) @ w_s            # sum_h w_h * ReLU(.)


def index_scores(qI, w, kI, total_len, rows=None) -> np.ndarray:
    """Indexer scores for every query token.

    qI [B,S,HI,DI], w [B,S,HI], kI [B,cap,DI], total_len [B] (T_b).
    Returns float64 [B,S,cap]; entries past a query's visible length are NaN.
    ``rows`` optionally restricts the work to a list of (b, s) pairs (the
    others stay NaN) for workloads too large to score in full on a CPU.
    """
    B, S = qI.shape[:2]
    cap = kI.shape[1]
    out = np.full((B, S, cap), np.nan)
    todo = rows if rows is not None else [(b, s) for b in range(B) for s in range(S)]
    for b, s in todo:
        n = visible_len(int(total_len[b]), S, s)
        out[b, s, :n] = index_scores_row(qI[b, s], w[b, s], kI[b], n)
    return out


# ---------------------------------------------------------------------------
# top-k selection (R3) -- PR #33802 Summary item 2 (radix partial top-k over
# 2,048-key chunks + final merge-and-emit); the chunking only changes speed,
# not the selected set, so the oracle selects over the whole row at once.
# ---------------------------------------------------------------------------
def topk_select_row(scores: np.ndarray, k: int) -> np.ndarray:
    """Select min(k, n) indices of the highest values of a 1-D array.

    Values are compared exactly (pass fp32 values as float64 to compare fp32
    numbers bit for bit); -0.0 equals +0.0; among equal values the lower index
    wins. Returns int64 [k]: the selected indices ascending, then -1s.
    """
    v = np.asarray(scores, dtype=np.float64) + 0.0   # -0.0 + 0.0 == +0.0
    n = v.shape[0]
    if np.isnan(v).any():
        raise ValueError("NaN scores have no defined order")
    keff = min(k, n)
    # sort by value descending, then index ascending
    order = np.lexsort((np.arange(n), -v))
    sel = np.sort(order[:keff])
    out = np.full(k, -1, dtype=np.int64)
    out[:keff] = sel
    return out


def topk(scores, total_len, k: int, rows=None) -> np.ndarray:
    """Top-k for every query row of a [B,S,cap] score tensor (only the visible
    prefix of each row takes part). Returns int64 [B,S,k]."""
    B, S = scores.shape[:2]
    out = np.full((B, S, k), -1, dtype=np.int64)
    todo = rows if rows is not None else [(b, s) for b in range(B) for s in range(S)]
    for b, s in todo:
        n = visible_len(int(total_len[b]), S, s)
        out[b, s] = topk_select_row(scores[b, s, :n], k)
    return out


# ---------------------------------------------------------------------------
# sparse GQA attention (R4, R5) -- PR #33997 Description item 2 (prefill and
# grouped decode over the selected rows), PR #33802 Summary item 1 (INT8 cache)
# ---------------------------------------------------------------------------
def dequantize(codes: np.ndarray, scale) -> np.ndarray:
    """K^ = code * scale per token and head (R5); scale None means the cache
    already stores values (BF16/FP16)."""
    if scale is None:
        return codes
    return codes * scale[..., None]


def attend_row(q_h: np.ndarray, Kg: np.ndarray, Vg: np.ndarray,
               scale: float) -> np.ndarray:
    """Exact softmax attention of one query head over a set of rows.

    q_h [D], Kg/Vg [m, D] (dequantised selected rows). Returns float64 [D].
    """
    logits = scale * (Kg @ q_h)
    mx = logits.max()
    p = np.exp(logits - mx)
    p /= p.sum()
    return p @ Vg


def sparse_attention(q, k, v, idx, num_kv_heads: int, k_scale=None,
                     v_scale=None, softmax_scale: float = 0.0,
                     rows=None) -> np.ndarray:
    """Softmax attention of each query head over its query token's selected
    rows.

    q [B,S,Hq,D]; k, v [B,cap,Hkv,D] (values, or INT8 codes with k_scale /
    v_scale [B,cap,Hkv]); idx [B,S,k] (selected indices, -1 = unused).
    Returns float64 [B,S,Hq,D] (rows not in ``rows`` stay NaN).
    """
    B, S, Hq, D = q.shape
    G = Hq // num_kv_heads
    scale = softmax_scale if softmax_scale else 1.0 / np.sqrt(D)
    out = np.full(q.shape, np.nan)
    todo = rows if rows is not None else [(b, s) for b in range(B) for s in range(S)]
    for b, s in todo:
        sel = idx[b, s]
        sel = sel[sel >= 0]
        Kb = dequantize(k[b, sel], None if k_scale is None else k_scale[b, sel])
        Vb = dequantize(v[b, sel], None if v_scale is None else v_scale[b, sel])
        for h in range(Hq):
            g = h // G
            out[b, s, h] = attend_row(q[b, s, h], Kb[:, g], Vb[:, g], scale)
    return out


def sparse_attention_aux(q, k, v, idx, num_kv_heads: int, k_aux, v_aux, total_len,
                         k_scale=None, v_scale=None, softmax_scale: float = 0.0,
                         rows=None) -> np.ndarray:
    """Sparse attention with floating auxiliary K/V for the new tokens (R14).

    As sparse_attention, except that a selected key t of sequence b with
    t >= T_b - S takes its K and V from k_aux / v_aux [B,S,Hkv,D] at row
    t - (T_b - S), as the values given (no conversion to the cache type).
    Returns float64 [B,S,Hq,D] (rows not in ``rows`` stay NaN).
    """
    B, S, Hq, D = q.shape
    G = Hq // num_kv_heads
    scale = softmax_scale if softmax_scale else 1.0 / np.sqrt(D)
    out = np.full(q.shape, np.nan)
    todo = rows if rows is not None else [(b, s) for b in range(B) for s in range(S)]
    for b, s in todo:
        past = int(total_len[b]) - S          # the first new token's position
        sel = idx[b, s]
        sel = sel[sel >= 0]
        Kb = dequantize(k[b, sel], None if k_scale is None else k_scale[b, sel])
        Vb = dequantize(v[b, sel], None if v_scale is None else v_scale[b, sel])
        for j, t in enumerate(sel):
            if t >= past:
                Kb[j] = k_aux[b, t - past]
                Vb[j] = v_aux[b, t - past]
        for h in range(Hq):
            g = h // G
            out[b, s, h] = attend_row(q[b, s, h], Kb[:, g], Vb[:, g], scale)
    return out


# ---------------------------------------------------------------------------
# the whole step
# ---------------------------------------------------------------------------
def sparse_attention_step(inp: dict, num_kv_heads: int, top_k: int,
                          softmax_scale: float = 0.0, rows=None) -> dict:
    """Indexer -> top-k -> sparse attention for one batch of query tokens.

    ``inp`` holds float64 arrays qI, w, kI, q, k, v, k_scale, v_scale (None
    unless INT8) and total_len. Returns dict(scores, idx, out).
    """
    T = inp["total_len"]
    scores = index_scores(inp["qI"], inp["w"], inp["kI"], T, rows=rows)
    idx = topk(scores, T, top_k, rows=rows)
    out = sparse_attention(inp["q"], inp["k"], inp["v"], idx, num_kv_heads,
                           inp.get("k_scale"), inp.get("v_scale"),
                           softmax_scale, rows=rows)
    return {"scores": scores, "idx": idx, "out": out}


# ---------------------------------------------------------------------------
# cache append (R11)
# ---------------------------------------------------------------------------
def quantize_row_int8(x) -> tuple:
    """One token's KV-head row (any length) -> (int8 codes, fp32 scale), with
    every decision in fp32 as R11 states."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0.0)
    scale = np.float32(amax / np.float32(127.0))
    if scale == np.float32(0.0):
        return np.zeros(x32.shape, dtype=np.int8), np.float32(0.0)
    q = np.rint(x32 / scale).astype(np.float32)          # fp32 division, ties to even
    return np.clip(q, -127, 127).astype(np.int8), scale


def round_to(values, dtype: str) -> np.ndarray:
    """float64 values rounded (nearest, ties to even) to bf16 / fp16 / fp32 and
    returned as float64. Uses torch's CPU casts as the rounding routine."""
    import torch
    t = torch.as_tensor(np.asarray(values, dtype=np.float64))
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[dtype]
    return t.to(torch.float32).to(tdt).to(torch.float64).numpy()


def cache_append(kI, k, v, k_scale, v_scale, kI_new, k_new, v_new, total_len, kv_dtype: str):
    """Write the S new tokens of every sequence into copies of the caches (R11).

    kI [B,cap,64], k/v [B,cap,Hkv,128] (INT8: codes as float64), k_scale /
    v_scale [B,cap,Hkv] (INT8 only, else None); kI_new [B,S,64], k_new / v_new
    [B,S,Hkv,128] exact float64 values; total_len [B]. Returns the updated
    (kI, k, v, k_scale, v_scale).
    """
    kI, k, v = kI.copy(), k.copy(), v.copy()
    k_scale = None if k_scale is None else k_scale.copy()
    v_scale = None if v_scale is None else v_scale.copy()
    B, S = k_new.shape[0], k_new.shape[1]
    Hkv = k_new.shape[2]
    for b in range(B):
        for s in range(S):
            t = int(total_len[b]) - S + s                    # R1: the last S rows
            if t < 0:
                raise ValueError("new tokens precede the cache start")
            kI[b, t] = kI_new[b, s]                          # bf16 to bf16: a copy
            for g in range(Hkv):
                for dst, dsc, src in ((k, k_scale, k_new), (v, v_scale, v_new)):
                    if kv_dtype == "int8":
                        codes, sc = quantize_row_int8(src[b, s, g])
                        dst[b, t, g] = codes.astype(np.float64)
                        dsc[b, t, g] = float(sc)
                    else:
                        dst[b, t, g] = round_to(src[b, s, g], kv_dtype)
    return kI, k, v, k_scale, v_scale


# ---------------------------------------------------------------------------
# paged caches (R12)
# ---------------------------------------------------------------------------
def gather_pages(pool, table, block_size: int, total_len):
    """Logical [B, cap, ...] cache of a paged pool: row t of sequence b is
    pool[table[b, t // block_size] * block_size + t % block_size] for
    t < total_len[b]; rows past a sequence's length are zero (never read)."""
    pool = np.asarray(pool)
    table = np.asarray(table)
    B, per_seq = table.shape
    cap = per_seq * block_size
    out = np.zeros((B, cap) + pool.shape[1:], dtype=np.float64)
    for b in range(B):
        for t in range(int(total_len[b])):
            out[b, t] = pool[table[b, t // block_size] * block_size + t % block_size]
    return out


# ---------------------------------------------------------------------------
# RMSNorm + rotary embedding (R13)
# ---------------------------------------------------------------------------
def rmsnorm_rotary(x, gamma, eps: float, cos, sin, positions, rotary_dim: int):
    """x [N, H, D] (exact values of the stored input), gamma [D], cos / sin
    [max_pos, rotary_dim / 2], positions [N]. Returns float64 [N, H, D]:
    per head vector, RMS normalisation with weight gamma, then the rotate-half
    rotation of the first rotary_dim dims by the token's cached angle."""
    x = np.asarray(x, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    y = x / np.sqrt(ms + eps) * gamma
    out = y.copy()
    h = rotary_dim // 2
    if h == 0:
        return out
    pos = np.asarray(positions, dtype=np.int64)
    c = np.asarray(cos, dtype=np.float64)[pos][:, None, :]     # [N, 1, h]
    s = np.asarray(sin, dtype=np.float64)[pos][:, None, :]
    a, b = y[..., :h], y[..., h:rotary_dim]
    out[..., :h] = a * c - b * s
    out[..., h:rotary_dim] = b * c + a * s
    return out
