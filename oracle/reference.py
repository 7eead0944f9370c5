"""Plain fp64 CPU oracle for chunked prefill attention with past.

TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the bench's
CPU-baseline / reference leg import this module.  It shares no code with the
CUDA library and never calls it.

Sources (page title, section):
  [P1] "functiongemma: chunk prefill-with-past graph gemma_prefill_with_past"
       (SKaiNET-transformers PR 417) -- Why; Change (additive); Validation.
  [P2] "[quanization] Enable prefill-decode modeling" (Samsung TICO issue 586)
       -- Runtime behavior; Mask/cache layout used in the runtime.
  [P4] "Pad the chunked-prefill tail for sliding-window models"
       (cactus PR 716) -- Problem; Fix; review sweep table; Declined with rationale.

Readings taken where the pages are silent (each is listed with its reason in
the design notes):
  rotate-half pairing (d, d+D/2); fp32 multiply / add / subtract with no fused
  multiply-add, rounded to bf16 to nearest-even; scale = 1/sqrt(D) unless
  given; an additive mask entry <= -1e29 is "masked"; a row with no unmasked
  key outputs zeros; implicit visibility: past slot j visible iff j < L and
  (L+i) - j < W; chunk row t visible iff t < n, t <= i (causal) and |i - t| < W;
  W = 0 disables the window; key columns are past slots first, then chunk rows.

bf16 tensors are passed as numpy uint16 arrays of raw bit patterns.

A cache may hold fp16 instead of bf16 (kv="f16"; the padded-tail page
mentions a runtime option that stores the KV cache in fp16).  Reading taken:
the rotation arithmetic is unchanged and only its final rounding is to fp16;
V rows are converted bf16 -> fp16 to nearest-even; the attention then sees Q
and the chunk keys rotated to fp16 as well (one precision for all products),
and values in fp16.  fp16 cache arrays are uint16 bit patterns too.

Parity: every function here is pinned by tests/test_oracle_pins.py and
tests/test_oracle_invariants.py (closed forms, invariants, a library routine
on the special cases that reduce to textbook attention, brute force).
"""
from __future__ import annotations

import numpy as np

MASKED = -1e30          # the additive value the pages give for "masked" [P1, Change]
MASK_LIMIT = -1e29      # an entry at or below this counts as masked

__all__ = [
    "MASKED", "MASK_LIMIT", "bf16_to_f32", "f32_to_bf16", "f16_to_f32", "f32_to_f16", "rope_rotate",
    "visible", "explicit_mask", "attend", "chunk_prefill_attn", "decode_step",
    "kv_append_global", "kv_append_sliding", "snapshot_padded_append",
    "rollback_padded_append", "select_argmax", "kv_to_f32", "to_kv",
]


# ---------------------------------------------------------------- bf16 bits

def bf16_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact widening)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32)
    return (b << np.uint32(16)).view(np.float32)


def f32_to_bf16(x) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest, ties to even (finite inputs)."""
    u = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def f16_to_f32(bits) -> np.ndarray:
    """IEEE half bit patterns -> float32 (exact widening)."""
    return np.ascontiguousarray(np.asarray(bits, dtype=np.uint16)).view(np.float16).astype(np.float32)


def f32_to_f16(x) -> np.ndarray:
    """float32 -> IEEE half bit patterns, round to nearest, ties to even
    (numpy's IEEE conversion; beyond the half range it gives +-inf)."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def kv_to_f32(bits, kv: str = "bf16") -> np.ndarray:
    """Cache-format bit patterns (bf16 or f16) -> float32."""
    return bf16_to_f32(bits) if kv == "bf16" else f16_to_f32(bits)


def to_kv(bf16_bits, kv: str = "bf16") -> np.ndarray:
    """bf16 bit patterns in the cache format (f16: nearest-even conversion)."""
    return np.asarray(bf16_bits, dtype=np.uint16) if kv == "bf16" else f32_to_f16(bf16_to_f32(bf16_bits))


# ---------------------------------------------------------------- RoPE

def rope_rotate(x_bits, cos, sin, out: str = "bf16") -> np.ndarray:
    """Rotate bf16 rows with per-row cos/sin tables; returns bf16 bits (or f16
    bits with out="f16": the same fp32 values, rounded to half).

    [P1, Change]: RoPE from per-position [C, headDim] cos/sin tables.
    [P2, Runtime behavior]: position_embeddings = (cos_t, sin_t).
    With x the bf16 row widened to fp32 and h = D/2, for d < h:
        y[d]   = bf16( x[d]   * cos[d]   - x[d+h] * sin[d]   )
        y[d+h] = bf16( x[d+h] * cos[d+h] + x[d]   * sin[d+h] )
    each product and the sum/difference rounded to fp32 separately.
    cos/sin broadcast against x's leading axes; their last axis is D.
    """
    x = bf16_to_f32(x_bits)
    c = np.asarray(cos, dtype=np.float32)
    s = np.asarray(sin, dtype=np.float32)
    h = x.shape[-1] // 2
    lo, hi = x[..., :h], x[..., h:]
    y_lo = np.subtract(np.multiply(lo, c[..., :h]), np.multiply(hi, s[..., :h]))
    y_hi = np.add(np.multiply(hi, c[..., h:]), np.multiply(lo, s[..., h:]))
    y = np.concatenate([y_lo, y_hi], axis=-1)
    return f32_to_bf16(y) if out == "bf16" else f32_to_f16(y)


# ---------------------------------------------------------------- masks

def visible(L: int, n: int, C: int, P: int, window: int, causal: int, sink: int = 0) -> np.ndarray:
    """Boolean [C, P+C]: which key columns query row i may attend to.

    [P1, Change]: the mask carries the causal band inside the chunk, the zero
    padding and the sliding window.  [P2, Mask/cache layout]: past tokens are
    packed into the first past_len slots; unfilled slots stay masked; the
    current token is visible.  Query row i sits at position L + i; past slot j
    at position j; chunk row t at position L + t.

    Sinks ("Pad the chunked-prefill tail for sliding-window models", Fix and
    review: the sliding cache keeps S pinned sink rows in slots [0, S) and
    compacts the rest chronologically).  Reading: the pinned rows are visible
    to every query row whatever the window; a non-sink slot j holds the token
    L - j rows before the chunk (compaction keeps the newest rows contiguous
    and ending at slot L - 1), so the window rule on L + i - j applies to it
    unchanged.  sink = 0 is the plain rule.
    """
    i = np.arange(C)[:, None]
    pos_q = L + i
    j = np.arange(P)[None, :]
    past = j < L
    t = np.arange(C)[None, :]
    chunk = t < n
    if causal:
        chunk = chunk & (t <= i)
    if window > 0:
        past = past & ((np.abs(pos_q - j) < window) | (j < sink))
        chunk = chunk & (np.abs(pos_q - (L + t)) < window)
    return np.concatenate([np.broadcast_to(past, (C, P)),
                           np.broadcast_to(chunk, (C, C))], axis=1)


def explicit_mask(L: int, n: int, C: int, P: int, window: int, causal: int, sink: int = 0) -> np.ndarray:
    """The additive fp32 mask [C, P+C] a caller builds: 0 = attend, -1e30 = masked [P1]."""
    return np.where(visible(L, n, C, P, window, causal, sink), np.float32(0.0),
                    np.float32(MASKED)).astype(np.float32)


# ---------------------------------------------------------------- attention

def attend(q, keys, values, add_mask, scale: float) -> np.ndarray:
    """Softmax attention of query rows over key rows under an additive mask, fp64.

    z[r, c] = scale * <q_r, k_c> + mask[r, c]; the softmax runs over the
    columns whose mask entry is above -1e29; a row with no such column
    returns zeros.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(keys, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64)
    m = np.asarray(add_mask, dtype=np.float64)
    z = (q @ k.T) * scale + m
    live = m > MASK_LIMIT
    out = np.zeros((q.shape[0], v.shape[1]), dtype=np.float64)
    for r in range(q.shape[0]):
        cols = np.nonzero(live[r])[0]
        if cols.size == 0:
            continue
        zr = z[r, cols]
        w = np.exp(zr - zr.max())
        out[r] = (w @ v[cols]) / w.sum()
    return out


def chunk_prefill_attn(q, k_new, v_new, cos, sin, cache_k, cache_v, P, past_len, n_real,
                       window=0, causal=1, mask=None, scale=None, sel_row=None, sink=0, kv="bf16"):
    """One chunk of C rows attending over P cached slots plus the chunk itself.

    [P1, Change]: heads-first [heads, C, headDim] Q/K/V, RoPE from the cos/sin
    tables, attention over past + C keys with a per-head additive mask
    [1, nHeads, C, past+C], K/V extended by the chunk, one-hot select of a row.
    GQA: q head h reads kv head h // (Hq // Hkv).

    q [B,Hq,C,D], k_new/v_new [B,Hkv,C,D]: bf16 bits; cache_k/cache_v
    [B,Hkv,>=P,D]: bits in the cache format kv ("bf16" or "f16").
    cos/sin [B,C,D] fp32.  mask: None (implicit from past_len, n_real, window,
    causal, sink) or fp32 [B,Hq,C,P+C].  Returns (out fp64 [B,Hq,C,D],
    out_sel fp64 [B,Hq*D] or None).
    """
    q = np.asarray(q)
    B, Hq, C, D = q.shape
    Hkv = np.asarray(k_new).shape[1]
    G = Hq // Hkv
    sc = (1.0 / np.sqrt(D)) if scale is None or scale <= 0 else float(scale)
    cos = np.asarray(cos, dtype=np.float32)
    sin = np.asarray(sin, dtype=np.float32)
    q_rot = kv_to_f32(rope_rotate(q, cos[:, None], sin[:, None], kv), kv).astype(np.float64)
    k_rot = kv_to_f32(rope_rotate(k_new, cos[:, None], sin[:, None], kv), kv).astype(np.float64)
    v_chk = kv_to_f32(to_kv(v_new, kv), kv).astype(np.float64)
    out = np.zeros((B, Hq, C, D), dtype=np.float64)
    for b in range(B):
        L, n = int(past_len[b]), int(n_real[b])
        implicit = None if mask is not None else explicit_mask(L, n, C, P, window, causal, sink)
        for h in range(Hq):
            kvh = h // G
            keys = np.concatenate([kv_to_f32(cache_k[b, kvh, :P], kv).astype(np.float64),
                                   k_rot[b, kvh]], axis=0)
            vals = np.concatenate([kv_to_f32(cache_v[b, kvh, :P], kv).astype(np.float64),
                                   v_chk[b, kvh]], axis=0)
            add = implicit if mask is None else np.asarray(mask[b, h], dtype=np.float32)
            out[b, h] = attend(q_rot[b, h], keys, vals, add, sc)
    out_sel = None
    if sel_row is not None:
        out_sel = np.stack([out[b, :, int(sel_row[b]), :].reshape(Hq * D) for b in range(B)])
    return out, out_sel


def decode_step(q, k_new, v_new, cos, sin, cache_k, cache_v, P, past_len, window=0, sink=0, kv="bf16"):
    """One-token decode: the C = 1 case.

    [P2, Mask/cache layout]: the mask unmasks the valid past slots and the
    current token's own slot; no causal mask is built inside decode.
    """
    B = np.asarray(q).shape[0]
    ones = np.ones(B, dtype=np.int64)
    out, _ = chunk_prefill_attn(q, k_new, v_new, cos, sin, cache_k, cache_v, P,
                                past_len, ones, window=window, causal=0, sink=sink, kv=kv)
    return out


def select_argmax(out_sel_f32) -> np.ndarray:
    """Index of the largest fp32 value per row, lowest index on ties."""
    return np.argmax(np.asarray(out_sel_f32, dtype=np.float32), axis=-1)


# ---------------------------------------------------------------- caches

def kv_append_global(cache_k, cache_v, length, k_new, v_new, cos, sin, n_rows, kv="bf16"):
    """Append the rotated chunk K and the chunk V after the cached rows (in place).

    [P2, Runtime behavior]: the runtime writes each step's KV into external
    cache buffers; past tokens stay packed into the first slots.  Rows
    [0, n_b) of the chunk go to slots [len_b, len_b + n_b) and len_b grows by
    n_b.  A sequence whose rows do not fit (len_b + n_b > capacity) is left
    unchanged and reported.  Returns the list of overflowing sequences.
    kv: the cache format ("bf16" or "f16").
    """
    cap = cache_k.shape[2]
    k_rot = rope_rotate(k_new, np.asarray(cos)[:, None], np.asarray(sin)[:, None], kv)
    v_kv = to_kv(v_new, kv)
    overflow = []
    for b in range(cache_k.shape[0]):
        L, n = int(length[b]), int(n_rows[b])
        if L + n > cap:
            overflow.append(b)
            continue
        cache_k[b, :, L:L + n] = k_rot[b, :, :n]
        cache_v[b, :, L:L + n] = v_kv[b, :, :n]
        length[b] = L + n
    return overflow


def kv_append_sliding(cache_k, cache_v, length, k_new, v_new, cos, sin, n_rows,
                      window: int, sink: int = 0, kv="bf16"):
    """Append to a sliding-window cache that compacts chronologically (in place).

    [P4, Fix]: sliding caches compact chronologically on eviction; the oldest
    window rows go first; sink rows stay pinned.  The cache holds at most W
    rows: S sink rows, then the newest rows in order.  Appending n rows evicts
    e = max(0, len + n - W) rows [S, S+e), shifts the rest down and writes the
    n rows at the end; len becomes min(len + n, W).  n must be <= W - S;
    sequences breaking that are left unchanged and returned.
    """
    W, S = int(window), int(sink)
    k_rot = rope_rotate(k_new, np.asarray(cos)[:, None], np.asarray(sin)[:, None], kv)
    v_kv = to_kv(v_new, kv)
    bad = []
    for b in range(cache_k.shape[0]):
        L, n = int(length[b]), int(n_rows[b])
        if n > W - S or L > W:
            bad.append(b)
            continue
        e = max(0, L + n - W)
        for cache, new in ((cache_k, k_rot), (cache_v, v_kv)):
            rows = np.concatenate([cache[b, :, :min(S, L)], cache[b, :, S + e:L], new[b, :, :n]],
                                  axis=1)
            cache[b, :, :rows.shape[1]] = rows
        length[b] = L - e + n
    return bad


def snapshot_padded_append(cache_k, cache_v, length, n_real, C: int, window: int, sink: int = 0):
    """Save the rows a padded append would evict beyond an exact append.

    [P4, Fix]: a padded append over-evicts up to pad_count of the oldest window
    rows; snapshot_cache_padded_append saves them before the padded execute.
    Guard [P4, review]: windows with W <= C + S are rejected.
    With e_pad = max(0, len + C - W) and e_ex = max(0, len + n - W), the saved
    rows are [S + e_ex, S + e_pad).  Returns a snapshot record.
    """
    W, S = int(window), int(sink)
    if W <= C + S:
        raise ValueError("window too small for a padded append")
    snap = []
    for b in range(cache_k.shape[0]):
        L, n = int(length[b]), int(n_real[b])
        e_pad = max(0, L + C - W)
        e_ex = max(0, L + n - W)
        snap.append(dict(n=n, e_ex=e_ex, e_pad=e_pad,
                         k=cache_k[b, :, S + e_ex:S + e_pad].copy(),
                         v=cache_v[b, :, S + e_ex:S + e_pad].copy()))
    return snap


def rollback_padded_append(cache_k, cache_v, length, snap, C: int, sink: int = 0):
    """Undo the pad part of a padded append (in place).

    [P4, Fix]: rollback_cache_padded_append reinserts the saved rows and drops
    the pad rows, leaving the cache byte-identical to an unpadded append.
    Rows [len - (C - n), len) are the pads and are dropped; the saved rows go
    back in at slot S ahead of the surviving rows.  Bytes past the final length
    are left as they are ([P4, Declined with rationale]: no consumer reads past
    the length).
    """
    S = int(sink)
    for b in range(cache_k.shape[0]):
        s = snap[b]
        keep = int(length[b]) - (C - s["n"])
        for cache, saved in ((cache_k, s["k"]), (cache_v, s["v"])):
            rows = np.concatenate([cache[b, :, :min(S, keep)], saved, cache[b, :, S:keep]], axis=1)
            cache[b, :, :rows.shape[1]] = rows
        length[b] = keep + s["k"].shape[1]
