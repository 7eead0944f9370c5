"""Invariants the pages fix, checked on the oracle at brute-force sizes (CPU only).

(a) N tokens fed as padded chunks == one full causal pass == N one-token decode
    steps ("must reproduce the token the all-positions redecode graph gives";
    the C = 64 and C = 32 chunkings agree -- functiongemma chunk prefill-with-past,
    Validation; prefill and decode connect cleanly -- TICO prefill-decode
    modeling).
(b) padded append + rollback == exact append, byte for byte, over eviction,
    overshoot and sink cases (cactus padded tail, Fix and unit tests).
(c) the explicit per-head mask and the implicit (past_len, n_real, window,
    causal) description give the same result.
    plus: a sliding cache fed by exact appends holds the sinks and then the
    newest rows in order (closed form, independent of the compaction code);
    and the implicit mask's slot -> position reading with sinks agrees with
    the absolute positions the sliding cache actually stores.
"""
import numpy as np
import pytest

import oracle as O
from synth import normal_bf16, rope_tables, bf16_bits


def stream(T, Hq, Hkv, D, tag):
    q = bf16_bits(normal_bf16((1, Hq, T, D), 0, tag + "/q"))
    k = bf16_bits(normal_bf16((1, Hkv, T, D), 0, tag + "/k"))
    v = bf16_bits(normal_bf16((1, Hkv, T, D), 0, tag + "/v"))
    return q, k, v


def chunk_of(x, s, e, C):
    """Rows [s, e) of a [1, H, T, D] stream, zero-padded to C rows."""
    out = np.zeros(x.shape[:2] + (C,) + x.shape[3:], dtype=x.dtype)
    out[:, :, :e - s] = x[:, :, s:e]
    return out


def tables(pos0, C, D, base=10000.0):
    c, s = rope_tables(np.arange(pos0, pos0 + C)[None, :], D, base)
    return c.numpy(), s.numpy()


def run_chunked_global(q, k, v, sizes, C, window=0, kv="bf16"):
    _, Hq, T, D = q.shape
    Hkv = k.shape[1]
    cap = T + C
    ck = np.zeros((1, Hkv, cap, D), dtype=np.uint16)
    cv = np.zeros_like(ck)
    length = np.zeros(1, dtype=np.int64)
    outs, s = [], 0
    for n in sizes:
        L = int(length[0])
        cos, sin = tables(L, C, D)
        qc, kc, vc = chunk_of(q, s, s + n, C), chunk_of(k, s, s + n, C), chunk_of(v, s, s + n, C)
        out, _ = O.chunk_prefill_attn(qc, kc, vc, cos, sin, ck, cv, L, [L], [n],
                                      window=window, causal=1, kv=kv)
        outs.append(out[:, :, :n])
        assert O.kv_append_global(ck, cv, length, kc, vc, cos, sin, [n], kv=kv) == []
        s += n
    assert s == T
    return np.concatenate(outs, axis=2), ck, cv, length


@pytest.mark.parametrize("D,Hq,Hkv,window,kv", [(16, 4, 1, 0, "bf16"), (32, 4, 2, 0, "bf16"), (16, 2, 2, 5, "bf16"),
                                                (16, 4, 1, 0, "f16"), (32, 4, 2, 5, "f16")])
def test_invariant_a_chunks_equal_full_pass_equal_decode(D, Hq, Hkv, window, kv):
    T = 23
    q, k, v = stream(T, Hq, Hkv, D, f"inv_a/{D}/{Hkv}/{window}")
    full, fk, fv, fl = run_chunked_global(q, k, v, [T], T, window, kv)
    for sizes, C in (([8, 8, 7], 8), ([5, 5, 5, 5, 3], 8), ([16, 7], 16), ([3, 11, 9], 12)):
        out, ck, cv, cl = run_chunked_global(q, k, v, sizes, C, window, kv)
        assert np.max(np.abs(out - full)) < 1e-12
        assert cl[0] == fl[0] == T
        assert np.array_equal(ck[:, :, :T], fk[:, :, :T]) and np.array_equal(cv[:, :, :T], fv[:, :, :T])
    # decode: T one-token steps, each followed by its append
    cap = T + 1
    dk = np.zeros((1, Hkv, cap, D), dtype=np.uint16)
    dv = np.zeros_like(dk)
    length = np.zeros(1, dtype=np.int64)
    outs = []
    for t in range(T):
        cos, sin = tables(t, 1, D)
        out = O.decode_step(q[:, :, t:t + 1], k[:, :, t:t + 1], v[:, :, t:t + 1], cos, sin,
                            dk, dv, t, [t], window=window, kv=kv)
        outs.append(out)
        O.kv_append_global(dk, dv, length, k[:, :, t:t + 1], v[:, :, t:t + 1], cos, sin, [1], kv=kv)
    dec = np.concatenate(outs, axis=2)
    assert np.max(np.abs(dec - full)) < 1e-12
    assert np.array_equal(dk[:, :, :T], fk[:, :, :T]) and np.array_equal(dv[:, :, :T], fv[:, :, :T])


def test_invariant_a_sliding_cache_matches_windowed_full_pass():
    """A compacting window cache (W rows) fed chunk by chunk gives the windowed full pass."""
    D, Hq, Hkv, W, C, T = 16, 2, 1, 12, 4, 29
    q, k, v = stream(T, Hq, Hkv, D, "inv_a/slide")
    full, *_ = run_chunked_global(q, k, v, [T], T, window=W)
    ck = np.zeros((1, Hkv, W, D), dtype=np.uint16)
    cv = np.zeros_like(ck)
    length = np.zeros(1, dtype=np.int64)
    outs, s = [], 0
    while s < T:
        n = min(C, T - s)
        L = int(length[0])
        cos, sin = tables(s, C, D)        # absolute positions of the chunk rows
        qc, kc, vc = chunk_of(q, s, s + n, C), chunk_of(k, s, s + n, C), chunk_of(v, s, s + n, C)
        out, _ = O.chunk_prefill_attn(qc, kc, vc, cos, sin, ck, cv, W, [L], [n], window=W, causal=1)
        outs.append(out[:, :, :n])
        assert O.kv_append_sliding(ck, cv, length, kc, vc, cos, sin, [n], W) == []
        s += n
    assert np.max(np.abs(np.concatenate(outs, axis=2) - full)) < 1e-12


def rows(T, D, tag):
    k = bf16_bits(normal_bf16((1, 1, T, D), 0, tag + "/k"))
    v = bf16_bits(normal_bf16((1, 1, T, D), 0, tag + "/v"))
    return k, v


def test_sliding_closed_form_sinks_then_newest():
    D, W, S = 8, 10, 2
    T = 37
    k, v = rows(T, D, "slide_closed")
    ck = np.zeros((1, 1, W, D), dtype=np.uint16); cv = np.zeros_like(ck)
    length = np.zeros(1, dtype=np.int64)
    zc = np.ones((1, 8, D), np.float32); zs = np.zeros((1, 8, D), np.float32)  # identity rotation
    s = 0
    for n in [3, 1, 4, 8, 2, 8, 5, 6]:
        O.kv_append_sliding(ck, cv, length, k[:, :, s:s + n], v[:, :, s:s + n],
                            zc[:, :n], zs[:, :n], [n], W, S)
        s += n
        keep = list(range(min(S, s))) + list(range(max(S, s - (W - S)), s))
        assert int(length[0]) == len(keep)
        assert np.array_equal(ck[0, 0, :len(keep)], k[0, 0, keep])
        assert np.array_equal(cv[0, 0, :len(keep)], v[0, 0, keep])


@pytest.mark.parametrize("W,S", [(10, 0), (10, 2), (12, 3), (7, 1)])
def test_sink_mask_matches_positions_in_the_sliding_cache(W, S):
    """The implicit mask with sinks, against brute force over absolute positions.

    The cache is fed by the oracle's own sliding append with each row's token
    position stored in its V bits; before every chunk the mask from visible()
    must equal: pinned sink slot (j < S), or a token within the window of the
    query's position; chunk keys causal and within the window."""
    D = 4
    T = 60
    zc = np.ones((1, 16, D), np.float32); zs = np.zeros((1, 16, D), np.float32)
    ck = np.zeros((1, 1, W, D), dtype=np.uint16); cv = np.zeros_like(ck)
    length = np.zeros(1, dtype=np.int64)
    s = 0
    for n in [3, 1, 4, 6, 2, 6, 5, 1, 6, 3, 6, 4, 6, 2]:
        if n > W - S:
            n = W - S
        C = 6
        L = int(length[0])
        pos_slot = cv[0, 0, :L, 0].astype(np.int64)          # absolute positions in the cache
        vis = O.visible(L, n, C, W, W, 1, S)                 # P = W slot columns
        for i in range(C):
            pos_q = s + i
            for j in range(W):
                want = j < L and (j < S or pos_q - pos_slot[j] < W)
                assert bool(vis[i, j]) == want, (W, S, s, i, j)
            for t in range(C):
                want = t < n and t <= i and (i - t) < W
                assert bool(vis[i, W + t]) == want, (W, S, s, i, t)
        newk = np.zeros((1, 1, n, D), np.uint16)
        newv = np.zeros((1, 1, n, D), np.uint16)
        newv[0, 0, :, 0] = np.arange(s, s + n)
        O.kv_append_sliding(ck, cv, length, newk, newv, zc[:, :n], zs[:, :n], [n], W, S)
        s += n
        if s >= T:
            break
    assert s > 2 * W   # eviction happened many times


def test_sink_zero_is_the_plain_mask():
    for L, n, C, P, W in [(5, 3, 4, 8, 4), (8, 4, 4, 8, 3), (0, 4, 4, 6, 2)]:
        assert np.array_equal(O.visible(L, n, C, P, W, 1, 0), O.visible(L, n, C, P, W, 1))


@pytest.mark.parametrize("S", [0, 2])
def test_invariant_b_padded_append_rollback_equals_exact(S):
    D, W, C = 4, 24, 8
    ident_c = np.ones((1, C, D), np.float32)
    ident_s = np.zeros((1, C, D), np.float32)
    k0, v0 = rows(W, D, f"inv_b/{S}/cache")
    kn, vn = rows(C, D, f"inv_b/{S}/new")
    cases = 0
    for L0 in range(0, W + 1):
        for n in range(0, C + 1):
            kc = kn.copy(); vc = vn.copy()
            kc[:, :, n:] = 0; vc[:, :, n:] = 0          # zero pads
            ek, ev = k0.copy(), v0.copy(); el = np.array([L0])
            O.kv_append_sliding(ek, ev, el, kc, vc, ident_c, ident_s, [n], W, S)
            pk, pv = k0.copy(), v0.copy(); pl = np.array([L0])
            snap = O.snapshot_padded_append(pk, pv, pl, [n], C, W, S)
            O.kv_append_sliding(pk, pv, pl, kc, vc, ident_c, ident_s, [C], W, S)
            O.rollback_padded_append(pk, pv, pl, snap, C, S)
            assert pl[0] == el[0] == min(L0 + n, W)
            Lf = int(el[0])
            assert np.array_equal(pk[:, :, :Lf], ek[:, :, :Lf]), (L0, n)
            assert np.array_equal(pv[:, :, :Lf], ev[:, :, :Lf]), (L0, n)
            cases += 1
    assert cases == (W + 1) * (C + 1)


def test_padded_guard_rejects_small_window():
    ck = np.zeros((1, 1, 10, 4), np.uint16)
    with pytest.raises(ValueError):
        O.snapshot_padded_append(ck, ck.copy(), np.array([3]), [2], 8, 10, 2)


def test_global_append_overflow_leaves_sequence_unchanged():
    ck = np.zeros((2, 1, 6, 4), np.uint16); cv = ck.copy()
    length = np.array([4, 1])
    k, v = rows(3, 4, "overflow")
    k = np.concatenate([k, k]); v = np.concatenate([v, v])
    c = np.ones((2, 3, 4), np.float32); s = np.zeros((2, 3, 4), np.float32)
    assert O.kv_append_global(ck, cv, length, k, v, c, s, [3, 3]) == [0]
    assert list(length) == [4, 4]
    assert np.all(ck[0] == 0) and np.array_equal(ck[1, :, 1:4], k[1, :, :3])


@pytest.mark.parametrize("window,causal", [(0, 1), (7, 1), (0, 0), (5, 0)])
def test_invariant_c_explicit_equals_implicit(window, causal):
    B, Hq, Hkv, C, D, P = 2, 4, 2, 8, 16, 13
    q = bf16_bits(normal_bf16((B, Hq, C, D), 0, "inv_c/q"))
    k = bf16_bits(normal_bf16((B, Hkv, C, D), 0, "inv_c/k"))
    v = bf16_bits(normal_bf16((B, Hkv, C, D), 0, "inv_c/v"))
    ck = bf16_bits(normal_bf16((B, Hkv, P, D), 0, "inv_c/ck"))
    cv = bf16_bits(normal_bf16((B, Hkv, P, D), 0, "inv_c/cv"))
    L, n = [9, 13], [5, 8]
    cos, sin = [t.numpy() for t in rope_tables(np.array(L)[:, None] + np.arange(C), D, 1e4)]
    imp, sel_i = O.chunk_prefill_attn(q, k, v, cos, sin, ck, cv, P, L, n, window, causal,
                                      sel_row=[4, 7])
    mask = np.stack([np.stack([O.explicit_mask(L[b], n[b], C, P, window, causal)] * Hq)
                     for b in range(B)])
    exp, sel_e = O.chunk_prefill_attn(q, k, v, cos, sin, ck, cv, P, L, n, mask=mask,
                                      sel_row=[4, 7])
    assert np.array_equal(imp, exp) and np.array_equal(sel_i, sel_e)
    assert np.array_equal(sel_i[1].reshape(Hq, D), imp[1, :, 7])


def test_f16_cache_holds_rotated_keys_rounded_to_half():
    """The f16 cache's key rows are the bf16 path's fp32 rotation rounded to half
    (closed form against the rotation done with exact fp64 products, within one
    fp32 rounding), values are the bf16 rows converted exactly; and attention over
    the f16 cache differs from the bf16 one only by rounding."""
    D, Hkv, C = 32, 2, 6
    k = bf16_bits(normal_bf16((1, Hkv, C, D), 0, "f16c/k"))
    v = bf16_bits(normal_bf16((1, Hkv, C, D), 0, "f16c/v"))
    cos, sin = tables(100, C, D)
    ck = np.zeros((1, Hkv, C, D), np.uint16); cv = ck.copy(); ln = np.zeros(1, np.int64)
    O.kv_append_global(ck, cv, ln, k, v, cos, sin, [C], kv="f16")
    x = O.bf16_to_f32(k).astype(np.float64)
    h = D // 2
    c64, s64 = cos.astype(np.float64)[None, None], sin.astype(np.float64)[None, None]
    exact = np.concatenate([x[..., :h] * c64[..., :h] - x[..., h:] * s64[..., :h],
                            x[..., h:] * c64[..., h:] + x[..., :h] * s64[..., h:]], axis=-1)
    got = O.f16_to_f32(ck).astype(np.float64)
    assert np.all(np.abs(got - exact) <= np.abs(exact) * 2.0 ** -11 + 2.0 ** -24 + 4 * 2.0 ** -24 * np.abs(x).max())
    assert np.array_equal(O.f16_to_f32(cv), O.bf16_to_f32(v))
    q, kk, vv = stream(9, 4, 2, 32, "f16c/attn")
    cos2, sin2 = tables(0, 9, 32)
    e = np.zeros((1, 2, 0, 32), np.uint16)
    a16, _ = O.chunk_prefill_attn(q, kk, vv, cos2, sin2, e, e, 0, [0], [9], kv="f16")
    a32, _ = O.chunk_prefill_attn(q, kk, vv, cos2, sin2, e, e, 0, [0], [9], kv="bf16")
    assert 0 < np.abs(a16 - a32).max() < 2e-2
