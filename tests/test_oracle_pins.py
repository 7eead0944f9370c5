"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test ties one oracle function to a hand-worked value, a closed form, an
invariant, or a library routine on a special case, so that a dropped term, a
wrong sign, a wrong index or a transposed operand fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O
from synth import normal_bf16, rope_tables, bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows[key] = vals
    return rows


def f64(bits):
    return O.bf16_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------------ bf16

def test_bf16_round_trip_and_rne_matches_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(200000).astype(np.float32) * np.float32(37.0)
    # exact ties: bf16 value + half an ulp
    base = O.bf16_to_f32(O.f32_to_bf16(x[:1000]))
    ties = (base.view(np.uint32) + np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties, np.float32([0.0, -0.0, 1.0, -3.5])])
    ours = O.f32_to_bf16(x)
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, lib)
    assert np.array_equal(O.f32_to_bf16(O.bf16_to_f32(ours)), ours)


def test_f16_conversions_match_torch():
    """fp32 -> fp16 nearest-even (ties, subnormals, overflow) and fp16 -> fp32
    widening of every bit pattern, against torch's conversions."""
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * np.float32(3e3),
                        rng.standard_normal(10000).astype(np.float32) * np.float32(1e-5),
                        np.float32([0.0, -0.0, 65504.0, 65520.0, 7e4, -7e4, 6.1e-5, 5.96e-8, 1e-9])])
    base = O.f16_to_f32(O.f32_to_f16(x[:1000]))
    ulp = np.abs(np.spacing(base.astype(np.float16)).astype(np.float32))
    ties = base + ulp * np.float32(0.5)          # exactly halfway between two halves
    x = np.concatenate([x, ties])
    ours = O.f32_to_f16(x)
    lib = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, lib)
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    wide = O.f16_to_f32(bits)
    lib_w = torch.from_numpy(bits.view(np.int16)).view(torch.float16).float().numpy()
    same = (wide.view(np.uint32) == lib_w.view(np.uint32)) | (np.isnan(wide) & np.isnan(lib_w))
    assert same.all()


def test_cache_format_helpers():
    """bf16 -> f16 conversion is exact inside the half range; bf16 stays as is."""
    v = bf16_bits(normal_bf16((4, 64), 0, "pin/to_kv"))
    assert np.array_equal(O.to_kv(v, "bf16"), v)
    h = O.to_kv(v, "f16")
    assert np.array_equal(O.kv_to_f32(h, "f16"), O.bf16_to_f32(v))   # N(0,1) values fit fp16 exactly


# ------------------------------------------------------------------ RoPE

def test_rope_hand_worked_example():
    g = read_golden("rope_rotate_half_d4.txt")
    x = O.f32_to_bf16(np.float32([float(v) for v in g["x"]]))
    cos = np.float32([float(v) for v in g["cos"]])
    sin = np.float32([float(v) for v in g["sin"]])
    y = O.bf16_to_f32(O.rope_rotate(x, cos, sin))
    assert np.array_equal(y, np.float32([float(v) for v in g["y"]]))


def test_rope_position_zero_is_identity():
    x = bf16_bits(normal_bf16((3, 5, 64), 0, "pin/rope0"))
    cos, sin = rope_tables(np.zeros((5,)), 64, 10000.0)
    assert np.all(cos.numpy() == 1.0) and np.all(sin.numpy() == 0.0)
    assert np.array_equal(O.rope_rotate(x, cos.numpy(), sin.numpy()), x)
    # in the half format the same rows, converted exactly
    assert np.array_equal(O.f16_to_f32(O.rope_rotate(x, cos.numpy(), sin.numpy(), "f16")), O.bf16_to_f32(x))


@pytest.mark.parametrize("D,out", [(64, "bf16"), (128, "bf16"), (256, "bf16"), (128, "f16"), (256, "f16")])
def test_rope_matches_complex_rotation(D, out):
    """Pair (x_d, x_{d+D/2}) as z = x_d + i x_{d+D/2}; RoPE multiplies z by cos + i sin."""
    x = bf16_bits(normal_bf16((7, D), 0, f"pin/rope_c{D}"))
    pos = np.arange(7) * 131 + 5
    cos, sin = [t.numpy() for t in rope_tables(pos, D, 10000.0)]
    y = O.kv_to_f32(O.rope_rotate(x, cos, sin, out), out).astype(np.float64)
    h = D // 2
    xf = f64(x)
    z = (xf[:, :h] + 1j * xf[:, h:]) * (cos[:, :h].astype(np.float64) + 1j * sin[:, :h].astype(np.float64))
    exact = np.concatenate([z.real, z.imag], axis=1)
    # fp32 rounding of two products and their sum (<= 3 * 2^-24 * (|a| + |b|)),
    # then one bf16 rounding (<= half a bf16 ulp of the larger of the two values)
    pair = np.concatenate([np.abs(xf[:, :h]) + np.abs(xf[:, h:])] * 2, axis=1)
    top = np.maximum(np.abs(exact), np.abs(y))
    mant = 7 if out == "bf16" else 10   # stored mantissa bits of the output format
    ulp = np.exp2(np.floor(np.log2(np.maximum(top, 2.0 ** -14))) - mant)
    assert np.all(np.abs(y - exact) <= 0.5 * ulp + 3 * 2.0 ** -24 * pair)
    # and the tolerance is tight enough that a wrong sign or pairing would fail
    wrong = np.concatenate([z.real, -z.imag], axis=1)
    assert np.any(np.abs(y - wrong) > 0.5 * ulp + 3 * 2.0 ** -24 * pair)


def test_rope_relative_position_and_pair_norm():
    D = 128
    q = bf16_bits(normal_bf16((D,), 0, "pin/rel_q"))
    k = bf16_bits(normal_bf16((D,), 0, "pin/rel_k"))
    def rot(x, p):
        c, s = rope_tables(np.array([p]), D, 10000.0)
        return f64(O.rope_rotate(x, c.numpy()[0], s.numpy()[0]))
    ref = rot(q, 40) @ rot(k, 13)
    for shift in (1, 7, 250, 1000):
        assert abs(rot(q, 40 + shift) @ rot(k, 13 + shift) - ref) < 0.15
    # the wrong relative offset gives a clearly different product
    assert abs(rot(q, 41) @ rot(k, 13) - ref) > 0.15 or abs(rot(q, 45) @ rot(k, 13) - ref) > 0.15
    y = rot(q, 777)
    xf = f64(q)
    h = D // 2
    n_in = xf[:h] ** 2 + xf[h:] ** 2
    n_out = y[:h] ** 2 + y[h:] ** 2
    assert np.allclose(n_out, n_in, rtol=2e-2, atol=1e-3)


# ------------------------------------------------------------------ masks

@pytest.mark.parametrize("L,n,C,P,W,causal", [
    (48, 12, 16, 48, 0, 1), (800, 52, 64, 800, 512, 1), (0, 8, 8, 0, 0, 1),
    (30, 5, 8, 40, 0, 1), (20, 8, 8, 24, 6, 1), (20, 8, 8, 24, 6, 0), (3, 8, 8, 16, 0, 0),
])
def test_visible_by_position_difference(L, n, C, P, W, causal):
    """Re-derive every entry from key positions: past slot j at position j, chunk row t at L+t."""
    vis = O.visible(L, n, C, P, W, causal)
    assert vis.shape == (C, P + C)
    for i in range(C):
        pq = L + i
        for c in range(P + C):
            if c < P:
                exists, pk = c < L, c
            else:
                exists, pk = (c - P) < n, L + (c - P)
            ok = exists and (not causal or pk <= pq) and (W == 0 or abs(pq - pk) < W)
            assert vis[i, c] == ok, (i, c)


def test_visible_counts_closed_form():
    # causal, no window: row i sees L + min(i, n-1) + 1 keys (pad rows see L + n)
    L, n, C, P = 37, 11, 16, 50
    vis = O.visible(L, n, C, P, 0, 1)
    for i in range(C):
        assert vis[i].sum() == L + min(i + 1, n)
    # window W: a real row at position p sees min(W, p + 1) keys (page-1 window is 512)
    L, n, C, P, W = 800, 52, 64, 800, 512
    vis = O.visible(L, n, C, P, W, 1)
    for i in range(n):
        assert vis[i].sum() == min(W, L + i + 1)
    g = read_golden("page1_call_signature.txt")
    assert vis.shape[1] == int(g["mask_shape"][3])


def test_explicit_mask_values():
    m = O.explicit_mask(5, 3, 4, 6, 0, 1)
    assert m.dtype == np.float32
    assert set(np.unique(m).tolist()) == {0.0, np.float32(-1e30)}
    assert np.array_equal(m == 0, O.visible(5, 3, 4, 6, 0, 1))


# ------------------------------------------------------------------ attention

def test_attend_single_visible_key_returns_its_value():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((6, 16)); k = rng.standard_normal((9, 16)); v = rng.standard_normal((9, 16))
    mask = np.full((6, 9), O.MASKED)
    for r in range(6):
        mask[r, (3 * r + 1) % 9] = 0.0
    out = O.attend(q, k, v, mask, 0.25)
    for r in range(6):
        assert np.array_equal(out[r], v[(3 * r + 1) % 9])


def test_attend_zero_query_is_mean_of_visible_values():
    rng = np.random.default_rng(3)
    k = rng.standard_normal((20, 8)); v = rng.standard_normal((20, 8))
    vis = rng.random((5, 20)) < 0.4
    vis[:, 0] = True
    mask = np.where(vis, 0.0, O.MASKED)
    out = O.attend(np.zeros((5, 8)), k, v, mask, 1.0)
    for r in range(5):
        assert np.allclose(out[r], v[vis[r]].mean(axis=0), rtol=0, atol=1e-13)


def test_attend_row_without_visible_key_is_zero():
    rng = np.random.default_rng(4)
    mask = np.full((2, 5), O.MASKED); mask[1, 2] = 0.0
    out = O.attend(rng.standard_normal((2, 4)), rng.standard_normal((5, 4)),
                   rng.standard_normal((5, 4)), mask, 1.0)
    assert np.all(out[0] == 0.0) and np.any(out[1] != 0.0)


def test_attend_matches_library_sdpa_with_bool_mask():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((12, 32)); k = rng.standard_normal((30, 32)); v = rng.standard_normal((30, 32))
    vis = rng.random((12, 30)) < 0.5
    vis[:, 7] = True
    add = np.where(vis, 0.0, O.MASKED)
    ours = O.attend(q, k, v, add, 1.0 / math.sqrt(32))
    lib = F.scaled_dot_product_attention(torch.from_numpy(q)[None], torch.from_numpy(k)[None],
                                         torch.from_numpy(v)[None],
                                         attn_mask=torch.from_numpy(vis)[None])[0].numpy()
    assert np.allclose(ours, lib, rtol=0, atol=1e-12)


def test_chunk_with_empty_past_is_textbook_causal_gqa_attention():
    """L = 0, no pads, causal: the step reduces to causal SDPA on the rotated Q/K with GQA."""
    B, Hq, Hkv, C, D = 2, 8, 2, 24, 64
    q = normal_bf16((B, Hq, C, D), 0, "pin/sdpa_q")
    k = normal_bf16((B, Hkv, C, D), 0, "pin/sdpa_k")
    v = normal_bf16((B, Hkv, C, D), 0, "pin/sdpa_v")
    cos, sin = rope_tables(np.tile(np.arange(C), (B, 1)), D, 10000.0)
    empty = np.zeros((B, Hkv, 0, D), dtype=np.uint16)
    out, _ = O.chunk_prefill_attn(bf16_bits(q), bf16_bits(k), bf16_bits(v), cos.numpy(), sin.numpy(),
                                  empty, empty, 0, [0] * B, [C] * B, causal=1)
    # library side: rotate with the complex form (independent of the oracle's code)
    def rot(x):
        xf = torch.from_numpy(f64(bf16_bits(x)))
        h = D // 2
        c = torch.from_numpy(cos.numpy().astype(np.float64))[:, None]
        s = torch.from_numpy(sin.numpy().astype(np.float64))[:, None]
        z = torch.complex(xf[..., :h], xf[..., h:]) * torch.complex(c[..., :h], s[..., :h])
        y = torch.cat([z.real, z.imag], dim=-1).float().to(torch.bfloat16)   # stored as bf16
        return y.double()
    lib = F.scaled_dot_product_attention(rot(q), rot(k), torch.from_numpy(f64(bf16_bits(v))),
                                         is_causal=True, enable_gqa=True).numpy()
    # the complex product is exact; the oracle rounds the products to fp32 first:
    # rare 1-ulp bf16 differences in the rotated inputs move outputs by ~1e-3 at most
    assert np.max(np.abs(out - lib)) < 2e-2
    assert np.sqrt(np.sum((out - lib) ** 2) / np.sum(lib ** 2)) < 2e-3


def test_page1_signature_counts():
    """One chunk call of the 18-layer spec: tokens, 2 tables per RoPE base, K and V per
    layer, one mask per layer type, select -> 44 arguments; 36 K/V + logits -> 37 results."""
    g = read_golden("page1_call_signature.txt")
    layers = int(g["layers"][0])
    types = {("sliding" if l % 2 == 0 else "global") for l in range(layers)}
    bases = {10000.0 if t == "sliding" else 1e6 for t in types}
    args = 1 + 2 * len(bases) + 2 * layers + len(types) + 1
    results = 2 * layers + 1
    assert args == int(g["args"][0]) and results == int(g["results"][0])
    assert int(g["select_row"][0]) == int(g["real"][0]) - 1


# ------------------------------------------------------------------ selected-row argmax

def test_select_argmax_hand_placed_maxima_and_ties():
    """One row per case, maxima placed by hand: the pick is per row along the
    last axis, in fp32 (two values 2^-20 apart, equal once rounded to bf16,
    still order), and the lowest index wins a tie."""
    rows = np.full((4, 12), -3.0, dtype=np.float32)
    rows[0, 9] = 5.0                                   # a single maximum late in the row
    rows[1, 2] = rows[1, 7] = 4.0                      # a tie: the lower index
    rows[2, 4] = np.float32(1.0) + np.float32(2.0 ** -20)
    rows[2, 3] = 1.0                                   # bf16 would round both to 1.0
    rows[3, :] = 0.5                                   # every value equal: index 0
    got = O.select_argmax(rows)
    assert got.shape == (4,)
    assert got.tolist() == [9, 2, 4, 0]
    assert O.f32_to_bf16(rows[2, 3:5]).tolist()[0] == O.f32_to_bf16(rows[2, 3:5]).tolist()[1]
    # a batch of rows against a per-row scan written out here
    rng = np.random.default_rng(11)
    x = rng.standard_normal((6, 40)).astype(np.float32)
    x[:, 5] = x[:, 17] = x.max(axis=1) + 1.0
    want = [min(j for j in range(40) if x[r, j] == x[r].max()) for r in range(6)]
    assert O.select_argmax(x).tolist() == want == [5] * 6


# ------------------------------------------------------------------ fp16 cache reading

def test_f16_reading_at_position_zero_equals_bf16_reading():
    """Tables at position 0 (cos 1, sin 0) leave every key unrotated, and
    N(0,1) bf16 values convert to half exactly: the fp16-cache reading then
    sees the same numbers as the bf16 one, so the outputs are equal."""
    B, Hq, Hkv, C, D, P = 1, 4, 2, 6, 32, 9
    q = bf16_bits(normal_bf16((B, Hq, C, D), 0, "pin/f16z_q"))
    k = bf16_bits(normal_bf16((B, Hkv, C, D), 0, "pin/f16z_k"))
    v = bf16_bits(normal_bf16((B, Hkv, C, D), 0, "pin/f16z_v"))
    ck = bf16_bits(normal_bf16((B, Hkv, P, D), 0, "pin/f16z_ck"))
    cv = bf16_bits(normal_bf16((B, Hkv, P, D), 0, "pin/f16z_cv"))
    cos = np.ones((B, C, D), dtype=np.float32)
    sin = np.zeros((B, C, D), dtype=np.float32)
    a32, _ = O.chunk_prefill_attn(q, k, v, cos, sin, ck, cv, P, [7], [5])
    a16, _ = O.chunk_prefill_attn(q, k, v, cos, sin, O.to_kv(ck, "f16"), O.to_kv(cv, "f16"), P, [7], [5],
                                  kv="f16")
    assert np.array_equal(a32, a16)


def test_f16_reading_matches_library_sdpa_on_half_operands():
    """General positions: the fp16-cache reading is fp64 softmax attention over
    Q and the chunk keys rotated to half, the half cache rows and the chunk
    values converted to half.  The half operands are formed here with torch's
    own conversions from an fp64 complex rotation (a different route from the
    oracle's fp32 arithmetic, so single half-ulp differences may appear) and
    the attention by the library's SDPA with GQA and a boolean mask.  On these
    seeded inputs both routes give the same half operands, so the outputs
    agree to fp64 rounding; a bf16 rounding of Q or of the chunk keys in place
    of half moves them by ~3e-3."""
    B, Hq, Hkv, C, D, P, L, n = 1, 8, 2, 10, 64, 21, 17, 8
    q = normal_bf16((B, Hq, C, D), 0, "pin/f16s_q")
    k = normal_bf16((B, Hkv, C, D), 0, "pin/f16s_k")
    v = normal_bf16((B, Hkv, C, D), 0, "pin/f16s_v")
    ck = normal_bf16((B, Hkv, P, D), 0, "pin/f16s_ck").half()
    cv = normal_bf16((B, Hkv, P, D), 0, "pin/f16s_cv").half()
    cos, sin = rope_tables(L + np.arange(C)[None, :], D, 10000.0)
    h16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    out, _ = O.chunk_prefill_attn(bf16_bits(q), bf16_bits(k), bf16_bits(v), cos.numpy(), sin.numpy(),
                                  h16(ck), h16(cv), P, [L], [n], kv="f16")

    def rot_half(x):
        xf = x.double()
        h = D // 2
        c = cos.double()[:, None]
        s = sin.double()[:, None]
        z = torch.complex(xf[..., :h], xf[..., h:]) * torch.complex(c[..., :h], s[..., :h])
        return torch.cat([z.real, z.imag], dim=-1).half().double()

    keys = torch.cat([ck.double(), rot_half(k)], dim=2)
    vals = torch.cat([cv.double(), v.half().double()], dim=2)
    vis = torch.from_numpy(O.visible(L, n, C, P, 0, 1))
    lib = F.scaled_dot_product_attention(rot_half(q), keys, vals, attn_mask=vis[None, None],
                                         enable_gqa=True).numpy()
    assert np.max(np.abs(out - lib)) < 1e-9
    # and the half reading is not the bf16 one: rounding to half moved it
    b16, _ = O.chunk_prefill_attn(bf16_bits(q), bf16_bits(k), bf16_bits(v), cos.numpy(), sin.numpy(),
                                  bf16_bits(ck.bfloat16()), bf16_bits(cv.bfloat16()), P, [L], [n])
    assert np.max(np.abs(b16 - out)) > 0
