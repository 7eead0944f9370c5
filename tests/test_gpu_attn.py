"""GPU parity of chunk-prefill attention and decode against the fp64 oracle.

Outputs within max-abs 1e-2 and rel-L2 3e-3 of the oracle; the explicit and
implicit forms of one 0 / -1e30 mask bitwise identical on every path; two runs
bitwise identical; selected-row argmax exact unless the oracle's top-2 gap is
within tolerance.
Sources: "functiongemma: chunk prefill-with-past graph gemma_prefill_with_past"
(Change: RoPE tables, per-head additive mask over past + C keys, one-hot select;
Validation: 800 cached + 52-token chunk, C = 64, select row 51) and
"[quanization] Enable prefill-decode modeling" (Mask/cache layout).
"""
import numpy as np
import pytest
import torch

import oracle as O
from synth import WORKLOADS, Workload, make_chunk_inputs, make_cache, normal_bf16, rope_tables
from harness import (lib, assert_close, check_argmax, oracle_attn, explicit_masks,
                     assert_explicit_matches, sample_rows, oracle_rows)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_gpu(cpa, inp, ck, cv, P, window=0, causal=True, mask=None, sel_row=None, want_sel=True,
            kind=0, wsize=0, sink=0):
    d = lambda t: None if t is None else t.to(DEV)
    cache = cpa.KVCache(d(ck), d(cv), d(inp["past_len"]).clone(), kind, wsize, sink)
    err = cpa.new_error_word()
    out, sel = cpa.chunk_prefill_attn(d(inp["q"]), d(inp["k"]), d(inp["v"]), d(inp["cos"]), d(inp["sin"]),
                                      cache, P, past_len=d(inp["past_len"]), n_real=d(inp["n_real"]),
                                      window=window, causal=causal, mask=d(mask), sel_row=d(sel_row),
                                      want_sel=want_sel, err=err)
    torch.cuda.synchronize()
    return out, sel, err


def small(name, B, Hq, Hkv, D, C, P, L, n, window=0, causal=1, seed=0):
    return Workload(name, B=B, Hq=Hq, Hkv=Hkv, D=D, C=C, P=P, cap=P + C, past=L, n_real=n,
                    window=window, causal=causal, seed=seed)


CASES = [
    WORKLOADS["tiny"],
    small("s_d128_g4", 2, 8, 2, 128, 40, 300, ("uniform", 0, 300), ("uniform", 1, 40)),
    small("s_d64_g1", 3, 2, 2, 64, 130, 257, ("uniform", 0, 257), ("uniform", 0, 130)),
    small("s_d256_g8", 1, 8, 1, 256, 128, 512, ("fixed", 512), ("fixed", 127), window=512),
    small("s_win_small", 2, 4, 1, 128, 64, 200, ("uniform", 50, 200), ("uniform", 30, 64), window=37),
    small("s_noncausal_win", 2, 4, 2, 64, 33, 100, ("uniform", 0, 100), ("uniform", 1, 33), window=9, causal=0),
    small("s_noncausal", 1, 4, 4, 128, 17, 140, ("fixed", 139), ("fixed", 17), causal=0),
    small("s_g16", 1, 16, 1, 128, 20, 64, ("fixed", 64), ("fixed", 20)),
    small("s_empty_past", 2, 4, 1, 128, 96, 0, ("fixed", 0), ("uniform", 0, 96)),
    small("d_decode", 3, 8, 2, 128, 1, 700, ("uniform", 1, 700), ("fixed", 1), causal=0),
    small("d_decode_win", 2, 8, 2, 64, 1, 900, ("uniform", 300, 900), ("fixed", 1), window=100, causal=0),
    small("d_decode_g16", 2, 16, 1, 128, 1, 257, ("uniform", 0, 257), ("fixed", 1), causal=0),
    small("d_decode_g32", 1, 32, 1, 128, 1, 300, ("fixed", 299), ("fixed", 1), causal=0),
    # edge shapes: one chunk row per packed tile row (G = 128), a long prefill
    # without past, D = 256 without grouping, a ragged C of 1 row past a tile
    small("e_g128", 1, 128, 1, 64, 8, 100, ("fixed", 100), ("fixed", 7)),
    small("e_prefill_1024", 1, 8, 8, 128, 1024, 0, ("fixed", 0), ("fixed", 1000)),
    small("e_d256_g1", 2, 2, 2, 256, 200, 130, ("uniform", 0, 130), ("uniform", 1, 200)),
    small("e_ragged_129", 2, 4, 2, 128, 129, 257, ("uniform", 0, 257), ("fixed", 129)),
    small("e_all_pad", 2, 8, 2, 128, 64, 64, ("fixed", 0), ("fixed", 0)),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_attention_matches_oracle_and_explicit_matches_implicit(w):
    cpa = lib()
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    out_i, sel_i, err = run_gpu(cpa, inp, ck, cv, w.P, w.window, bool(w.causal))
    assert int(err[0]) == 0
    ref, ref_sel = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                               inp["past_len"], inp["n_real"], w.window, w.causal,
                               sel_row=(inp["n_real"] - 1).clamp(min=0))
    assert_close(out_i, ref, w.name)
    if (inp["n_real"] > 0).all():
        assert_close(sel_i.view(w.B, w.Hq, w.D).to(torch.bfloat16), ref_sel.reshape(w.B, w.Hq, w.D), w.name + "/sel")
        check_argmax(sel_i, ref_sel, w.name)
    mask = explicit_masks(inp["past_len"].numpy(), inp["n_real"].numpy(), w.C, w.P, w.Hq, w.window, w.causal)
    out_e, sel_e, err = run_gpu(cpa, inp, ck, cv, w.P, mask=mask)
    assert int(err[0]) == 0
    assert_close(out_e, ref, w.name + "/explicit")
    assert_explicit_matches(out_e, out_i, w.name)
    out_2, _, _ = run_gpu(cpa, inp, ck, cv, w.P, w.window, bool(w.causal))
    assert torch.equal(out_2.view(torch.int16), out_i.view(torch.int16)), "not deterministic"


GENERAL_MASK_CASES = [
    small("g_pair_d128", 2, 8, 2, 128, 96, 300, ("uniform", 0, 300), ("uniform", 1, 96)),
    small("g_pair_d64_odd", 2, 8, 2, 64, 61, 203, ("uniform", 0, 203), ("uniform", 1, 61)),
    small("g_single_d256", 1, 4, 1, 256, 64, 300, ("fixed", 250), ("fixed", 60)),
    small("g_decode", 3, 8, 2, 128, 1, 700, ("uniform", 1, 700), ("fixed", 1), causal=0),
]


@pytest.mark.parametrize("w", GENERAL_MASK_CASES, ids=lambda w: w.name)
def test_general_additive_mask(w):
    """Mask entries other than 0 and -1e30: a negative bias on the visible keys
    that differs per head and row, added to the scaled scores like any mask
    value ("functiongemma: chunk prefill-with-past graph", Change: the
    caller-supplied additive mask).  Head 0 keeps the plain 0 / -1e30 form, so
    both forms meet in one call; P and C not multiples of 4 in one case."""
    cpa = lib()
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    base = explicit_masks(inp["past_len"].numpy(), inp["n_real"].numpy(), w.C, w.P, w.Hq, w.window, w.causal)
    bias = normal_bf16(tuple(base.shape), w.seed, "mask_bias").float().abs() * -2.0
    mask = torch.where(base == 0, bias, base)
    mask[:, 0] = base[:, 0]
    sel = (inp["n_real"] - 1).clamp(min=0)
    out, sel_out, err = run_gpu(cpa, inp, ck, cv, w.P, mask=mask, sel_row=sel)
    assert int(err[0]) == 0
    ref, ref_sel = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                               inp["past_len"], inp["n_real"], mask=mask, sel_row=sel)
    assert_close(out, ref, w.name)
    check_argmax(sel_out, ref_sel, w.name)
    # the bias matters: the plain mask gives another answer
    ref0, _ = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                          inp["past_len"], inp["n_real"], mask=base)
    assert np.abs(ref0 - ref).max() > 1e-2


SINK_CASES = [
    # (workload over a full or nearly full sliding window cache of W = P rows, sink rows S)
    (small("k_pair_d128", 2, 8, 2, 128, 64, 256, ("uniform", 200, 256), ("uniform", 1, 64), window=256), 4),
    (small("k_single_d256", 1, 8, 1, 256, 128, 512, ("fixed", 512), ("fixed", 127), window=512), 2),
    (small("k_single_d64", 2, 4, 1, 64, 16, 96, ("uniform", 80, 96), ("uniform", 1, 16), window=96), 3),
    (small("k_decode", 4, 8, 2, 128, 1, 512, ("uniform", 400, 512), ("fixed", 1), window=300, causal=0), 4),
    (small("k_decode_g32", 1, 32, 1, 128, 1, 300, ("fixed", 300), ("fixed", 1), window=200, causal=0), 5),
]


@pytest.mark.parametrize("w,S", SINK_CASES, ids=lambda x: x.name if hasattr(x, "name") else str(x))
def test_sink_aware_implicit_mask(w, S):
    """A sliding cache with S pinned sink rows and the implicit mask: the sink
    slots stay visible whatever the window (the oracle's reading of the pinned
    rows in "Pad the chunked-prefill tail for sliding-window models"); the
    explicit mask built from the same rule gives the same output."""
    cpa = lib()
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    out_i, sel_i, err = run_gpu(cpa, inp, ck, cv, w.P, w.window, bool(w.causal), kind=cpa.SLIDING, wsize=w.P,
                                sink=S)
    assert int(err[0]) == 0
    ref, ref_sel = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                               inp["past_len"], inp["n_real"], w.window, w.causal,
                               sel_row=(inp["n_real"] - 1).clamp(min=0), sink=S)
    assert_close(out_i, ref, w.name)
    check_argmax(sel_i, ref_sel, w.name)
    # the sinks matter here: without them the oracle's answer differs
    ref0, _ = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                          inp["past_len"], inp["n_real"], w.window, w.causal, sink=0)
    assert np.abs(ref0 - ref).max() > 1e-3
    mask = explicit_masks(inp["past_len"].numpy(), inp["n_real"].numpy(), w.C, w.P, w.Hq, w.window, w.causal, S)
    out_e, _, err = run_gpu(cpa, inp, ck, cv, w.P, mask=mask, kind=cpa.SLIDING, wsize=w.P, sink=S)
    assert int(err[0]) == 0
    assert_close(out_e, ref, w.name + "/explicit")
    assert_explicit_matches(out_e, out_i, w.name)


DEAD_CASES = [
    # two-tile kernel (D 128 and 64), single-tile kernel (D 128, D 256), decode kernel, G > 16 decode
    small("dead_pair_d128", 2, 8, 2, 128, 96, 400, ("uniform", 10, 300), ("uniform", 40, 96)),
    small("dead_pair_d64", 2, 8, 1, 64, 64, 333, ("uniform", 50, 333), ("uniform", 20, 64)),
    small("dead_single_d128", 2, 8, 2, 128, 32, 400, ("uniform", 10, 300), ("uniform", 5, 32)),
    small("dead_single_d256", 1, 8, 1, 256, 64, 520, ("fixed", 301), ("fixed", 45), window=200),
    small("dead_decode", 3, 8, 2, 128, 1, 700, ("uniform", 1, 699), ("fixed", 1), causal=0),
    small("dead_decode_g32", 1, 32, 1, 128, 1, 300, ("fixed", 219), ("fixed", 1), causal=0),
]
# bit patterns written into dead rows: quiet and all-ones NaNs, +inf, -inf
NONFINITE = {torch.bfloat16: (0x7FC0, 0xFFFF, 0x7F80, 0xFF80), torch.float16: (0x7E00, 0xFFFF, 0x7C00, 0xFC00)}


def fill_nonfinite(t, rows_from, dims=2):
    """Cycle the non-finite patterns of t's dtype over rows [rows_from[b], end)
    of dimension `dims` of every sequence b (in place, on a host tensor)."""
    pats = NONFINITE[t.dtype]
    bits = t.view(torch.int16)
    for b in range(t.shape[0]):
        r0 = int(rows_from[b])
        n = t.shape[dims] - r0
        if n <= 0:
            continue
        vals = torch.tensor([pats[k % len(pats)] for k in range(n)], dtype=torch.int32).to(torch.int16)
        shape = [1] * t.dim()
        shape[dims] = n
        bits[b].narrow(dims - 1, r0, n).copy_(vals.view(shape[1:]).expand_as(bits[b].narrow(dims - 1, r0, n)))


@pytest.mark.parametrize("kv", ["bf16", "f16"])
@pytest.mark.parametrize("w", DEAD_CASES, ids=lambda w: w.name)
def test_implicit_ignores_dead_rows_whatever_their_bits(w, kv):
    """Cache slots at or past past_len hold no promised bytes ("Pad the
    chunked-prefill tail for sliding-window models", Declined with rationale:
    nothing reads past the current length), and chunk pad rows are not keys.
    Filling them with NaN and infinity patterns must not change one bit of
    the implicit-mask output, on every attention path and cache format; the
    output stays within tolerance of the oracle, which never reads them."""
    cpa = lib()
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    if kv == "f16":
        ck, cv = ck.to(torch.float16), cv.to(torch.float16)
    out1, _, err1 = run_gpu(cpa, inp, ck, cv, w.P, w.window, bool(w.causal))
    ck2, cv2 = ck.clone(), cv.clone()
    fill_nonfinite(ck2, inp["past_len"])
    fill_nonfinite(cv2, inp["past_len"])
    inp2 = dict(inp)
    inp2["k"], inp2["v"] = inp["k"].clone(), inp["v"].clone()
    fill_nonfinite(inp2["k"], inp["n_real"])   # chunk pad rows too
    fill_nonfinite(inp2["v"], inp["n_real"])
    out2, _, err2 = run_gpu(cpa, inp2, ck2, cv2, w.P, w.window, bool(w.causal))
    assert int(err1[0]) == 0 and int(err2[0]) == 0
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16)), f"{w.name}/{kv}: dead rows leaked"
    ref, _ = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P, inp["past_len"],
                         inp["n_real"], w.window, w.causal)
    assert_close(out2, ref, f"{w.name}/{kv}")


def test_page1_shape_eighteen_layers_explicit_masks():
    """800 cached positions + a 52-token chunk padded to 64, select row 51, 18 layers
    alternating a 512-position window (base 1e4) and global attention (base 1e6),
    one explicit [1, 4, 64, 864] mask and one cos/sin pair per layer type."""
    cpa = lib()
    w = WORKLOADS["page1"]
    L = w.past_lens(); n = w.n_reals()
    masks, tabs = {}, {}
    for kind, W, base in (("sliding", 512, 1e4), ("global", 0, 1e6)):
        masks[kind] = explicit_masks(L.numpy(), n.numpy(), w.C, w.P, w.Hq, W, 1)
        tabs[kind] = rope_tables(L.numpy()[:, None] + np.arange(w.C)[None, :], w.D, base)
    # per-type sharing: 1 (tokens) + 2 bases x 2 tables + 18 x (K, V) + 2 masks + 1 select = 44
    assert 1 + 2 * len(tabs) + 2 * w.layers + len(masks) + 1 == 44
    sel = torch.full((w.B,), 51, dtype=torch.int32)
    for layer in range(w.layers):
        kind = "sliding" if layer % 2 == 0 else "global"
        inp = make_chunk_inputs(w, layer=layer)
        inp["cos"], inp["sin"] = tabs[kind]
        ck, cv = make_cache(w, layer=layer)
        out, sel_out, err = run_gpu(cpa, inp, ck, cv, w.P, mask=masks[kind], sel_row=sel)
        assert int(err[0]) == 0
        ref, ref_sel = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                                   L, n, mask=masks[kind], sel_row=sel)
        assert_close(out, ref, f"page1/L{layer}")
        check_argmax(sel_out, ref_sel, f"page1/L{layer}")
        # the implicit description of the same mask gives the same bits
        out_i, _, _ = run_gpu(cpa, inp, ck, cv, w.P, window=512 if kind == "sliding" else 0, sel_row=sel)
        assert torch.equal(out_i.view(torch.int16), out.view(torch.int16)), f"page1/L{layer} implicit"


def run_full(cpa, w, device_gen=False, explicit=False):
    """Run the full workload on the GPU.  `explicit`: pass the mask as an
    explicit [B, Hq, C, P+C] tensor, each sequence's rows built by the
    oracle's mask function and repeated over the heads on the device."""
    dev = DEV if device_gen else "cpu"
    inp = make_chunk_inputs(w, device=dev)
    ck, cv = make_cache(w, device=dev)
    d = lambda t: t.to(DEV)
    mask = None
    if explicit:
        rows = [torch.from_numpy(O.explicit_mask(int(inp["past_len"][b]), int(inp["n_real"][b]), w.C, w.P,
                                                 w.window, w.causal).astype(np.float32)) for b in range(w.B)]
        mask = torch.stack(rows).to(DEV)[:, None].expand(w.B, w.Hq, w.C, w.P + w.C).contiguous()
    cache = cpa.KVCache(d(ck), d(cv), d(inp["past_len"]).clone())
    err = cpa.new_error_word()
    out, sel = cpa.chunk_prefill_attn(d(inp["q"]), d(inp["k"]), d(inp["v"]), d(inp["cos"]), d(inp["sin"]),
                                      cache, w.P, past_len=d(inp["past_len"]), n_real=d(inp["n_real"]),
                                      causal=bool(w.causal), mask=mask, want_sel=True, err=err)
    del mask
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    return out, inp, ck, cv


def check_every_group(w, out, inp, ck, cv, salt=0):
    """Every (sequence, kv head) group against the oracle on sampled rows:
    the first, an inner and the last row of every query tile and the last
    real row, for every q head of the group."""
    G = w.Hq // w.Hkv
    R = max(1, 128 // G)
    host = lambda t: t.detach().cpu()
    out_h = host(out)
    for b in range(w.B):
        L, n = int(inp["past_len"][b]), int(inp["n_real"][b])
        rows = sample_rows(w.C, R, n, salt + b)
        q_b, k_b, v_b = host(inp["q"][b]), host(inp["k"][b]), host(inp["v"][b])
        cos_b, sin_b = host(inp["cos"][b]), host(inp["sin"][b])
        for kvh in range(w.Hkv):
            hs = slice(kvh * G, (kvh + 1) * G)
            ref = oracle_rows(q_b[hs], k_b[kvh], v_b[kvh], cos_b, sin_b, host(ck[b, kvh, :L]),
                              host(cv[b, kvh, :L]), L, n, rows, w.window, w.causal)
            assert_close(out_h[b, hs][:, rows], ref, f"{w.name}/b{b}/kvh{kvh}")


RANDOM_MASK_CASES = [
    small("r_pair_d128", 2, 8, 2, 128, 96, 300, ("fixed", 300), ("fixed", 96)),
    small("r_pair_d64_odd", 2, 8, 2, 64, 61, 203, ("fixed", 203), ("fixed", 61)),
    small("r_single_d256", 1, 4, 1, 256, 64, 300, ("fixed", 300), ("fixed", 64)),
]


@pytest.mark.parametrize("w", RANDOM_MASK_CASES, ids=lambda w: w.name)
def test_explicit_mask_without_implicit_form(w):
    """A 0 / -1e30 mask that no (past_len, n_real, window) describes: entries
    visible at random (a third of them), a band of past tiles masked for every
    row, and some rows with no visible key at all.  Every key position of a
    tile meets its own visibility bit, so a wrong bit order fails here."""
    cpa = lib()
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    g = torch.Generator().manual_seed(1234)
    vis = torch.rand((w.B, w.Hq, w.C, w.P + w.C), generator=g) < 0.33
    vis[..., 128:256] = False                      # a whole key tile dead for every row
    vis[:, :, 5] = False                           # row 5 of every head sees nothing
    mask = torch.where(vis, torch.tensor(0.0), torch.tensor(-1e30))
    sel = torch.full((w.B,), w.C - 1, dtype=torch.int32)
    out, sel_out, err = run_gpu(cpa, inp, ck, cv, w.P, mask=mask, sel_row=sel)
    assert int(err[0]) == 0
    ref, ref_sel = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                               inp["past_len"], inp["n_real"], mask=mask, sel_row=sel)
    assert_close(out, ref, w.name)
    assert torch.all(out[:, :, 5] == 0)
    check_argmax(sel_out, ref_sel, w.name)


@pytest.mark.parametrize("w", [CASES[1], CASES[2], CASES[4], CASES[16]], ids=lambda w: w.name)
def test_explicit_mask_without_bit_copy_gives_same_bits(w):
    """With only cpa_attn_workspace_size bytes (no room for the mask's bit
    copy) the two-tile path reads the fp32 values of every visited tile; the
    output bits are the same as with the copy and as the implicit form's."""
    cpa = lib()
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    mask = explicit_masks(inp["past_len"].numpy(), inp["n_real"].numpy(), w.C, w.P, w.Hq, w.window, w.causal)
    small_ws = cpa.attn_workspace_size(w.B, w.Hq, w.Hkv, w.D, w.C, w.P)
    assert small_ws < cpa.attn_workspace_size_mask(w.B, w.Hq, w.Hkv, w.D, w.C, w.P)
    d = lambda t: t.to(DEV)
    outs = []
    for ws, m in ((small_ws, mask), (None, mask), (small_ws, None)):
        cache = cpa.KVCache(d(ck), d(cv), d(inp["past_len"]).clone())
        err = cpa.new_error_word()
        kw = {} if ws is None else {"workspace": torch.empty(ws, dtype=torch.uint8, device=DEV)}
        out, _ = cpa.chunk_prefill_attn(d(inp["q"]), d(inp["k"]), d(inp["v"]), d(inp["cos"]), d(inp["sin"]),
                                        cache, w.P, past_len=d(inp["past_len"]), n_real=d(inp["n_real"]),
                                        window=w.window, causal=bool(w.causal), mask=None if m is None else d(m),
                                        err=err, **kw)
        torch.cuda.synchronize()
        assert int(err[0]) == 0
        outs.append(out)
    assert_explicit_matches(outs[0], outs[2], w.name + "/no bit copy")
    assert_explicit_matches(outs[1], outs[2], w.name + "/bit copy")


def test_packed_batch_full_size_every_group():
    """Every (sequence, kv head) group of the packed batch (B 16, 32/8 heads,
    D 128, past U[0, 4095], C 128), 13 rows of each of its 32 q heads."""
    cpa = lib()
    w = WORKLOADS["packed_batch"]
    out, inp, ck, cv = run_full(cpa, w)
    check_every_group(w, out, inp, ck, cv)


def test_packed_batch_full_size_explicit_mask_every_group():
    """The packed batch with its 1.1 GB explicit fp32 mask, in the launch
    configuration the bench times: every group against the oracle, and the
    whole output bitwise equal to the implicit form's."""
    cpa = lib()
    w = WORKLOADS["packed_batch"]
    out_e, inp, ck, cv = run_full(cpa, w, device_gen=True, explicit=True)
    check_every_group(w, out_e, inp, ck, cv, salt=3)
    del ck, cv
    out_i, _, _, _ = run_full(cpa, w, device_gen=True)
    assert_explicit_matches(out_e, out_i, "packed_batch/all units")


def test_whole_block_deal_every_unit():
    """64 sequences, 16/4 heads, D 64, C 64, past lengths uniform on [128, 384]:
    256 (sequence, kv head) blocks of 5 to 7 key tiles (switch cost included)
    for about 150 one-CTA teams.  The largest block fits the even split's share
    plus the cut cost, and the deal (largest first, rounds of alternating
    direction) gives no team more than that, so every unit is finished whole by
    one CTA.  Every row against the oracle; the explicit form of the same mask
    gives the same bits."""
    cpa = lib()
    w = small("whole_deal", 64, 16, 4, 64, 64, 384, ("uniform", 128, 384), ("uniform", 1, 64))
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    out, sel, err = run_gpu(cpa, inp, ck, cv, w.P)
    assert int(err[0]) == 0
    ref, ref_sel = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                               inp["past_len"], inp["n_real"], sel_row=inp["n_real"] - 1)
    assert_close(out, ref, w.name)
    check_argmax(sel, ref_sel, w.name)
    mask = explicit_masks(inp["past_len"], inp["n_real"], w.C, w.P, w.Hq, 0, 1)
    out_e, _, err = run_gpu(cpa, inp, ck, cv, w.P, mask=mask)
    assert int(err[0]) == 0
    assert_explicit_matches(out_e, out, w.name)


def test_planned_walk_even_split_fallback():
    """80 (sequence, kv head) blocks for 74-76 two-CTA teams (20 sequences,
    32/4 heads, D 128, C 64), 19 sequences with pasts of 200 to 380 rows and
    one with 4000: the largest block (36 tiles with the switch cost) exceeds
    the even split's share plus the cut cost, so the plan keeps the even split
    inside the planned-order walk and cuts that block between teams.  Every
    row (each sees at least 200 keys) against the oracle; the explicit form of
    the same mask takes the same plan and gives the same bits."""
    cpa = lib()
    w = small("plan_fallback", 20, 32, 4, 128, 64, 4096, ("uniform", 200, 380), ("uniform", 1, 64))
    L = w.past_lens().clone()
    L[7] = 4000
    inp = make_chunk_inputs(w, past_len=L)
    ck, cv = make_cache(w)
    out, sel, err = run_gpu(cpa, inp, ck, cv, w.P)
    assert int(err[0]) == 0
    ref, ref_sel = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                               inp["past_len"], inp["n_real"], sel_row=inp["n_real"] - 1)
    assert_close(out, ref, w.name)
    check_argmax(sel, ref_sel, w.name)
    mask = explicit_masks(inp["past_len"], inp["n_real"], w.C, w.P, w.Hq, 0, 1)
    out_e, _, err = run_gpu(cpa, inp, ck, cv, w.P, mask=mask)
    assert int(err[0]) == 0
    assert_explicit_matches(out_e, out, w.name)


def test_long_context_full_size_every_group():
    """All 32 (sequence, kv head) groups of the long-context chunk (B 4, 32/8
    heads, D 128, past 32768, C 512): the plan cuts these units between the
    CTAs of a team and merges their pieces, so every group and every query
    tile is checked."""
    cpa = lib()
    w = WORKLOADS["long_ctx"]
    out, inp, ck, cv = run_full(cpa, w, device_gen=True)
    check_every_group(w, out, inp, ck, cv)


def test_decode_full_size_every_group():
    """Every q head of all 64 decode sequences (past U[1024, 32768])."""
    cpa = lib()
    w = WORKLOADS["decode"]
    inp = make_chunk_inputs(w, device=DEV)
    ck, cv = make_cache(w, device=DEV)
    cache = cpa.KVCache(ck, cv, inp["past_len"].clone())
    err = cpa.new_error_word()
    out, _ = cpa.decode_step(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], cache, w.P,
                             past_len=inp["past_len"], n_real=inp["n_real"], err=err)
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    G = w.Hq // w.Hkv
    Ls = inp["past_len"].cpu().numpy()
    u16 = lambda t: t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    out_h = out.cpu()
    for b in range(w.B):
        L = int(Ls[b])
        for kvh in range(w.Hkv):
            hs = slice(kvh * G, (kvh + 1) * G)
            ref = O.decode_step(u16(inp["q"][b:b + 1, hs]), u16(inp["k"][b:b + 1, kvh:kvh + 1]),
                                u16(inp["v"][b:b + 1, kvh:kvh + 1]), inp["cos"][b:b + 1].cpu().numpy(),
                                inp["sin"][b:b + 1].cpu().numpy(), u16(ck[b:b + 1, kvh:kvh + 1, :L]),
                                u16(cv[b:b + 1, kvh:kvh + 1, :L]), L, [L])
            assert_close(out_h[b:b + 1, hs], ref, f"decode/b{b}/kvh{kvh}")


def test_out_of_range_lengths_are_flagged_and_clamped():
    cpa = lib()
    w = small("bad_len", 2, 4, 1, 64, 8, 32, ("fixed", 10), ("fixed", 8))
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    inp["past_len"] = torch.tensor([40, 5], dtype=torch.int32)   # 40 > P = 32
    inp["n_real"] = torch.tensor([8, 9], dtype=torch.int32)      # 9 > C = 8
    out, _, err = run_gpu(cpa, inp, ck, cv, w.P, want_sel=False)
    e = int(err[0])
    assert e & cpa.EBIT["PAST_GT_SPAN"] and e & cpa.EBIT["NREAL_GT_C"]
    ref, _ = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                         torch.tensor([32, 5]), torch.tensor([8, 8]))
    assert_close(out, ref, "clamped")
