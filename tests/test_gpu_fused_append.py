"""cpa_chunk_prefill_attn_append: attention and global append in one call.

The call must give exactly what cpa_chunk_prefill_attn followed by
cpa_kv_append gives ("functiongemma: chunk prefill-with-past graph", Change:
the keys and values are extended by the chunk; "[quanization] Enable
prefill-decode modeling", Runtime behavior: the runtime writes the new K/V
into its buffers): the same output and selected-row bits, the same cache
bytes, the same lengths and error bits.  Every attention path is covered (the
two-tile kernel, the single-tile kernel with a cluster merge and with the
combine kernel, the one-token decode kernel), with past_len passed as its own
tensor and as the cache's own len, an explicit mask, n_rows different from
n_real, and a sequence whose append overflows the cache.  The fused call is
also compared with the fp64 oracle directly (attention then global append):
outputs within the attention tolerance, the selected-row argmax by the tie
rule, cache rows [0, len) and len bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle as O
from synth import Workload, make_chunk_inputs, make_cache, bf16_bits
from harness import lib, explicit_masks, oracle_attn, assert_close, check_argmax, bits16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def case(name, B, Hq, Hkv, D, C, P, past, n, cap=None):
    return Workload(name, B=B, Hq=Hq, Hkv=Hkv, D=D, C=C, P=P, cap=cap or P + C, past=past, n_real=n)


CASES = [
    case("fa_pair_d128", 2, 8, 2, 128, 40, 300, ("uniform", 0, 300), ("uniform", 1, 40)),
    case("fa_pair_d64", 1, 8, 1, 64, 100, 200, ("fixed", 150), ("fixed", 77)),
    case("fa_single_d256", 1, 4, 1, 256, 64, 800, ("fixed", 800), ("fixed", 52)),
    case("fa_single_d64_small", 2, 4, 1, 64, 16, 48, ("uniform", 0, 48), ("uniform", 1, 16)),
    case("fa_single_g32_c1", 2, 32, 1, 128, 1, 4096, ("uniform", 1000, 4096), ("fixed", 1)),
    case("fa_decode", 4, 8, 2, 128, 1, 1024, ("uniform", 1, 1024), ("fixed", 1)),
    # more blocks than one-CTA teams, of similar cost: whole blocks dealt to the teams
    case("fa_whole_deal", 48, 16, 4, 128, 64, 384, ("uniform", 128, 384), ("uniform", 1, 64)),
]


def run(cpa, w, fused, alias, mask=None, n_rows=None, len0=None):
    inp = {k: v.to(DEV) for k, v in make_chunk_inputs(w).items()}
    ck, cv = (t.to(DEV) for t in make_cache(w))
    L = inp["past_len"] if len0 is None else len0.to(DEV)
    cache = cpa.KVCache(ck, cv, L.clone())
    past = cache.len if alias else inp["past_len"]
    rows = inp["n_real"] if n_rows is None else n_rows.to(DEV)
    err = cpa.new_error_word()
    kw = dict(past_len=past, n_real=inp["n_real"], mask=None if mask is None else mask.to(DEV), want_sel=True,
              err=err)
    if fused:
        out, sel = cpa.chunk_prefill_attn_append(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], cache, w.P,
                                                 rows, **kw)
    else:
        out, sel = cpa.chunk_prefill_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], cache, w.P, **kw)
        cpa.kv_append(cache, inp["k"], inp["v"], inp["cos"], inp["sin"], rows, err=err)
    torch.cuda.synchronize()
    return out, sel, cache.k, cache.v, cache.len, err


def same(a, b):
    bits = lambda t: t.contiguous().view(torch.uint8) if t.dtype != torch.int32 else t
    for name, x, y in zip(("out", "sel", "k", "v", "len", "err"), a, b):
        assert torch.equal(bits(x), bits(y)), name


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("alias", [False, True], ids=["past_len", "past_is_len"])
def test_fused_equals_attention_then_append(w, alias):
    cpa = lib()
    ref = run(cpa, w, fused=False, alias=False)
    got = run(cpa, w, fused=True, alias=alias)
    same(got, ref)
    n = make_chunk_inputs(w)["n_real"].to(DEV)
    assert torch.equal(got[4], make_chunk_inputs(w)["past_len"].to(DEV) + n)
    assert int(got[5][0]) == 0


def test_fused_with_explicit_mask():
    cpa = lib()
    w = CASES[2]
    L, n = w.past_lens(), w.n_reals()
    mask = explicit_masks(L.numpy(), n.numpy(), w.C, w.P, w.Hq, 512, 1)
    same(run(cpa, w, fused=True, alias=False, mask=mask), run(cpa, w, fused=False, alias=False, mask=mask))


def test_fused_rows_differ_from_n_real():
    cpa = lib()
    w = CASES[0]
    rows = torch.tensor([3, 40], dtype=torch.int32)
    same(run(cpa, w, fused=True, alias=False, n_rows=rows), run(cpa, w, fused=False, alias=False, n_rows=rows))


@pytest.mark.parametrize("w", [CASES[0], CASES[2]], ids=lambda w: w.name)
def test_fused_overflow_leaves_sequence_untouched(w):
    cpa = lib()
    # the last sequence starts 5 rows short of capacity: its append overflows
    L = w.past_lens().clone()
    L[-1] = w.cap - 5
    ref = run(cpa, w, fused=False, alias=False, len0=L)
    got = run(cpa, w, fused=True, alias=False, len0=L)
    same(got, ref)
    assert int(got[4][-1]) == w.cap - 5
    assert int(got[5][0]) & cpa.EBIT["CAPACITY"]


def oracle_fused(w, inp, ck, cv, L0, rows, mask=None, len0=None):
    """The oracle's attention (past lengths L0) over the cache as it is before
    the append, then its global append of rows [0, rows[b]) after len0 (L0 by
    default) cached rows; the cache format follows ck's dtype."""
    kv = "f16" if ck.dtype == torch.float16 else "bf16"
    sel = (inp["n_real"] - 1).clamp(min=0)
    ref, ref_sel = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P, L0,
                               inp["n_real"], mask=mask, sel_row=sel)
    k_np, v_np = bits16(ck).copy(), bits16(cv).copy()
    length = (L0 if len0 is None else len0).numpy().astype(np.int64).copy()
    over = O.kv_append_global(k_np, v_np, length, bf16_bits(inp["k"]), bf16_bits(inp["v"]), inp["cos"].numpy(),
                              inp["sin"].numpy(), rows.numpy(), kv=kv)
    return ref, ref_sel, k_np, v_np, length, over


def check_against_oracle(cpa, w, got, inp, ck, cv, L0, rows, mask=None, len0=None):
    out, sel, gk, gv, glen, err = got
    ref, ref_sel, k_np, v_np, length, over = oracle_fused(w, inp, ck, cv, L0, rows, mask, len0)
    assert_close(out, ref, w.name + "/fused out")
    if (inp["n_real"] > 0).all():
        check_argmax(sel, ref_sel, w.name + "/fused sel")
    assert glen.cpu().numpy().tolist() == length.tolist()
    gk16, gv16 = bits16(gk), bits16(gv)
    for b in range(w.B):
        n = int(length[b])
        assert np.array_equal(gk16[b, :, :n], k_np[b, :, :n]), f"{w.name}: cache K of sequence {b}"
        assert np.array_equal(gv16[b, :, :n], v_np[b, :, :n]), f"{w.name}: cache V of sequence {b}"
    e = int(err[0])
    assert bool(e & cpa.EBIT["CAPACITY"]) == bool(over), (e, over)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fused_matches_oracle(w):
    cpa = lib()
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    got = run(cpa, w, fused=True, alias=True)
    check_against_oracle(cpa, w, got, inp, ck, cv, inp["past_len"], inp["n_real"])


def test_fused_matches_oracle_explicit_mask_rows_and_overflow():
    """The single-tile case with an explicit 512-window mask, the two-tile
    case with n_rows != n_real and a sequence that overflows its cache."""
    cpa = lib()
    w = CASES[2]
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    mask = explicit_masks(inp["past_len"].numpy(), inp["n_real"].numpy(), w.C, w.P, w.Hq, 512, 1)
    got = run(cpa, w, fused=True, alias=False, mask=mask)
    check_against_oracle(cpa, w, got, inp, ck, cv, inp["past_len"], inp["n_real"], mask=mask)

    w = CASES[0]
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    rows = torch.tensor([3, 40], dtype=torch.int32)
    got = run(cpa, w, fused=True, alias=False, n_rows=rows)
    check_against_oracle(cpa, w, got, inp, ck, cv, inp["past_len"], rows)

    # the cache of the last sequence holds cap - 5 rows: its append overflows
    # (the attention still reads past_len rows)
    L = w.past_lens().clone()
    L[-1] = w.cap - 5
    got = run(cpa, w, fused=True, alias=False, len0=L)
    check_against_oracle(cpa, w, got, inp, ck, cv, inp["past_len"], inp["n_real"], len0=L)
