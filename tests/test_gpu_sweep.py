"""A seeded sweep of chunk-attention shapes on the GPU against the fp64 oracle.

The shapes are drawn once from a fixed seed and named in the test ids: batch 1
or 2, one or two kv heads, groups of 1 to 16 query heads, head dims 64 / 128 /
256, chunks of 1 to 200 rows (ragged against every tile size), pasts of 0 to 700
slots with per-sequence lengths, per-sequence real-row counts down to zero,
causal and not, with and without a window.  Every kernel path is met (two-tile,
single-tile with and without a cluster merge, one-token decode).  Each case
runs the implicit mask and the explicit mask built from the same rule
("functiongemma: chunk prefill-with-past graph", Change: per-head additive mask
over past + C keys) and checks both against the oracle (max-abs 1e-2, rel-L2
3e-3), the selected-row argmax, and the two masks against each other
(bitwise).
"""
import numpy as np
import pytest
import torch

from synth import Workload, make_chunk_inputs, make_cache
from harness import (lib, assert_close, check_argmax, oracle_attn, explicit_masks,
                     assert_explicit_matches)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def draw_cases(n=48, seed=20261202):
    rng = np.random.RandomState(seed)
    cases = []
    for k in range(n):
        D = int(rng.choice([64, 128, 256]))
        Hkv = int(rng.choice([1, 2]))
        G = int(rng.choice([1, 2, 4, 8, 16]))
        C = int(rng.choice([1, 5, 17, 33, 64, 100, 129, 200]))
        P = int(rng.choice([0, 1, 63, 128, 300, 700]))
        B = int(rng.randint(1, 3))
        causal = int(rng.rand() < 0.8)
        window = int(rng.choice([0, 0, 0, 37, 200]))
        past = ("uniform", int(rng.randint(0, P)), P) if P > 0 else ("fixed", 0)
        name = f"sw{k}_B{B}_g{G}x{Hkv}_D{D}_C{C}_P{P}_w{window}_c{causal}"
        cases.append(Workload(name, B=B, Hq=Hkv * G, Hkv=Hkv, D=D, C=C, P=P, cap=P + C, past=past,
                              n_real=("uniform", 0, C), window=window, causal=causal, seed=k))
    return cases


CASES = draw_cases()


def run(cpa, inp, ck, cv, w, mask=None):
    d = lambda t: None if t is None else t.to(DEV)
    cache = cpa.KVCache(d(ck), d(cv), d(inp["past_len"]).clone())
    err = cpa.new_error_word()
    sel = (inp["n_real"] - 1).clamp(min=0)
    out, out_sel = cpa.chunk_prefill_attn(d(inp["q"]), d(inp["k"]), d(inp["v"]), d(inp["cos"]), d(inp["sin"]),
                                          cache, w.P, past_len=d(inp["past_len"]), n_real=d(inp["n_real"]),
                                          window=w.window, causal=bool(w.causal), mask=d(mask), sel_row=d(sel),
                                          want_sel=True, err=err)
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    return out, out_sel, sel


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_sweep_matches_oracle(w):
    cpa = lib()
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    out, out_sel, sel = run(cpa, inp, ck, cv, w)
    ref, ref_sel = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                               inp["past_len"], inp["n_real"], w.window, w.causal, sel_row=sel)
    assert_close(out, ref, w.name)
    if (inp["n_real"] > 0).all():
        check_argmax(out_sel, ref_sel, w.name)
    mask = explicit_masks(inp["past_len"].numpy(), inp["n_real"].numpy(), w.C, w.P, w.Hq, w.window, w.causal)
    out_e, _, _ = run(cpa, inp, ck, cv, w, mask=mask)
    assert_close(out_e, ref, w.name + "/explicit")
    assert_explicit_matches(out_e, out, w.name)


@pytest.mark.parametrize("w", CASES[::3], ids=lambda w: w.name)
def test_sweep_fp16_cache_matches_oracle(w):
    """Every third drawn shape over an fp16 KV cache (the bf16 N(0,1) cache
    values convert exactly), against the oracle's fp16 reading: products in
    fp16, P rounded to half ("Pad the chunked-prefill tail for sliding-window
    models", Declined with rationale: the fp16 KV-cache runtime option)."""
    cpa = lib()
    inp = make_chunk_inputs(w)
    ck, cv = (t.to(torch.float16) for t in make_cache(w))
    out, out_sel, sel = run(cpa, inp, ck, cv, w)
    ref, ref_sel = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                               inp["past_len"], inp["n_real"], w.window, w.causal, sel_row=sel)
    assert_close(out, ref, w.name + "/f16")
    if (inp["n_real"] > 0).all():
        check_argmax(out_sel, ref_sel, w.name + "/f16")


@pytest.mark.parametrize("w", [w for w in CASES if w.C > 1][::2], ids=lambda w: w.name)
def test_sweep_fused_append_equals_attention_then_append(w):
    """cpa_chunk_prefill_attn_append on every second drawn chunk shape gives
    exactly the bits of attention followed by cpa_kv_append: output, selected
    row, cache bytes, lengths and error word ("functiongemma: chunk
    prefill-with-past graph", Change: K/V extended by the chunk)."""
    from test_gpu_fused_append import run as run_pair, same
    cpa = lib()
    same(run_pair(cpa, w, fused=True, alias=True), run_pair(cpa, w, fused=False, alias=False))
