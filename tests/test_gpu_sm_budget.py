"""Attention on a partial SM budget, alone and beside a decode batch on another stream.

`sm_budget` sizes a call's grids for fewer SMs than the device has and holds
its follow-up kernels back until its attention grid ends, so that a decode
batch issued on a second stream runs on the remaining SMs: the mixed
prefill + decode batch of chunked-prefill serving ("functiongemma: chunk
prefill-with-past graph", Change: chunk cost scales with C, so prefill chunks
and decode tokens share a step).  The budget changes only the split of the work
(the stream-K cuts of the two-tile kernel, the split count of the others), so
outputs stay within the attention tolerance of the fp64 oracle, and a call
with a fixed budget is bitwise reproducible whatever runs beside it.
"""
import numpy as np
import pytest
import torch

from synth import Workload, make_chunk_inputs, make_cache
from harness import lib, assert_close, check_argmax, oracle_attn, bits16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def wl(name, B, Hq, Hkv, D, C, P, past, n, causal=1, window=0, seed=0):
    return Workload(name, B=B, Hq=Hq, Hkv=Hkv, D=D, C=C, P=P, cap=P + C, past=past, n_real=n,
                    causal=causal, window=window, seed=seed)


CASES = [
    wl("pair_d128", 2, 8, 2, 128, 200, 700, ("uniform", 0, 700), ("uniform", 1, 200), seed=1),
    wl("pair_d64_window", 2, 16, 2, 64, 129, 300, ("uniform", 0, 300), ("uniform", 0, 129), window=200, seed=2),
    wl("single_d256", 1, 4, 2, 256, 33, 500, ("fixed", 400), ("fixed", 33), seed=3),
    wl("decode_g8", 3, 16, 2, 128, 1, 900, ("uniform", 1, 900), ("fixed", 1), causal=0, seed=4),
]


def run(cpa, w, inp, ck, cv, budget, stream=None):
    d = lambda t: t.to(DEV)
    cache = cpa.KVCache(d(ck), d(cv), d(inp["past_len"]).clone())
    err = cpa.new_error_word()
    sel = d((inp["n_real"] - 1).clamp(min=0))
    f = cpa.decode_step if w.C == 1 else cpa.chunk_prefill_attn
    out, out_sel = f(d(inp["q"]), d(inp["k"]), d(inp["v"]), d(inp["cos"]), d(inp["sin"]), cache, w.P,
                     past_len=d(inp["past_len"]), n_real=d(inp["n_real"]), window=w.window,
                     causal=bool(w.causal), sel_row=sel, want_sel=True, err=err, sm_budget=budget, stream=stream)
    return out, out_sel, err


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
@pytest.mark.parametrize("budget", [1, 3, 37, 151])
def test_budget_matches_oracle(w, budget):
    cpa = lib()
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    out, out_sel, err = run(cpa, w, inp, ck, cv, budget)
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    sel = (inp["n_real"] - 1).clamp(min=0)
    ref, ref_sel = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                               inp["past_len"], inp["n_real"], w.window, w.causal, sel_row=sel)
    assert_close(out, ref, f"{w.name}/budget{budget}")
    if (inp["n_real"] > 0).all():
        check_argmax(out_sel, ref_sel, f"{w.name}/budget{budget}")


def test_budget_at_or_above_the_device_is_the_whole_device():
    cpa = lib()
    w = CASES[0]
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    outs = [run(cpa, w, inp, ck, cv, b)[0] for b in (0, sms, sms + 100)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert np.array_equal(bits16(o), bits16(outs[0]))


def test_prefill_on_budget_beside_decode_on_second_stream():
    """A 4-sequence, 512-row chunk over 4096 past slots on 100 SMs (high-priority
    stream) while a 16-sequence decode batch runs on a second stream: each output
    is bitwise the one its call gives alone, and the prefill output is within
    the oracle's tolerance on sampled (sequence, kv head) groups."""
    cpa = lib()
    pw = wl("mixed_prefill", 4, 32, 8, 128, 512, 4096, ("uniform", 1024, 4096), ("fixed", 512), seed=11)
    dw = wl("mixed_decode", 16, 32, 8, 128, 1, 8192, ("uniform", 1, 8192), ("fixed", 1), causal=0, seed=12)
    # inputs resident on the device first, so that the two calls' launches overlap
    pin, din = ({k: v.to(DEV) for k, v in make_chunk_inputs(w).items()} for w in (pw, dw))
    pk, pv = (t.to(DEV) for t in make_cache(pw))
    dk, dv = (t.to(DEV) for t in make_cache(dw))
    solo_p = run(cpa, pw, pin, pk, pv, 100)
    solo_d = run(cpa, dw, din, dk, dv, 0)
    torch.cuda.synchronize()
    sa = torch.cuda.Stream(priority=-1)
    sb = torch.cuda.Stream(priority=0)
    # every tensor of each call is made and used on that call's stream
    with torch.cuda.stream(sa):
        both_p = run(cpa, pw, pin, pk, pv, 100, stream=sa)
    with torch.cuda.stream(sb):
        both_d = run(cpa, dw, din, dk, dv, 0, stream=sb)
    torch.cuda.synchronize()
    for r in (solo_p, solo_d, both_p, both_d):
        assert int(r[2][0]) == 0
    assert np.array_equal(bits16(both_p[0]), bits16(solo_p[0]))
    assert torch.equal(both_p[1], solo_p[1])
    assert np.array_equal(bits16(both_d[0]), bits16(solo_d[0]))
    assert torch.equal(both_d[1], solo_d[1])
    G = pw.Hq // pw.Hkv
    for b, kvh in ((0, 0), (3, 7)):
        hs = slice(kvh * G, (kvh + 1) * G)
        sub = {k: v[b:b + 1] for k, v in pin.items()}
        L = int(sub["past_len"][0])
        ref, _ = oracle_attn(sub["q"][:, hs], sub["k"][:, kvh:kvh + 1], sub["v"][:, kvh:kvh + 1], sub["cos"],
                             sub["sin"], pk[b:b + 1, kvh:kvh + 1, :L], pv[b:b + 1, kvh:kvh + 1, :L], L,
                             sub["past_len"], sub["n_real"], 0, 1)
        assert_close(both_p[0][b:b + 1, hs], ref, f"mixed/b{b}/kvh{kvh}")


def test_negative_budget_is_refused():
    cpa = lib()
    w = CASES[0]
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    with pytest.raises(cpa.CpaError) as e:
        run(cpa, w, inp, ck, cv, -1)
    assert e.value.status == 2   # CPA_ERR_SHAPE
