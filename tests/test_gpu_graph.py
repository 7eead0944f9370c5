"""The page-1 call shape as one CUDA graph.

"functiongemma: chunk prefill-with-past graph gemma_prefill_with_past" (Change;
Validation) runs the whole 18-layer chunk prefill as one compiled call: 800
cached positions, a 52-token chunk padded to 64, row 51 selected, layers
alternating a 512-position window (base 1e4) and global attention (base 1e6),
one explicit mask and one cos/sin pair per layer type.  Here each layer is an
attention call plus a global append through the C ABI, and the 18 layers are
captured once into a CUDA graph and replayed.  Replays must give the same bits
as the eager calls (outputs, selected rows, cache bytes and lengths), replay
after replay, and the outputs must match the oracle.
"""
import numpy as np
import pytest
import torch

from synth import WORKLOADS, make_chunk_inputs, make_cache, rope_tables
from harness import lib, explicit_masks, oracle_attn, assert_close, check_argmax

pytestmark = pytest.mark.gpu
DEV = "cuda"


def build_layers(cpa):
    w = WORKLOADS["page1"]
    L, n = w.past_lens(), w.n_reals()
    shared = {}
    for kind, W, base in (("sliding", 512, 1e4), ("global", 0, 1e6)):
        cos, sin = rope_tables(L.numpy()[:, None] + np.arange(w.C)[None, :], w.D, base)
        shared[kind] = dict(mask=explicit_masks(L.numpy(), n.numpy(), w.C, w.P, w.Hq, W, 1), cos=cos, sin=sin)
    layers = []
    for layer in range(w.layers):
        kind = "sliding" if layer % 2 == 0 else "global"
        inp = make_chunk_inputs(w, layer=layer)
        ck, cv = make_cache(w, layer=layer)
        layers.append(dict(kind=kind, host=inp, ck0=ck, cv0=cv,
                           q=inp["q"].to(DEV), k=inp["k"].to(DEV), v=inp["v"].to(DEV),
                           cache=cpa.KVCache(ck.to(DEV), cv.to(DEV), inp["past_len"].to(DEV).clone()),
                           out=torch.empty((w.B, w.Hq, w.C, w.D), dtype=torch.bfloat16, device=DEV),
                           sel=torch.empty((w.B, w.Hq * w.D), dtype=torch.float32, device=DEV)))
    dev_shared = {k: {n_: t.to(DEV) for n_, t in v.items()} for k, v in shared.items()}
    ctx = dict(w=w, L=L, n=n, shared=shared, dshared=dev_shared,
               len0=L.to(DEV), n_real=n.to(DEV), past=L.to(DEV),
               sel_row=torch.full((w.B,), 51, dtype=torch.int32, device=DEV),
               ws=torch.empty(max(1, cpa.attn_workspace_size(w.B, w.Hq, w.Hkv, w.D, w.C, w.P)),
                              dtype=torch.uint8, device=DEV),
               err=cpa.new_error_word())
    return ctx, layers


def reset(layers, ctx):
    for ly in layers:
        ly["cache"].k.copy_(ly["ck0"], non_blocking=True)
        ly["cache"].v.copy_(ly["cv0"], non_blocking=True)
        ly["cache"].len.copy_(ctx["len0"])


def run_layers(cpa, ctx, layers):
    w = ctx["w"]
    for ly in layers:
        sh = ctx["dshared"][ly["kind"]]
        cpa.chunk_prefill_attn(ly["q"], ly["k"], ly["v"], sh["cos"], sh["sin"], ly["cache"], w.P,
                               past_len=ctx["past"], n_real=ctx["n_real"], mask=sh["mask"],
                               sel_row=ctx["sel_row"], out=ly["out"], out_sel=ly["sel"], workspace=ctx["ws"],
                               err=ctx["err"])
        cpa.kv_append(ly["cache"], ly["k"], ly["v"], sh["cos"], sh["sin"], ctx["n_real"], err=ctx["err"])


def snapshot(layers):
    return [(ly["out"].clone(), ly["sel"].clone(), ly["cache"].k.clone(), ly["cache"].v.clone(),
             ly["cache"].len.clone()) for ly in layers]


def test_page1_eighteen_layers_as_one_cuda_graph():
    cpa = lib()
    ctx, layers = build_layers(cpa)
    w = ctx["w"]
    reset(layers, ctx)
    run_layers(cpa, ctx, layers)            # eager (also sets kernel attributes before capture)
    torch.cuda.synchronize()
    assert int(ctx["err"][0]) == 0
    eager = snapshot(layers)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_layers(cpa, ctx, layers)
    for rep in range(2):
        reset(layers, ctx)
        for ly in layers:
            ly["out"].zero_()
            ly["sel"].zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(ctx["err"][0]) == 0
        for l, (ly, e) in enumerate(zip(layers, eager)):
            got = (ly["out"], ly["sel"], ly["cache"].k, ly["cache"].v, ly["cache"].len)
            for name, a, b in zip(("out", "sel", "k", "v", "len"), got, e):
                assert torch.equal(a.view(torch.uint8) if a.dtype != torch.int32 else a,
                                   b.view(torch.uint8) if b.dtype != torch.int32 else b), (rep, l, name)
        assert int(layers[0]["cache"].len[0]) == int(ctx["L"][0]) + int(ctx["n"][0])

    # the graph's outputs against the oracle, one layer of each type
    sel = torch.full((w.B,), 51, dtype=torch.int32)
    for l in (0, 1):
        ly = layers[l]
        sh = ctx["shared"][ly["kind"]]
        h = ly["host"]
        ref, ref_sel = oracle_attn(h["q"], h["k"], h["v"], sh["cos"], sh["sin"], ly["ck0"], ly["cv0"], w.P,
                                   ctx["L"], ctx["n"], mask=sh["mask"], sel_row=sel)
        assert_close(ly["out"], ref, f"page1 graph/L{l}")
        check_argmax(ly["sel"], ref_sel, f"page1 graph/L{l}")
