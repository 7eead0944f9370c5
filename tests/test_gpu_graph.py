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


@pytest.mark.parametrize("D,window", [(256, 0), (256, 96), (128, 0)])
def test_chunk_sequence_in_one_graph_reads_each_previous_append(D, window):
    """Chunked prefill as one CUDA graph: four chunks, each an attention call
    whose past length is the cache's own length, then the chunk's append.  In
    a graph the launches follow one another with no host gap, so every chunk
    must see exactly the rows and length the previous chunk's append wrote
    ("functiongemma: chunk prefill-with-past graph", Change: K/V extended by
    the chunk).  Each chunk's output is checked against the oracle run chunk
    by chunk, and the final cache bytes and lengths exactly."""
    import oracle as O
    from synth import normal_bf16, bf16_bits
    from harness import bits16
    cpa = lib()
    B, Hq, Hkv, C, NCH = 2, 8, 2, 64, 4
    L0 = np.array([37, 100])
    cap = int(L0.max()) + NCH * C
    ck = normal_bf16((B, Hkv, cap, D), 0, f"seqgraph/{D}/ck")
    cv = normal_bf16((B, Hkv, cap, D), 0, f"seqgraph/{D}/cv")
    chunks = []
    for c in range(NCH):
        pos = L0[:, None] + c * C + np.arange(C)[None, :]
        cos, sin = rope_tables(pos, D, 10000.0)
        chunks.append(dict(q=normal_bf16((B, Hq, C, D), 0, f"seqgraph/{D}/{c}/q"),
                           k=normal_bf16((B, Hkv, C, D), 0, f"seqgraph/{D}/{c}/k"),
                           v=normal_bf16((B, Hkv, C, D), 0, f"seqgraph/{D}/{c}/v"), cos=cos, sin=sin))
    dev = [{k: t.to(DEV) for k, t in ch.items()} for ch in chunks]
    full = torch.full((B,), C, dtype=torch.int32, device=DEV)
    cache = cpa.KVCache(ck.to(DEV), cv.to(DEV), torch.from_numpy(L0.astype(np.int32)).to(DEV))
    outs = [torch.empty((B, Hq, C, D), dtype=torch.bfloat16, device=DEV) for _ in range(NCH)]
    ws = torch.empty(max(1, cpa.attn_workspace_size(B, Hq, Hkv, D, C, cap)), dtype=torch.uint8, device=DEV)
    err = cpa.new_error_word()

    def run():
        for c in range(NCH):
            x = dev[c]
            cpa.chunk_prefill_attn(x["q"], x["k"], x["v"], x["cos"], x["sin"], cache, cap, past_len=cache.len,
                                   n_real=full, window=window, out=outs[c], workspace=ws, err=err)
            cpa.kv_append(cache, x["k"], x["v"], x["cos"], x["sin"], full, err=err)

    def reset():
        cache.k.copy_(ck.to(DEV))
        cache.v.copy_(cv.to(DEV))
        cache.len.copy_(torch.from_numpy(L0.astype(np.int32)).to(DEV))

    run()                                   # eager warm-up (kernel attributes before capture)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    reset()
    with torch.cuda.graph(g):
        run()
    # the oracle, chunk by chunk over its own copy of the cache
    ok_, ov_ = bits16(ck).copy(), bits16(cv).copy()
    olen = L0.astype(np.int64).copy()
    refs = []
    for c in range(NCH):
        x = chunks[c]
        ref, _ = O.chunk_prefill_attn(bf16_bits(x["q"]), bf16_bits(x["k"]), bf16_bits(x["v"]), x["cos"].numpy(),
                                      x["sin"].numpy(), ok_, ov_, cap, olen.copy(), np.full(B, C), window=window,
                                      causal=1)
        refs.append(ref)
        assert O.kv_append_global(ok_, ov_, olen, bf16_bits(x["k"]), bf16_bits(x["v"]), x["cos"].numpy(),
                                  x["sin"].numpy(), np.full(B, C)) == []
    for rep in range(3):
        reset()
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(err[0]) == 0
        for c in range(NCH):
            assert_close(outs[c], refs[c], f"chunk graph D{D} w{window} rep{rep} chunk{c}")
        assert cache.len.cpu().numpy().tolist() == olen.tolist()
        assert np.array_equal(bits16(cache.k), ok_) and np.array_equal(bits16(cache.v), ov_)


def test_prepared_calls_equal_plain_calls():
    """The page-1 layers run eagerly through prepared calls (arguments bound
    once, then only enqueued) give the same bits as the plain binding:
    outputs, selected rows, cache bytes and lengths."""
    cpa = lib()
    ctx, layers = build_layers(cpa)
    reset(layers, ctx)
    run_layers(cpa, ctx, layers)
    torch.cuda.synchronize()
    plain = snapshot(layers)
    w = ctx["w"]
    calls = []
    for ly in layers:
        sh = ctx["dshared"][ly["kind"]]
        calls.append(cpa.prepare_chunk_prefill_attn(
            ly["q"], ly["k"], ly["v"], sh["cos"], sh["sin"], ly["cache"], w.P, past_len=ctx["past"],
            n_real=ctx["n_real"], mask=sh["mask"], sel_row=ctx["sel_row"], out=ly["out"], out_sel=ly["sel"],
            workspace=ctx["ws"], err=ctx["err"]))
        calls.append(cpa.prepare_kv_append(ly["cache"], ly["k"], ly["v"], sh["cos"], sh["sin"], ctx["n_real"],
                                           err=ctx["err"]))
    for rep in range(2):
        reset(layers, ctx)
        for ly in layers:
            ly["out"].zero_()
            ly["sel"].zero_()
        for call in calls:
            call()
        torch.cuda.synchronize()
        assert int(ctx["err"][0]) == 0
        for l, (ly, e) in enumerate(zip(layers, plain)):
            got = (ly["out"], ly["sel"], ly["cache"].k, ly["cache"].v, ly["cache"].len)
            for name, a, b in zip(("out", "sel", "k", "v", "len"), got, e):
                assert torch.equal(a.view(torch.uint8) if a.dtype != torch.int32 else a,
                                   b.view(torch.uint8) if b.dtype != torch.int32 else b), (rep, l, name)


@pytest.mark.parametrize("D,window", [(256, 0), (256, 96), (128, 0)])
def test_outputs_fed_back_as_queries_in_one_graph(D, window):
    """Each chunk's query is the previous chunk's output tensor, with the
    appends in between, all captured in one CUDA graph: every call must read
    what the call before it wrote, with no host gap between the launches.
    The replays equal a run with a device sync after every call, bit for
    bit; the first chunk (all inputs synthetic) also matches the oracle."""
    from synth import normal_bf16
    cpa = lib()
    B, Hq, Hkv, C, NCH = 2, 8, 2, 64, 4
    L0 = np.array([37, 100])
    cap = int(L0.max()) + NCH * C
    ck = normal_bf16((B, Hkv, cap, D), 0, f"fedback/{D}/ck")
    cv = normal_bf16((B, Hkv, cap, D), 0, f"fedback/{D}/cv")
    q0 = normal_bf16((B, Hq, C, D), 0, f"fedback/{D}/q0")
    ks = [normal_bf16((B, Hkv, C, D), 0, f"fedback/{D}/{c}/k").to(DEV) for c in range(NCH)]
    vs = [normal_bf16((B, Hkv, C, D), 0, f"fedback/{D}/{c}/v").to(DEV) for c in range(NCH)]
    tabs = [tuple(t.to(DEV) for t in rope_tables(L0[:, None] + c * C + np.arange(C)[None, :], D, 10000.0))
            for c in range(NCH)]
    full = torch.full((B,), C, dtype=torch.int32, device=DEV)
    cache = cpa.KVCache(ck.to(DEV), cv.to(DEV), torch.from_numpy(L0.astype(np.int32)).to(DEV))
    qin = q0.to(DEV)
    outs = [torch.empty((B, Hq, C, D), dtype=torch.bfloat16, device=DEV) for _ in range(NCH)]
    ws = torch.empty(max(1, cpa.attn_workspace_size(B, Hq, Hkv, D, C, cap)), dtype=torch.uint8, device=DEV)
    err = cpa.new_error_word()

    def run(sync):
        for c in range(NCH):
            q = qin if c == 0 else outs[c - 1]
            cos, sin = tabs[c]
            cpa.chunk_prefill_attn(q, ks[c], vs[c], cos, sin, cache, cap, past_len=cache.len, n_real=full,
                                   window=window, out=outs[c], workspace=ws, err=err)
            if sync:
                torch.cuda.synchronize()
            cpa.kv_append(cache, ks[c], vs[c], cos, sin, full, err=err)
            if sync:
                torch.cuda.synchronize()

    def reset():
        cache.k.copy_(ck.to(DEV))
        cache.v.copy_(cv.to(DEV))
        cache.len.copy_(torch.from_numpy(L0.astype(np.int32)).to(DEV))
        for o in outs:
            o.zero_()

    reset()
    run(sync=True)
    assert int(err[0]) == 0
    ref = [o.clone() for o in outs] + [cache.k.clone(), cache.v.clone(), cache.len.clone()]
    cos0, sin0 = (t.cpu() for t in tabs[0])
    oref, _ = oracle_attn(q0, ks[0].cpu(), vs[0].cpu(), cos0, sin0, ck, cv, cap,
                          torch.from_numpy(L0.astype(np.int32)), torch.full((B,), C, dtype=torch.int32), window, 1)
    assert_close(outs[0], oref, f"fed back D{D} w{window} chunk 0")
    g = torch.cuda.CUDAGraph()
    reset()
    with torch.cuda.graph(g):
        run(sync=False)
    for rep in range(3):
        reset()
        g.replay()
        torch.cuda.synchronize()
        assert int(err[0]) == 0
        got = outs + [cache.k, cache.v, cache.len]
        for k, (a, b) in enumerate(zip(got, ref)):
            assert torch.equal(a.view(torch.uint8) if a.dtype != torch.int32 else a,
                               b.view(torch.uint8) if b.dtype != torch.int32 else b), (rep, k)
