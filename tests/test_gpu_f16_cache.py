"""An fp16 KV cache on the GPU, against the oracle's fp16 reading.

"Pad the chunked-prefill tail for sliding-window models" (Declined with
rationale) names a runtime option that keeps the KV cache in fp16.  With
cpa_cache.dtype = CPA_KV_F16: appends round the fp32 key rotation to half and
convert values to half (bit-exact against the oracle, global and sliding,
through a padded tail with snapshot and rollback); the attention runs its
products in fp16 on every path (two-tile, single-tile with and without a
cluster, decode, explicit mask, fused append) and matches the oracle within
the attention tolerance; explicit and implicit masks give the same bits; the
fused attention + append matches the oracle's fp16 reading and its half
append directly.
"""
import numpy as np
import pytest
import torch

import oracle as O
from synth import Workload, make_chunk_inputs, make_cache, normal_bf16, rope_tables, bf16_bits, uniform_int
from harness import (lib, assert_close, check_argmax, oracle_attn, explicit_masks, bits16,
                     assert_explicit_matches)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def small(name, B, Hq, Hkv, D, C, P, L, n, window=0, causal=1):
    return Workload(name, B=B, Hq=Hq, Hkv=Hkv, D=D, C=C, P=P, cap=P + C, past=L, n_real=n, window=window,
                    causal=causal)


CASES = [
    small("h_pair_d128", 2, 8, 2, 128, 40, 300, ("uniform", 0, 300), ("uniform", 1, 40)),
    small("h_pair_d64", 2, 4, 1, 64, 130, 257, ("uniform", 0, 257), ("uniform", 1, 130)),
    small("h_single_d256", 1, 8, 1, 256, 128, 512, ("fixed", 512), ("fixed", 127), window=512),
    small("h_single_small", 2, 4, 1, 64, 16, 48, ("uniform", 0, 48), ("uniform", 1, 16)),
    small("h_single_g32_c1", 2, 32, 1, 128, 1, 600, ("uniform", 100, 600), ("fixed", 1), causal=0),
    small("h_decode", 3, 8, 2, 128, 1, 700, ("uniform", 1, 700), ("fixed", 1), causal=0),
    small("h_decode_d64_win", 2, 8, 2, 64, 1, 900, ("uniform", 300, 900), ("fixed", 1), window=100, causal=0),
    # more (sequence, kv head) blocks than one-CTA teams, all of similar cost:
    # the plan deals whole blocks to the teams (the planned-order walk)
    small("h_whole_deal_d64", 64, 16, 4, 64, 64, 384, ("uniform", 128, 384), ("uniform", 1, 64)),
    small("h_whole_deal_d128", 48, 16, 4, 128, 64, 384, ("uniform", 128, 384), ("uniform", 1, 64)),
    # the page-1 call shape: two query tiles of 8 splits, each split taken by
    # two CTAs that divide D (clusters of 16)
    small("h_page1_d256", 1, 4, 1, 256, 64, 800, ("fixed", 800), ("fixed", 52)),
]


def run_gpu(cpa, inp, ck, cv, P, window=0, causal=True, mask=None):
    d = lambda t: None if t is None else t.to(DEV)
    cache = cpa.KVCache(d(ck), d(cv), d(inp["past_len"]).clone())
    err = cpa.new_error_word()
    out, sel = cpa.chunk_prefill_attn(d(inp["q"]), d(inp["k"]), d(inp["v"]), d(inp["cos"]), d(inp["sin"]), cache, P,
                                      past_len=d(inp["past_len"]), n_real=d(inp["n_real"]), window=window,
                                      causal=causal, mask=d(mask), want_sel=True, err=err)
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    return out, sel


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_f16_cache_attention_matches_oracle(w):
    cpa = lib()
    inp = make_chunk_inputs(w)
    ck, cv = (t.to(torch.float16) for t in make_cache(w))   # N(0,1) bf16 values convert exactly
    out, sel = run_gpu(cpa, inp, ck, cv, w.P, w.window, bool(w.causal))
    ref, ref_sel = oracle_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], ck, cv, w.P,
                               inp["past_len"], inp["n_real"], w.window, w.causal,
                               sel_row=(inp["n_real"] - 1).clamp(min=0))
    assert_close(out, ref, w.name)
    check_argmax(sel, ref_sel, w.name)
    mask = explicit_masks(inp["past_len"].numpy(), inp["n_real"].numpy(), w.C, w.P, w.Hq, w.window, w.causal)
    out_e, _ = run_gpu(cpa, inp, ck, cv, w.P, mask=mask)
    assert_close(out_e, ref, w.name + "/explicit")
    assert_explicit_matches(out_e, out, w.name)


@pytest.mark.parametrize("D,Hkv", [(64, 1), (128, 4), (256, 2)])
def test_f16_global_append_bit_exact(D, Hkv):
    cpa = lib()
    B, C, cap = 6, 24, 80
    L0 = uniform_int(0, cap - C, B, 0, f"h_ga/{D}/L").numpy()
    n = uniform_int(0, C, B, 0, f"h_ga/{D}/n").numpy()
    ck = normal_bf16((B, Hkv, cap, D), 0, f"h_ga/{D}/ck").to(torch.float16)
    cv = normal_bf16((B, Hkv, cap, D), 0, f"h_ga/{D}/cv").to(torch.float16)
    k = normal_bf16((B, Hkv, C, D), 0, f"h_ga/{D}/k")
    v = normal_bf16((B, Hkv, C, D), 0, f"h_ga/{D}/v")
    cos, sin = rope_tables(L0[:, None] + np.arange(C)[None, :], D, 10000.0)
    ok_, ov_ = bits16(ck).copy(), bits16(cv).copy()
    olen = L0.astype(np.int64).copy()
    assert O.kv_append_global(ok_, ov_, olen, bf16_bits(k), bf16_bits(v), cos.numpy(), sin.numpy(), n,
                              kv="f16") == []
    gk, gv = ck.to(DEV), cv.to(DEV)
    glen = torch.from_numpy(L0.astype(np.int32)).to(DEV)
    cache = cpa.KVCache(gk, gv, glen)
    err = cpa.kv_append(cache, k.to(DEV), v.to(DEV), cos.to(DEV), sin.to(DEV), torch.from_numpy(n.astype(np.int32)).to(DEV))
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    assert np.array_equal(glen.cpu().numpy(), olen)
    assert np.array_equal(bits16(gk), ok_) and np.array_equal(bits16(gv), ov_)


@pytest.mark.parametrize("prefix,tail", [(1, 9), (7, 127), (7, 2)])
def test_f16_sliding_padded_tail_equals_exact_append(prefix, tail):
    """Full chunks into a 512-row fp16 window cache, then a padded tail with
    snapshot -> padded append -> rollback: bytes equal the oracle's exact appends."""
    cpa = lib()
    B, Hkv, D, W, C = 1, 1, 128, 512, 128
    gk = torch.zeros((B, Hkv, W, D), dtype=torch.float16, device=DEV)
    cache = cpa.KVCache(gk, gk.clone(), torch.zeros(B, dtype=torch.int32, device=DEV), cpa.SLIDING, W, 0)
    scratch = torch.empty(cpa.cache_scratch_size(cache, C), dtype=torch.uint8, device=DEV)
    ok_ = np.zeros((B, Hkv, W, D), np.uint16); ov_ = ok_.copy(); ol = np.zeros(B, np.int64)
    s = 0
    for c in range(prefix + 1):
        n = C if c < prefix else tail
        k = normal_bf16((B, Hkv, C, D), 0, f"h_sl/{c}/k")
        v = normal_bf16((B, Hkv, C, D), 0, f"h_sl/{c}/v")
        k[:, :, n:] = 0
        v[:, :, n:] = 0
        cos, sin = rope_tables(np.arange(s, s + C)[None, :], D, 10000.0)
        nr = torch.tensor([n], dtype=torch.int32, device=DEV)
        full = torch.tensor([C], dtype=torch.int32, device=DEV)
        if n < C:
            err = cpa.kv_snapshot_padded_append(cache, nr, C, scratch)
            cpa.kv_append(cache, k.to(DEV), v.to(DEV), cos.to(DEV), sin.to(DEV), full, scratch=scratch, err=err)
            cpa.kv_rollback_padded_append(cache, C, scratch, err=err)
        else:
            err = cpa.kv_append(cache, k.to(DEV), v.to(DEV), cos.to(DEV), sin.to(DEV), nr, scratch=scratch)
        torch.cuda.synchronize()
        assert int(err[0]) == 0
        O.kv_append_sliding(ok_, ov_, ol, bf16_bits(k), bf16_bits(v), cos.numpy(), sin.numpy(), [n], W, kv="f16")
        s += n
    Lf = int(ol[0])
    assert int(cache.len[0]) == Lf
    assert np.array_equal(bits16(cache.k)[:, :, :Lf], ok_[:, :, :Lf])
    assert np.array_equal(bits16(cache.v)[:, :, :Lf], ov_[:, :, :Lf])


@pytest.mark.parametrize("w", [CASES[0], CASES[2], CASES[5], CASES[-2], CASES[-1]], ids=lambda w: w.name)
def test_f16_fused_append_equals_attention_then_append(w):
    cpa = lib()
    inp = {k: v.to(DEV) for k, v in make_chunk_inputs(w).items()}
    outs = []
    for fused in (False, True):
        ck, cv = (t.to(torch.float16).to(DEV) for t in make_cache(w))
        cache = cpa.KVCache(ck, cv, inp["past_len"].clone())
        err = cpa.new_error_word()
        kw = dict(past_len=inp["past_len"], n_real=inp["n_real"], window=w.window, causal=bool(w.causal), err=err)
        if fused:
            out, _ = cpa.chunk_prefill_attn_append(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], cache, w.P,
                                                   inp["n_real"], **kw)
        else:
            out, _ = cpa.chunk_prefill_attn(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], cache, w.P, **kw)
            cpa.kv_append(cache, inp["k"], inp["v"], inp["cos"], inp["sin"], inp["n_real"], err=err)
        torch.cuda.synchronize()
        assert int(err[0]) == 0
        outs.append((out, cache.k, cache.v, cache.len))
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int16) if a.dtype != torch.int32 else a,
                           b.view(torch.int16) if b.dtype != torch.int32 else b)
    # and the fused call against the oracle directly: its fp16 reading of the
    # attention, then its global append in half (cache rows [0, len) and len exact)
    out, gk, gv, glen = outs[1]
    host = {k: v.cpu() for k, v in inp.items()}
    ck, cv = (t.to(torch.float16) for t in make_cache(w))
    ref, _ = oracle_attn(host["q"], host["k"], host["v"], host["cos"], host["sin"], ck, cv, w.P,
                         host["past_len"], host["n_real"], w.window, w.causal)
    assert_close(out, ref, w.name + "/f16 fused")
    ok_, ov_ = bits16(ck).copy(), bits16(cv).copy()
    ol = host["past_len"].numpy().astype(np.int64).copy()
    assert O.kv_append_global(ok_, ov_, ol, bf16_bits(host["k"]), bf16_bits(host["v"]), host["cos"].numpy(),
                              host["sin"].numpy(), host["n_real"].numpy(), kv="f16") == []
    assert glen.cpu().numpy().tolist() == ol.tolist()
    for b in range(w.B):
        n = int(ol[b])
        assert np.array_equal(bits16(gk)[b, :, :n], ok_[b, :, :n])
        assert np.array_equal(bits16(gv)[b, :, :n], ov_[b, :, :n])
