"""The attention entry point for callers that cannot allocate device memory.

cpa_chunk_prefill_attn_noalloc serves code that has no way to obtain a
workspace: work recorded during CUDA graph capture, runtimes that plan every
buffer once from static shapes, and plugins inside a framework that owns the
allocator.  Its split-KV partials live in the library's fixed 16 MiB array.
This test calls it through the C ABI twice in a row, on two problems that both
need split-KV partials, and checks each output against the regular entry point
(which takes a caller workspace) within the attention tolerance.  It also
checks that a problem needing more than 16 MiB of partials is refused.
"""
import pytest
import torch

from synth import Workload, make_chunk_inputs, make_cache
from harness import lib, compare, MAX_ABS, REL_L2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def case(name, B, Hq, Hkv, D, C, P, past, n):
    return Workload(name, B=B, Hq=Hq, Hkv=Hkv, D=D, C=C, P=P, cap=P + C, past=past, n_real=n)


def run(cpa, w, noalloc):
    inp = {k: v.to(DEV) for k, v in make_chunk_inputs(w).items()}
    ck, cv = (t.to(DEV) for t in make_cache(w))
    cache = cpa.KVCache(ck, cv, inp["past_len"].clone())
    err = cpa.new_error_word()
    f = cpa.chunk_prefill_attn_noalloc if noalloc else cpa.chunk_prefill_attn
    out, _ = f(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], cache, w.P, past_len=inp["past_len"],
               n_real=inp["n_real"], err=err)
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    return out


def test_noalloc_matches_regular_entry_point_two_calls_in_a_row():
    cpa = lib()
    decode_like = case("noalloc_decode", 8, 32, 8, 128, 1, 4096, ("uniform", 100, 4096), ("fixed", 1))
    prefill = case("noalloc_prefill", 2, 8, 2, 128, 40, 300, ("uniform", 0, 300), ("uniform", 1, 40))
    for w in (decode_like, prefill):
        need = cpa.attn_workspace_size(w.B, w.Hq, w.Hkv, w.D, w.C, w.P)
        assert 0 < need <= 16 << 20, (w.name, need)
    got = [run(cpa, w, noalloc=True) for w in (decode_like, prefill)]   # two calls in a row
    for w, out in zip((decode_like, prefill), got):
        ref = run(cpa, w, noalloc=False).double().cpu().numpy()
        max_abs, rel = compare(out, ref, w.name)
        assert max_abs <= MAX_ABS and rel <= REL_L2, (w.name, max_abs, rel)


def test_noalloc_refuses_problems_beyond_its_array():
    cpa = lib()
    B, Hq, Hkv, D, P = 128, 32, 8, 128, 32768   # a decode batch whose split-KV partials need ~18 MiB
    assert cpa.attn_workspace_size(B, Hq, Hkv, D, 1, P) > 16 << 20
    q = torch.zeros((B, Hq, 1, D), dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros((B, Hkv, 1, D), dtype=torch.bfloat16, device=DEV)
    tab = torch.zeros((B, 1, D), dtype=torch.float32, device=DEV)
    ck = torch.zeros((B, Hkv, 8, D), dtype=torch.bfloat16, device=DEV)   # never read: refused first
    length = torch.zeros((B,), dtype=torch.int32, device=DEV)
    cache = cpa.KVCache(ck, ck, length)
    with pytest.raises(cpa.CpaError) as e:
        cpa.chunk_prefill_attn_noalloc(q, kv, kv, tab, tab, cache, P, past_len=length, n_real=length + 1)
    assert e.value.status == 6
