"""The attention entry point for callers that cannot allocate device memory.

cpa_chunk_prefill_attn_noalloc serves code that has no way to obtain a
workspace: work recorded during CUDA graph capture, runtimes that plan every
buffer once from static shapes, and plugins inside a framework that owns the
allocator.  Its split-KV partials live in the library's fixed 16 MiB array.
This test calls it through the C ABI twice in a row, on two problems that both
need split-KV partials, and checks each output against the regular entry point
(which takes a caller workspace): both run the same geometry and arithmetic,
so the outputs must be bitwise identical.  A two-tile problem whose partials
only fit the array on a partial SM budget must run with that budget and be
refused without it; a problem needing more than 16 MiB is refused.
"""
import pytest
import torch

from synth import Workload, make_chunk_inputs, make_cache
from harness import lib

pytestmark = pytest.mark.gpu
DEV = "cuda"
ARRAY_BYTES = 16 << 20


def case(name, B, Hq, Hkv, D, C, P, past, n):
    return Workload(name, B=B, Hq=Hq, Hkv=Hkv, D=D, C=C, P=P, cap=P + C, past=past, n_real=n)


def run(cpa, w, noalloc, sm_budget=0):
    inp = {k: v.to(DEV) for k, v in make_chunk_inputs(w).items()}
    ck, cv = (t.to(DEV) for t in make_cache(w))
    cache = cpa.KVCache(ck, cv, inp["past_len"].clone())
    err = cpa.new_error_word()
    f = cpa.chunk_prefill_attn_noalloc if noalloc else cpa.chunk_prefill_attn
    out, _ = f(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], cache, w.P, past_len=inp["past_len"],
               n_real=inp["n_real"], err=err, sm_budget=sm_budget)
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    return out


def same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_noalloc_matches_regular_entry_point_two_calls_in_a_row():
    cpa = lib()
    decode_like = case("noalloc_decode", 8, 32, 8, 128, 1, 4096, ("uniform", 100, 4096), ("fixed", 1))
    prefill = case("noalloc_prefill", 2, 8, 2, 128, 40, 300, ("uniform", 0, 300), ("uniform", 1, 40))
    for w in (decode_like, prefill):
        need = cpa.attn_workspace_size(w.B, w.Hq, w.Hkv, w.D, w.C, w.P)
        assert 0 < need <= ARRAY_BYTES, (w.name, need)
    got = [run(cpa, w, noalloc=True) for w in (decode_like, prefill)]   # two calls in a row
    for w, out in zip((decode_like, prefill), got):
        assert same_bits(out, run(cpa, w, noalloc=False)), w.name


def test_noalloc_sizes_the_call_for_its_sm_budget():
    """Two-tile partial slots scale with the persistent grid: on the whole GPU
    this problem needs more than the array, on 32 SMs it fits."""
    cpa = lib()
    w = case("noalloc_budget", 4, 16, 4, 128, 256, 4096, ("uniform", 1000, 4096), ("uniform", 1, 256))
    assert cpa.attn_workspace_size(w.B, w.Hq, w.Hkv, w.D, w.C, w.P) > ARRAY_BYTES
    with pytest.raises(cpa.CpaError) as e:
        run(cpa, w, noalloc=True)
    assert e.value.status == 6
    budget = 32
    got = [run(cpa, w, noalloc=True, sm_budget=budget) for _ in range(2)]
    ref = run(cpa, w, noalloc=False, sm_budget=budget)
    assert same_bits(got[0], ref) and same_bits(got[1], ref)


def test_noalloc_refuses_problems_beyond_its_array():
    cpa = lib()
    B, Hq, Hkv, D, P = 128, 32, 8, 128, 32768   # a decode batch whose split-KV partials need ~18 MiB
    assert cpa.attn_workspace_size(B, Hq, Hkv, D, 1, P) > ARRAY_BYTES
    q = torch.zeros((B, Hq, 1, D), dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros((B, Hkv, 1, D), dtype=torch.bfloat16, device=DEV)
    tab = torch.zeros((B, 1, D), dtype=torch.float32, device=DEV)
    ck = torch.zeros((B, Hkv, 8, D), dtype=torch.bfloat16, device=DEV)   # never read: refused first
    length = torch.zeros((B,), dtype=torch.int32, device=DEV)
    cache = cpa.KVCache(ck, ck, length)
    with pytest.raises(cpa.CpaError) as e:
        cpa.chunk_prefill_attn_noalloc(q, kv, kv, tab, tab, cache, P, past_len=length, n_real=length + 1)
    assert e.value.status == 6
