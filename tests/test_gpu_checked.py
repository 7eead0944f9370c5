"""The checked build of the library (libcpa_checked.so) on the GPU.

compute-sanitizer is not available, so the library is also built with
CPA_BOUNDS_CHECK: every global index the kernels compute is range-checked and
an index outside its buffer sets CPA_EBIT_BOUNDS (the access is skipped, never
made).  The drawn sweep shapes (every attention path, both mask forms, fp16
caches, the fused append) and the sliding-window append, snapshot and rollback
run through it here: the error word must stay 0 and every output and cache
byte must equal the regular library's, so the checks neither fire nor change
a result.

The same build carries CPA_TEST_HOOKS: its pipeline waits give up after 20 ms,
and cpa_test_drop_tile() makes the two-tile kernel's producer withhold one
K/V tile copy.  The consumer's bounded wait must then run out, the call must
report CPA_EBIT_TIMEOUT, and the next call must run normally on the same
context (failure detection without a GPU fault).
"""
import pytest
import torch

from synth import Workload, make_chunk_inputs, make_cache
from harness import lib, explicit_masks, bits16
from test_gpu_sweep import CASES

pytestmark = pytest.mark.gpu
DEV = "cuda"


def attn(cpa, w, inp, ck, cv, mask=None, fused=False, err=None):
    d = lambda t: None if t is None else t.to(DEV)
    cache = cpa.KVCache(d(ck), d(cv), d(inp["past_len"]).clone())
    err = cpa.new_error_word() if err is None else err
    kw = dict(past_len=d(inp["past_len"]), n_real=d(inp["n_real"]), window=w.window, causal=bool(w.causal),
              mask=d(mask), sel_row=d((inp["n_real"] - 1).clamp(min=0)), want_sel=True, err=err)
    if fused:
        out, sel = cpa.chunk_prefill_attn_append(d(inp["q"]), d(inp["k"]), d(inp["v"]), d(inp["cos"]),
                                                 d(inp["sin"]), cache, w.P, d(inp["n_real"]), **kw)
    else:
        out, sel = cpa.chunk_prefill_attn(d(inp["q"]), d(inp["k"]), d(inp["v"]), d(inp["cos"]), d(inp["sin"]),
                                          cache, w.P, **kw)
    torch.cuda.synchronize()
    return out, sel, cache, int(err[0])


def both(cpa, fn):
    """fn() through the checked build, then through the library."""
    with cpa.using_library("checked"):
        checked = fn()
    return checked, fn()


def same(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


@pytest.mark.parametrize("w", CASES[::2], ids=lambda w: w.name)
def test_checked_build_sweep(w):
    cpa = lib()
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    mask = explicit_masks(inp["past_len"].numpy(), inp["n_real"].numpy(), w.C, w.P, w.Hq, w.window, w.causal)
    for m in (None, mask):
        (o1, s1, _, e1), (o2, s2, _, e2) = both(cpa, lambda: attn(cpa, w, inp, ck, cv, mask=m))
        assert e1 == 0 and e2 == 0, (w.name, e1)
        assert same(o1, o2) and same(s1, s2), w.name
    ck16, cv16 = ck.to(torch.float16), cv.to(torch.float16)
    (o1, _, _, e1), (o2, _, _, e2) = both(cpa, lambda: attn(cpa, w, inp, ck16, cv16))
    assert e1 == 0 and same(o1, o2), w.name + "/f16"
    if w.C > 1:
        (o1, _, c1, e1), (o2, _, c2, e2) = both(cpa, lambda: attn(cpa, w, inp, ck, cv, fused=True))
        assert e1 == 0 and e2 == 0 and same(o1, o2), w.name + "/fused"
        assert same(c1.k, c2.k) and same(c1.v, c2.v) and torch.equal(c1.len, c2.len), w.name + "/fused cache"


@pytest.mark.parametrize("S,len0,n", [(0, 20, 5), (2, 24, 8), (2, 23, 3), (0, 7, 8)])
def test_checked_build_sliding_flows(S, len0, n):
    """Sliding append with compaction, and snapshot -> padded append ->
    rollback, on a window of 24 rows (the eviction, overshoot and sink cases)."""
    cpa = lib()
    B, Hkv, D, C, W = 2, 2, 64, 8, 24
    w = Workload("chk_slide", B=B, Hq=Hkv, Hkv=Hkv, D=D, C=C, P=W, cap=W, past=("fixed", len0),
                 n_real=("fixed", n))
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)

    def flow():
        cache = cpa.KVCache(ck.to(DEV), cv.to(DEV), torch.full((B,), len0, dtype=torch.int32, device=DEV),
                            cpa.SLIDING, W, S)
        err = cpa.new_error_word()
        scratch = torch.empty(cpa.cache_scratch_size(cache, C), dtype=torch.uint8, device=DEV)
        d = {k: v.to(DEV) for k, v in inp.items()}
        cpa.kv_snapshot_padded_append(cache, d["n_real"], C, scratch, err=err)
        cpa.kv_append(cache, d["k"], d["v"], d["cos"], d["sin"], torch.full((B,), C, dtype=torch.int32,
                                                                             device=DEV), scratch=scratch, err=err)
        cpa.kv_rollback_padded_append(cache, C, scratch, err=err)
        cpa.kv_append(cache, d["k"], d["v"], d["cos"], d["sin"], d["n_real"], scratch=scratch, err=err)
        torch.cuda.synchronize()
        return cache, int(err[0])

    (c1, e1), (c2, e2) = both(cpa, flow)
    assert e1 == 0 and e2 == 0
    assert torch.equal(c1.len, c2.len)
    for b in range(B):
        L = int(c1.len[b])
        assert (bits16(c1.k[b, :, :L]) == bits16(c2.k[b, :, :L])).all()
        assert (bits16(c1.v[b, :, :L]) == bits16(c2.v[b, :, :L])).all()


def test_bounded_wait_runs_out_and_the_context_recovers():
    """The two-tile kernel's producer withholds every CTA's first K/V tile:
    the consumer's wait runs out after 20 ms, the call sets CPA_EBIT_TIMEOUT
    and returns; the next call on the same context is exact again."""
    cpa = lib()
    w = Workload("chk_timeout", B=2, Hq=8, Hkv=2, D=128, C=64, P=200, cap=264, past=("uniform", 0, 200),
                 n_real=("uniform", 1, 64))
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    with cpa.using_library("checked") as so:
        so.cpa_test_drop_tile(0)
        try:
            _, _, _, e = attn(cpa, w, inp, ck, cv)
        finally:
            so.cpa_test_drop_tile(-1)
        assert e & cpa.EBIT["TIMEOUT"], e
        assert not e & cpa.EBIT["BOUNDS"], e
        o1, s1, _, e1 = attn(cpa, w, inp, ck, cv)
    o2, s2, _, e2 = attn(cpa, w, inp, ck, cv)
    assert e1 == 0 and e2 == 0
    assert same(o1, o2) and same(s1, s2)
