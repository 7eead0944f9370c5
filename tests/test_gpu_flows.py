"""Whole flows from the pages, on the GPU through the C ABI, checked step by step
against the fp64 oracle.

(a) One token stream fed as one full causal pass, as padded chunks, and as
    one-token decode steps gives bit-identical global-cache bytes and outputs
    within tolerance of the oracle ("functiongemma: chunk prefill-with-past
    graph", Validation: one chunk call reproduces the all-positions result;
    "[quanization] Enable prefill-decode modeling": prefill and decode connect).
(b) The sliding-window padded tail ("Pad the chunked-prefill tail for
    sliding-window models", Problem / Fix): a 1023-token prompt as 7 full
    128-row chunks into a 512-row window cache plus a 127-token tail padded to
    128 with snapshot -> attention -> padded append -> rollback; and the tail
    sweep 2..40 after 1 chunk (overshoot) and after 7 chunks (eviction).  Cache
    bytes are bit-exact against the oracle and against the unpadded (scalar)
    tail; attention outputs are within tolerance.
"""
import numpy as np
import pytest
import torch

import oracle as O
from synth import normal_bf16, rope_tables, bf16_bits
from harness import lib, assert_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def tables(pos0, C, D, base=10000.0):
    c, s = rope_tables(np.arange(pos0, pos0 + C)[None, :], D, base)
    return c, s


def padded(x, s, e, C):
    out = torch.zeros(x.shape[:2] + (C,) + x.shape[3:], dtype=x.dtype)
    out[:, :, :e - s] = x[:, :, s:e]
    return out


def test_invariant_a_full_chunked_decode_on_gpu():
    cpa = lib()
    T, Hq, Hkv, D = 300, 8, 2, 128
    q = normal_bf16((1, Hq, T, D), 0, "flow_a/q")
    k = normal_bf16((1, Hkv, T, D), 0, "flow_a/k")
    v = normal_bf16((1, Hkv, T, D), 0, "flow_a/v")
    cap = T + 128
    d = lambda t: t.to(DEV)

    def new_cache():
        z = torch.zeros((1, Hkv, cap, D), dtype=torch.bfloat16, device=DEV)
        return cpa.KVCache(z, z.clone(), torch.zeros(1, dtype=torch.int32, device=DEV))

    # oracle: the full causal pass and its cache
    cos, sin = tables(0, T, D)
    ref, _ = O.chunk_prefill_attn(bf16_bits(q), bf16_bits(k), bf16_bits(v), cos.numpy(), sin.numpy(),
                                  np.zeros((1, Hkv, 0, D), np.uint16), np.zeros((1, Hkv, 0, D), np.uint16),
                                  0, [0], [T], causal=1)
    ok_ = np.zeros((1, Hkv, cap, D), np.uint16); ov_ = ok_.copy(); ol = np.zeros(1, np.int64)
    O.kv_append_global(ok_, ov_, ol, bf16_bits(k), bf16_bits(v), cos.numpy(), sin.numpy(), [T])

    results = {}
    for name, sizes, C in (("full", [T], T), ("chunks", [128, 128, 44], 128), ("chunks64", [64] * 4 + [44], 64)):
        cache = new_cache()
        outs, s = [], 0
        for n in sizes:
            L = int(cache.len[0])
            cs, sn = tables(L, C, D)
            qc, kc, vc = padded(q, s, s + n, C), padded(k, s, s + n, C), padded(v, s, s + n, C)
            nr = torch.tensor([n], dtype=torch.int32, device=DEV)
            out, _ = cpa.chunk_prefill_attn(d(qc), d(kc), d(vc), d(cs), d(sn), cache, L,
                                            past_len=cache.len.clone(), n_real=nr)
            cpa.kv_append(cache, d(kc), d(vc), d(cs), d(sn), nr)
            outs.append(out[:, :, :n])
            s += n
        torch.cuda.synchronize()
        results[name] = (torch.cat(outs, dim=2), cache)
    cache = new_cache()
    outs = []
    for t in range(T):
        cs, sn = tables(t, 1, D)
        one = torch.ones(1, dtype=torch.int32, device=DEV)
        out, _ = cpa.decode_step(d(q[:, :, t:t + 1]), d(k[:, :, t:t + 1]), d(v[:, :, t:t + 1]), d(cs), d(sn),
                                 cache, t, past_len=cache.len.clone(), n_real=one)
        cpa.kv_append(cache, d(k[:, :, t:t + 1]), d(v[:, :, t:t + 1]), d(cs), d(sn), one)
        outs.append(out)
    torch.cuda.synchronize()
    results["decode"] = (torch.cat(outs, dim=2), cache)

    for name, (out, cache) in results.items():
        assert int(cache.len[0]) == T, name
        assert np.array_equal(bf16_bits(cache.k)[:, :, :T], ok_[:, :, :T]), name
        assert np.array_equal(bf16_bits(cache.v)[:, :, :T], ov_[:, :, :T]), name
        assert_close(out, ref, f"flow_a/{name}")


def run_sliding_flow(cpa, prefix, tail, padded_tail=True, Hq=8, D=256, W=512, C=128, c_tail=None):
    """GPU and oracle side by side: `prefix` full chunks, then a tail of `tail`
    tokens (a chunk padded to `c_tail` rows, default C, with snapshot/rollback,
    or scalar decode steps)."""
    c_tail = c_tail or C
    Hkv = 1
    N = prefix * C + tail
    q = normal_bf16((1, Hq, N, D), 0, "flow_b/q")
    k = normal_bf16((1, Hkv, N, D), 0, "flow_b/k")
    v = normal_bf16((1, Hkv, N, D), 0, "flow_b/v")
    d = lambda t: t.to(DEV)
    gk = torch.zeros((1, Hkv, W, D), dtype=torch.bfloat16, device=DEV)
    cache = cpa.KVCache(gk, gk.clone(), torch.zeros(1, dtype=torch.int32, device=DEV), cpa.SLIDING, W, 0)
    scratch = torch.empty(cpa.cache_scratch_size(cache, C), dtype=torch.uint8, device=DEV)
    ok_ = np.zeros((1, Hkv, W, D), np.uint16); ov_ = ok_.copy(); ol = np.zeros(1, np.int64)
    worst = 0.0

    def attend(s, n, Cc, causal=1):
        nonlocal worst
        L = int(ol[0])
        cs, sn = tables(s, Cc, D)
        qc, kc, vc = padded(q, s, s + n, Cc), padded(k, s, s + n, Cc), padded(v, s, s + n, Cc)
        nr = torch.tensor([n], dtype=torch.int32, device=DEV)
        if Cc == 1:
            out, _ = cpa.decode_step(d(qc), d(kc), d(vc), d(cs), d(sn), cache, W, past_len=cache.len.clone(),
                                     n_real=nr, window=W)
        else:
            out, _ = cpa.chunk_prefill_attn(d(qc), d(kc), d(vc), d(cs), d(sn), cache, W,
                                            past_len=cache.len.clone(), n_real=nr, window=W, causal=bool(causal))
        ref, _ = O.chunk_prefill_attn(bf16_bits(qc), bf16_bits(kc), bf16_bits(vc), cs.numpy(), sn.numpy(), ok_, ov_,
                                      W, [L], [n], window=W, causal=causal if Cc > 1 else 0)
        assert_close(out[:, :, :n], ref[:, :, :n], f"flow_b/s{s}")
        return qc, kc, vc, cs, sn, nr

    s = 0
    for _ in range(prefix):
        _, kc, vc, cs, sn, nr = attend(s, C, C)
        cpa.kv_append(cache, d(kc), d(vc), d(cs), d(sn), nr, scratch=scratch)
        O.kv_append_sliding(ok_, ov_, ol, bf16_bits(kc), bf16_bits(vc), cs.numpy(), sn.numpy(), [C], W)
        s += C
    if tail:
        if padded_tail:
            nr = torch.tensor([tail], dtype=torch.int32, device=DEV)
            full = torch.tensor([c_tail], dtype=torch.int32, device=DEV)
            err = cpa.kv_snapshot_padded_append(cache, nr, c_tail, scratch)
            _, kc, vc, cs, sn, _ = attend(s, tail, c_tail)
            cpa.kv_append(cache, d(kc), d(vc), d(cs), d(sn), full, scratch=scratch, err=err)
            cpa.kv_rollback_padded_append(cache, c_tail, scratch, err=err)
            torch.cuda.synchronize()
            assert int(err[0]) == 0
            O.kv_append_sliding(ok_, ov_, ol, bf16_bits(kc), bf16_bits(vc), cs.numpy(), sn.numpy(), [tail], W)
        else:
            for t in range(tail):
                _, kc, vc, cs, sn, nr = attend(s + t, 1, 1)
                cpa.kv_append(cache, d(kc), d(vc), d(cs), d(sn), nr, scratch=scratch)
                O.kv_append_sliding(ok_, ov_, ol, bf16_bits(kc), bf16_bits(vc), cs.numpy(), sn.numpy(), [1], W)
    torch.cuda.synchronize()
    Lf = int(ol[0])
    assert int(cache.len[0]) == Lf == min(N, W)
    assert np.array_equal(bf16_bits(cache.k)[:, :, :Lf], ok_[:, :, :Lf])
    assert np.array_equal(bf16_bits(cache.v)[:, :, :Lf], ov_[:, :, :Lf])
    return bf16_bits(cache.k)[:, :, :Lf], bf16_bits(cache.v)[:, :, :Lf]


def test_sliding_1023_token_prompt_padded_tail_equals_scalar_tail():
    cpa = lib()
    kp, vp = run_sliding_flow(cpa, 7, 127, padded_tail=True)
    ks, vs = run_sliding_flow(cpa, 7, 127, padded_tail=False)
    assert np.array_equal(kp, ks) and np.array_equal(vp, vs)


@pytest.mark.parametrize("prefix", [1, 7])
@pytest.mark.parametrize("tail", [2, 4, 8, 9, 10, 16, 24, 32, 40])
def test_sliding_tail_sweep(prefix, tail):
    cpa = lib()
    run_sliding_flow(cpa, prefix, tail, padded_tail=True, Hq=4, D=128)


@pytest.mark.parametrize("tail", [2, 9, 20, 33, 100])
def test_sliding_tail_padded_to_plan_bucket(tail):
    """The tail chunk size cpa_tail_plan picks from buckets {16, 32, 64, 128}
    ("Pad the chunked-prefill tail for sliding-window models", follow-ups: a
    small tail-chunk variant): the padded tail in that bucket leaves the same
    cache bytes as the oracle's exact append and as the scalar tail."""
    cpa = lib()
    mode, c_pad = cpa.tail_plan(tail, 128, 512, 0, [16, 32, 64, 128], crossover=2)
    assert mode == cpa.TAIL_PADDED and c_pad >= tail and c_pad == max(16, 1 << (tail - 1).bit_length())
    kp, vp = run_sliding_flow(cpa, 7, tail, padded_tail=True, c_tail=c_pad)
    ks, vs = run_sliding_flow(cpa, 7, tail, padded_tail=False)
    assert np.array_equal(kp, ks) and np.array_equal(vp, vs)
