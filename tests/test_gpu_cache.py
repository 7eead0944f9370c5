"""GPU parity of the cache operations against the oracle: bit-exact bytes.

Global append with fused RoPE ("[quanization] Enable prefill-decode modeling",
Runtime behavior: the runtime writes each step's K/V into external cache
buffers); sliding append, snapshot and rollback ("Pad the chunked-prefill tail
for sliding-window models", Fix: padded append + rollback leaves the cache
byte-identical to an unpadded prefill, including eviction, overshoot and sink
cases).
"""
import numpy as np
import pytest
import torch

import oracle as O
from synth import normal_bf16, rope_tables, bf16_bits, uniform_int
from harness import lib, cache_bytes

pytestmark = pytest.mark.gpu
DEV = "cuda"


def chunk(B, Hkv, C, D, tag, pos0):
    k = normal_bf16((B, Hkv, C, D), 0, tag + "/k")
    v = normal_bf16((B, Hkv, C, D), 0, tag + "/v")
    pos = np.asarray(pos0)[:, None] + np.arange(C)[None, :]
    cos, sin = rope_tables(pos, D, 10000.0)
    return k, v, cos, sin


@pytest.mark.parametrize("D,Hkv", [(64, 1), (128, 8), (256, 2)])
def test_global_append_bit_exact(D, Hkv):
    cpa = lib()
    B, C, cap = 9, 24, 80
    L0 = uniform_int(0, cap - C, B, 0, f"ga/{D}/L").numpy()
    n = uniform_int(0, C, B, 0, f"ga/{D}/n").numpy()
    L0[3] = cap - 5          # this one overflows when n[3] > 5
    n[3] = 11
    ck = normal_bf16((B, Hkv, cap, D), 0, f"ga/{D}/ck")
    cv = normal_bf16((B, Hkv, cap, D), 0, f"ga/{D}/cv")
    k, v, cos, sin = chunk(B, Hkv, C, D, f"ga/{D}", L0)
    # oracle
    ok_, ov_ = cache_bytes(ck).copy(), cache_bytes(cv).copy()
    olen = L0.astype(np.int64).copy()
    over = O.kv_append_global(ok_, ov_, olen, bf16_bits(k), bf16_bits(v), cos.numpy(), sin.numpy(), n)
    assert over == [3]
    # GPU
    gk, gv = ck.to(DEV), cv.to(DEV)
    glen = torch.from_numpy(L0.astype(np.int32)).to(DEV)
    cache = cpa.KVCache(gk, gv, glen)
    err = cpa.kv_append(cache, k.to(DEV), v.to(DEV), cos.to(DEV), sin.to(DEV),
                        torch.from_numpy(n.astype(np.int32)).to(DEV))
    torch.cuda.synchronize()
    assert int(err[0]) == cpa.EBIT["CAPACITY"]
    assert np.array_equal(glen.cpu().numpy(), olen)
    assert np.array_equal(cache_bytes(gk), ok_) and np.array_equal(cache_bytes(gv), ov_)


def test_global_append_strided_cache_view():
    """A cache that is a view into a larger buffer (stride_s > D, stride_h padded)."""
    cpa = lib()
    B, Hkv, D, C, cap = 3, 2, 128, 16, 40
    big_k = normal_bf16((B, Hkv + 1, cap, D + 64), 0, "gs/bk").to(DEV)
    big_v = normal_bf16((B, Hkv + 1, cap, D + 64), 0, "gs/bv").to(DEV)
    gk, gv = big_k[:, :Hkv, :, :D], big_v[:, :Hkv, :, :D]
    L0 = np.array([0, 7, 24])
    n = np.array([16, 3, 16])
    k, v, cos, sin = chunk(B, Hkv, C, D, "gs", L0)
    ok_ = cache_bytes(gk.contiguous()).copy(); ov_ = cache_bytes(gv.contiguous()).copy()
    olen = L0.copy()
    O.kv_append_global(ok_, ov_, olen, bf16_bits(k), bf16_bits(v), cos.numpy(), sin.numpy(), n)
    before_pad = cache_bytes(big_k[:, :, :, D:].contiguous())
    glen = torch.from_numpy(L0.astype(np.int32)).to(DEV)
    cpa.kv_append(cpa.KVCache(gk, gv, glen), k.to(DEV), v.to(DEV), cos.to(DEV), sin.to(DEV),
                  torch.from_numpy(n.astype(np.int32)).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(cache_bytes(gk.contiguous()), ok_)
    assert np.array_equal(cache_bytes(gv.contiguous()), ov_)
    assert np.array_equal(cache_bytes(big_k[:, :, :, D:].contiguous()), before_pad)
    assert np.array_equal(glen.cpu().numpy(), olen)


@pytest.mark.parametrize("S", [0, 2])
@pytest.mark.parametrize("D", [64, 256])
def test_sliding_padded_append_rollback_sweep(S, D):
    """Every (len0, n) pair at once, one sequence each: padded append + rollback
    must equal the exact append byte for byte, and both must equal the oracle."""
    cpa = lib()
    W, C, Hkv = 24, 8, 2
    cases = [(L0, n) for L0 in range(W + 1) for n in range(C + 1)]
    B = len(cases)
    L0 = np.array([c[0] for c in cases]); n = np.array([c[1] for c in cases])
    ck = normal_bf16((B, Hkv, W, D), 0, f"sl/{S}/{D}/ck")
    cv = normal_bf16((B, Hkv, W, D), 0, f"sl/{S}/{D}/cv")
    k, v, cos, sin = chunk(B, Hkv, C, D, f"sl/{S}/{D}", L0)
    pad = torch.arange(C)[None, :] >= torch.from_numpy(n)[:, None]
    k.masked_fill_(pad[:, None, :, None], 0); v.masked_fill_(pad[:, None, :, None], 0)
    # oracle exact append
    ek, ev = cache_bytes(ck).copy(), cache_bytes(cv).copy()
    elen = L0.copy()
    assert O.kv_append_sliding(ek, ev, elen, bf16_bits(k), bf16_bits(v), cos.numpy(), sin.numpy(), n, W, S) == []
    dev = lambda t: t.to(DEV)
    n_d = torch.from_numpy(n.astype(np.int32)).to(DEV)
    full_d = torch.full((B,), C, dtype=torch.int32, device=DEV)
    # GPU exact append
    xk, xv = dev(ck), dev(cv)
    xlen = torch.from_numpy(L0.astype(np.int32)).to(DEV)
    xc = cpa.KVCache(xk, xv, xlen, cpa.SLIDING, W, S)
    scratch = torch.empty(cpa.cache_scratch_size(xc, C), dtype=torch.uint8, device=DEV)
    err = cpa.kv_append(xc, dev(k), dev(v), dev(cos), dev(sin), n_d, scratch=scratch)
    # GPU padded append + rollback
    pk, pv = dev(ck), dev(cv)
    plen = torch.from_numpy(L0.astype(np.int32)).to(DEV)
    pc = cpa.KVCache(pk, pv, plen, cpa.SLIDING, W, S)
    scratch2 = torch.empty(cpa.cache_scratch_size(pc, C), dtype=torch.uint8, device=DEV)
    cpa.kv_snapshot_padded_append(pc, n_d, C, scratch2, err=err)
    cpa.kv_append(pc, dev(k), dev(v), dev(cos), dev(sin), full_d, scratch=scratch2, err=err)
    cpa.kv_rollback_padded_append(pc, C, scratch2, err=err)
    torch.cuda.synchronize()
    assert int(err[0]) == 0
    assert np.array_equal(xlen.cpu().numpy(), elen) and np.array_equal(plen.cpu().numpy(), elen)
    gx, gxv, gp, gpv = cache_bytes(xk), cache_bytes(xv), cache_bytes(pk), cache_bytes(pv)
    for b in range(B):
        Lf = int(elen[b])
        assert np.array_equal(gx[b, :, :Lf], ek[b, :, :Lf]), ("exact", cases[b])
        assert np.array_equal(gxv[b, :, :Lf], ev[b, :, :Lf]), ("exact v", cases[b])
        assert np.array_equal(gp[b, :, :Lf], ek[b, :, :Lf]), ("padded", cases[b])
        assert np.array_equal(gpv[b, :, :Lf], ev[b, :, :Lf]), ("padded v", cases[b])


def test_sliding_guards_and_errors():
    cpa = lib()
    W, C, Hkv, D = 16, 8, 1, 64
    ck = torch.zeros((2, Hkv, W, D), dtype=torch.bfloat16, device=DEV)
    cv = torch.zeros_like(ck)
    length = torch.tensor([3, 16], dtype=torch.int32, device=DEV)
    c = cpa.KVCache(ck, cv, length, cpa.SLIDING, W, 8)  # W <= C + S
    scratch = torch.empty(cpa.cache_scratch_size(c, C), dtype=torch.uint8, device=DEV)
    with pytest.raises(cpa.CpaError) as e:
        cpa.kv_snapshot_padded_append(c, torch.tensor([1, 1], dtype=torch.int32, device=DEV), C, scratch)
    assert e.value.status == 5
    # rollback without a snapshot: flagged, cache untouched
    c2 = cpa.KVCache(ck, cv, length, cpa.SLIDING, W, 0)
    scratch.zero_()
    err = cpa.kv_rollback_padded_append(c2, C, scratch)
    torch.cuda.synchronize()
    assert int(err[0]) & cpa.EBIT["SNAPSHOT"]
    assert length.cpu().tolist() == [3, 16]
