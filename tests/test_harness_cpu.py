"""The GPU tests' row-sampled oracle (harness.oracle_rows) against the oracle's
whole-chunk function, on the CPU: the sampled rows of one (sequence, kv head)
group must equal the corresponding rows of oracle.chunk_prefill_attn exactly,
for causal, windowed and non-causal masks, an empty past and pad rows."""
import numpy as np
import pytest
import torch

import oracle as O
from synth import Workload, make_chunk_inputs, make_cache, bf16_bits
from harness import sample_rows, oracle_rows


@pytest.mark.parametrize("L,n,window,causal", [(37, 20, 0, 1), (0, 24, 0, 1), (50, 13, 9, 1), (40, 24, 11, 0)])
def test_oracle_rows_equal_chunk_prefill_rows(L, n, window, causal):
    w = Workload("harness_rows", B=1, Hq=8, Hkv=2, D=32, C=24, P=64, cap=88, past=("fixed", L),
                 n_real=("fixed", n), window=window, causal=causal)
    inp = make_chunk_inputs(w)
    ck, cv = make_cache(w)
    full, _ = O.chunk_prefill_attn(bf16_bits(inp["q"]), bf16_bits(inp["k"]), bf16_bits(inp["v"]),
                                   inp["cos"].numpy(), inp["sin"].numpy(), bf16_bits(ck), bf16_bits(cv), w.P,
                                   [L], [n], window=window, causal=causal)
    G = w.Hq // w.Hkv
    rows = sample_rows(w.C, 128 // G, n)
    assert rows[0] == 0 and rows[-1] == w.C - 1 and (n == 0 or n - 1 in rows)
    for kvh in range(w.Hkv):
        hs = slice(kvh * G, (kvh + 1) * G)
        got = oracle_rows(inp["q"][0, hs], inp["k"][0, kvh], inp["v"][0, kvh], inp["cos"][0], inp["sin"][0],
                          ck[0, kvh, :L], cv[0, kvh, :L], L, n, rows, window, causal)
        assert np.array_equal(got, full[0, hs][:, rows])


def test_sample_rows_cover_every_query_tile():
    rows = sample_rows(512, 32, 500)
    tiles = {r // 32 for r in rows}
    assert tiles == set(range(16))
    assert 499 in rows and all(0 <= r < 512 for r in rows)
