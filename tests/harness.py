"""Shared helpers of the GPU parity tests: run the CUDA path through the C-ABI
binding and the fp64 oracle on the same seeded bytes, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from synth import bf16_bits

MAX_ABS = 1e-2     # attention output tolerance, max |gpu - oracle|
REL_L2 = 3e-3      # attention output tolerance, ||gpu - oracle|| / ||oracle||
ARGMAX_GAP = 2e-2  # oracle top-1 minus top-2 gap above which the argmax must match exactly


def lib():
    import chunked_prefill_attention_rope_gb300 as cpa
    from chunked_prefill_attention_rope_gb300.build import build
    build()
    return cpa


def compare(gpu_bf16: torch.Tensor, ref: np.ndarray, what: str = ""):
    """max-abs and rel-L2 of a bf16 GPU tensor against an fp64 oracle array."""
    g = gpu_bf16.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    d = np.abs(g - ref)
    max_abs = float(d.max()) if d.size else 0.0
    den = float(np.sqrt(np.sum(ref ** 2)))
    rel = float(np.sqrt(np.sum(d ** 2)) / den) if den > 0 else max_abs
    return max_abs, rel


def assert_close(gpu_bf16, ref, what=""):
    max_abs, rel = compare(gpu_bf16, ref, what)
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    return max_abs, rel


def assert_explicit_matches(out_e, out_i, what=""):
    """Outputs of the explicit and the implicit form of one 0 / -1e30 mask:
    bitwise identical on every path.  Both forms visit the same key tiles in
    the same order with the same work split, and each tile's scores meet the
    same arithmetic: a 0 entry leaves the score as it is and a masked entry
    gives -inf, exactly as the implicit predicate does."""
    assert torch.equal(out_e.view(torch.int16), out_i.view(torch.int16)), f"{what}: explicit != implicit"


def check_argmax(gpu_sel: torch.Tensor, ref_sel: np.ndarray, what=""):
    """Selected-row argmax: exact when the oracle's top-2 gap exceeds ARGMAX_GAP;
    otherwise the GPU's pick must be one of the near-tied oracle maxima."""
    g = gpu_sel.detach().float().cpu().numpy()
    r32 = ref_sel.astype(np.float32)
    for b in range(r32.shape[0]):
        gi = int(O.select_argmax(g[b]))
        ri = int(O.select_argmax(r32[b]))
        top2 = np.sort(r32[b])[-2:]
        gap = float(top2[1] - top2[0])
        if gap > ARGMAX_GAP:
            assert gi == ri, f"{what}: argmax {gi} != oracle {ri} (gap {gap:.3e})"
        else:
            assert r32[b, ri] - r32[b, gi] <= ARGMAX_GAP, f"{what}: argmax {gi} not near-tied with {ri}"


def cache_bytes(t: torch.Tensor) -> np.ndarray:
    return bf16_bits(t)


def bits16(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns (bf16 or fp16 tensors) as a uint16 numpy array."""
    assert t.dtype in (torch.bfloat16, torch.float16)
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_attn(q, k_new, v_new, cos, sin, ck, cv, P, past_len, n_real, window=0, causal=1,
                mask=None, sel_row=None, sink=0):
    """Run the oracle on host copies of torch tensors (the cache format follows
    the cache tensors' dtype)."""
    f = lambda t: None if t is None else t.detach().cpu()
    L = f(past_len).numpy() if past_len is not None else None
    n = f(n_real).numpy() if n_real is not None else None
    m = None if mask is None else f(mask).numpy()
    s = None if sel_row is None else f(sel_row).numpy()
    kv = "f16" if ck.dtype == torch.float16 else "bf16"
    return O.chunk_prefill_attn(bf16_bits(q), bf16_bits(k_new), bf16_bits(v_new), f(cos).numpy(),
                                f(sin).numpy(), bits16(ck), bits16(cv), P, L, n,
                                window=window, causal=causal, mask=m, sel_row=s, sink=sink, kv=kv)


def explicit_masks(past_len, n_real, C, P, Hq, window, causal, sink=0):
    """[B, Hq, C, P+C] fp32 additive masks built by the oracle's mask function."""
    B = len(past_len)
    out = np.zeros((B, Hq, C, P + C), dtype=np.float32)
    for b in range(B):
        out[b] = O.explicit_mask(int(past_len[b]), int(n_real[b]), C, P, window, causal, sink)[None]
    return torch.from_numpy(out)


def sample_rows(C, R, n, salt=0):
    """Chunk rows to check in one (sequence, kv head) group: the first, one
    inner and the last row of every R-row query tile, plus the last real row."""
    rows = set()
    for t0 in range(0, C, R):
        hi = min(t0 + R, C)
        rows.update((t0, t0 + (7 * (t0 // R) + 5 + salt) % (hi - t0), hi - 1))
    if n > 0:
        rows.add(n - 1)
    return sorted(rows)


def oracle_rows(q, k_new, v_new, cos, sin, ck, cv, L, n, rows, window=0, causal=1):
    """fp64 outputs of chunk rows `rows` of one (sequence, kv head) group,
    composed from the oracle's own steps: RoPE of the sampled query rows and of
    every chunk key, the implicit mask's rows, and softmax attention.  Inputs
    are host tensors of one group: q [G, C, D], k_new/v_new [C, D], cos/sin
    [C, D], cache rows ck/cv [L, D] (the L valid past slots; slots past L are
    masked and never read).  Returns [G, len(rows), D]."""
    G, C, D = q.shape
    rows = np.asarray(rows)
    c = cos.numpy()
    s = sin.numpy()
    k_rot = O.bf16_to_f32(O.rope_rotate(bf16_bits(k_new), c, s)).astype(np.float64)
    keys = np.concatenate([O.bf16_to_f32(bf16_bits(ck)).astype(np.float64), k_rot], axis=0)
    vals = np.concatenate([O.bf16_to_f32(bf16_bits(cv)).astype(np.float64),
                           O.bf16_to_f32(bf16_bits(v_new)).astype(np.float64)], axis=0)
    m = O.explicit_mask(L, n, C, L, window, causal)[rows]
    out = np.zeros((G, len(rows), D))
    for g in range(G):
        qr = O.bf16_to_f32(O.rope_rotate(bf16_bits(q[g, rows]), c[rows], s[rows])).astype(np.float64)
        out[g] = O.attend(qr, keys, vals, m, 1.0 / np.sqrt(D))
    return out
