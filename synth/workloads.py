"""Seeded synthetic workloads for chunked prefill attention with past.

Every tensor is drawn from its own torch generator, seeded from (seed, tag), so
any tensor can be regenerated alone.  bf16 data is N(0,1) drawn in fp32 and
rounded to bf16 by torch.  The cos/sin tables are the per-position inputs that
the caller supplies to the attention step ("RoPE from per-position [C, headDim]
cos/sin tables", functiongemma chunk prefill-with-past graph, Change section;
"position_embeddings = (cos_t, sin_t)", TICO prefill-decode modeling, Runtime
behavior): angle = pos * base^(-2k/D) in fp64, cos/sin in fp64, stored as fp32,
both halves of a row holding the same frequencies.

Nothing in this module rotates, masks, attends or edits a cache.
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Optional

import numpy as np
import torch

__all__ = [
    "tag_seed", "normal_bf16", "uniform_int", "rope_tables", "bf16_bits",
    "Workload", "WORKLOADS", "make_chunk_inputs", "make_cache",
]


def tag_seed(seed: int, tag: str) -> int:
    """A 63-bit generator seed derived from a workload seed and a tensor tag."""
    h = zlib.crc32(f"{seed}/{tag}".encode()) ^ (zlib.adler32(tag.encode()) << 32)
    return (h ^ (seed * 0x9E3779B97F4A7C15)) & 0x7FFFFFFFFFFFFFFF


def normal_bf16(shape, seed: int, tag: str, device="cpu") -> torch.Tensor:
    """N(0,1) values drawn in fp32 and rounded to bf16."""
    g = torch.Generator(device=device)
    g.manual_seed(tag_seed(seed, tag))
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)


def uniform_int(lo: int, hi: int, n: int, seed: int, tag: str) -> torch.Tensor:
    """n integers uniform on [lo, hi] (both ends included), int32, on the CPU."""
    g = torch.Generator(device="cpu")
    g.manual_seed(tag_seed(seed, tag))
    return torch.randint(lo, hi + 1, (n,), generator=g, dtype=torch.int64).to(torch.int32)


def rope_tables(positions, D: int, base: float):
    """cos, sin tables [*positions.shape, D] as fp32 (computed in fp64)."""
    pos = np.asarray(positions, dtype=np.float64)
    k = np.arange(D // 2, dtype=np.float64)
    inv_freq = base ** (-(2.0 * k) / D)
    ang = pos[..., None] * inv_freq
    ang = np.concatenate([ang, ang], axis=-1)
    return (torch.from_numpy(np.cos(ang).astype(np.float32)),
            torch.from_numpy(np.sin(ang).astype(np.float32)))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw bf16 bit patterns of a tensor as a uint16 numpy array (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and draw recipe of one attention workload."""
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    C: int                      # chunk rows, pads included
    P: int                      # past span: cache slot columns the step may see
    cap: int                    # cache capacity in rows
    past: tuple                 # ("fixed", L) or ("uniform", lo, hi)
    n_real: tuple               # ("fixed", n) or ("uniform", lo, hi)
    window: int = 0
    causal: int = 1
    base: float = 10000.0
    seed: int = 0
    kind: str = "global"        # "global" or "sliding"
    sink: int = 0
    layers: int = 1
    note: str = ""

    def past_lens(self) -> torch.Tensor:
        if self.past[0] == "fixed":
            return torch.full((self.B,), self.past[1], dtype=torch.int32)
        return uniform_int(self.past[1], self.past[2], self.B, self.seed, self.name + "/past_len")

    def n_reals(self) -> torch.Tensor:
        if self.n_real[0] == "fixed":
            return torch.full((self.B,), self.n_real[1], dtype=torch.int32)
        return uniform_int(self.n_real[1], self.n_real[2], self.B, self.seed, self.name + "/n_real")


WORKLOADS = {
    # B=1, 4 q / 1 kv heads, D=64, 48 cached rows, a 16-row chunk with 12 real rows.
    "tiny": Workload("tiny", B=1, Hq=4, Hkv=1, D=64, C=16, P=48, cap=64,
                     past=("fixed", 48), n_real=("fixed", 12)),
    # The page-1 call shape: 800 cached positions and a 64-row chunk with 52 real
    # rows, 18 layers alternating a 512-position window (base 1e4) and global
    # attention (base 1e6), explicit per-head masks [1, 4, 64, 864].
    "page1": Workload("page1", B=1, Hq=4, Hkv=1, D=256, C=64, P=800, cap=864,
                      past=("fixed", 800), n_real=("fixed", 52), layers=18),
    # Sliding-window cache (512 rows) fed in 128-row chunks; 1023-token prompt.
    "sliding_tail": Workload("sliding_tail", B=1, Hq=8, Hkv=1, D=256, C=128, P=512,
                             cap=512, past=("fixed", 512), n_real=("fixed", 127),
                             window=512, kind="sliding"),
    # Packed static cache batch: 16 sequences, past uniform on [0, 4095].
    "packed_batch": Workload("packed_batch", B=16, Hq=32, Hkv=8, D=128, C=128, P=4096,
                             cap=4224, past=("uniform", 0, 4095), n_real=("fixed", 128)),
    # Long context: 4 sequences with 32768 cached rows, a 512-row chunk.
    "long_ctx": Workload("long_ctx", B=4, Hq=32, Hkv=8, D=128, C=512, P=32768,
                         cap=33280, past=("fixed", 32768), n_real=("fixed", 512)),
    # One-token decode for 64 sequences, past uniform on [1024, 32768].
    "decode": Workload("decode", B=64, Hq=32, Hkv=8, D=128, C=1, P=32768, cap=32769,
                       past=("uniform", 1024, 32768), n_real=("fixed", 1)),
}


def make_chunk_inputs(w: Workload, layer: int = 0, device="cpu",
                      past_len: Optional[torch.Tensor] = None,
                      n_real: Optional[torch.Tensor] = None,
                      base: Optional[float] = None, pos0: Optional[torch.Tensor] = None):
    """Q [B,Hq,C,D], K/V chunk [B,Hkv,C,D] (bf16, pad rows zero), cos/sin [B,C,D] fp32.

    Row i of sequence b sits at absolute position pos0[b] + i (pos0 defaults to
    past_len).  Pad rows (i >= n_real[b]) of Q, K and V are zero.
    """
    L = w.past_lens() if past_len is None else past_len.to(torch.int32).cpu()
    n = w.n_reals() if n_real is None else n_real.to(torch.int32).cpu()
    p0 = L if pos0 is None else pos0.to(torch.int32).cpu()
    tag = f"{w.name}/L{layer}"
    q = normal_bf16((w.B, w.Hq, w.C, w.D), w.seed, tag + "/q", device)
    k = normal_bf16((w.B, w.Hkv, w.C, w.D), w.seed, tag + "/k", device)
    v = normal_bf16((w.B, w.Hkv, w.C, w.D), w.seed, tag + "/v", device)
    rows = torch.arange(w.C, device=device)
    pad = rows[None, :] >= n.to(device)[:, None]          # [B, C]
    for t in (q, k, v):
        t.masked_fill_(pad[:, None, :, None], 0)
    positions = p0.numpy().astype(np.int64)[:, None] + np.arange(w.C)[None, :]
    cos, sin = rope_tables(positions, w.D, w.base if base is None else base)
    return dict(q=q, k=k, v=v, cos=cos.to(device), sin=sin.to(device),
                past_len=L.to(device), n_real=n.to(device))


def make_cache(w: Workload, layer: int = 0, device="cpu", fill_rows: Optional[int] = None):
    """Cache K/V [B,Hkv,cap,D] bf16, every row N(0,1) (dead rows included)."""
    tag = f"{w.name}/L{layer}"
    rows = w.cap if fill_rows is None else fill_rows
    k = normal_bf16((w.B, w.Hkv, rows, w.D), w.seed, tag + "/cache_k", device)
    v = normal_bf16((w.B, w.Hkv, rows, w.D), w.seed, tag + "/cache_v", device)
    return k, v
