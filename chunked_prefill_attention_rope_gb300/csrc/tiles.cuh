// Key-tile bookkeeping shared by the attention kernels.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace cpa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMaskedLog2 = -1e30f * kLog2e;  // the masked score, in log2 units
constexpr float kEmptyRow = -1e28f;              // running max below this: no visible key yet

// Key tiles live in one index space known on the host: tiles [0, Tc) are chunk
// tiles (chunk rows [t*BN, t*BN + BN)), tiles [Tc, Tc + Tp) are past tiles
// (slots [(t-Tc)*BN, ...)).  Split s owns the fixed index range
// [s*T/S, (s+1)*T/S) and visits the live tiles inside it.  The implicit mask
// makes the live set two intervals (with sink slots, the past interval starts
// at slot 0 and the tiles between the sinks and the window are visited,
// fully masked); with an explicit mask every tile is live.
// Because the ranges do not depend on the mask, the explicit and implicit
// descriptions of one mask split the keys identically; the extra tiles the
// explicit path visits are fully masked and contribute exactly zero.
struct TilePlan {
  int L, n;       // clamped past length and real rows of this sequence
  int Tc;         // chunk tiles in the index space
  int cb, ce;     // chunk tiles visited: index range [cb, ce)
  int pb, pe;     // past tiles visited: index range [pb, pe)
  __device__ __forceinline__ int count() const { return (ce - cb) + (pe - pb); }
  __device__ __forceinline__ int index(int q) const { return q < ce - cb ? cb + q : pb + (q - (ce - cb)); }
};

// Live key tiles for query rows [i_min, i_max] of sequence b, restricted to the
// tile index range [r0, r1).
template <int BN>
__device__ __forceinline__ TilePlan plan_tiles_range(const AttnParams& p, int b, int i_min, int i_max, long long r0,
                                                     long long r1) {
  TilePlan t;
  int L = p.past_len ? p.past_len[b] : p.P;
  int n = p.n_real ? p.n_real[b] : p.C;
  t.L = min(max(L, 0), p.P);
  t.n = min(max(n, 0), p.C);
  t.Tc = (p.C + BN - 1) / BN;
  const int Tp = (p.P + BN - 1) / BN;
  int c0 = 0, c1 = t.Tc, q0 = 0, q1 = Tp;
  if (!p.mask) {
    const int W = p.window;
    const int t_lo = W > 0 ? max(0, i_min - W + 1) : 0;
    const int t_hi = p.causal ? min(t.n, i_max + 1) : (W > 0 ? min(t.n, i_max + W) : t.n);
    const int j_lo = (W > 0 && p.sink <= 0) ? max(0, t.L + i_min - W + 1) : 0;
    const int j_hi = t.L;
    c0 = t_lo / BN;
    c1 = t_hi > t_lo ? (t_hi + BN - 1) / BN : c0;
    q0 = j_lo / BN;
    q1 = j_hi > j_lo ? (j_hi + BN - 1) / BN : q0;
  }
  const int lo = static_cast<int>(r0 < 0 ? 0 : r0);
  const int hi = static_cast<int>(r1 > (1LL << 30) ? (1LL << 30) : r1);
  t.cb = max(c0, lo);
  t.ce = max(t.cb, min(c1, hi));
  t.pb = max(t.Tc + q0, lo);
  t.pe = max(t.pb, min(t.Tc + q1, hi));
  return t;
}

// Live key tiles of split `split` (of p.splits): split s owns [s*T/S, (s+1)*T/S).
template <int BN>
__device__ __forceinline__ TilePlan plan_tiles(const AttnParams& p, int b, int i_min, int i_max, int split) {
  const long long T = (p.C + BN - 1) / BN + (p.P + BN - 1) / BN;
  return plan_tiles_range<BN>(p, b, i_min, i_max, T * split / p.splits, T * (split + 1) / p.splits);
}

// All live key tiles of query rows [i_min, i_max] of sequence b.
template <int BN>
__device__ __forceinline__ TilePlan plan_whole(const AttnParams& p, int b, int i_min, int i_max) {
  return plan_tiles_range<BN>(p, b, i_min, i_max, 0, 1LL << 30);
}

// Bits [a, b) of a 32-bit word (a and b clipped to [0, 32]).
__device__ __forceinline__ uint32_t bit_range(int a, int b) {
  a = min(max(a, 0), 32);
  b = min(max(b, 0), 32);
  const uint32_t below_b = b >= 32 ? 0xffffffffu : ((1u << b) - 1u);
  const uint32_t below_a = a >= 32 ? 0xffffffffu : ((1u << a) - 1u);
  return below_b & ~below_a;
}

// Visible key interval of query row i, relative to a tile's first key
// (implicit mask): keys e with lo <= e < hi are visible.
struct RowSpan {
  int past_lo, ch_lo, ch_hi, L, sinkL;
  __device__ __forceinline__ void init(const AttnParams& p, const TilePlan& tp, int i, bool valid) {
    const int W = p.window;
    L = valid ? tp.L : 0;
    past_lo = W > 0 ? max(0, tp.L + i - W + 1) : 0;
    ch_lo = W > 0 ? max(0, i - W + 1) : 0;
    ch_hi = !valid ? 0 : (p.causal ? min(tp.n, i + 1) : (W > 0 ? min(tp.n, i + W) : tp.n));
    sinkL = min(p.sink, L);
  }
  // Keys e of the tile with lo <= e < hi, or e < sk (pinned sink slots), are visible.
  __device__ __forceinline__ void tile(bool chunk, int base, int& lo, int& hi, int& sk) const {
    lo = (chunk ? ch_lo : past_lo) - base;
    hi = (chunk ? ch_hi : L) - base;
    sk = chunk ? 0 : sinkL - base;
  }
};

// Rows of key tile [base, base + BN) that the implicit mask never shows to any
// query row but that the tile copy fills from memory: cache slots in [L, P)
// (dead rows: nothing promises their bytes) and chunk pad rows in [n, C).
// Rows at or past P (or C) arrive as zeros from the copy.  Returns [z0, z1)
// relative to the tile (empty when z0 >= z1).  P is exactly zero for these
// keys, but 0 times a non-finite value is not zero, so the kernels clear
// these rows of the V tile before the P V product.
template <int BN>
__device__ __forceinline__ void dead_rows(const AttnParams& p, const TilePlan& tp, bool chunk, int base, int& z0,
                                          int& z1) {
  z0 = max((chunk ? tp.n : tp.L) - base, 0);
  z1 = min((chunk ? p.C : p.P) - base, BN);
}

// Zero rows [r0, r1) of a 128-byte-swizzled tile stored as D/64 blocks of
// `rows` rows x 128 bytes (the swizzle only permutes 16-byte chunks inside a
// row), by `nthreads` threads of which this is `tid`.
template <int D>
__device__ __forceinline__ void zero_tile_rows(uint8_t* tile, int rows, int r0, int r1, int tid, int nthreads) {
  constexpr int kChunks = D / 8;  // 16-byte chunks per row
  const int n = (r1 - r0) * kChunks;
#pragma unroll 1
  for (int k = tid; k < n; k += nthreads) {
    const int r = r0 + k / kChunks, c = k % kChunks;
    *reinterpret_cast<uint4*>(tile + (c / 8) * (rows * 128) + r * 128 + (c % 8) * 16) = make_uint4(0, 0, 0, 0);
  }
}

// Fused append, device side: write rotated key chunk pair (lo, hi) and the
// value chunks of chunk row i of (b, kv head h) into the cache, if the
// sequence has room (len + n <= cap) and i < n.
__device__ __forceinline__ void fused_append_pair(const AttnParams& p, int b, int h, int i, int kc,
                                                  uint4 lo, uint4 hi) {
  const int n = min(max(p.app_n[b], 0), p.C);
  const int L = p.app_len[b];
  if (L < 0 || L + n > p.app_cap || i >= n) return;
  const int D = p.D;
  const size_t dst = static_cast<size_t>(b) * p.app_sb + static_cast<size_t>(h) * p.app_sh +
                     static_cast<size_t>(L + i) * p.app_ss;
  const size_t src = ((static_cast<size_t>(b) * p.Hkv + h) * p.C + i) * D;
  if (!in_bounds(static_cast<long long>(dst), D, p.n_app, p.err) ||
      !in_bounds(static_cast<long long>(src), D, n_chunk(p), p.err))
    return;
  *reinterpret_cast<uint4*>(p.app_k + dst + kc * 8) = lo;
  *reinterpret_cast<uint4*>(p.app_k + dst + D / 2 + kc * 8) = hi;
  uint4 vl = *reinterpret_cast<const uint4*>(p.v_new + src + kc * 8);
  uint4 vh = *reinterpret_cast<const uint4*>(p.v_new + src + D / 2 + kc * 8);
  if (p.f16) {  // an fp16 cache: the rotated keys are half already; convert the values
    vl = bf16x8_to_f16x8(vl);
    vh = bf16x8_to_f16x8(vh);
  }
  *reinterpret_cast<uint4*>(p.app_v + dst + kc * 8) = vl;
  *reinterpret_cast<uint4*>(p.app_v + dst + D / 2 + kc * 8) = vh;
}

// Fused append: advance len (or flag the sequence that has no room); one
// thread per sequence, after every reader of len.
__device__ __forceinline__ void fused_append_len(const AttnParams& p, int b) {
  const int raw = p.app_n[b];
  const int n = min(max(raw, 0), p.C);
  if (raw != n) set_err(p.err, CPA_EBIT_NREAL_GT_C);
  const int L = p.app_len[b];
  if (L >= 0 && L + n <= p.app_cap) p.app_len[b] = L + n;
  else set_err(p.err, CPA_EBIT_CAPACITY);
}

}  // namespace cpa
