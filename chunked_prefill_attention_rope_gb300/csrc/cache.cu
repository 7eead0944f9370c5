// KV-cache bookkeeping kernels: global append with fused RoPE, sliding-window
// append with chronological compaction, and the padded-append snapshot /
// rollback pair ("Pad the chunked-prefill tail for sliding-window models", Fix).
//
// Every kernel moves whole 16-byte chunks with coalesced vector loads/stores.
// Row moves whose source and destination ranges overlap (compaction, the
// rollback's shift) go through caller scratch in two launches, so no CTA can
// overwrite a row another CTA has yet to read.  Per-sequence lengths are read
// by the first launch of a pair and passed to the second through a header in
// scratch; only the second launch writes `len`.
#include "common.cuh"
#include "kernels.h"

namespace cpa {

namespace {

constexpr int kThreads = 256;
constexpr int32_t kSnapMagic = 0x43504153;

struct Hdr {
  int32_t v[8];
};

// 16-byte chunk i (element index) of a buffer of n elements; checked builds
// range-check it (see common.cuh).
__device__ __forceinline__ uint4 ld16(const uint16_t* base, size_t i, long long n, int32_t* err) {
  return ld16_chk(base, static_cast<long long>(i), n, err);
}
__device__ __forceinline__ void st16(uint16_t* base, size_t i, long long n, uint4 v, int32_t* err) {
  st16_chk(base, static_cast<long long>(i), n, v, err);
}

__device__ __forceinline__ size_t crow(const CacheView& c, int b, int h, int s) {
  return static_cast<size_t>(b) * c.sb + static_cast<size_t>(h) * c.sh + static_cast<size_t>(s) * c.ss;
}

// Rotate K row i of the chunk (pair kc) and copy V row i, writing cache slot `dst`
// in the cache format (bf16, or half for an fp16 cache).
__device__ __forceinline__ void put_new_row(const CacheView& c, const ChunkView& x, int b, int h, int i,
                                            int dst, int kc, int Hkv, int D, int C) {
  const size_t src = ((static_cast<size_t>(b) * Hkv + h) * C + i) * D;
  if (!in_bounds((static_cast<long long>(b) * C + i) * D, D, x.n_tab, c.err)) return;
  uint4 lo = ld16(x.k, src + kc * 8, x.n_kv, c.err);
  uint4 hi = ld16(x.k, src + D / 2 + kc * 8, x.n_kv, c.err);
  const float* cr = x.cos + (static_cast<size_t>(b) * C + i) * D;
  const float* sr = x.sin + (static_cast<size_t>(b) * C + i) * D;
  uint4 vl = ld16(x.v, src + kc * 8, x.n_kv, c.err), vh = ld16(x.v, src + D / 2 + kc * 8, x.n_kv, c.err);
  if (c.f16) {
    rope_pair<true>(lo, hi, cr + kc * 8, sr + kc * 8, cr + D / 2 + kc * 8, sr + D / 2 + kc * 8);
    vl = bf16x8_to_f16x8(vl);
    vh = bf16x8_to_f16x8(vh);
  } else {
    rope_pair(lo, hi, cr + kc * 8, sr + kc * 8, cr + D / 2 + kc * 8, sr + D / 2 + kc * 8);
  }
  const size_t d = crow(c, b, h, dst);
  st16(c.k, d + kc * 8, c.extent, lo, c.err);
  st16(c.k, d + D / 2 + kc * 8, c.extent, hi, c.err);
  st16(c.v, d + kc * 8, c.extent, vl, c.err);
  st16(c.v, d + D / 2 + kc * 8, c.extent, vh, c.err);
}

__device__ __forceinline__ int clamp_rows(int n, int C, int32_t* err, bool report) {
  if (n < 0 || n > C) {
    if (report) set_err(err, CPA_EBIT_NREAL_GT_C);
    n = min(max(n, 0), C);
  }
  return n;
}

// ---------------------------------------------------------------- global append

__global__ void global_append_rows(CacheView c, ChunkView x, int B, int Hkv, int D, int C, int32_t* err) {
  grid_launch_dependents();  // the next launch may be scheduled; it waits for this grid
  grid_dependency_wait();    // everything the launches before this one wrote
  const int HP = D / 16;
  const unsigned total = static_cast<unsigned>(B) * Hkv * C * HP;  // < 2^31 (host)
  const int sh = __ffs(HP) - 1;  // HP is a power of two
  for (unsigned it = blockIdx.x * blockDim.x + threadIdx.x; it < total; it += gridDim.x * blockDim.x) {
    const int kc = static_cast<int>(it & (HP - 1));
    unsigned r = it >> sh;
    const int i = static_cast<int>(r % C);
    r /= C;
    const int h = static_cast<int>(r % Hkv);
    const int b = static_cast<int>(r / Hkv);
    const bool first = (h == 0 && i == 0 && kc == 0);
    const int n = clamp_rows(x.n_rows[b], C, err, first);
    const int L = c.len[b];
    if (L < 0 || L + n > c.cap) {
      if (first) set_err(err, CPA_EBIT_CAPACITY);
      continue;
    }
    if (i >= n) continue;
    put_new_row(c, x, b, h, i, L + i, kc, Hkv, D, C);
  }
}

__global__ void global_append_len(CacheView c, const int32_t* n_rows, int B, int C) {
  grid_launch_dependents();  // the next launch may be scheduled; it waits for this grid
  grid_dependency_wait();    // everything the launches before this one wrote
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int n = min(max(n_rows[b], 0), C);
  const int L = c.len[b];
  if (L >= 0 && L + n <= c.cap) c.len[b] = L + n;
}

// ---------------------------------------------------------------- sliding append

// Pass 1: decide (L, n, e) per sequence and copy the rows that survive an
// eviction ([S + e, L)) into staging.
__global__ void sliding_stage(CacheView c, const int32_t* n_rows, int B, int Hkv, int D, int C,
                              Hdr* hdr, uint16_t* stage_k, uint16_t* stage_v, int32_t* err) {
  grid_launch_dependents();  // the next launch may be scheduled; it waits for this grid
  grid_dependency_wait();    // everything the launches before this one wrote
  const int W = c.window, S = c.sink;
  const int CH = D / 8;
  const unsigned total = static_cast<unsigned>(B) * Hkv * W * CH;  // < 2^31 (host)
  const int sh = __ffs(CH) - 1;  // CH is a power of two
  for (unsigned it = blockIdx.x * blockDim.x + threadIdx.x; it < total; it += gridDim.x * blockDim.x) {
    const int cc = static_cast<int>(it & (CH - 1));
    unsigned r = it >> sh;
    const int row = static_cast<int>(r % W);
    r /= W;
    const int h = static_cast<int>(r % Hkv);
    const int b = static_cast<int>(r / Hkv);
    const bool first = (h == 0 && row == 0 && cc == 0);
    const int n = clamp_rows(n_rows[b], C, err, first);
    const int L = c.len[b];
    const bool ok = L >= 0 && L <= W && n <= W - S;
    const int e = max(0, L + n - W);
    if (first) {
      hdr[b].v[0] = L;
      hdr[b].v[1] = n;
      hdr[b].v[2] = e;
      hdr[b].v[3] = ok ? 1 : 0;
      if (!ok) set_err(err, CPA_EBIT_SLIDING_N);
    }
    const int cnt = max(0, L - S - e);
    if (!ok || e == 0 || row >= cnt) continue;
    const size_t s = crow(c, b, h, S + e + row) + cc * 8;
    const size_t d = ((static_cast<size_t>(b) * Hkv + h) * W + row) * D + cc * 8;
    const long long nst = static_cast<long long>(B) * Hkv * W * D;
    st16(stage_k, d, nst, ld16(c.k, s, c.extent, c.err), c.err);
    st16(stage_v, d, nst, ld16(c.v, s, c.extent, c.err), c.err);
  }
}

// Pass 2: survivors from staging to [S, L - e), the new rows (rotated K) to
// [L - e, L - e + n), then len = L - e + n.
__global__ void sliding_commit(CacheView c, ChunkView x, int B, int Hkv, int D, int C, const Hdr* hdr,
                               const uint16_t* stage_k, const uint16_t* stage_v) {
  grid_launch_dependents();  // the next launch may be scheduled; it waits for this grid
  grid_dependency_wait();    // everything the launches before this one wrote
  const int W = c.window, S = c.sink;
  const int HP = D / 16;
  const int rows = W + C;
  const unsigned total = static_cast<unsigned>(B) * Hkv * rows * HP;  // < 2^31 (host)
  const int sh = __ffs(HP) - 1;  // HP is a power of two
  for (unsigned it = blockIdx.x * blockDim.x + threadIdx.x; it < total; it += gridDim.x * blockDim.x) {
    const int kc = static_cast<int>(it & (HP - 1));
    unsigned r = it >> sh;
    const int rr = static_cast<int>(r % rows);
    r /= rows;
    const int h = static_cast<int>(r % Hkv);
    const int b = static_cast<int>(r / Hkv);
    const int L = hdr[b].v[0], n = hdr[b].v[1], e = hdr[b].v[2];
    if (!hdr[b].v[3]) continue;
    if (h == 0 && rr == 0 && kc == 0) c.len[b] = L - e + n;
    if (rr < W) {
      const int cnt = max(0, L - S - e);
      if (e == 0 || rr >= cnt) continue;
      const size_t s = ((static_cast<size_t>(b) * Hkv + h) * W + rr) * D;
      const size_t d = crow(c, b, h, S + rr);
      const long long nst = static_cast<long long>(B) * Hkv * W * D;
      st16(c.k, d + kc * 8, c.extent, ld16(stage_k, s + kc * 8, nst, c.err), c.err);
      st16(c.k, d + D / 2 + kc * 8, c.extent, ld16(stage_k, s + D / 2 + kc * 8, nst, c.err), c.err);
      st16(c.v, d + kc * 8, c.extent, ld16(stage_v, s + kc * 8, nst, c.err), c.err);
      st16(c.v, d + D / 2 + kc * 8, c.extent, ld16(stage_v, s + D / 2 + kc * 8, nst, c.err), c.err);
    } else {
      const int t = rr - W;
      if (t >= n) continue;
      put_new_row(c, x, b, h, t, L - e + t, kc, Hkv, D, C);
    }
  }
}

// ---------------------------------------------------------------- snapshot / rollback

// Save rows [S + e_ex, S + e_pad): the rows a padded append of C rows evicts
// beyond an exact append of n rows.
__global__ void snapshot_kernel(CacheView c, const int32_t* n_real, int B, int Hkv, int D, int C, Hdr* hdr,
                                uint16_t* saved_k, uint16_t* saved_v, int32_t* err) {
  grid_launch_dependents();  // the next launch may be scheduled; it waits for this grid
  grid_dependency_wait();    // everything the launches before this one wrote
  const int W = c.window, S = c.sink;
  const int CH = D / 8;
  const unsigned total = static_cast<unsigned>(B) * Hkv * C * CH;  // < 2^31 (host)
  const int sh = __ffs(CH) - 1;  // CH is a power of two
  for (unsigned it = blockIdx.x * blockDim.x + threadIdx.x; it < total; it += gridDim.x * blockDim.x) {
    const int cc = static_cast<int>(it & (CH - 1));
    unsigned r = it >> sh;
    const int row = static_cast<int>(r % C);
    r /= C;
    const int h = static_cast<int>(r % Hkv);
    const int b = static_cast<int>(r / Hkv);
    const bool first = (h == 0 && row == 0 && cc == 0);
    const int n = clamp_rows(n_real[b], C, err, first);
    const int L = c.len[b];
    const bool ok = L >= 0 && L <= W;
    const int e_pad = max(0, L + C - W);
    const int e_ex = max(0, L + n - W);
    if (first) {
      hdr[b].v[0] = L;
      hdr[b].v[1] = n;
      hdr[b].v[2] = e_ex;
      hdr[b].v[3] = e_pad;
      hdr[b].v[4] = ok ? 1 : 0;
      hdr[b].v[5] = kSnapMagic;
      if (!ok) set_err(err, CPA_EBIT_SLIDING_N);
    }
    if (!ok || row >= e_pad - e_ex) continue;
    const size_t s = crow(c, b, h, S + e_ex + row) + cc * 8;
    const size_t d = ((static_cast<size_t>(b) * Hkv + h) * C + row) * D + cc * 8;
    const long long nsv = static_cast<long long>(B) * Hkv * C * D;
    st16(saved_k, d, nsv, ld16(c.k, s, c.extent, c.err), c.err);
    st16(saved_v, d, nsv, ld16(c.v, s, c.extent, c.err), c.err);
  }
}

// Rollback pass 1: check the cache length against the snapshot, then stage the
// rows [S, keep) that must move right by d = e_pad - e_ex.
__global__ void rollback_stage(CacheView c, int B, int Hkv, int D, int C, const Hdr* snap, Hdr* roll,
                               uint16_t* stage_k, uint16_t* stage_v, int32_t* err) {
  grid_launch_dependents();  // the next launch may be scheduled; it waits for this grid
  grid_dependency_wait();    // everything the launches before this one wrote
  const int W = c.window, S = c.sink;
  const int CH = D / 8;
  const unsigned total = static_cast<unsigned>(B) * Hkv * W * CH;  // < 2^31 (host)
  const int sh = __ffs(CH) - 1;  // CH is a power of two
  for (unsigned it = blockIdx.x * blockDim.x + threadIdx.x; it < total; it += gridDim.x * blockDim.x) {
    const int cc = static_cast<int>(it & (CH - 1));
    unsigned r = it >> sh;
    const int row = static_cast<int>(r % W);
    r /= W;
    const int h = static_cast<int>(r % Hkv);
    const int b = static_cast<int>(r / Hkv);
    const bool first = (h == 0 && row == 0 && cc == 0);
    const int L0 = snap[b].v[0], n = snap[b].v[1], e_ex = snap[b].v[2], e_pad = snap[b].v[3];
    const int len_p = c.len[b];
    const bool good = snap[b].v[5] == kSnapMagic && snap[b].v[4] == 1 && len_p == L0 + C - e_pad;
    const int keep = len_p - (C - n);
    const int d = e_pad - e_ex;
    if (first) {
      roll[b].v[0] = keep;
      roll[b].v[1] = d;
      roll[b].v[2] = good ? 1 : 0;
      if (!good) set_err(err, CPA_EBIT_SNAPSHOT);
    }
    if (!good || d == 0 || row >= keep - S) continue;
    const size_t s = crow(c, b, h, S + row) + cc * 8;
    const size_t o = ((static_cast<size_t>(b) * Hkv + h) * W + row) * D + cc * 8;
    const long long nst = static_cast<long long>(B) * Hkv * W * D;
    st16(stage_k, o, nst, ld16(c.k, s, c.extent, c.err), c.err);
    st16(stage_v, o, nst, ld16(c.v, s, c.extent, c.err), c.err);
  }
}

// Rollback pass 2: staged rows to [S + d, keep + d), saved rows to [S, S + d),
// len = keep + d; the snapshot record is retired.
__global__ void rollback_commit(CacheView c, int B, int Hkv, int D, int C, Hdr* snap, const Hdr* roll,
                                const uint16_t* stage_k, const uint16_t* stage_v, const uint16_t* saved_k,
                                const uint16_t* saved_v) {
  grid_launch_dependents();  // the next launch may be scheduled; it waits for this grid
  grid_dependency_wait();    // everything the launches before this one wrote
  const int W = c.window, S = c.sink;
  const int CH = D / 8;
  const int rows = W + C;
  const unsigned total = static_cast<unsigned>(B) * Hkv * rows * CH;  // < 2^31 (host)
  const int sh = __ffs(CH) - 1;  // CH is a power of two
  for (unsigned it = blockIdx.x * blockDim.x + threadIdx.x; it < total; it += gridDim.x * blockDim.x) {
    const int cc = static_cast<int>(it & (CH - 1));
    unsigned r = it >> sh;
    const int rr = static_cast<int>(r % rows);
    r /= rows;
    const int h = static_cast<int>(r % Hkv);
    const int b = static_cast<int>(r / Hkv);
    const int keep = roll[b].v[0], d = roll[b].v[1];
    if (!roll[b].v[2]) continue;
    if (h == 0 && rr == 0 && cc == 0) {
      c.len[b] = keep + d;
      snap[b].v[5] = 0;
    }
    if (d == 0) continue;
    if (rr < W) {
      if (rr >= keep - S) continue;
      const size_t s = ((static_cast<size_t>(b) * Hkv + h) * W + rr) * D + cc * 8;
      const size_t o = crow(c, b, h, S + d + rr) + cc * 8;
      const long long nst = static_cast<long long>(B) * Hkv * W * D;
      st16(c.k, o, c.extent, ld16(stage_k, s, nst, c.err), c.err);
      st16(c.v, o, c.extent, ld16(stage_v, s, nst, c.err), c.err);
    } else {
      const int t = rr - W;
      if (t >= d) continue;
      const size_t s = ((static_cast<size_t>(b) * Hkv + h) * C + t) * D + cc * 8;
      const size_t o = crow(c, b, h, S + t) + cc * 8;
      const long long nsv = static_cast<long long>(B) * Hkv * C * D;
      st16(c.k, o, c.extent, ld16(saved_k, s, nsv, c.err), c.err);
      st16(c.v, o, c.extent, ld16(saved_v, s, nsv, c.err), c.err);
    }
  }
}

int grid_for(long long items) {
  long long blocks = (items + kThreads - 1) / kThreads;
  if (blocks < 1) blocks = 1;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  return static_cast<int>(blocks);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

SlidingScratch sliding_scratch_layout(int B, int Hkv, int D, int C, int W) {
  SlidingScratch L;
  size_t off = 0;
  const size_t hdr = align256(static_cast<size_t>(B) * sizeof(Hdr));
  L.hdr_append = off; off += hdr;
  L.hdr_snap = off; off += hdr;
  L.hdr_roll = off; off += hdr;
  const size_t saved = align256(static_cast<size_t>(B) * Hkv * C * D * 2);
  L.saved_k = off; off += saved;
  L.saved_v = off; off += saved;
  const size_t stage = align256(static_cast<size_t>(B) * Hkv * W * D * 2);
  L.stage_k = off; off += stage;
  L.stage_v = off; off += stage;
  L.total = off;
  return L;
}

cudaError_t launch_global_append(const CacheView& c, const ChunkView& x, int B, int Hkv, int D, int C,
                                 int32_t* err, cudaStream_t s) {
  const long long items = static_cast<long long>(B) * Hkv * C * (D / 16);
  cudaError_t e = launch_dependent(global_append_rows, grid_for(items), dim3(kThreads), 0, s, c, x, B, Hkv, D, C, err);
  if (e != cudaSuccess) return e;
  return launch_dependent(global_append_len, dim3((B + 127) / 128), dim3(128), 0, s, c, x.n_rows, B, C);
}

cudaError_t launch_sliding_append(const CacheView& c, const ChunkView& x, int B, int Hkv, int D, int C,
                                  uint8_t* scratch, int32_t* err, cudaStream_t s) {
  const SlidingScratch L = sliding_scratch_layout(B, Hkv, D, C, c.window);
  Hdr* hdr = reinterpret_cast<Hdr*>(scratch + L.hdr_append);
  uint16_t* sk = reinterpret_cast<uint16_t*>(scratch + L.stage_k);
  uint16_t* sv = reinterpret_cast<uint16_t*>(scratch + L.stage_v);
  const long long items1 = static_cast<long long>(B) * Hkv * c.window * (D / 8);
  cudaError_t e = launch_dependent(sliding_stage, grid_for(items1), dim3(kThreads), 0, s, c, x.n_rows, B, Hkv, D, C,
                                   hdr, sk, sv, err);
  if (e != cudaSuccess) return e;
  const long long items2 = static_cast<long long>(B) * Hkv * (c.window + C) * (D / 16);
  return launch_dependent(sliding_commit, grid_for(items2), dim3(kThreads), 0, s, c, x, B, Hkv, D, C,
                          static_cast<const Hdr*>(hdr), static_cast<const uint16_t*>(sk),
                          static_cast<const uint16_t*>(sv));
}

cudaError_t launch_snapshot(const CacheView& c, const int32_t* n_real, int B, int Hkv, int D, int C,
                            uint8_t* scratch, int32_t* err, cudaStream_t s) {
  const SlidingScratch L = sliding_scratch_layout(B, Hkv, D, C, c.window);
  const long long items = static_cast<long long>(B) * Hkv * C * (D / 8);
  return launch_dependent(snapshot_kernel, grid_for(items), dim3(kThreads), 0, s, c, n_real, B, Hkv, D, C,
                          reinterpret_cast<Hdr*>(scratch + L.hdr_snap), reinterpret_cast<uint16_t*>(scratch + L.saved_k),
                          reinterpret_cast<uint16_t*>(scratch + L.saved_v), err);
}

cudaError_t launch_rollback(const CacheView& c, int B, int Hkv, int D, int C, uint8_t* scratch, int32_t* err,
                            cudaStream_t s) {
  const SlidingScratch L = sliding_scratch_layout(B, Hkv, D, C, c.window);
  Hdr* snap = reinterpret_cast<Hdr*>(scratch + L.hdr_snap);
  Hdr* roll = reinterpret_cast<Hdr*>(scratch + L.hdr_roll);
  uint16_t* sk = reinterpret_cast<uint16_t*>(scratch + L.stage_k);
  uint16_t* sv = reinterpret_cast<uint16_t*>(scratch + L.stage_v);
  const long long items1 = static_cast<long long>(B) * Hkv * c.window * (D / 8);
  cudaError_t e = launch_dependent(rollback_stage, grid_for(items1), dim3(kThreads), 0, s, c, B, Hkv, D, C,
                                   static_cast<const Hdr*>(snap), roll, sk, sv, err);
  if (e != cudaSuccess) return e;
  const long long items2 = static_cast<long long>(B) * Hkv * (c.window + C) * (D / 8);
  return launch_dependent(rollback_commit, grid_for(items2), dim3(kThreads), 0, s, c, B, Hkv, D, C, snap,
                          static_cast<const Hdr*>(roll), static_cast<const uint16_t*>(sk),
                          static_cast<const uint16_t*>(sv), reinterpret_cast<const uint16_t*>(scratch + L.saved_k),
                          reinterpret_cast<const uint16_t*>(scratch + L.saved_v));
}

}  // namespace cpa
