// C-ABI entry points (include/cpa.h): host-side validation, TMA descriptors,
// split-KV policy and kernel launches.  Nothing here allocates device memory
// or synchronises.
#include <math.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#ifdef CPA_TEST_HOOKS
#include "../../include/cpa_test.h"
#endif

using namespace cpa;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 4-D bf16 map {D, rows, heads, batch} with a {64, box_rows, box_heads, 1} box, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int D, int rows, int heads, int batch, int64_t s_row,
              int64_t s_head, int64_t s_batch, int box_rows, int box_heads = 1) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows > 0 ? rows : 1),
                        static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(s_row) * 2, static_cast<cuuint64_t>(s_head) * 2,
                           static_cast<cuuint64_t>(s_batch) * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(box_heads), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checked build's test hook: the key tile whose copy each two-tile CTA
// withholds (-1: none); the regular build never withholds one.
#ifdef CPA_TEST_HOOKS
std::atomic<int> g_test_drop_tile{-1};
int test_drop_tile() { return g_test_drop_tile.load(std::memory_order_relaxed); }
#else
int test_drop_tile() { return -1; }
#endif

// SM count of the current device, queried once per device (devices 0-63).
int num_sms() {
  static std::atomic<int> cached[64];
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && (n = cached[dev].load(std::memory_order_relaxed)) > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

enum Path { kPathSingle = 0, kPathPair = 1, kPathDecode = 2 };

struct Geometry {
  int G, R, nq, splits, path;
  bool cluster;  // single-tile splits merged inside a thread-block cluster
  int dsplit;    // CTAs per split in that cluster (2: they divide D)
  PairTeams teams;
};

// Kernel path and work split for these sizes.  The host cannot see per-sequence
// lengths without a sync, so every choice depends only on the shapes.
//   pair   (D = 64/128, at least two query tiles): persistent CTAs, one per SM
//          at most, balanced on the device by stream-K (no split-KV).
//   decode (C = 1) and single-tile chunks: split-KV, each split owning a fixed
//          range of the key-tile index space (see tiles.cuh); splits grow while
//          the grid is under two waves, and one-query-tile calls cap a CTA at
//          about 32 (decode kernel) or 16 (single-tile kernel) key tiles of the
//          longest possible past.
Geometry geometry(int B, int Hq, int Hkv, int D, int C, int P, int sm_budget = 0) {
  Geometry g;
  g.G = Hq / Hkv;
  g.R = 128 / g.G;
  g.nq = (C + g.R - 1) / g.R;
  g.teams = PairTeams{};
  g.cluster = false;
  g.dsplit = 1;
  const int dev_sms = num_sms();
  const int sms = sm_budget > 0 && sm_budget < dev_sms ? sm_budget : dev_sms;
  if (attn_uses_pair(D, g.nq) && !attn_uses_decode(D, C, g.G)) {
    g.path = kPathPair;
    g.splits = 1;
    g.teams = pair_teams(B, Hkv, g.nq, P, C, sms);
    return g;
  }
  g.path = attn_uses_decode(D, C, g.G) ? kPathDecode : kPathSingle;
  const int bn = attn_block_n(D);
  const int max_tiles = (P + bn - 1) / bn + (C + bn - 1) / bn;
  const long long ctas = static_cast<long long>(B) * Hkv * g.nq;
  int s = 1;
  while (ctas * s < 2LL * sms && s * 2 <= max_tiles) s *= 2;
  // one query tile per (sequence, kv head): enough splits that a CTA sees at
  // most ~32 key tiles of the longest past on the decode kernel (measured
  // best of 8/16/32/64/128 on a 64-sequence batch), ~16 on the single-tile one
  const int per_cta = g.path == kPathDecode ? 32 : 16;
  if (g.nq == 1 && max_tiles > 32) s = max(s, (max_tiles + per_cta - 1) / per_cta);
  g.splits = max(1, min(s, max(1, max_tiles)));
  g.cluster = g.path == kPathSingle && (g.splits == 2 || g.splits == 4 || g.splits == 8) &&
              attn_cluster_ok(D, g.splits);
  // D = 256 over 8 splits: the merge's exchange of 128 KB of fp32 rows per CTA
  // through distributed shared memory bounds the call, so each split is taken
  // by two CTAs that divide D (each sends half), in clusters of 16, when all of
  // those clusters can be resident at once (not every GPC holds 16 CTAs, and
  // a second wave of them costs more than the exchange saves)
  if (g.cluster && g.splits == 8 && D == 256 && ctas * 16 <= sms && ctas <= attn_max_clusters(D, 16)) g.dsplit = 2;
  return g;
}

// Workspace of the decode and single-tile paths: split-KV partials (when
// combine_kernel merges them), then, on the single-tile path, the rotated
// queries and chunk keys and (fp16 cache) the converted chunk values.
struct SingleWorkspace {
  size_t part_o, part_lse, q_rot, k_rot, v_cvt, total;
};
SingleWorkspace single_workspace(const Geometry& g, int B, int Hq, int Hkv, int D, int C) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  SingleWorkspace w{};
  size_t off = 0;
  if (g.splits > 1 && !g.cluster) {
    const size_t rows = static_cast<size_t>(B) * Hq * C;
    w.part_o = off;
    off += al(static_cast<size_t>(g.splits) * rows * D * sizeof(float));
    w.part_lse = off;
    off += al(static_cast<size_t>(g.splits) * rows * sizeof(float));
  }
  if (g.path == kPathSingle) {
    w.q_rot = off;  // the rotated queries (in half for an fp16 cache)
    off += al(static_cast<size_t>(B) * Hq * C * D * 2);
    w.k_rot = off;
    off += al(static_cast<size_t>(B) * Hkv * C * D * 2);
    w.v_cvt = off;  // fp16 cache: the chunk values in half
    off += al(static_cast<size_t>(B) * Hkv * C * D * 2);
  }
  w.total = off;
  return w;
}

// Bytes of workspace for these sizes; `mask_bits`: with room for the two-tile
// path's bit copy of an explicit mask (the other paths need no more for it).
size_t workspace_bytes(const Geometry& g, int B, int Hq, int Hkv, int D, int C, int P, bool mask_bits = false) {
  if (g.path == kPathPair) {
    const PairWorkspace w = pair_workspace(B, Hq, Hkv, D, C, P, g.teams);
    return mask_bits ? w.total_bits : w.total;
  }
  return single_workspace(g, B, Hq, Hkv, D, C).total;
}

bool valid_d(int D) { return D == 64 || D == 128 || D == 256; }

cpa_status check_cache(const cpa_cache* c, int D) {
  if (!c || !c->k || !c->v || !c->len) return CPA_ERR_NULL;
  if (c->cap < 1 || c->stride_s < D || c->stride_h < 1 || c->stride_b < 1) return CPA_ERR_SHAPE;
  if (!aligned16(c->k) || !aligned16(c->v) || !aligned16(c->len)) return CPA_ERR_ALIGN;
  if (c->stride_s % 8 || c->stride_h % 8 || c->stride_b % 8) return CPA_ERR_ALIGN;
  if (c->kind != CPA_CACHE_GLOBAL && c->kind != CPA_CACHE_SLIDING) return CPA_ERR_SHAPE;
  if (c->dtype != CPA_KV_BF16 && c->dtype != CPA_KV_F16) return CPA_ERR_UNSUPPORTED;
  if (c->kind == CPA_CACHE_SLIDING) {
    if (c->window < 1 || c->window > c->cap || c->sink < 0 || c->sink >= c->window) return CPA_ERR_SHAPE;
  }
  return CPA_OK;
}

// Elements spanned by a [B, Hkv, cap, D] view with these strides.
long long view_extent(const cpa_cache* c, int B, int Hkv, int D) {
  return static_cast<long long>(B - 1) * c->stride_b + static_cast<long long>(Hkv - 1) * c->stride_h +
         static_cast<long long>(c->cap - 1) * c->stride_s + D;
}

CacheView view_of(const cpa_cache* c, int B, int Hkv, int D, int32_t* err) {
  CacheView v;
  v.extent = view_extent(c, B, Hkv, D);
  v.err = err;
  v.k = static_cast<uint16_t*>(c->k);
  v.v = static_cast<uint16_t*>(c->v);
  v.sb = c->stride_b;
  v.sh = c->stride_h;
  v.ss = c->stride_s;
  v.len = c->len;
  v.cap = c->cap;
  v.window = c->kind == CPA_CACHE_SLIDING ? c->window : c->cap;
  v.sink = c->kind == CPA_CACHE_SLIDING ? c->sink : 0;
  v.f16 = c->dtype == CPA_KV_F16 ? 1 : 0;
  return v;
}

cpa_status attn_impl(const cpa_attn_args* a, cudaStream_t stream, bool decode, const int32_t* app_n = nullptr) {
  if (!a) return CPA_ERR_NULL;
  if (!a->q || !a->k_new || !a->v_new || !a->cos || !a->sin || !a->out || !a->err) return CPA_ERR_NULL;
  if (a->B < 1 || a->Hq < 1 || a->Hkv < 1 || a->C < 1 || a->P < 0) return CPA_ERR_SHAPE;
  if (a->Hq % a->Hkv != 0 || a->Hq / a->Hkv > 128) return CPA_ERR_SHAPE;
  if (!valid_d(a->D)) return CPA_ERR_UNSUPPORTED;
  if (decode && a->C != 1) return CPA_ERR_SHAPE;
  if (a->window < 0 || a->sm_budget < 0) return CPA_ERR_SHAPE;
  const cpa_status cs = check_cache(a->cache, a->D);
  if (cs != CPA_OK) return cs;
  if (a->P > a->cache->cap) return CPA_ERR_SHAPE;
  if (!a->mask && (!a->past_len || !a->n_real)) return CPA_ERR_NULL;
  if (a->out_sel && !a->sel_row && !a->n_real) return CPA_ERR_NULL;
  if (!aligned16(a->q) || !aligned16(a->k_new) || !aligned16(a->v_new) || !aligned16(a->cos) ||
      !aligned16(a->sin) || !aligned16(a->out) || (a->out_sel && !aligned16(a->out_sel)) ||
      (a->mask && !aligned16(a->mask)) || !aligned16(a->err))
    return CPA_ERR_ALIGN;
  if (static_cast<long long>(a->B) * a->Hq * a->C * a->D > (1LL << 40)) return CPA_ERR_SHAPE;
  // the RoPE pre-passes index their items (rows x 16-byte chunk pairs, four
  // heads per item) in 32 bits
  if (static_cast<long long>(a->B) * (a->Hq + a->Hkv + 3) * a->C * (a->D / 16) >= (1LL << 31)) return CPA_ERR_SHAPE;

  const Geometry g = geometry(a->B, a->Hq, a->Hkv, a->D, a->C, a->P, a->sm_budget);
  const size_t need = workspace_bytes(g, a->B, a->Hq, a->Hkv, a->D, a->C, a->P);
  if (need > 0 && (!a->workspace || a->workspace_bytes < need || !aligned16(a->workspace)))
    return CPA_ERR_WORKSPACE;

  const int bn = attn_uses_decode(a->D, a->C, g.G) ? 64 : attn_block_n(a->D);
  CUtensorMap maps[5];
  const cpa_cache* c = a->cache;
  const int64_t cs_ = static_cast<int64_t>(a->C) * a->D;
  if (!make_map(&maps[0], c->k, a->D, a->P, a->Hkv, a->B, c->stride_s, c->stride_h, c->stride_b, bn) ||
      !make_map(&maps[1], c->v, a->D, a->P, a->Hkv, a->B, c->stride_s, c->stride_h, c->stride_b, bn) ||
      !make_map(&maps[2], a->k_new, a->D, a->C, a->Hkv, a->B, a->D, cs_, cs_ * a->Hkv, bn) ||
      !make_map(&maps[3], a->v_new, a->D, a->C, a->Hkv, a->B, a->D, cs_, cs_ * a->Hkv, bn))
    return CPA_ERR_CUDA;

  AttnParams p{};
  p.B = a->B;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.D = a->D;
  p.C = a->C;
  p.P = a->P;
  p.G = g.G;
  p.R = g.R;
  p.nq = g.nq;
  p.splits = g.splits;
  p.cluster = g.cluster ? 1 : 0;
  p.dsplit = g.dsplit;
  const double scale = a->scale > 0.f ? static_cast<double>(a->scale) : 1.0 / sqrt(static_cast<double>(a->D));
  p.sl2 = static_cast<float>(scale * 1.4426950408889634);
  p.inv_scale = static_cast<float>(1.0 / scale);
  p.q = static_cast<const uint16_t*>(a->q);
  p.cos = a->cos;
  p.sin = a->sin;
  p.mask = a->mask;
  p.past_len = a->past_len;
  p.n_real = a->n_real;
  p.sel_row = a->sel_row;
  p.window = a->window;
  p.causal = a->causal ? 1 : 0;
  p.f16 = c->dtype == CPA_KV_F16 ? 1 : 0;
  p.sink = (!a->mask && a->cache->kind == CPA_CACHE_SLIDING) ? a->cache->sink : 0;
  p.out = static_cast<uint16_t*>(a->out);
  p.hold_dependents = a->sm_budget > 0 && a->sm_budget < num_sms() ? 1 : 0;
  p.out_sel = a->out_sel;
  p.err = a->err;
  p.k_new = static_cast<const uint16_t*>(a->k_new);
  p.v_new = static_cast<const uint16_t*>(a->v_new);
  p.test_drop_tile = test_drop_tile();
  if (app_n && g.path != kPathDecode) {
    p.n_app = view_extent(c, a->B, a->Hkv, a->D);
    p.app_n = app_n;
    p.app_k = static_cast<uint16_t*>(c->k);
    p.app_v = static_cast<uint16_t*>(c->v);
    p.app_sb = c->stride_b;
    p.app_sh = c->stride_h;
    p.app_ss = c->stride_s;
    p.app_len = c->len;
    p.app_cap = c->cap;
  }
  if (g.path == kPathPair) {
    const PairTeams& t = g.teams;
    p.pairs = t.pairs;
    p.units = a->B * a->Hkv * t.pairs;
    p.team = t.team;
    p.nblk = t.nblk;
    p.blocks = t.blocks;
    p.teams = t.teams;
    p.ctas = t.ctas;
    uint8_t* w = static_cast<uint8_t*>(a->workspace);
    const PairWorkspace L = pair_workspace(a->B, a->Hq, a->Hkv, a->D, a->C, a->P, t);
    p.ustart = reinterpret_cast<int32_t*>(w + L.ustart);
    // the plan depends on the shapes and the visited tiles only, whatever the
    // mask form, so that both forms of one mask split the work alike
    p.perm = t.perm ? 1 : 0;
    p.ntiles = (a->C + 127) / 128 + (a->P + 127) / 128;
    if (a->mask) {
      p.tcls = w + L.tcls;
      p.hull = reinterpret_cast<int4*>(w + L.hull);
      // the mask's bit copy when the caller's workspace has room for it
      p.mbits = a->workspace_bytes >= L.total_bits ? reinterpret_cast<uint4*>(w + L.mbits) : nullptr;
    }
    p.uorder = reinterpret_cast<int32_t*>(w + L.uorder);
    p.upos = reinterpret_cast<int32_t*>(w + L.upos);
    p.tlo = reinterpret_cast<int32_t*>(w + L.tlo);
    p.part_o = reinterpret_cast<float*>(w + L.part_o);
    p.part_lse = reinterpret_cast<float*>(w + L.part_lse);
    p.n_part = static_cast<long long>(t.ctas) * 2 * 256 * a->D;
    p.ptag = reinterpret_cast<int32_t*>(w + L.ptag);
    p.q_rot = reinterpret_cast<uint16_t*>(w + L.q_rot);
    p.k_rot = reinterpret_cast<uint16_t*>(w + L.k_rot);
    p.v_cvt = reinterpret_cast<uint16_t*>(w + L.v_cvt);
    // chunk keys and queries come from the rotated copies the pre-pass writes
    // (and, for an fp16 cache, the chunk values from its half copy)
    CUtensorMap pm[5] = {maps[0], maps[1], maps[2], maps[3], maps[4]};
    if (!make_map(&pm[2], p.k_rot, a->D, a->C, a->Hkv, a->B, a->D, cs_, cs_ * a->Hkv, bn) ||
        !make_map(&pm[4], p.q_rot, a->D, a->C, a->Hq, a->B, a->D, cs_, cs_ * a->Hq, g.R, g.G) ||
        (p.f16 && !make_map(&pm[3], p.v_cvt, a->D, a->C, a->Hkv, a->B, a->D, cs_, cs_ * a->Hkv, bn)))
      return CPA_ERR_CUDA;
    return launch_attn_pair5(pm, p, stream) == cudaSuccess ? CPA_OK : CPA_ERR_CUDA;
  }
  const SingleWorkspace L = single_workspace(g, a->B, a->Hq, a->Hkv, a->D, a->C);
  uint8_t* w = static_cast<uint8_t*>(a->workspace);
  if (g.splits > 1 && !g.cluster) {
    p.part_o = reinterpret_cast<float*>(w + L.part_o);
    p.part_lse = reinterpret_cast<float*>(w + L.part_lse);
    p.n_part = static_cast<long long>(g.splits) * a->B * a->Hq * a->C * a->D;
  }
  if (g.path == kPathSingle) {
    // Q rows and chunk keys from the pre-pass's rotated copies (Q box {64, R, G, 1})
    p.q_rot = reinterpret_cast<uint16_t*>(w + L.q_rot);
    p.k_rot = reinterpret_cast<uint16_t*>(w + L.k_rot);
    p.v_cvt = reinterpret_cast<uint16_t*>(w + L.v_cvt);
    if (!make_map(&maps[4], p.q_rot, a->D, a->C, a->Hq, a->B, a->D, cs_, cs_ * a->Hq, g.R, g.G) ||
        !make_map(&maps[2], p.k_rot, a->D, a->C, a->Hkv, a->B, a->D, cs_, cs_ * a->Hkv, bn) ||
        (p.f16 && !make_map(&maps[3], p.v_cvt, a->D, a->C, a->Hkv, a->B, a->D, cs_, cs_ * a->Hkv, bn)))
      return CPA_ERR_CUDA;
  }
  if (launch_attn(maps, p, stream) != cudaSuccess) return CPA_ERR_CUDA;
  if (app_n) {
    // the rows were written by the RoPE pre-pass; advance len after the
    // attention (one token: the separate append kernels after the attention)
    const cudaError_t e =
        g.path == kPathDecode
            ? launch_global_append(view_of(c, a->B, a->Hkv, a->D, a->err),
                                   ChunkView{static_cast<const uint16_t*>(a->k_new),
                                             static_cast<const uint16_t*>(a->v_new), a->cos, a->sin, app_n,
                                             static_cast<long long>(a->B) * a->Hkv * a->C * a->D,
                                             static_cast<long long>(a->B) * a->C * a->D},
                                   a->B, a->Hkv, a->D, a->C, a->err, stream)
            : launch_fused_append_len(p, stream);
    if (e != cudaSuccess) return CPA_ERR_CUDA;
  }
  return CPA_OK;
}

// The cache kernels index their items (rows x 16-byte chunks) in 32 bits.
bool items_fit(int B, int Hkv, long long rows, int D) {
  return static_cast<long long>(B) * Hkv * rows * (D / 8) < (1LL << 31);
}

cpa_status chunk_check(const void* k_new, const void* v_new, const float* cos, const float* sin,
                       const int32_t* n_rows, int B, int Hkv, int D, int C, int32_t* err) {
  if (!k_new || !v_new || !cos || !sin || !n_rows || !err) return CPA_ERR_NULL;
  if (B < 1 || Hkv < 1 || C < 1) return CPA_ERR_SHAPE;
  if (!valid_d(D)) return CPA_ERR_UNSUPPORTED;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(cos) || !aligned16(sin) || !aligned16(err))
    return CPA_ERR_ALIGN;
  return CPA_OK;
}

}  // namespace

namespace cpa {

size_t attn_workspace_need(const cpa_attn_args* a) {
  if (!a || a->B < 1 || a->Hq < 1 || a->Hkv < 1 || a->C < 1 || a->P < 0 || a->Hq % a->Hkv ||
      a->Hq / a->Hkv > 128 || !valid_d(a->D) || a->sm_budget < 0)
    return 0;
  const Geometry g = geometry(a->B, a->Hq, a->Hkv, a->D, a->C, a->P, a->sm_budget);
  return workspace_bytes(g, a->B, a->Hq, a->Hkv, a->D, a->C, a->P);
}

}  // namespace cpa

extern "C" {

cpa_status cpa_chunk_prefill_attn(const cpa_attn_args* args, cpa_stream stream) {
  return attn_impl(args, reinterpret_cast<cudaStream_t>(stream), false);
}

cpa_status cpa_decode_step(const cpa_attn_args* args, cpa_stream stream) {
  return attn_impl(args, reinterpret_cast<cudaStream_t>(stream), true);
}

cpa_status cpa_chunk_prefill_attn_append(const cpa_attn_args* args, const int32_t* n_rows, cpa_stream stream) {
  if (!args || !n_rows) return CPA_ERR_NULL;
  if (args->cache && args->cache->kind != CPA_CACHE_GLOBAL) return CPA_ERR_UNSUPPORTED;
  if (!aligned16(n_rows)) return CPA_ERR_ALIGN;
  return attn_impl(args, reinterpret_cast<cudaStream_t>(stream), false, n_rows);
}

size_t cpa_attn_workspace_size(int B, int Hq, int Hkv, int D, int C, int P) {
  if (B < 1 || Hq < 1 || Hkv < 1 || C < 1 || P < 0 || Hq % Hkv || Hq / Hkv > 128 || !valid_d(D)) return 0;
  return workspace_bytes(geometry(B, Hq, Hkv, D, C, P), B, Hq, Hkv, D, C, P);
}

size_t cpa_attn_workspace_size_mask(int B, int Hq, int Hkv, int D, int C, int P) {
  if (B < 1 || Hq < 1 || Hkv < 1 || C < 1 || P < 0 || Hq % Hkv || Hq / Hkv > 128 || !valid_d(D)) return 0;
  return workspace_bytes(geometry(B, Hq, Hkv, D, C, P), B, Hq, Hkv, D, C, P, true);
}

size_t cpa_cache_scratch_size(const cpa_cache* cache, int B, int Hkv, int D, int C) {
  if (!cache || cache->kind != CPA_CACHE_SLIDING || B < 1 || Hkv < 1 || C < 1 || !valid_d(D)) return 0;
  return sliding_scratch_layout(B, Hkv, D, C, cache->window).total;
}

cpa_status cpa_kv_append(const cpa_cache* cache, const void* k_new, const void* v_new, const float* cos,
                         const float* sin, const int32_t* n_rows, int B, int Hkv, int D, int C, void* scratch,
                         size_t scratch_bytes, int32_t* err, cpa_stream stream) {
  cpa_status st = chunk_check(k_new, v_new, cos, sin, n_rows, B, Hkv, D, C, err);
  if (st != CPA_OK) return st;
  if ((st = check_cache(cache, D)) != CPA_OK) return st;
  if (!items_fit(B, Hkv, static_cast<long long>(C) + (cache->kind == CPA_CACHE_SLIDING ? cache->window : 0), D))
    return CPA_ERR_SHAPE;
  const CacheView cv = view_of(cache, B, Hkv, D, err);
  ChunkView x{static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new), cos, sin, n_rows,
              static_cast<long long>(B) * Hkv * C * D, static_cast<long long>(B) * C * D};
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (cache->kind == CPA_CACHE_GLOBAL) {
    e = launch_global_append(cv, x, B, Hkv, D, C, err, s);
  } else {
    const size_t need = sliding_scratch_layout(B, Hkv, D, C, cache->window).total;
    if (!scratch || scratch_bytes < need || !aligned16(scratch)) return CPA_ERR_WORKSPACE;
    e = launch_sliding_append(cv, x, B, Hkv, D, C, static_cast<uint8_t*>(scratch), err, s);
  }
  return e == cudaSuccess ? CPA_OK : CPA_ERR_CUDA;
}

cpa_status cpa_kv_snapshot_padded_append(const cpa_cache* cache, const int32_t* n_real, int B, int Hkv, int D,
                                         int C, void* scratch, size_t scratch_bytes, int32_t* err,
                                         cpa_stream stream) {
  if (!n_real || !err) return CPA_ERR_NULL;
  if (B < 1 || Hkv < 1 || C < 1) return CPA_ERR_SHAPE;
  if (!valid_d(D)) return CPA_ERR_UNSUPPORTED;
  cpa_status st = check_cache(cache, D);
  if (st != CPA_OK) return st;
  if (cache->kind != CPA_CACHE_SLIDING) return CPA_ERR_UNSUPPORTED;
  if (cache->window <= C + cache->sink) return CPA_ERR_WINDOW_TOO_SMALL;
  const size_t need = sliding_scratch_layout(B, Hkv, D, C, cache->window).total;
  if (!scratch || scratch_bytes < need || !aligned16(scratch)) return CPA_ERR_WORKSPACE;
  if (!items_fit(B, Hkv, static_cast<long long>(C) + cache->window, D)) return CPA_ERR_SHAPE;
  return launch_snapshot(view_of(cache, B, Hkv, D, err), n_real, B, Hkv, D, C, static_cast<uint8_t*>(scratch), err,
                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CPA_OK
             : CPA_ERR_CUDA;
}

cpa_status cpa_kv_rollback_padded_append(const cpa_cache* cache, int B, int Hkv, int D, int C, void* scratch,
                                         size_t scratch_bytes, int32_t* err, cpa_stream stream) {
  if (!err) return CPA_ERR_NULL;
  if (B < 1 || Hkv < 1 || C < 1) return CPA_ERR_SHAPE;
  if (!valid_d(D)) return CPA_ERR_UNSUPPORTED;
  cpa_status st = check_cache(cache, D);
  if (st != CPA_OK) return st;
  if (cache->kind != CPA_CACHE_SLIDING) return CPA_ERR_UNSUPPORTED;
  if (cache->window <= C + cache->sink) return CPA_ERR_WINDOW_TOO_SMALL;
  const size_t need = sliding_scratch_layout(B, Hkv, D, C, cache->window).total;
  if (!scratch || scratch_bytes < need || !aligned16(scratch)) return CPA_ERR_WORKSPACE;
  if (!items_fit(B, Hkv, static_cast<long long>(C) + cache->window, D)) return CPA_ERR_SHAPE;
  return launch_rollback(view_of(cache, B, Hkv, D, err), B, Hkv, D, C, static_cast<uint8_t*>(scratch), err,
                         reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CPA_OK
             : CPA_ERR_CUDA;
}

cpa_status cpa_tail_plan(int t, int C, int window, int sink, const int32_t* buckets, int n_buckets,
                         int crossover, int force, int32_t* mode, int32_t* c_pad) {
  if (!mode || !c_pad) return CPA_ERR_NULL;
  if (C < 1 || t < 1 || t > C || window < 0 || sink < 0 || n_buckets < 0) return CPA_ERR_SHAPE;
  if (n_buckets > 0 && !buckets) return CPA_ERR_NULL;
  if (force < CPA_TAIL_AUTO || force > CPA_TAIL_FORCE_PADDED) return CPA_ERR_SHAPE;
  for (int i = 0; i < n_buckets; ++i) {
    if (buckets[i] < 1 || buckets[i] > C) return CPA_ERR_SHAPE;
    if (i > 0 && buckets[i] <= buckets[i - 1]) return CPA_ERR_SHAPE;
  }
  *mode = CPA_TAIL_SCALAR;
  *c_pad = t;
  if (force == CPA_TAIL_FORCE_SCALAR) return CPA_OK;
  if (force == CPA_TAIL_AUTO && t < (crossover > 0 ? crossover : CPA_TAIL_CROSSOVER_DEFAULT)) return CPA_OK;
  // smallest runnable bucket holding the tail whose padded append the window can snapshot
  const int n = n_buckets > 0 ? n_buckets : 1;
  for (int i = 0; i < n; ++i) {
    const int cp = n_buckets > 0 ? buckets[i] : C;
    if (cp < t) continue;
    if (window > 0 && window <= cp + sink) continue;
    *mode = CPA_TAIL_PADDED;
    *c_pad = cp;
    return CPA_OK;
  }
  return force == CPA_TAIL_FORCE_PADDED ? CPA_ERR_WINDOW_TOO_SMALL : CPA_OK;
}

const char* cpa_status_str(cpa_status s) {
  switch (s) {
    case CPA_OK: return "ok";
    case CPA_ERR_NULL: return "a required pointer is NULL";
    case CPA_ERR_SHAPE: return "a size is out of range or inconsistent";
    case CPA_ERR_ALIGN: return "a pointer or stride is misaligned";
    case CPA_ERR_UNSUPPORTED: return "unsupported configuration";
    case CPA_ERR_WINDOW_TOO_SMALL: return "sliding window too small for a padded append (W <= C + S)";
    case CPA_ERR_WORKSPACE: return "workspace or scratch too small";
    case CPA_ERR_CUDA: return "CUDA launch error";
  }
  return "unknown status";
}

const char* cpa_version(void) { return "cpa 0.1 (sm_103a)"; }

#ifdef CPA_TEST_HOOKS
void cpa_test_drop_tile(int tile) { g_test_drop_tile.store(tile, std::memory_order_relaxed); }
#endif

}  // extern "C"
