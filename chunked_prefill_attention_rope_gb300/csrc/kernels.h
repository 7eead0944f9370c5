// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/cpa.h"

namespace cpa {

// Raises a kernel's dynamic shared-memory limit once per device.  The
// attribute belongs to the current device's context, so each device keeps
// its own bit (devices 0-63; beyond that the attribute is set on every
// launch).  Two host threads racing on one device both set it, which is
// harmless.
struct SmemAttr {
  std::atomic<uint64_t> done{0};
  cudaError_t ensure(const void* kern, int bytes, bool nonportable_cluster = false) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t(1) << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && nonportable_cluster)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
  }
};

// Workspace bytes the attention call described by `a` needs, sized for its
// own sm_budget (0 for sizes the call would reject).  This is the minimum: an
// explicit mask on the two-tile path runs faster with more (see
// cpa_attn_workspace_size_mask).
size_t attn_workspace_need(const cpa_attn_args* a);

// Launch `kern` as a programmatic dependent of the grid before it on the
// stream: it may start while that grid runs and must call
// grid_dependency_wait() before reading that grid's results.
template <typename... Params, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

struct AttnParams {
  int B, Hq, Hkv, D, C, P, G, R, nq, splits;
  float sl2;  // softmax scale * log2(e)
  const uint16_t* q;
  const float* cos;
  const float* sin;
  const float* mask;
  const int32_t* past_len;
  const int32_t* n_real;
  const int32_t* sel_row;
  int window, causal;
  int sink;  // implicit mask: past slots [0, sink) stay visible whatever the window
  uint16_t* out;
  float* out_sel;
  float* part_o;    // split-KV partials [splits][B][Hq][C][D] or null
  float* part_lse;  // [splits][B][Hq][C]
  int32_t* err;
  // persistent team-aligned stream-K path (two query tiles per work unit)
  int32_t* ustart;  // [blocks + 1] exclusive prefix sum of block costs, in walk order
  int perm;         // blocks walked in the planned order uorder, team ranges in tlo
  int32_t* uorder;  // [blocks] block at each walk position (perm)
  int32_t* upos;    // [blocks] walk position of each block (perm)
  int32_t* tlo;     // [teams + 3] first cost position of each team's range, the total,
                    // then 1 when whole blocks were dealt, then whether a block is empty (perm)
  int units;        // B * Hkv * pairs
  int pairs;        // query-tile pairs per (sequence, kv head)
  int team;         // CTAs per team = pairs per block
  int nblk;         // blocks per (sequence, kv head)
  int blocks;       // B * Hkv * nblk
  int teams;        // teams of CTAs
  int ctas;         // persistent CTAs = teams * team
  int hold_dependents;  // SM budget below the device: follow-up kernels launch only as the grid ends
  const uint16_t* k_new;  // chunk keys before RoPE [B, Hkv, C, D]
  uint16_t* q_rot;        // rotated queries [B, Hq, C, D] (workspace)
  uint16_t* k_rot;        // rotated chunk keys [B, Hkv, C, D] (workspace)
  int32_t* ptag;          // [2 * ctas] unit of each CTA's partial slots (-1: none)
  int f16;                // fp16 KV cache: every product runs in fp16 (else bf16)
  uint16_t* v_cvt;        // fp16 KV cache: the chunk values in fp16 (workspace)
  int cluster;            // single-tile path: the splits of a query tile form one
                          // thread-block cluster and merge their partials in-kernel
  int dsplit;             // single-tile cluster: 1, or 2 when each split is taken by a
                          // CTA pair that divides D between them for P V and the merge
  // Fused global append (app_n non-null): the rotated chunk keys and the
  // values of rows [0, n_b) go to cache slots [len_b, len_b + n_b) from the
  // RoPE pre-pass; len is advanced after the attention has read it.
  const uint16_t* v_new;  // chunk values [B, Hkv, C, D]
  const int32_t* app_n;   // [B] rows to append, or null
  uint16_t* app_k;
  uint16_t* app_v;
  int64_t app_sb, app_sh, app_ss;  // cache strides in elements
  int32_t* app_len;
  int app_cap;
  // Explicit mask on the two-tile path: mask_scan_kernel classifies every
  // (block, key tile) and the plan visits the tiles between each block's
  // first and last tile holding a visible entry (the implicit mask's tile
  // intervals when the mask is the implicit one written out).
  float inv_scale;   // 1 / softmax scale: a finite bias b enters as s + b / scale
  int ntiles;        // key tiles per block: chunk tiles, then past tiles
  uint8_t* tcls;     // [blocks * ntiles] tile classes (kTileDead / kTileBinary / kTileGeneral)
  int4* hull;        // [blocks] visited tiles: chunk [x, y), past [z, w) in the tile index space
  uint4* mbits;      // [B, Hq, ntiles, C] visibility bits of each row and tile, or null
  // Checked builds: element counts of the buffers whose size the shapes alone
  // do not give, and the test hook.
  long long n_part;     // part_o elements (part_lse holds n_part / D)
  long long n_app;      // fused append: elements the cache's K (and V) view spans
  int test_drop_tile;   // K/V tile whose copy each CTA withholds (-1: none)
};

// Element counts of an attention call's buffers (checked builds).
__host__ __device__ inline long long n_qo(const AttnParams& p) {  // q, out, rotated q
  return static_cast<long long>(p.B) * p.Hq * p.C * p.D;
}
__host__ __device__ inline long long n_chunk(const AttnParams& p) {  // k_new, v_new, rotated k, half v
  return static_cast<long long>(p.B) * p.Hkv * p.C * p.D;
}
__host__ __device__ inline long long n_tab(const AttnParams& p) {  // cos, sin
  return static_cast<long long>(p.B) * p.C * p.D;
}
__host__ __device__ inline long long n_mask(const AttnParams& p) {
  return static_cast<long long>(p.B) * p.Hq * p.C * (static_cast<long long>(p.P) + p.C);
}
__host__ __device__ inline long long n_sel(const AttnParams& p) {  // out_sel
  return static_cast<long long>(p.B) * p.Hq * p.D;
}
__host__ __device__ inline long long n_bits(const AttnParams& p) {  // mbits (uint4)
  return static_cast<long long>(p.B) * p.Hq * p.ntiles * p.C;
}


// Team-aligned stream-K layout for these sizes, and its workspace.
struct PairTeams {
  int pairs, team, nblk, blocks, teams, ctas;
  int perm;  // the plan may reorder blocks (whole-block deal); implicit masks without sinks only
};
PairTeams pair_teams(int B, int Hkv, int nq, int P, int C, int num_sms);
struct PairWorkspace {
  size_t ustart, uorder, upos, tlo, part_o, part_lse, ptag, q_rot, k_rot, v_cvt, tcls, hull, total;
  size_t mbits, total_bits;  // the explicit mask's bit copy goes last: [total, total_bits)
};
PairWorkspace pair_workspace(int B, int Hq, int Hkv, int D, int C, int P, const PairTeams& t);
// maps for the pair path: cache K, cache V, rotated chunk K, chunk V, rotated Q
// (dims {D, C, Hq, B}, box {64, R, G, 1}).
cudaError_t launch_attn_pair5(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream);

int attn_block_n(int D);
// Largest split count whose partials the single-tile kernel merges inside a
// thread-block cluster (portable cluster size).
constexpr int kMaxClusterSplits = 8;
constexpr int kMaxClusterSize = 16;  // CTAs: splits x dsplit
// True when clusters of `cluster_size` single-tile CTAs of head dim D can run
// on the current device (checked once per device and size).
bool attn_cluster_ok(int D, int cluster_size);
// Clusters of that size that can be resident at once (0: none fits).
int attn_max_clusters(int D, int cluster_size);
// True when the two-query-tile kernel (256 packed rows per CTA) serves these sizes.
inline bool attn_uses_pair(int D, int nq) { return (D == 64 || D == 128) && nq >= 2; }
// True when the warp-MMA decode kernel (64-key tiles, G <= 16 rows) serves these sizes.
inline bool attn_uses_decode(int D, int C, int G) { return C == 1 && (D == 64 || D == 128) && G <= 16; }
cudaError_t launch_attn_decode(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream);
// maps: cache K, cache V (dims {D, P, Hkv, B}), chunk K, chunk V (dims {D, C, Hkv, B}),
// all bf16, box {64, block_n, 1, 1}, 128-byte swizzle; for the single-tile
// kernel also raw Q (dims {D, C, Hq, B}, box {64, R, G, 1}).
cudaError_t launch_attn(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream);
// Fused append's length update as a programmatic dependent of the attention.
cudaError_t launch_fused_append_len(const AttnParams& p, cudaStream_t stream);

struct CacheView {
  uint16_t* k;
  uint16_t* v;
  int64_t sb, sh, ss;  // strides in elements
  int32_t* len;
  int cap, window, sink;
  int f16;             // elements are IEEE half (else bf16)
  long long extent;    // elements the K (and V) view spans (checked builds)
  int32_t* err;        // the call's error word (checked builds)
};

struct ChunkView {
  const uint16_t* k;  // [B, Hkv, C, D]
  const uint16_t* v;
  const float* cos;   // [B, C, D]
  const float* sin;
  const int32_t* n_rows;
  long long n_kv, n_tab;  // elements of k (and v) and of cos (and sin) (checked builds)
};

// Scratch layout of a sliding cache (byte offsets from the scratch base).
struct SlidingScratch {
  size_t hdr_append, hdr_snap, hdr_roll, saved_k, saved_v, stage_k, stage_v, total;
};
SlidingScratch sliding_scratch_layout(int B, int Hkv, int D, int C, int W);

cudaError_t launch_global_append(const CacheView& c, const ChunkView& x, int B, int Hkv, int D, int C,
                                 int32_t* err, cudaStream_t s);
cudaError_t launch_sliding_append(const CacheView& c, const ChunkView& x, int B, int Hkv, int D, int C,
                                  uint8_t* scratch, int32_t* err, cudaStream_t s);
cudaError_t launch_snapshot(const CacheView& c, const int32_t* n_real, int B, int Hkv, int D, int C,
                            uint8_t* scratch, int32_t* err, cudaStream_t s);
cudaError_t launch_rollback(const CacheView& c, int B, int Hkv, int D, int C, uint8_t* scratch,
                            int32_t* err, cudaStream_t s);

}  // namespace cpa
