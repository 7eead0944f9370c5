// Chunk-prefill attention for head dims 64 and 128: two query tiles per work
// unit, persistent CTAs with stream-K balancing.
//
// Same computation as attn_kernel ("functiongemma: chunk prefill-with-past
// graph", Change: RoPE'd queries attend over past + chunk keys under an
// additive mask), organised for the tensor core:
//
//   * Work unit = 256 packed query rows of one (sequence, kv head): query tiles
//     Q0 and Q1 of 128 rows that share every K/V tile.
//   * Team-aligned stream-K.  The CTAs form teams of `team` CTAs; member m
//     of a team handles pair blk*team + m of each block of pairs of one
//     (sequence, kv head).  The planning CTA of prep_kernel counts the live key tiles of
//     every block (lengths live on the device) and prefix-sums them with a
//     unit-switch cost.  Each team takes an equal contiguous range of that
//     sequence; its members walk the same key tiles of the same block in
//     lockstep, so every K/V tile a team loads is shared through L2 by all
//     the pairs of the block.  A member finishes whole units directly and
//     writes partial results only for the units cut at its team's range ends;
//     merge_units_kernel combines those in fixed order and zero-fills units
//     without live keys.
//   * RoPE: prep_kernel rotates the chunk's queries and keys once per call
//     (coalesced, the same fp32 rounding as the cache append) into the
//     workspace; the attention kernel TMA-loads rotated Q tiles and chunk-K
//     tiles from there, so no tile is rotated twice and no load waits on a
//     table lookup inside the pipeline.
//   * TMEM (512 columns): S0 [0,128), S1 [128,256), O0 and O1 after them.  P
//     (bf16) is written back over the first 64 columns of its S buffer and fed
//     to the P V product straight from tensor memory.
//   * The MMA warp interleaves the two tiles: while softmax 0 works on S0 of
//     key tile j, the tensor core runs P1 V(j-1) and S1 = Q1 K(j), and vice versa.
//   * Softmax loads a row of S from TMEM in one batch, takes the row max with
//     three-input max, and forms 2^(scale*log2e*s - m) with one packed fused
//     multiply-add per two scores (masked scores are -inf and give exactly 0).
//
// Warps: 0-3 softmax for Q0, 4-7 softmax for Q1 (warp w owns TMEM lanes
// 32*(w%4)..+31), 8 K/V TMA producer, 9 MMA issuer, 10 Q TMA loader, 11 idle
// (it completes the aux warpgroup for the register split).  Every
// role walks the same segment sequence and counts tiles globally, so barrier
// phases carry across unit boundaries.
#include <type_traits>

#include "tiles.cuh"

namespace cpa {

namespace {

constexpr int kBN = 128;
constexpr int kThreadsPair = 384;
// Register split (setmaxnreg): the launch gives every thread 168 registers
// (384 x 168 = 64512).  The aux warpgroup (warps 8-11) drops to 96 (104 at
// D = 128, whose producer and MMA issuer keep more state), freeing 128 x 72
// = 9216 (128 x 64 = 8192); the two softmax warpgroups rise to 200, taking
// 2 x 128 x 32 = 8192, so the increase never waits on the pool.
constexpr int kRegsSoftmax = 200;
template <int D>
struct RegsAux {
  static constexpr int value = D == 128 ? 104 : 96;
};
static_assert(2 * 128 * (kRegsSoftmax - 168) <= 128 * (168 - RegsAux<128>::value), "register split");
constexpr int kUnitRows = 256;
// A unit switch (Q reload, epilogue, pipeline refill) costs about this many key
// tiles (per-CTA cycle counts fitted over key tiles and segments: ~3); the
// stream-K split charges it to every non-empty unit.
constexpr int kSwitchCost = 3;
// A cut unit costs its second piece another switch and goes through the merge
// kernel; a plan that deals whole blocks is kept while its busiest team has at
// most this many key tiles more than the even split's share.
constexpr int kCutCost = 2 * kSwitchCost;
// Whole-block deal: key tiles prefetched into L2 this far ahead of the copies.
constexpr int kPrefetchTiles = 4;

template <int D>
struct PairCfg {
  static constexpr int kStages = D == 64 ? 4 : 2;
  static constexpr int kQBytes = 128 * D * 2;
  static constexpr int kKBytes = kBN * D * 2;
  static constexpr int kVBytes = kBN * D * 2;
  static constexpr int kQ = 0;  // Q0, then Q1
  static constexpr int kK = 2 * kQBytes;
  static constexpr int kV = kK + kStages * kKBytes;
  static constexpr int kBars = kV + kStages * kVBytes;
  static constexpr int kOCol = 2 * kBN;  // O0 at [256, 256 + D), O1 at [256 + D, 256 + 2D)
  static_assert(kOCol + 2 * D <= 512, "TMEM columns");
  // a 4 KB staging tile per softmax warp (32 rows x 32 fp32 columns) for the
  // epilogue's coalesced stores
  static constexpr int kStage = kBars + 256;
  static constexpr int kStageEnd = kStage + 8 * 32 * 32 * 4;
};

struct __align__(8) PairBars {
  uint64_t k_full[4], v_full[4], kv_empty[4];
  uint64_t k_empty[4];  // K stage free (its S = Q K products done); kv_empty then frees V only
  uint64_t v_ready[4];  // implicit mask: V tile landed and its dead rows cleared (warp 11)
  uint64_t s_full[2], p_full[2], o_done[2], q_full[2], q_free[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

template <int D>
constexpr int pair_smem_bytes() {
  static_assert(sizeof(PairBars) <= 256, "barrier block");
  return PairCfg<D>::kStageEnd + 1024;
}
static_assert(pair_smem_bytes<128>() <= 227 * 1024, "shared memory");

struct Unit {
  int b, kvh, pair;
};

// Block g = (b, kvh, blk): pairs [blk*team, (blk+1)*team) of one (sequence, kv head).
struct Block {
  int b, kvh, blk;
};

__device__ __forceinline__ Block block_of(const AttnParams& p, int g) {
  Block x;
  x.blk = g % p.nblk;
  x.kvh = (g / p.nblk) % p.Hkv;
  x.b = g / (p.nblk * p.Hkv);
  return x;
}

__device__ __forceinline__ int block_index(const AttnParams& p, const Block& x) {
  return (x.b * p.Hkv + x.kvh) * p.nblk + x.blk;
}

// Live key tiles of all rows of a block: the tiles its members walk together.
// Explicit mask: the chunk tiles and the past tiles from the first to the
// last one holding a visible entry for some row of the block (mask_scan_kernel
// and the plan find them); for a mask that writes out the implicit one these
// are exactly the implicit mask's tile intervals, so both forms visit the same
// tiles and split the work alike.
__device__ __forceinline__ TilePlan block_plan(const AttnParams& p, const Block& x) {
  const int i_min = x.blk * p.team * 2 * p.R;
  const int i_max = min(i_min + p.team * 2 * p.R, p.C) - 1;
  TilePlan t = plan_whole<kBN>(p, x.b, i_min, i_max);
  if (p.mask) {
    const int gi = block_index(p, x);
    const int4 h = in_bounds(gi, 1, p.blocks, p.err) ? p.hull[gi] : make_int4(0, 0, t.Tc, t.Tc);
    t.cb = h.x;
    t.ce = h.y;
    t.pb = h.z;
    t.pe = h.w;
  }
  return t;
}

__device__ __forceinline__ Unit unit_of(const AttnParams& p, int u) {
  Unit x;
  x.pair = u % p.pairs;
  x.kvh = (u / p.pairs) % p.Hkv;
  x.b = u / (p.pairs * p.Hkv);
  return x;
}

__device__ __forceinline__ int unit_id(const AttnParams& p, int b, int kvh, int pair) {
  return (b * p.Hkv + kvh) * p.pairs + pair;
}

// First tile of CTA c's range in the concatenated tile sequence of T tiles.
__device__ __forceinline__ long long cta_lo(long long T, int c, int ctas) { return T * c / ctas; }

// Largest u in [0, U) with start[u] <= x (the unit holding tile x when x < T).
__device__ __forceinline__ int unit_at(const int32_t* start, int U, long long x) {
  int lo = 0, hi = U - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (start[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Walks the (block, first tile, end tile) segments of a team's range of cost
// positions, for one member: segments whose pair does not exist are skipped.
// PERM: the blocks are walked in the planned order p.uorder and team t's
// range is [p.tlo[t], p.tlo[t + 1]) (a whole-block deal or the even split);
// otherwise blocks are in index order and the ranges split the costs evenly.
template <bool PERM>
struct SegWalk {
  using Pos = typename std::conditional<PERM, int, long long>::type;  // tlo holds 32-bit positions
  const int32_t* start;
  int NB, g, member;
  Pos lo, hi;
  const AttnParams* pp;
  __device__ __forceinline__ void init(const AttnParams& p, int cta) {
    pp = &p;
    start = p.ustart;
    NB = p.blocks;
    member = cta % p.team;
    const int t = cta / p.team;
    if (PERM) {
      lo = p.tlo[t];
      hi = p.tlo[t + 1];
    } else {
      const long long T = start[NB];
      lo = cta_lo(T, t, p.teams);
      hi = cta_lo(T, t + 1, p.teams);
    }
    g = lo < hi ? unit_at(start, NB, lo) : NB;
  }
  // Next segment holding at least one key tile of this member's unit; false
  // when the range is exhausted.  Block g spans cost positions
  // [start[g], start[g+1]): first the switch cost, then one per key tile.
  __device__ __forceinline__ bool next(int& unit, Block& blk, int& a, int& e) {
    while (g < NB && start[g] < hi) {
      const Pos t0 = start[g] + kSwitchCost, s1 = start[g + 1];
      const int cur = g++;
      const Pos aa = lo > t0 ? lo : t0;
      const Pos ee = hi < s1 ? hi : s1;
      if (ee <= aa) continue;
      const int gb = PERM ? pp->uorder[cur] : cur;
      if (!in_bounds(gb, 1, NB, pp->err)) continue;
      const Block x = block_of(*pp, gb);
      const int pair = x.blk * pp->team + member;
      if (pair >= pp->pairs) continue;
      blk = x;
      unit = unit_id(*pp, x.b, x.kvh, pair);
      a = static_cast<int>(aa - t0);
      e = static_cast<int>(ee - t0);
      return true;
    }
    return false;
  }
};

}  // namespace

constexpr int kPrepThreads = 256;
constexpr int kPrepHeads = 4;  // heads rotated per item with one table load (two CTAs per SM)

// Blocks the whole-block plan can order (their costs sit in shared memory).
constexpr int kPlanSortMax = 1024;

// Key tiles of block u plus the switch cost (0 for a block without live tiles).
// The first block of each sequence also checks the sequence's lengths, which
// the plan loads here anyway.
__device__ __forceinline__ int block_cost(const AttnParams& p, int u) {
  const Block x = block_of(p, u);
  if (x.kvh == 0 && x.blk == 0) {
    if (p.past_len && (p.past_len[x.b] < 0 || p.past_len[x.b] > p.P)) set_err(p.err, CPA_EBIT_PAST_GT_SPAN);
    if (p.n_real && (p.n_real[x.b] < 0 || p.n_real[x.b] > p.C)) set_err(p.err, CPA_EBIT_NREAL_GT_C);
  }
  const int n = block_plan(p, x).count();
  return n > 0 ? n + kSwitchCost : 0;
}

// Exclusive prefix sum of cost(k) over k in [0, n) into out[0..n] (out[n] =
// total), by one CTA of kPrepThreads threads; returns the total.
template <typename Cost>
__device__ int prefix_costs(int n, Cost cost, int32_t* out) {
  __shared__ int32_t warp_sums[kPrepThreads / 32];
  __shared__ int32_t carry;
  constexpr int kWarps = kPrepThreads / 32;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
  for (int base = 0; base < n; base += kPrepThreads) {
    const int u = base + threadIdx.x;
    const int c = u < n ? cost(u) : 0;
    int incl = c;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int w = lane < kWarps ? warp_sums[lane] : 0;
#pragma unroll
      for (int o = 1; o < kWarps; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += v;
      }
      if (lane < kWarps) warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + carry;
    if (u < n) out[u] = before + incl - c;
    __syncthreads();
    if (threadIdx.x == kPrepThreads - 1) carry = before + incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) out[n] = carry;
  return carry;
}

// First position of team t's blocks when `nb` blocks, sorted by cost, are
// dealt to `teams` teams in rounds of alternating direction (round r gives
// sorted position r*teams + j to team j, or to team teams-1-j when r is odd).
__device__ __forceinline__ int deal_start(int t, int nb, int teams) {
  const int R = nb / teams, rem = nb % teams;
  return t * R + ((R & 1) == 0 ? min(t, rem) : max(0, t - (teams - rem)));
}

// Cost of every block (its live key tiles plus the switch cost) and the
// exclusive prefix sum of the costs, by one CTA of kPrepThreads threads.
// With p.perm, blocks are first dealt whole to the teams, largest first in
// rounds of alternating direction; that deal is kept when its busiest team
// carries at most the even split's share plus kCutCost, and then no unit is
// cut (no partial rows, nothing to merge).  Otherwise, and always without
// p.perm, the teams split the costs in index order evenly.  With p.perm the
// walk order goes to p.uorder (and its inverse to p.upos) and the team ranges
// to p.tlo.
__device__ void plan_units(const AttnParams& p) {
  if (!p.perm) {
    prefix_costs(p.blocks, [&](int u) { return block_cost(p, u); }, p.ustart);
    return;
  }
  __shared__ int32_t cost[kPlanSortMax];
  __shared__ int32_t order[kPlanSortMax];
  __shared__ int32_t total, biggest, busiest;
  const int NB = p.blocks, teams = p.teams;  // NB <= kPlanSortMax (host)
  if (threadIdx.x == 0) {
    total = 0;
    biggest = 0;
    busiest = 0;
  }
  __syncthreads();
  int sum = 0, mx = 0;
  for (int u = threadIdx.x; u < NB; u += kPrepThreads) {
    const int c = block_cost(p, u);
    cost[u] = c;
    sum += c;
    mx = max(mx, c);
  }
  atomicAdd(&total, sum);
  atomicMax(&biggest, mx);
  __syncthreads();
  const int T = total;
  const int even = (T + teams - 1) / teams + kCutCost;
  bool whole = biggest <= even;
  if (whole) {
    for (int u = threadIdx.x; u < NB; u += kPrepThreads) {
      const int c = cost[u];
      int rank = 0;  // position in decreasing cost, ties by block index
      for (int v = 0; v < NB; ++v) rank += (cost[v] > c) || (cost[v] == c && v < u);
      const int r = rank / teams, j = rank % teams;
      order[deal_start((r & 1) ? teams - 1 - j : j, NB, teams) + r] = u;
    }
    __syncthreads();
    int worst = 0;
    for (int t = threadIdx.x; t < teams; t += kPrepThreads) {
      int load = 0;
      for (int k = deal_start(t, NB, teams), e = deal_start(t + 1, NB, teams); k < e; ++k) load += cost[order[k]];
      worst = max(worst, load);
    }
    atomicMax(&busiest, worst);
    __syncthreads();
    whole = busiest <= even;  // the same value in every thread
  }
  if (!whole) {
    for (int k = threadIdx.x; k < NB; k += kPrepThreads) order[k] = k;
    __syncthreads();
  }
  for (int k = threadIdx.x; k < NB; k += kPrepThreads) {
    p.uorder[k] = order[k];
    st_chk(p.upos, order[k], NB, k, p.err);
  }
  prefix_costs(NB, [&](int k) { return cost[order[k]]; }, p.ustart);
  __syncthreads();  // ustart, written by other threads of this CTA
  for (int t = threadIdx.x; t <= teams; t += kPrepThreads)
    p.tlo[t] = t == teams ? T
                          : (whole ? p.ustart[deal_start(t, NB, teams)]
                                   : static_cast<int32_t>(static_cast<long long>(T) * t / teams));
  int empty = 0;  // blocks without a live key tile (their units are zero-filled by the merge)
  for (int u = threadIdx.x; u < NB; u += kPrepThreads) empty += cost[u] == 0;
  empty = __syncthreads_count(empty > 0);
  if (threadIdx.x == 0) {
    p.tlo[teams + 1] = whole ? 1 : 0;  // whole blocks: no unit is cut
    p.tlo[teams + 2] = empty;          // threads that saw an empty block
  }
}

// Classes of a key tile of one block under an explicit mask.
enum : uint8_t {
  kTileDead = 0,     // no entry above -1e29 (every key masked for every row)
  kTileBinary = 1,   // every entry 0 or at most -1e29: the pages' 0 / -1e30 form
  kTileGeneral = 2,  // some entry is a finite bias (or not a number)
};

constexpr int kScanThreads = 256;
constexpr int kScanBatch = 8;  // mask rows a warp has in flight

// Explicit mask pre-pass of the two-tile path.  One CTA per (block, key
// tile) reads that tile's entries of every mask row of the block once: a
// warp takes one row's 128 keys per load, four consecutive keys per lane.
// It records the tile's class and, when p.mbits is set, each row's
// visibility bits: word j, bit l holds key 4 l + j of the tile, set when the
// entry is exactly 0 (the attention tests bit (q % 4, q / 4) for key q).
// Keys past the row's end (P or C) read as masked.
__global__ void __launch_bounds__(kScanThreads, 4) mask_scan_kernel(const AttnParams p) {
  grid_launch_dependents();
  grid_dependency_wait();  // the mask may come from the work before this call
  const int T = p.ntiles;
  const int g = blockIdx.x / T, t = blockIdx.x % T;
  const Block x = block_of(p, g);
  const int Tc = (p.C + kBN - 1) / kBN;
  const bool chunk = t < Tc;
  const int base = (chunk ? t : t - Tc) * kBN;
  const int lim = (chunk ? p.C : p.P) - base;
  const size_t moff = chunk ? static_cast<size_t>(p.P) + base : static_cast<size_t>(base);
  const size_t stride = static_cast<size_t>(p.P) + p.C;
  const int i0 = x.blk * p.team * 2 * p.R;
  const int ni = min(i0 + p.team * 2 * p.R, p.C) - i0;  // chunk rows of the block
  const int rows = p.G * ni;                             // mask rows: heads x chunk rows
  const bool vec = (p.P % 4 == 0) && (p.C % 4 == 0);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int k0 = 4 * lane;
  bool live = false, general = false;
  for (int r0 = warp * 32; r0 < rows; r0 += kScanThreads) {
    // lane l owns row r0 + l: its head and chunk row, and its offset in the
    // mask (one division per 32 rows; each row's offset reaches the warp by
    // shuffle)
    const int rl = r0 + lane;
    const int hl = x.kvh * p.G + rl / ni, il = i0 + rl % ni;
    const long long ro_l = (static_cast<long long>(x.b * p.Hq + hl) * p.C + il) * stride + moff;
    uint4 mine = make_uint4(0u, 0u, 0u, 0u);  // bits of row r0 + lane
    for (int j0 = 0; j0 < 32 && r0 + j0 < rows; j0 += kScanBatch) {
      float v[kScanBatch][4];
#pragma unroll
      for (int u = 0; u < kScanBatch; ++u) {
        const long long ro = __shfl_sync(0xffffffffu, ro_l, j0 + u);
        v[u][0] = v[u][1] = v[u][2] = v[u][3] = -1e30f;
        if (r0 + j0 + u < rows && in_bounds(ro, lim, n_mask(p), p.err)) {
          const float* row = p.mask + ro;
          if (vec) {
            if (k0 < lim) {
              const float4 f = __ldg(reinterpret_cast<const float4*>(row + k0));
              v[u][0] = f.x;
              v[u][1] = f.y;
              v[u][2] = f.z;
              v[u][3] = f.w;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (k0 + e < lim) v[u][e] = __ldg(row + k0 + e);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kScanBatch; ++u) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float m = v[u][e];
          live |= m > -1e29f;
          general |= !(m == 0.f || m <= -1e29f);
          w[e] = __ballot_sync(0xffffffffu, m == 0.f);
        }
        if (lane == j0 + u) mine = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    if (p.mbits && rl < rows)
      st_chk(p.mbits, (static_cast<long long>(x.b * p.Hq + hl) * T + t) * p.C + il, n_bits(p), mine, p.err);
  }
  live = __syncthreads_or(live);
  general = __syncthreads_or(general);
  if (threadIdx.x == 0) p.tcls[blockIdx.x] = !live ? kTileDead : (general ? kTileGeneral : kTileBinary);
}

// Explicit mask: each block's visited tiles (first to last non-dead chunk
// tile, and likewise for the past tiles) from the scan's classes, by one CTA
// of kPrepThreads threads, before the plan prices the blocks.
__device__ void explicit_hulls(const AttnParams& p) {
  const int T = p.ntiles, Tc = (p.C + kBN - 1) / kBN;
  for (int g = threadIdx.x; g < p.blocks; g += kPrepThreads) {
    const uint8_t* c = p.tcls + static_cast<size_t>(g) * T;
    int cb = 0, ce = 0, pb = Tc, pe = Tc;
    for (int t = 0; t < Tc; ++t)
      if (c[t] != kTileDead) {
        if (ce == 0) cb = t;
        ce = t + 1;
      }
    for (int t = Tc; t < T; ++t)
      if (c[t] != kTileDead) {
        if (pe == Tc) pb = t;
        pe = t + 1;
      }
    p.hull[g] = make_int4(cb, ce, pb, pe);
  }
  __syncthreads();  // the hulls, read by other threads of this CTA
}

// CTA 0 plans (plan_units); the others rotate the chunk's queries and
// keys into the workspace.  An item is one (sequence, chunk row, chunk pair)
// and up to four heads of the combined list [query heads, key heads]: the
// table values of its row are loaded once and the four heads' loads are
// issued together.  A warp covers four consecutive rows of each head, so
// every load and store is a contiguous 512-byte run per head.
__global__ void __launch_bounds__(kPrepThreads, 2) prep_kernel(const AttnParams p) {
  grid_launch_dependents();
  grid_dependency_wait();  // launched as a dependent: whatever the launches before it wrote
  if (blockIdx.x == 0) {  // the first CTA to start plans, alongside the rotations
    if (p.mask) explicit_hulls(p);
    plan_units(p);
    // and marks the attention's partial-result slots empty (it reads them
    // only after waiting for this grid)
    for (int k = threadIdx.x; k < 2 * p.ctas; k += blockDim.x) st_chk(p.ptag, k, 2LL * p.ctas, -1, p.err);
    return;
  }
  const int D = p.D;
  const int HP = D / 16;  // 8-element chunk pairs (d, d + D/2) per row: 4, 8 or 16
  const int hp_shift = D == 64 ? 2 : (D == 128 ? 3 : 4);
  const int HH = p.Hq + p.Hkv;
  const int groups = (HH + kPrepHeads - 1) / kPrepHeads;
  // item index in 32 bits (the host keeps B * groups * C * HP below 2^31):
  // a 64-bit division per item had made this pass issue-bound
  const unsigned total = static_cast<unsigned>(p.B) * groups * p.C * HP;
  const unsigned stride = (gridDim.x - 1) * blockDim.x;
  for (unsigned it = (blockIdx.x - 1) * blockDim.x + threadIdx.x; it < total; it += stride) {
    const int kc = static_cast<int>(it & (HP - 1));
    unsigned t = it >> hp_shift;
    const unsigned Cu = static_cast<unsigned>(p.C);
    const int i = static_cast<int>(t % Cu);
    t /= Cu;
    const int grp = static_cast<int>(t % static_cast<unsigned>(groups));
    const int b = static_cast<int>(t / static_cast<unsigned>(groups));
    const float* cr = p.cos + (static_cast<size_t>(b) * p.C + i) * D;
    const float* sr = p.sin + (static_cast<size_t>(b) * p.C + i) * D;
    if (!in_bounds((static_cast<long long>(b) * p.C + i) * D, D, n_tab(p), p.err)) continue;
    const RopeTab tab = rope_tab(cr + kc * 8, sr + kc * 8, cr + D / 2 + kc * 8, sr + D / 2 + kc * 8);
    uint4 lo[kPrepHeads], hi[kPrepHeads];
    size_t off[kPrepHeads];
#pragma unroll
    for (int u = 0; u < kPrepHeads; ++u) {
      const int hh = grp * kPrepHeads + u;
      if (hh >= HH) break;
      const bool is_q = hh < p.Hq;
      off[u] = is_q ? ((static_cast<size_t>(b) * p.Hq + hh) * p.C + i) * D
                    : ((static_cast<size_t>(b) * p.Hkv + (hh - p.Hq)) * p.C + i) * D;
      const uint16_t* src = (is_q ? p.q : p.k_new) + off[u];
      if (!in_bounds(static_cast<long long>(off[u]), D, is_q ? n_qo(p) : n_chunk(p), p.err)) {
        off[u] = ~size_t(0);  // skipped below
        lo[u] = hi[u] = make_uint4(0, 0, 0, 0);
        continue;
      }
      lo[u] = __ldg(reinterpret_cast<const uint4*>(src + kc * 8));
      hi[u] = __ldg(reinterpret_cast<const uint4*>(src + D / 2 + kc * 8));
    }
#pragma unroll
    for (int u = 0; u < kPrepHeads; ++u) {
      const int hh = grp * kPrepHeads + u;
      if (hh >= HH) break;
      if (kChecked && off[u] == ~size_t(0)) continue;
      if (p.f16) {
        rope_apply<true>(lo[u], hi[u], tab);
        if (hh >= p.Hq) {  // an fp16 cache: the chunk's values in half too
          const uint16_t* vs = p.v_new + off[u];
          uint16_t* vd = p.v_cvt + off[u];
          *reinterpret_cast<uint4*>(vd + kc * 8) = bf16x8_to_f16x8(__ldg(reinterpret_cast<const uint4*>(vs + kc * 8)));
          *reinterpret_cast<uint4*>(vd + D / 2 + kc * 8) =
              bf16x8_to_f16x8(__ldg(reinterpret_cast<const uint4*>(vs + D / 2 + kc * 8)));
        }
      } else {
        rope_apply(lo[u], hi[u], tab);
      }
      uint16_t* dst = (hh < p.Hq ? p.q_rot : p.k_rot) + off[u];
      *reinterpret_cast<uint4*>(dst + kc * 8) = lo[u];
      *reinterpret_cast<uint4*>(dst + D / 2 + kc * 8) = hi[u];
      if (p.app_n && hh >= p.Hq) fused_append_pair(p, b, hh - p.Hq, i, kc, lo[u], hi[u]);
    }
  }
}

// Explicit mask values of keys [k0, k0 + 32) of a tile for this thread's row
// (`mp`: the row at the tile's first key, or null), -1e30 at or past `lim`.
// `vec`: P and C are multiples of 4, so each row starts 16-byte aligned and no
// 16-byte vector straddles `lim`.  Checked builds: `mo` is mp's element
// offset in the mask of `mn` elements.
__device__ __forceinline__ void load_mask32(float (&mv)[32], const float* mp, int k0, int lim, bool vec,
                                            long long mo, long long mn, int32_t* err) {
  if (mp && k0 < lim && !in_bounds(mo + k0, min(32, lim - k0), mn, err)) mp = nullptr;
  if (vec) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float4 v = make_float4(-1e30f, -1e30f, -1e30f, -1e30f);
      if (mp && k0 + 4 * k < lim) v = __ldg(reinterpret_cast<const float4*>(mp + k0 + 4 * k));
      mv[4 * k] = v.x;
      mv[4 * k + 1] = v.y;
      mv[4 * k + 2] = v.z;
      mv[4 * k + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 32; ++q) mv[q] = (mp && k0 + q < lim) ? __ldg(mp + k0 + q) : -1e30f;
  }
}

// Where tile `t` of the plan starts in a mask row (`moff`) and how many of
// its keys the row holds (`lim`: keys at or past it are outside the row).
__device__ __forceinline__ void mask_span(const AttnParams& p, const TilePlan& tp, int t, size_t& moff, int& lim) {
  const bool chunk = t < tp.Tc;
  const int base = (chunk ? t : t - tp.Tc) * kBN;
  lim = chunk ? p.C - base : p.P - base;
  moff = chunk ? static_cast<size_t>(p.P) + base : static_cast<size_t>(base);
}

// SINK: the implicit mask also keeps pinned sink slots visible (a separate
// instantiation, so the common case carries none of that code).  F16: an
// fp16 KV cache, every product in fp16.
template <int D, bool EXPLICIT, bool SINK, bool F16, bool PERM>
__global__ void __launch_bounds__(kThreadsPair, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap map_kc, const __grid_constant__ CUtensorMap map_vc,
                     const __grid_constant__ CUtensorMap map_kn, const __grid_constant__ CUtensorMap map_vn,
                     const __grid_constant__ CUtensorMap map_q, const AttnParams p) {
  using CF = PairCfg<D>;
  constexpr int NS = CF::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PairBars* bars = reinterpret_cast<PairBars*>(smem + CF::kBars);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_ready[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 128);
      mbar_init(&bars->o_done[s], 1);
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_free[s], 128);
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  // the merge grid may be scheduled now (on a partial SM budget only as this
  // grid ends, leaving the other SMs to other streams); this grid's inputs
  // (plan, rotated Q and keys) come from prep_kernel, launched just before it
  if (!p.hold_dependents) grid_launch_dependents();
  // Global memory only after this wait: until it returns, launches before the
  // one just ahead of this grid (a previous call's work on the same
  // workspace or cache) may still be running.
  grid_dependency_wait();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  uint8_t* sK = smem + CF::kK;
  uint8_t* sV = smem + CF::kV;
  SegWalk<PERM> walk;
  walk.init(p, cta);

  if (warp >= 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(RegsAux<D>::value));
  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&map_kc);
      prefetch_tensormap(&map_vc);
      prefetch_tensormap(&map_kn);
      prefetch_tensormap(&map_vn);
      int g = 0;  // tiles issued (chunk keys come from the rotated copy behind map_kn)
      bool ok = true;
      int unit, a, e;
      Block bx;
      while (ok && walk.next(unit, bx, a, e)) {
        const Unit x = unit_of(p, unit);
        const TilePlan tp = block_plan(p, bx);
        for (int j = a; j < e; ++j, ++g) {
          const int st = g % NS;
          if (!(ok = mbar_wait(&bars->k_empty[st], ((g / NS) + 1) & 1, abort))) break;
          // checked build's test hook: no copy for this tile, so that the
          // consumer's bounded wait for it runs out
          if (kTestHooks && g == p.test_drop_tile) continue;
          const int t = tp.index(j);
          const bool chunk = t < tp.Tc;
          const int base = (chunk ? t : t - tp.Tc) * kBN;
          const CUtensorMap* mk = chunk ? &map_kn : &map_kc;
          const CUtensorMap* mv = chunk ? &map_vn : &map_vc;
          mbar_arrive_expect_tx(&bars->k_full[st], CF::kKBytes);
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk)
            tma_load_4d(sK + st * CF::kKBytes + blk * kBN * 128, mk, &bars->k_full[st], blk * 64, base, x.kvh, x.b);
          if (!(ok = mbar_wait(&bars->kv_empty[st], ((g / NS) + 1) & 1, abort))) break;
          mbar_arrive_expect_tx(&bars->v_full[st], CF::kVBytes);
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk)
            tma_load_4d(sV + st * CF::kVBytes + blk * kBN * 128, mv, &bars->v_full[st], blk * 64, base, x.kvh, x.b);
          if (PERM) {
            // Short segments whose tiles come cold from HBM: prefetch the
            // segment's next tiles into L2 (a few tiles ahead of the copies)
            for (int jp = (j == a ? j + 1 : j + kPrefetchTiles); jp <= j + kPrefetchTiles && jp < e; ++jp) {
              const int t2 = tp.index(jp);
              const bool chunk2 = t2 < tp.Tc;
              const int base2 = (chunk2 ? t2 : t2 - tp.Tc) * kBN;
#pragma unroll
              for (int blk = 0; blk < D / 64; ++blk) {
                tma_prefetch_4d(chunk2 ? &map_kn : &map_kc, blk * 64, base2, x.kvh, x.b);
                tma_prefetch_4d(chunk2 ? &map_vn : &map_vc, blk * 64, base2, x.kvh, x.b);
              }
            }
          }
        }
      }
      for (int j = max(0, g - NS); j < g; ++j) {  // let copies in flight land
        const int st = j % NS;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&bars->v_full[st], (j / NS) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
        while (!mbar_try_wait(&bars->k_full[st], (j / NS) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the tiles and waits, so that every descriptor and
    // TMEM address is a warp-uniform value; one lane, elected once, issues the
    // MMAs and their commits (a commit tracks the MMAs of the lane that
    // issues it).  Issuing from a lane-0-only loop instead cost ~64 clocks per
    // MMA, as much as an MMA's tensor work at N = 128.
    {
      const bool leader = elect_lane();
      constexpr uint32_t idesc_qk = idesc_16(128, kBN, false, F16);
      constexpr uint32_t idesc_pv = idesc_16(128, D, true, F16);
      const uint32_t q_addr = smem_u32(smem + CF::kQ);
      int g = 0, seg = 0;
      bool ok = true;
      auto k_ready = [&](const TilePlan&, int, int gg) -> bool {
        return warp_all(mbar_wait(&bars->k_full[gg % NS], (gg / NS) & 1, abort));
      };
      // Descriptors are formed once; the MMAs of a group step through them by
      // constant offsets (the start-address field is address / 16).
      const uint64_t qd0 = sdesc_sw128(q_addr, 16, 1024);
      const uint64_t kd0 = sdesc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t vd0 = sdesc_sw128(smem_u32(sV), kBN * 128, 1024);
      auto issue_qk = [&](int i, int gg) {
        const uint64_t qd = qd0 + static_cast<uint64_t>(i * (CF::kQBytes >> 4));
        const uint64_t kd = kd0 + static_cast<uint64_t>((gg % NS) * (CF::kKBytes >> 4));
        const uint32_t d_tm = tmem + i * kBN;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t qo = ((kk / 4) * (128 * 128) + (kk % 4) * 32) >> 4;
            const uint32_t ko = ((kk / 4) * (kBN * 128) + (kk % 4) * 32) >> 4;
            mma_bf16_ss(d_tm, qd + qo, kd + ko, idesc_qk, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[i]);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int i, int gg, bool first) {
        const uint64_t vd = vd0 + static_cast<uint64_t>((gg % NS) * (CF::kVBytes >> 4));
        const uint32_t d_tm = tmem + CF::kOCol + i * D;
        const uint32_t p_tm = tmem + i * kBN;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_bf16_ts(d_tm, p_tm + kk * 8, vd + static_cast<uint32_t>((kk * 2048) >> 4), idesc_pv,
                        (!first || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
      };
      auto commit = [&](uint64_t* bar) {
        if (leader) mma_commit(bar);
        __syncwarp();
      };
      int unit, a, e;
      Block bx;
      while (ok && walk.next(unit, bx, a, e)) {
        const TilePlan tp = block_plan(p, bx);
        const int n = e - a;
        if (!(ok = k_ready(tp, a, g) && warp_all(mbar_wait(&bars->q_full[0], seg & 1, abort)))) break;
        tc_fence_after();
        issue_qk(0, g);
        if (!(ok = warp_all(mbar_wait(&bars->q_full[1], seg & 1, abort)))) break;
        tc_fence_after();
        issue_qk(1, g);
        commit(&bars->k_empty[g % NS]);
        for (int jj = 0; jj < n; ++jj) {
          const int gt = g + jj;
          const int st = gt % NS;
          // V of this tile and K of the next: waited for while the softmax
          // still works on S (a wait costs the issuer ~200 clocks even on a
          // completed barrier), so that P alone gates the products below.
          // The next K is there by then: its stage was freed after the S = Q K
          // products of the tile before this one.
          if (!(ok = warp_all(mbar_wait(EXPLICIT ? &bars->v_full[st] : &bars->v_ready[st], (gt / NS) & 1, abort))))
            break;
          if (jj + 1 < n && !(ok = k_ready(tp, a + jj + 1, gt + 1))) break;
          if (!(ok = warp_all(mbar_wait(&bars->p_full[0], gt & 1, abort)))) break;
          tc_fence_after();
          issue_pv(0, gt, jj == 0);
          if (jj + 1 == n) commit(&bars->o_done[0]);
          else issue_qk(0, gt + 1);
          if (!(ok = warp_all(mbar_wait(&bars->p_full[1], gt & 1, abort)))) break;
          tc_fence_after();
          issue_pv(1, gt, jj == 0);
          commit(&bars->kv_empty[st]);
          if (jj + 1 == n) {
            commit(&bars->o_done[1]);
          } else {
            issue_qk(1, gt + 1);
            commit(&bars->k_empty[(gt + 1) % NS]);
          }
        }
        g += n;
        ++seg;
      }
      commit(&bars->mma_done);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&bars->mma_done, 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
    __syncwarp();
  } else if (warp == 10) {
    // ------------------------------------------------------------ Q TMA loader
    if (lane == 0) {
      prefetch_tensormap(&map_q);
      const uint32_t q_bytes = (D / 64) * 128 * p.R * p.G;
      int seg = 0, issued[2] = {-1, -1};  // last segment whose copy of each tile was issued
      bool ok = true;
      int unit, a, e;
      Block bx;
      while (ok && walk.next(unit, bx, a, e)) {
        const Unit x = unit_of(p, unit);
        for (int qi = 0; qi < 2 && ok; ++qi) {
          // the previous segment's S = Q K products of this tile have completed
          if (!(ok = mbar_wait(&bars->q_free[qi], (seg + 1) & 1, abort))) break;
          mbar_arrive_expect_tx(&bars->q_full[qi], q_bytes);
          uint8_t* sQ = smem + CF::kQ + qi * CF::kQBytes;
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk)
            tma_load_4d(sQ + blk * (128 * 128), &map_q, &bars->q_full[qi], blk * 64, (x.pair * 2 + qi) * p.R,
                        x.kvh * p.G, x.b);
          issued[qi] = seg;
        }
        ++seg;
      }
      for (int qi = 0; qi < 2; ++qi) {  // let copies in flight land (also those of a stopped segment)
        if (issued[qi] < 0) continue;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&bars->q_full[qi], issued[qi] & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (!EXPLICIT) {
    // ------------------------------------------------------------ V tile release (warp 11)
    // Implicit mask: once a V tile has landed, its dead rows (cache slots
    // past the length, chunk pad rows) are cleared, since P is exactly zero
    // there but 0 times a non-finite value is not; then the tile goes to the
    // P V products.  (With an explicit mask every visited row must hold
    // finite values and the products take the tile as it lands.)
    int g = 0;
    bool ok = true;
    int unit, a, e;
    Block bx;
    while (ok && walk.next(unit, bx, a, e)) {
      const TilePlan tp = block_plan(p, bx);
      for (int j = a; j < e; ++j, ++g) {
        const int st = g % NS;
        if (!(ok = warp_all(mbar_wait(&bars->v_full[st], (g / NS) & 1, abort)))) break;
        const int t = tp.index(j);
        const bool chunk = t < tp.Tc;
        int z0, z1;
        dead_rows<kBN>(p, tp, chunk, (chunk ? t : t - tp.Tc) * kBN, z0, z1);
        if (z0 < z1) {
          zero_tile_rows<D>(sV + st * CF::kVBytes, kBN, z0, z1, lane, 32);
          fence_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->v_ready[st]);
      }
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    // ------------------------------------------------------------ softmax (query tile qi)
    const int qi = warp / 4;
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lanes = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t s_col = tmem + lanes + qi * kBN;
    const uint32_t o_col = tmem + lanes + CF::kOCol + qi * D;
    const float sl2 = p.sl2;
    float4* mstage = reinterpret_cast<float4*>(smem + CF::kStage) + warp * 32 * 8;  // this warp's staging tile
    int g = 0, seg = 0;
    bool ok = true;
    int unit, a, e;
    Block bx;
    while (ok && walk.next(unit, bx, a, e)) {
      const Unit x = unit_of(p, unit);
      const TilePlan tp = block_plan(p, bx);
      const int qt = x.pair * 2 + qi;
      const int gr = row / p.R;
      const int i = qt * p.R + row % p.R;
      const bool valid = gr < p.G && i < p.C;
      const int h = x.kvh * p.G + (valid ? gr : 0);

      RowSpan span;
      span.init(p, tp, i, valid);
      const bool mask_vec = (p.P % 4 == 0) && (p.C % 4 == 0);
      const size_t mstride = static_cast<size_t>(p.P + p.C);
      const float* mrow = nullptr;
      if (EXPLICIT && valid) mrow = p.mask + (static_cast<size_t>(x.b * p.Hq + h) * p.C + i) * mstride;
      float m_run = kMaskedLog2, l_run = 0.f;
      const int n = e - a;
      for (int jj = 0; jj < n; ++jj) {
        const int gt = g + jj;
        const int t = tp.index(a + jj);
        const bool chunk = t < tp.Tc;
        const int base = (chunk ? t : t - tp.Tc) * kBN;
        int lo, hi, sk;
        span.tile(chunk, base, lo, hi, sk);
        // Explicit mask: the tile's class (one for every row of the block)
        // and, for a tile of 0 and masked entries, this row's visibility bits,
        // loaded before the wait on S.  Without a bit copy such tiles take the
        // fp32 values, which give the same result.
        int cls = kTileBinary;
        uint4 vb = make_uint4(0u, 0u, 0u, 0u);
        if (EXPLICIT) {
          cls = ld_chk(p.tcls, static_cast<long long>(block_index(p, bx)) * p.ntiles + t,
                       static_cast<long long>(p.blocks) * p.ntiles, p.err);
          if (cls == kTileBinary && !p.mbits) cls = kTileGeneral;
          if (cls == kTileBinary && valid)
            vb = ld_chk(p.mbits, (static_cast<long long>(x.b * p.Hq + h) * p.ntiles + t) * p.C + i, n_bits(p), p.err);
        }
        if (!(ok = warp_all(mbar_wait(&bars->s_full[qi], gt & 1, abort)))) break;
        tc_fence_after();
        if (jj + 1 == n) mbar_arrive(&bars->q_free[qi]);  // last S = Q K of the segment is done

        if (EXPLICIT && cls == kTileGeneral) {
          // Finite biases: s + bias / scale is written back over S (masked
          // keys -inf), so that the exponentials below form
          // 2^(scale*log2e*s + log2e*bias - m); an entry of 0 leaves s as it is.
          size_t moff;
          int lim;
          mask_span(p, tp, t, moff, lim);
          const float* mp = mrow ? mrow + moff : nullptr;
          const long long mo = mrow ? static_cast<long long>(mrow - p.mask) + static_cast<long long>(moff) : 0;
#pragma unroll 1
          for (int c = 0; c < kBN / 32; ++c) {
            float mc[32];
            load_mask32(mc, mp, 32 * c, lim, mask_vec, mo, n_mask(p), p.err);
            uint32_t r[32];
            tmem_ld32(s_col + 32 * c, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int q = 0; q < 32; ++q)
              r[q] = __float_as_uint(mc[q] > -1e29f ? __fmaf_rn(mc[q], p.inv_scale, __uint_as_float(r[q])) : -INFINITY);
            tmem_st32(s_col + 32 * c, r);
          }
          tmem_st_wait();
        }

        // Scores of this row: one batch of TMEM loads, masked keys set to -inf
        // (they give exactly 0 below).  The implicit mask masks by the row's
        // visible intervals, an explicit 0 / masked tile by its bits.
        float sc[kBN];
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) tmem_ld32f(s_col + 32 * c, sc + 32 * c);
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) tmem_ld_waitf(sc + 32 * c);
        if (!EXPLICIT) {
          if (__any_sync(0xffffffffu, lo > 0 || hi < kBN)) {
            if (!SINK || !__any_sync(0xffffffffu, sk > 0)) {
#pragma unroll
              for (int q = 0; q < kBN; ++q) sc[q] = (q >= lo && q < hi) ? sc[q] : -INFINITY;
            } else {
              // pinned sink slots: visible keys [0, sk) and [lo, hi), as one
              // 32-bit visibility word per 32 keys
#pragma unroll
              for (int c = 0; c < kBN / 32; ++c) {
                const uint32_t vis = bit_range(lo - 32 * c, hi - 32 * c) | bit_range(-32, sk - 32 * c);
#pragma unroll
                for (int q = 0; q < 32; ++q) sc[32 * c + q] = ((vis >> q) & 1u) ? sc[32 * c + q] : -INFINITY;
              }
            }
          }
        } else if (cls != kTileGeneral) {
          if (__any_sync(0xffffffffu, (vb.x & vb.y & vb.z & vb.w) != 0xffffffffu)) {
            const uint32_t vw[4] = {vb.x, vb.y, vb.z, vb.w};  // key q: word q % 4, bit q / 4
#pragma unroll
            for (int q = 0; q < kBN; ++q) sc[q] = ((vw[q & 3] >> (q >> 2)) & 1u) ? sc[q] : -INFINITY;
          }
        }
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int q = 0; q < kBN; q += 8) {
          m0 = fmax3(m0, sc[q], sc[q + 1]);
          m1 = fmax3(m1, sc[q + 2], sc[q + 3]);
          m2 = fmax3(m2, sc[q + 4], sc[q + 5]);
          m3 = fmax3(m3, sc[q + 6], sc[q + 7]);
        }
        const float mt = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
        const float m_tile = (mt == -INFINITY) ? kMaskedLog2 : __fmul_rn(mt, sl2);
        const float m_new = fmaxf(m_run, m_tile);
        const bool rescale = m_new > m_run + 8.f;
        float factor = 1.f;
        if (rescale) {
          factor = fast_exp2(m_run - m_new);
          m_run = m_new;
        }
        const bool live = m_run > kEmptyRow;
        if (jj > 0 && __any_sync(0xffffffffu, rescale)) {
          // O holds every earlier P V (the S = Q K that signalled s_full was issued after them)
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(o_col + 32 * c, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * factor);
            tmem_st32(o_col + 32 * c, o);
          }
        }
        // P = 2^(scale*log2e*s - m), summed in one fixed order (four packed
        // partial sums, for shorter add chains), written over S as bf16
        float2 accA = make_float2(0.f, 0.f), accB = accA, accC = accA, accD = accA;
        auto emit = [&](const float* pv, int c) {
          uint32_t w[16];
#pragma unroll
          for (int q = 0; q < 32; q += 8) {
            accA = fadd2(accA, make_float2(pv[q], pv[q + 1]));
            accB = fadd2(accB, make_float2(pv[q + 2], pv[q + 3]));
            accC = fadd2(accC, make_float2(pv[q + 4], pv[q + 5]));
            accD = fadd2(accD, make_float2(pv[q + 6], pv[q + 7]));
#pragma unroll
            for (int k = 0; k < 8; k += 2) w[(q + k) / 2] = pack16x2<F16>(pv[q + k], pv[q + k + 1]);
          }
          tmem_st16(s_col + 16 * c, w);
        };
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) {
          float* pv = sc + 32 * c;
          const float nm = live ? -m_run : -INFINITY;
#pragma unroll
          for (int q = 0; q < 32; q += 2) {
            const float2 y = ffma2(make_float2(pv[q], pv[q + 1]), make_float2(sl2, sl2), make_float2(nm, nm));
            pv[q] = fast_exp2(y.x);
            pv[q + 1] = fast_exp2(y.y);
          }
          emit(pv, c);
        }
        const float sum = __fadd_rn(__fadd_rn(__fadd_rn(accA.x, accA.y), __fadd_rn(accB.x, accB.y)), __fadd_rn(__fadd_rn(accC.x, accC.y), __fadd_rn(accD.x, accD.y)));
        tmem_st_wait();
        l_run = __fmaf_rn(l_run, factor, sum);
        tc_fence_before();
        mbar_arrive(&bars->p_full[qi]);
      }
      if (!ok) break;

      // -------------------------------------------------------- segment epilogue
      if (!(ok = warp_all(mbar_wait(&bars->o_done[qi], seg & 1, abort)))) break;
      tc_fence_after();
      const bool whole = a == 0 && e == tp.count();
      const bool empty = !(m_run > kEmptyRow);
      const float inv_l = empty ? 0.f : 1.f / l_run;
      const int sel = valid ? (p.sel_row ? p.sel_row[x.b] : tp.n - 1) : -1;
      const size_t orow = (static_cast<size_t>(x.b) * p.Hq + h) * p.C + i;
      // only a CTA's first and last segments can be partial: slots 0 and 1
      const int which = seg == 0 ? 0 : 1;
      const size_t slot = (static_cast<size_t>(cta) * 2 + which) * kUnitRows + qi * 128 + row;
      if (!whole && qi == 0 && row == 0) st_chk(p.ptag, 2 * cta + which, 2LL * p.ctas, unit, p.err);
      // Each 32-column chunk of the warp's 32 rows goes through the staging
      // tile (16-byte slots XOR-swizzled by row, conflict-free both ways) so
      // that the global stores are row-contiguous runs: 128 bytes per row for
      // the fp32 partial rows (consecutive slots), 64 bytes per row for the
      // bf16 output.
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o32[32];
        tmem_ld32(o_col + 32 * c, o32);
        tmem_ld_wait(o32);
        float o[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) o[q] = empty ? 0.f : __uint_as_float(o32[q]) * inv_l;
        __syncwarp();
        if (!whole) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mstage[lane * 8 + (k ^ (lane & 7))] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
          __syncwarp();
          // partial rows stay in L2 for merge_units_kernel while the K/V stream passes
          float* base = p.part_o + (slot - lane) * D + 32 * c;  // the warp's first row
          const uint64_t keep = l2_policy_keep();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int rr = 4 * j + (lane >> 3), k = lane & 7;
            if (in_bounds(static_cast<long long>(base - p.part_o) + rr * D + 4 * k, 4, p.n_part, p.err))
              st_global_hint(reinterpret_cast<float4*>(base + rr * D + 4 * k), mstage[rr * 8 + (k ^ (rr & 7))], keep);
          }
        } else {
          uint4* st4 = reinterpret_cast<uint4*>(mstage);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 wv;
            wv.x = pack_bf16x2(o[8 * k + 0], o[8 * k + 1]);
            wv.y = pack_bf16x2(o[8 * k + 2], o[8 * k + 3]);
            wv.z = pack_bf16x2(o[8 * k + 4], o[8 * k + 5]);
            wv.w = pack_bf16x2(o[8 * k + 6], o[8 * k + 7]);
            st4[lane * 4 + (k ^ ((lane >> 1) & 3))] = wv;
          }
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int rr = 8 * j + (lane >> 2), k = lane & 3;
            const bool ok_r = __shfl_sync(0xffffffffu, valid, rr);
            const unsigned long long orr = __shfl_sync(0xffffffffu, static_cast<unsigned long long>(orow), rr);
            const uint4 wv = st4[rr * 4 + (k ^ ((rr >> 1) & 3))];
            if (ok_r) st16_chk(p.out, static_cast<long long>(orr) * D + 32 * c + 8 * k, n_qo(p), wv, p.err);
          }
          if (p.out_sel && valid && i == sel &&
              in_bounds((static_cast<long long>(x.b) * p.Hq + h) * D + 32 * c, 32, n_sel(p), p.err)) {
            float* sd = p.out_sel + (static_cast<size_t>(x.b) * p.Hq + h) * D + 32 * c;
#pragma unroll
            for (int q = 0; q < 32; q += 4)
              *reinterpret_cast<float4*>(sd + q) = make_float4(o[q], o[q + 1], o[q + 2], o[q + 3]);
          }
        }
      }
      if (valid && !whole) st_chk(p.part_lse, slot, p.n_part / D, empty ? -INFINITY : m_run + __log2f(l_run), p.err);
      g += n;
      ++seg;
    }
  }

  __syncthreads();
  if (threadIdx.x == 0 && bars->abort) set_err(p.err, CPA_EBIT_TIMEOUT);
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Final rows of units cut between CTAs (merged in CTA order) and of units with
// no live key tile (zeros).  CTA (unit, group) handles 32 of the unit's 256
// rows, one per warp; units finished by a single CTA exit at once.
constexpr int kMaxCtas = 256;

constexpr int kMergeThreads = 256;
constexpr int kMergeRows = 64;  // rows of one unit per merge block
constexpr int kMergeRowBatch = 2;
constexpr int kMergePieceBatch = 2;

// One block per (unit, 64-row slab).  Warp 0 finds the unit's pieces (the
// partial-result slots tagged with the unit, in CTA order) with one load per
// lane; then each warp merges 8 rows, two rows and two pieces per batch with
// all their loads issued before any use.  Pieces combine in CTA order with a
// running maximum (one batch, and so the plain max-shifted weighted sum, when
// a unit has two pieces, the usual case).  Registers are capped at 64 so that
// four blocks fit an SM: the grid then runs in under two waves (at 90
// registers it took 3.4).
template <int D, bool PERM>
__global__ void __launch_bounds__(kMergeThreads, 4) merge_units_kernel(const AttnParams p) {
  __shared__ int piece_slot[kMaxCtas];  // partial-result slot of each piece, in CTA order
  __shared__ int n_pieces;
  constexpr int V = D / 32;  // floats per lane
  using Vec = typename std::conditional<V == 4, float4, float2>::type;
  const int unit = blockIdx.x;
  const Unit x = unit_of(p, unit);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  grid_dependency_wait();  // partials and tags of attn_pair_kernel
  if (p.app_n && blockIdx.x == 0 && blockIdx.y == 0)  // fused append: every reader of len is done
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) fused_append_len(p, b);
  // whole blocks dealt and none empty: no unit was cut, every row is written
  if (PERM && p.tlo[p.teams + 1] && p.tlo[p.teams + 2] == 0) return;
  if (warp == 0) {
    const int gnat = (x.b * p.Hkv + x.kvh) * p.nblk + x.pair / p.team;
    int gblk = PERM ? p.upos[gnat] : gnat;  // the block's place in the walk order
    if (!in_bounds(gblk, 1, p.blocks, p.err)) gblk = 0;
    const int member = x.pair % p.team;
    const long long s0 = p.ustart[gblk], s1 = p.ustart[gblk + 1];
    const long long T = p.ustart[p.blocks];
    int np = 0;
    if (PERM && s1 > s0 && p.tlo[p.teams + 1]) {
      np = -1;  // whole blocks were dealt: one CTA wrote every row of the unit
    } else if (s1 > s0) {
      // teams whose ranges meet [s0, s1): from the last team whose range starts
      // at or before s0 to the last one starting at or before s1 - 1; even
      // split: team t covers [floor(t T / teams), floor((t+1) T / teams)), and the
      // last team starting at or before x is floor(((x + 1) teams - 1) / T)
      const int t_first = PERM ? unit_at(p.tlo, p.teams, s0) : static_cast<int>(((s0 + 1) * p.teams - 1) / T);
      const int t_last = PERM ? unit_at(p.tlo, p.teams, s1 - 1) : static_cast<int>((s1 * p.teams - 1) / T);
      for (int t0 = t_first; t0 <= t_last; t0 += 32) {
        const int t = t0 + lane;
        int slot = -1;
        if (t <= t_last) {
          const int c = t * p.team + member;
          const int tag0 = ld_chk(p.ptag, 2LL * c, 2LL * p.ctas, p.err);
          const int tag1 = ld_chk(p.ptag, 2LL * c + 1, 2LL * p.ctas, p.err);
          slot = tag0 == unit ? 2 * c : (tag1 == unit ? 2 * c + 1 : -1);
        }
        const unsigned m = __ballot_sync(0xffffffffu, slot >= 0);
        if (slot >= 0) piece_slot[np + __popc(m & ((1u << lane) - 1u))] = slot;
        np += __popc(m);
      }
      if (np == 0) np = -1;  // one CTA did the whole unit and wrote it already
    }
    if (lane == 0) n_pieces = np;
  }
  __syncthreads();
  const int np = n_pieces;
  if (np < 0) return;
  const int n_real = p.n_real ? min(max(p.n_real[x.b], 0), p.C) : p.C;
  const int sel = p.sel_row ? p.sel_row[x.b] : n_real - 1;
  const uint64_t drop = l2_policy_drop();
  constexpr int kRowsPerWarp = kMergeRows / (kMergeThreads / 32);
  for (int j0 = 0; j0 < kRowsPerWarp; j0 += kMergeRowBatch) {
    int r[kMergeRowBatch], i[kMergeRowBatch], h[kMergeRowBatch];
    bool live[kMergeRowBatch];
#pragma unroll
    for (int u = 0; u < kMergeRowBatch; ++u) {
      r[u] = blockIdx.y * kMergeRows + (j0 + u) * (kMergeThreads / 32) + warp;
      const int qi = r[u] / 128, rr = r[u] % 128;
      const int gr = rr / p.R;
      i[u] = (x.pair * 2 + qi) * p.R + rr % p.R;
      h[u] = x.kvh * p.G + gr;
      live[u] = gr < p.G && i[u] < p.C;
    }
    float acc[kMergeRowBatch][V], m[kMergeRowBatch], wsum[kMergeRowBatch];
#pragma unroll
    for (int u = 0; u < kMergeRowBatch; ++u) {
      m[u] = -INFINITY;
      wsum[u] = 0.f;
#pragma unroll
      for (int q = 0; q < V; ++q) acc[u][q] = 0.f;
    }
    for (int k0 = 0; k0 < np; k0 += kMergePieceBatch) {
      float ls[kMergeRowBatch][kMergePieceBatch];
      Vec o[kMergeRowBatch][kMergePieceBatch];
#pragma unroll
      for (int u = 0; u < kMergeRowBatch; ++u)
#pragma unroll
        for (int k = 0; k < kMergePieceBatch; ++k) {
          ls[u][k] = -INFINITY;
          if (live[u] && k0 + k < np &&
              in_bounds((static_cast<long long>(piece_slot[k0 + k]) * kUnitRows + r[u]) * D, D, p.n_part, p.err)) {
            const size_t sidx = static_cast<size_t>(piece_slot[k0 + k]) * kUnitRows + r[u];
            ls[u][k] = p.part_lse[sidx];
            if constexpr (V == 4)  // the last read of these rows: let L2 drop them first
              o[u][k] = ld_global_hint(reinterpret_cast<const float4*>(p.part_o + sidx * D + lane * V), drop);
            else
              o[u][k] = *reinterpret_cast<const Vec*>(p.part_o + sidx * D + lane * V);
          }
        }
#pragma unroll
      for (int u = 0; u < kMergeRowBatch; ++u) {
        float bm = m[u];
#pragma unroll
        for (int k = 0; k < kMergePieceBatch; ++k) bm = fmaxf(bm, ls[u][k]);
        if (bm == -INFINITY) continue;
        if (bm != m[u]) {
          const float c = m[u] == -INFINITY ? 0.f : fast_exp2(m[u] - bm);
          wsum[u] *= c;
#pragma unroll
          for (int q = 0; q < V; ++q) acc[u][q] *= c;
          m[u] = bm;
        }
#pragma unroll
        for (int k = 0; k < kMergePieceBatch; ++k) {
          if (ls[u][k] == -INFINITY) continue;
          const float w = fast_exp2(ls[u][k] - bm);
          wsum[u] += w;
          const float* ov = reinterpret_cast<const float*>(&o[u][k]);
#pragma unroll
          for (int q = 0; q < V; ++q) acc[u][q] = __fmaf_rn(w, ov[q], acc[u][q]);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kMergeRowBatch; ++u) {
      if (!live[u]) continue;
      const size_t orow = (static_cast<size_t>(x.b) * p.Hq + h[u]) * p.C + i[u];
      if (!in_bounds(static_cast<long long>(orow) * D, D, n_qo(p), p.err)) continue;
      const bool sel_ok = in_bounds((static_cast<long long>(x.b) * p.Hq + h[u]) * D, D, n_sel(p), p.err);
      const float inv = wsum[u] > 0.f ? 1.f / wsum[u] : 0.f;
#pragma unroll
      for (int q = 0; q < V; q += 2) {
        const float o0 = acc[u][q] * inv, o1 = acc[u][q + 1] * inv;
        *reinterpret_cast<uint32_t*>(p.out + orow * D + lane * V + q) = pack_bf16x2(o0, o1);
        if (p.out_sel && i[u] == sel && sel_ok) {
          float* sd = p.out_sel + (static_cast<size_t>(x.b) * p.Hq + h[u]) * D + lane * V + q;
          sd[0] = o0;
          sd[1] = o1;
        }
      }
    }
  }
}

PairTeams pair_teams(int B, int Hkv, int nq, int P, int C, int num_sms) {
  PairTeams t;
  t.pairs = (nq + 1) / 2;
  const int sms = num_sms < kMaxCtas ? num_sms : kMaxCtas;
  t.team = t.pairs < sms ? t.pairs : sms;
  t.nblk = (t.pairs + t.team - 1) / t.team;
  t.blocks = B * Hkv * t.nblk;
  const long long max_cost = static_cast<long long>(t.blocks) *
                             ((P + kBN - 1) / kBN + (C + kBN - 1) / kBN + kSwitchCost);
  t.teams = static_cast<int>(max(1LL, min(static_cast<long long>(sms / t.team), max_cost)));
  t.ctas = t.teams * t.team;
  // small teams (chunks of at most 512 packed rows per (sequence, kv head))
  // and at least one block per team: the plan may deal whole blocks instead
  // of cutting them (with fewer blocks than teams the even split is kept)
  t.perm = t.team <= 2 && t.teams > 1 && t.blocks >= t.teams && t.blocks <= kPlanSortMax ? 1 : 0;
  return t;
}

PairWorkspace pair_workspace(int B, int Hq, int Hkv, int D, int C, int P, const PairTeams& t) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const int ctas = t.ctas;
  PairWorkspace w;
  size_t off = 0;
  w.ustart = off; off += al((static_cast<size_t>(t.blocks) + 1) * sizeof(int32_t));
  w.uorder = off; off += al(static_cast<size_t>(t.blocks) * sizeof(int32_t));
  w.upos = off; off += al(static_cast<size_t>(t.blocks) * sizeof(int32_t));
  w.tlo = off; off += al((static_cast<size_t>(t.teams) + 3) * sizeof(int32_t));  // + the whole-deal and empty flags
  w.part_o = off; off += al(static_cast<size_t>(ctas) * 2 * kUnitRows * D * sizeof(float));
  w.part_lse = off; off += al(static_cast<size_t>(ctas) * 2 * kUnitRows * sizeof(float));
  w.ptag = off; off += al(static_cast<size_t>(ctas) * 2 * sizeof(int32_t));
  w.q_rot = off; off += al(static_cast<size_t>(B) * Hq * C * D * 2);
  w.k_rot = off; off += al(static_cast<size_t>(B) * Hkv * C * D * 2);
  w.v_cvt = off; off += al(static_cast<size_t>(B) * Hkv * C * D * 2);  // fp16 cache: chunk values in half
  const size_t T = static_cast<size_t>((C + kBN - 1) / kBN + (P + kBN - 1) / kBN);
  w.tcls = off; off += al(static_cast<size_t>(t.blocks) * T);                  // explicit mask: tile classes
  w.hull = off; off += al(static_cast<size_t>(t.blocks) * 16);                 // explicit mask: tile hulls
  w.total = off;
  w.mbits = off; off += al(static_cast<size_t>(B) * Hq * T * C * 16);          // explicit mask: bit copy
  w.total_bits = off;
  return w;
}

template <int D, bool EXPLICIT, bool SINK, bool F16, bool PERM>
static cudaError_t launch_pair_t(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream) {
  constexpr int smem = pair_smem_bytes<D>();
  auto kern = attn_pair_kernel<D, EXPLICIT, SINK, F16, PERM>;
  static SmemAttr smem_attr;
  if (cudaError_t e = smem_attr.ensure(reinterpret_cast<const void*>(kern), smem); e != cudaSuccess) return e;
  const long long items = static_cast<long long>(p.B) * ((p.Hq + p.Hkv + kPrepHeads - 1) / kPrepHeads) * p.C *
                          (p.D / 16);
  const int rope_blocks =
      static_cast<int>(max(1LL, min(static_cast<long long>(65535) * 4, (items + kPrepThreads - 1) / kPrepThreads)));
  cudaError_t e;
  if (EXPLICIT) {  // classify the mask's tiles before the plan reads them
    e = launch_dependent(mask_scan_kernel, dim3(static_cast<unsigned>(p.blocks) * p.ntiles), dim3(kScanThreads), 0,
                         stream, p);
    if (e != cudaSuccess) return e;
  }
  e = launch_dependent(prep_kernel, dim3(rope_blocks + 1), dim3(kPrepThreads), 0, stream, p);
  if (e != cudaSuccess) return e;
  e = launch_dependent(kern, dim3(p.ctas), dim3(kThreadsPair), smem, stream, maps[0], maps[1], maps[2], maps[3],
                       maps[4], p);
  if (e != cudaSuccess) return e;
  return launch_dependent(merge_units_kernel<D, PERM>, dim3(p.units, kUnitRows / kMergeRows), dim3(kMergeThreads), 0,
                          stream, p);
}

// The walk (planned order or index order) follows the shapes alone, so the
// explicit and implicit forms of one mask take the same plan.
template <int D, bool F16, bool EXPLICIT, bool SINK>
static cudaError_t launch_pair_w(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream) {
  if (p.perm) return launch_pair_t<D, EXPLICIT, SINK, F16, true>(maps, p, stream);
  return launch_pair_t<D, EXPLICIT, SINK, F16, false>(maps, p, stream);
}

template <int D, bool F16>
static cudaError_t launch_pair_d(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream) {
  if (p.mask) return launch_pair_w<D, F16, true, false>(maps, p, stream);
  if (p.sink > 0) return launch_pair_w<D, F16, false, true>(maps, p, stream);
  return launch_pair_w<D, F16, false, false>(maps, p, stream);
}

cudaError_t launch_attn_pair5(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream) {
  switch (p.D) {
    case 64: return p.f16 ? launch_pair_d<64, true>(maps, p, stream) : launch_pair_d<64, false>(maps, p, stream);
    case 128: return p.f16 ? launch_pair_d<128, true>(maps, p, stream) : launch_pair_d<128, false>(maps, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cpa
