// Chunk-prefill attention with past on tcgen05 tensor cores (sm_103a).
//
// What it computes ("functiongemma: chunk prefill-with-past graph", Change):
// a chunk of C query rows, rotated with per-position cos/sin tables, attends
// over P cached key slots followed by the C chunk rows (chunk keys rotated with
// the same tables) under an additive mask; softmax-weighted values per row.
//
// Work decomposition.  One CTA owns 128 packed query rows of one (sequence b,
// kv head): R = floor(128 / G) chunk rows for each of the G query heads that
// share the kv head (row r <-> head g = r / R, chunk row i = i0 + r % R), so K
// and V tiles are loaded once for the whole GQA group.  Key tiles of BN keys
// are visited chunk tiles first, then past tiles; tiles that the implicit mask
// leaves fully masked for every row of the CTA are never visited.  A CTA may
// take only a slice of its key tiles (split-KV).  With S = 2, 4 or 8 splits,
// the splits of a query tile form one thread-block cluster: once every CTA
// of the cluster is done with its Q/K/V buffers, each thread stores its
// normalised row and log2-sum-exp straight from tensor memory into the
// shared memory of the CTA that owns the row's slice (CTA s owns rows
// [s*128/S, (s+1)*128/S)); after a second cluster barrier each CTA merges its
// slice from its own shared memory.  At D = 256 with 8 splits each split is
// taken by two CTAs (clusters of 16): both compute the same S and P, each
// forms P V for one half of D, and each half is exchanged and merged among
// the 8 CTAs that hold it, so a CTA sends half the bytes (the exchange, at
// ~10 bytes per clock per SM, bounds these calls).  Other split counts write
// the partials to the workspace and combine_kernel merges them.  Both merges
// take the splits in the same fixed order with the same arithmetic.
//
// Queries and chunk keys: rope_chunk_k_kernel rotates them once per call into
// the workspace (the append's arithmetic).  The attention grid is launched as
// a programmatic dependent of it, so its prologue (barriers, tensor memory)
// runs while the rows are rotated; it then waits for that grid before it reads
// anything of the call: the rotated Q tile, the lengths, any cached row.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: K and V tiles into a 2-stage shared-memory ring.
//   warp 1      tcgen05 issuer: S = Q K^T into one of two TMEM S buffers,
//               O += P V into the TMEM O accumulator; owns the TMEM allocation.
//   warps 2..5  softmax warpgroup: thread = TMEM lane = packed query row.
//               Applies the mask, keeps the running
//               max / sum in fp32 (log2 domain, rescaling O only when the max
//               grows by more than 2^8), writes P as bf16 (fp16 for an fp16
//               KV cache), and finally scales O by 1/l: into a shared-memory
//               staging tile from which whole rows are stored with coalesced
//               accesses, or, in a cluster, straight into the slice owner's
//               shared memory.
#include "tiles.cuh"

namespace cpa {

constexpr int kBM = 128;
constexpr int kStages = 2;
constexpr int kThreads = 192;

struct __align__(8) AttnBars {
  uint64_t k_full[kStages], v_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full, pv_done, q_full, mma_done;
  uint32_t tmem_base;
  int abort;
  int sel;  // the caller's selected row of this sequence, read once at the start
};

template <int D, int BN>
struct AttnSmem {
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kKBytes = BN * D * 2;
  static constexpr int kVBytes = BN * D * 2;
  static constexpr int kPBytes = kBM * BN * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kQBytes;
  static constexpr int kV = kK + kStages * kKBytes;
  static constexpr int kP = kV + kStages * kVBytes;
  static constexpr int kBars = kP + kPBytes;
  static constexpr int kTotal = kBars + static_cast<int>(sizeof(AttnBars));
  static constexpr int kAlloc = kTotal + 1024;  // room to align the base to 1024
  // Epilogue buffers over the Q/K/V buffers (free once the last product has
  // finished).  Without a cluster: a staging tile [128][D + 4] fp32 (a
  // 16-byte pad per row keeps row-per-thread float4 writes conflict-free) and
  // the rows' log2-sum-exp.  With a cluster of S: the receive buffer of this
  // CTA's slice, [S][D/4][128/S] float4 with the slot index XOR-swizzled by
  // the chunk index, then [S][128/S] log2-sum-exp.
  static constexpr int kStg = D + 4;
  static constexpr int kStgLse = kBM * kStg * 4;
  static_assert(kStgLse + kBM * 4 <= kP, "staging tile fits over Q, K and V");
  static constexpr int kRecvLse = kBM * D * 4;
  static_assert(kRecvLse + kBM * 4 <= kP, "receive buffer fits over Q, K and V");
  // Per-row tables over the P buffer: output row index (-1: no such row),
  // chunk row, (sequence, head) index.
  static constexpr int kTabRow = kP;
  static constexpr int kTabI = kTabRow + kBM * 8;
  static constexpr int kTabBh = kTabI + kBM * 4;
  static_assert(kTabBh + kBM * 4 <= kP + kPBytes, "row tables fit over P");
  static constexpr int kSCol = 0;               // S buffers at columns [0, 2*BN)
  static constexpr int kOCol = 2 * BN;          // O at columns [2*BN, 2*BN + D)
  static_assert(2 * BN + D <= 512, "TMEM columns");
  static_assert(kAlloc <= 232448, "shared memory");
};

template <int D, int BN, bool F16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap map_kc, const __grid_constant__ CUtensorMap map_vc,
                const __grid_constant__ CUtensorMap map_kn, const __grid_constant__ CUtensorMap map_vn,
                const __grid_constant__ CUtensorMap map_q, const AttnParams p) {
  using SM = AttnSmem<D, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  AttnBars* bars = reinterpret_cast<AttnBars*>(smem + SM::kBars);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // CTAs of a query tile: p.splits key splits, each taken by p.dsplit CTAs
  // that divide D for the P V products and the merge (cluster rank
  // dh * p.splits + split)
  const int per_q = p.splits * p.dsplit;
  const int qt = blockIdx.x / per_q;
  const int dh = (blockIdx.x % per_q) / p.splits;
  const int split = blockIdx.x % p.splits;
  const int DV = D / p.dsplit;  // value columns of this CTA: [dh * DV, dh * DV + DV)
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;

  // combine_kernel (if any) may be scheduled now, except on a partial SM
  // budget (then as this grid ends); it waits for this grid
  if (!p.hold_dependents) grid_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_empty[s], 128);
    }
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_barrier_init();
    prefetch_tensormap(&map_q);
  }
  // The Q tile's rows past the G * R packed rows, which the Q copy does not
  // write, stay zero.
  for (int item = threadIdx.x; item < (kBM - p.G * p.R) * (D / 8); item += kThreads) {
    const int r = p.G * p.R + item / (D / 8);
    const int c = item % (D / 8);
    *reinterpret_cast<uint4*>(smem + SM::kQ + (c / 8) * (kBM * 128) + sw128(r, c % 8)) = make_uint4(0, 0, 0, 0);
  }
  fence_async_smem();
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  uint8_t* sQ = smem + SM::kQ;
  uint8_t* sK = smem + SM::kK;
  uint8_t* sV = smem + SM::kV;
  uint8_t* sP = smem + SM::kP;

  // Nothing of the call's or the caller's memory is touched before this wait:
  // until it returns, the key pre-pass (which also rotates the queries) and,
  // through it, earlier launches may still be running.
  grid_dependency_wait();
  if (threadIdx.x == 0) {
    // the rotated Q rows of the G heads, head-major ({64, R, G, 1} boxes;
    // rows past the chunk arrive as zeros)
    mbar_arrive_expect_tx(&bars->q_full, static_cast<uint32_t>(D * p.R * p.G * 2));
#pragma unroll
    for (int blk = 0; blk < D / 64; ++blk)
      tma_load_4d(smem + SM::kQ + blk * kBM * 128, &map_q, &bars->q_full, blk * 64, qt * p.R, kvh * p.G, b);
    bars->sel = p.sel_row ? p.sel_row[b] : -1;
    if (kvh == 0 && blockIdx.x == 0) {
      if (p.past_len && (p.past_len[b] < 0 || p.past_len[b] > p.P)) set_err(p.err, CPA_EBIT_PAST_GT_SPAN);
      if (p.n_real && (p.n_real[b] < 0 || p.n_real[b] > p.C)) set_err(p.err, CPA_EBIT_NREAL_GT_C);
    }
  }
  const TilePlan tp = plan_tiles<BN>(p, b, qt * p.R, min(qt * p.R + p.R, p.C) - 1, split);
  const int my_nt = tp.count();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && my_nt > 0) {
      prefetch_tensormap(&map_kc);
      prefetch_tensormap(&map_vc);
      prefetch_tensormap(&map_kn);
      prefetch_tensormap(&map_vn);
      int issued = 0;
      for (int q = 0; q < my_nt; ++q) {
        const int st = q % kStages;
        if (!mbar_wait(&bars->kv_empty[st], ((q / kStages) + 1) & 1, abort)) break;
        const int j = tp.index(q);
        const bool chunk = j < tp.Tc;
        const int base = (chunk ? j : j - tp.Tc) * BN;
        const CUtensorMap* mk = chunk ? &map_kn : &map_kc;
        const CUtensorMap* mv = chunk ? &map_vn : &map_vc;
        mbar_arrive_expect_tx(&bars->k_full[st], SM::kKBytes);
#pragma unroll
        for (int blk = 0; blk < D / 64; ++blk)
          tma_load_4d(sK + st * SM::kKBytes + blk * BN * 128, mk, &bars->k_full[st], blk * 64, base, kvh, b);
        mbar_arrive_expect_tx(&bars->v_full[st], static_cast<uint32_t>(SM::kVBytes / p.dsplit));
        for (int blk = 0; blk < DV / 64; ++blk)
          tma_load_4d(sV + st * SM::kVBytes + blk * BN * 128, mv, &bars->v_full[st], dh * DV + blk * 64, base, kvh,
                      b);
        issued = q + 1;
      }
      // Before leaving, make sure no copy is still landing in shared memory.
      for (int q = max(0, issued - kStages); q < issued; ++q) {
        const int st = q % kStages;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&bars->v_full[st], (q / kStages) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
        while (!mbar_try_wait(&bars->k_full[st], (q / kStages) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the tiles and waits (descriptors stay warp-uniform);
    // one elected lane issues the MMAs and the commits that track them.
    {
      const bool leader = elect_lane();
      constexpr uint32_t idesc_qk = idesc_16(kBM, BN, false, F16);
      constexpr uint32_t idesc_pv_d = idesc_16(kBM, D, true, F16);
      constexpr uint32_t idesc_pv_h = idesc_16(kBM, D / 2, true, F16);
      const uint32_t idesc_pv = p.dsplit == 2 ? idesc_pv_h : idesc_pv_d;  // N = DV
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t p_addr = smem_u32(sP);
      bool ok = my_nt > 0 ? warp_all(mbar_wait(&bars->q_full, 0, abort)) : true;
      auto issue_pv = [&](int q) -> bool {
        const int st = q % kStages;
        if (!warp_all(mbar_wait(&bars->p_full, q & 1, abort))) return false;
        if (!warp_all(mbar_wait(&bars->v_full[st], (q / kStages) & 1, abort))) return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(sV + st * SM::kVBytes);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t a = sdesc_sw128(p_addr + (kk / 4) * (kBM * 128) + (kk % 4) * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(v_addr + kk * 2048, BN * 128, 1024);
            mma_bf16_ss(tmem + SM::kOCol, a, bd, idesc_pv, (q > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bars->pv_done);
          mma_commit(&bars->kv_empty[st]);
        }
        __syncwarp();
        return true;
      };
      for (int q = 0; ok && q < my_nt; ++q) {
        const int st = q % kStages;
        const int sb = q & 1;
        ok = warp_all(mbar_wait(&bars->k_full[st], (q / kStages) & 1, abort));
        if (!ok) break;
        ok = warp_all(mbar_wait(&bars->s_empty[sb], ((q >> 1) + 1) & 1, abort));
        if (!ok) break;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(sK + st * SM::kKBytes);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t a = sdesc_sw128(q_addr + (kk / 4) * (kBM * 128) + (kk % 4) * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(k_addr + (kk / 4) * (BN * 128) + (kk % 4) * 32, 16, 1024);
            mma_bf16_ss(tmem + SM::kSCol + sb * BN, a, bd, idesc_qk, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars->s_full[sb]);
        }
        __syncwarp();
        if (q > 0) ok = issue_pv(q - 1);
      }
      if (ok && my_nt > 0) issue_pv(my_nt - 1);
      // Every MMA issued above has finished once this barrier flips.
      if (leader) mma_commit(&bars->mma_done);
      __syncwarp();
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&bars->mma_done, 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warpgroup
    const int tid = threadIdx.x - 64;               // 0..127
    const int row = 32 * (warp & 3) + lane;         // TMEM lane owned by this thread
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int g = row / p.R;
    const int i = qt * p.R + row % p.R;
    const bool valid = g < p.G && i < p.C;
    const int h = kvh * p.G + (valid ? g : 0);


    // Visible key intervals of this row (implicit mask).
    const int W = p.window;
    const int past_lo = W > 0 ? max(0, tp.L + i - W + 1) : 0;
    const int ch_lo = W > 0 ? max(0, i - W + 1) : 0;
    const int ch_hi = p.causal ? min(tp.n, i + 1) : (W > 0 ? min(tp.n, i + W) : tp.n);
    const bool mask_vec = (p.P % 4 == 0) && (p.C % 4 == 0);
    const long long mrow_off = ((static_cast<long long>(b) * p.Hq + h) * p.C + i) * (static_cast<long long>(p.P) + p.C);
    const float* mrow = (p.mask && valid && in_bounds(mrow_off, static_cast<long long>(p.P) + p.C, n_mask(p), p.err))
                            ? p.mask + mrow_off
                            : nullptr;

    float m_run = kMaskedLog2, l_run = 0.f;
    bool ok = true;
    for (int q = 0; q < my_nt; ++q) {
      const int sb = q & 1;
      const int j = tp.index(q);
      const bool chunk = j < tp.Tc;
      const int base = (chunk ? j : j - tp.Tc) * BN;
      // Explicit mask values of this tile, loaded before the wait on S so
      // their latency hides behind the product (64-key tiles only: a 128-key
      // tile has no registers to spare).  With P and C multiples of 4 every
      // 16-byte vector of the row lies wholly inside or outside [0, lim).
      constexpr bool kMaskEarly = BN == 64;
      float mk[kMaskEarly ? BN : 1];
      if (kMaskEarly && mrow) {
        const int lim = chunk ? p.C : p.P;
        const float* mp = mrow + (chunk ? p.P + base : base);
        if (mask_vec) {
#pragma unroll
          for (int e = 0; e < (kMaskEarly ? BN : 4); e += 4) {
            float4 v = make_float4(-1e30f, -1e30f, -1e30f, -1e30f);
            if (base + e < lim) v = __ldg(reinterpret_cast<const float4*>(mp + e));
            mk[e] = v.x;
            mk[e + 1] = v.y;
            mk[e + 2] = v.z;
            mk[e + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < (kMaskEarly ? BN : 1); ++e) mk[e] = (base + e < lim) ? __ldg(mp + e) : -1e30f;
        }
      }
      if (!(ok = warp_all(mbar_wait(&bars->s_full[sb], (q >> 1) & 1, abort)))) break;
      tc_fence_after();
      float x[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r32[32];
        tmem_ld32(tmem + lane_base + SM::kSCol + sb * BN + 32 * c, r32);
        tmem_ld_wait(r32);
#pragma unroll
        for (int e = 0; e < 32; ++e) x[32 * c + e] = __uint_as_float(r32[e]);
      }
      tc_fence_before();
      mbar_arrive(&bars->s_empty[sb]);

      // scale + mask, in log2 units
      if (mrow) {
        const bool pastt = !chunk;
        const int lim = pastt ? p.P : p.C;
        const float* mp = mrow + (pastt ? base : p.P + base);
        if constexpr (kMaskEarly) {
#pragma unroll
          for (int e = 0; e < BN; ++e) x[e] = __fmaf_rn(x[e], p.sl2, __fmul_rn(mk[e], kLog2e));
        } else if (mask_vec) {
#pragma unroll
          for (int e = 0; e < BN; e += 4) {
            float4 v = make_float4(-1e30f, -1e30f, -1e30f, -1e30f);
            if (base + e < lim) v = __ldg(reinterpret_cast<const float4*>(mp + e));
            x[e] = __fmaf_rn(x[e], p.sl2, __fmul_rn(v.x, kLog2e));
            x[e + 1] = __fmaf_rn(x[e + 1], p.sl2, __fmul_rn(v.y, kLog2e));
            x[e + 2] = __fmaf_rn(x[e + 2], p.sl2, __fmul_rn(v.z, kLog2e));
            x[e + 3] = __fmaf_rn(x[e + 3], p.sl2, __fmul_rn(v.w, kLog2e));
          }
        } else {
#pragma unroll
          for (int e = 0; e < BN; ++e) {
            const float mv = (base + e < lim) ? __ldg(mp + e) : -1e30f;
            x[e] = __fmaf_rn(x[e], p.sl2, __fmul_rn(mv, kLog2e));
          }
        }
      } else {
        const int lo = (chunk ? ch_lo : past_lo) - base;
        const int hi = valid ? ((chunk ? ch_hi : tp.L) - base) : -1;
        const int sk = (valid && !chunk) ? min(p.sink, tp.L) - base : 0;  // pinned sink slots
#pragma unroll
        for (int e = 0; e < BN; ++e)
          x[e] = ((e >= lo && e < hi) || e < sk) ? __fmul_rn(x[e], p.sl2) : kMaskedLog2;
      }
      float mt = x[0];
#pragma unroll
      for (int e = 1; e < BN; ++e) mt = fmaxf(mt, x[e]);
      float m_use, factor = 1.f;
      bool rescale = false;
      if (q == 0) {
        m_use = mt;
      } else {
        const float m_new = fmaxf(m_run, mt);
        rescale = (m_new - m_run) > 8.f;
        m_use = rescale ? m_new : m_run;
        if (rescale) factor = fast_exp2(m_run - m_new);
      }
      float sum = 0.f;
#pragma unroll
      for (int e = 0; e < BN; ++e) {
        x[e] = fast_exp2(__fsub_rn(x[e], m_use));
        sum += x[e];
      }
      l_run = (q == 0) ? sum : __fmaf_rn(l_run, factor, sum);
      m_run = m_use;

      // P buffer and O are free once the previous P V has finished.
      if (q > 0) {
        if (!(ok = warp_all(mbar_wait(&bars->pv_done, (q - 1) & 1, abort)))) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c = 0; c < DV / 32; ++c) {
            uint32_t o32[32];
            const uint32_t ta = tmem + lane_base + SM::kOCol + 32 * c;
            tmem_ld32(ta, o32);
            tmem_ld_wait(o32);
#pragma unroll
            for (int e = 0; e < 32; ++e) o32[e] = __float_as_uint(__uint_as_float(o32[e]) * factor);
            tmem_st32(ta, o32);
          }
          tmem_st_wait();
        }
      }
#pragma unroll
      for (int c8 = 0; c8 < BN / 8; ++c8) {
        uint4 w;
        w.x = pack16x2<F16>(x[8 * c8 + 0], x[8 * c8 + 1]);
        w.y = pack16x2<F16>(x[8 * c8 + 2], x[8 * c8 + 3]);
        w.z = pack16x2<F16>(x[8 * c8 + 4], x[8 * c8 + 5]);
        w.w = pack16x2<F16>(x[8 * c8 + 6], x[8 * c8 + 7]);
        *reinterpret_cast<uint4*>(sP + (c8 / 8) * (kBM * 128) + sw128(row, c8 % 8)) = w;
      }
      if (!p.mask) {
        // dead V rows of this tile (cache slots past the length, chunk pad
        // rows) are cleared once the tile has landed, before the P V product
        int z0, z1;
        dead_rows<BN>(p, tp, chunk, base, z0, z1);
        if (z0 < z1) {
          const int st = q % kStages;
          if (!(ok = warp_all(mbar_wait(&bars->v_full[st], (q / kStages) & 1, abort)))) break;
          zero_tile_rows<D>(sV + st * SM::kVBytes, BN, z0, z1, tid, 128);
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }

    // ---------------------------------------------------------- epilogue
    if (ok && my_nt > 0) ok = warp_all(mbar_wait(&bars->pv_done, (my_nt - 1) & 1, abort));
    tc_fence_after();
    const bool empty = !(my_nt > 0 && ok && m_run > kEmptyRow);
    const float inv_l = empty ? 0.f : 1.f / l_run;
    // O / l of this row into the staging tile.  Every product has finished
    // (pv_done of the last tile) and every copy has been consumed, so the
    // Q, K and V buffers are free.
    long long* tab_row = reinterpret_cast<long long*>(smem + SM::kTabRow);
    int* tab_i = reinterpret_cast<int*>(smem + SM::kTabI);
    int* tab_bh = reinterpret_cast<int*>(smem + SM::kTabBh);
    const long long orow_me = (static_cast<long long>(b) * p.Hq + h) * p.C + i;
    const float lse_me = empty ? -INFINITY : m_run + __log2f(l_run);
    tab_row[row] = valid ? orow_me : -1;
    tab_i[row] = i;
    tab_bh[row] = b * p.Hq + h;
    if (!p.cluster) {
      float* stg = reinterpret_cast<float*>(smem);
#pragma unroll 1
      for (int c = 0; c < D / 32; c += 2) {
        uint32_t o0[32], o1[32];
        if (my_nt > 0) {
          tmem_ld32(tmem + lane_base + SM::kOCol + 32 * c, o0);
          tmem_ld32(tmem + lane_base + SM::kOCol + 32 * c + 32, o1);
          tmem_ld_wait(o0);
          tmem_ld_wait(o1);
        }
#pragma unroll
        for (int e = 0; e < 64; e += 4) {
          const uint32_t* oo = e < 32 ? o0 + e : o1 + (e - 32);
          float4 v;
          v.x = empty ? 0.f : __uint_as_float(oo[0]) * inv_l;
          v.y = empty ? 0.f : __uint_as_float(oo[1]) * inv_l;
          v.z = empty ? 0.f : __uint_as_float(oo[2]) * inv_l;
          v.w = empty ? 0.f : __uint_as_float(oo[3]) * inv_l;
          *reinterpret_cast<float4*>(stg + row * SM::kStg + 32 * c + e) = v;
        }
      }
      if (valid && p.part_o)
        st_chk(p.part_lse, static_cast<long long>(split) * p.B * p.Hq * p.C + orow_me, p.n_part / D, lse_me, p.err);
      named_bar_sync(1, 128);
      // This warp's own 32 rows, whole rows with lanes across D: bf16 output
      // (one split) or fp32 partials.  Row indices come from the table, four
      // rows per step.
      const int w = warp - 2;
      const int sel = p.sel_row ? bars->sel : tp.n - 1;
      const size_t part_base = static_cast<size_t>(split) * p.B * p.Hq * p.C;
#pragma unroll 4
      for (int k = 0; k < 32; ++k) {
        const int r = 32 * w + k;
        const long long orow = tab_row[r];
        if (orow < 0) continue;
        const float* src = stg + r * SM::kStg;
        if (!in_bounds(static_cast<long long>(p.part_o ? part_base + orow : orow) * D, D,
                       p.part_o ? p.n_part : n_qo(p), p.err))
          continue;
        if (p.part_o) {
          float* dst = p.part_o + (part_base + static_cast<size_t>(orow)) * D;
#pragma unroll
          for (int e = 4 * lane; e < D; e += 128)
            *reinterpret_cast<float4*>(dst + e) = *reinterpret_cast<const float4*>(src + e);
        } else {
          uint16_t* dst = p.out + static_cast<size_t>(orow) * D;
#pragma unroll
          for (int e = 4 * lane; e < D; e += 128) {
            const float4 v = *reinterpret_cast<const float4*>(src + e);
            *reinterpret_cast<uint2*>(dst + e) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
          }
          if (p.out_sel && tab_i[r] == sel && in_bounds(static_cast<long long>(tab_bh[r]) * D, D, n_sel(p), p.err)) {
            float* sd = p.out_sel + static_cast<size_t>(tab_bh[r]) * D;
#pragma unroll
            for (int e = 4 * lane; e < D; e += 128)
              *reinterpret_cast<float4*>(sd + e) = *reinterpret_cast<const float4*>(src + e);
          }
        }
      }
    } else {
      // Cluster merge, step 1: once every CTA is done with its Q/K/V
      // buffers (barrier A), push this row to its slice owner.
      const int S = p.splits;
      const int rows_per = kBM / S;
      const int owner = row / rows_per, slot = row % rows_per;
      named_bar_sync(1, 128);
      asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
      const uint32_t dst = dsmem_addr(smem_u32(smem), dh * S + owner);
      dsmem_st(dst + SM::kRecvLse + 4u * (split * rows_per + slot), lse_me);
#pragma unroll 1
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t o32[32];
        if (my_nt > 0) {
          tmem_ld32(tmem + lane_base + SM::kOCol + 32 * c, o32);
          tmem_ld_wait(o32);
        }
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const int e = 8 * c + q4;  // float4 chunk index along D
          float4 v;
          v.x = empty ? 0.f : __uint_as_float(o32[4 * q4 + 0]) * inv_l;
          v.y = empty ? 0.f : __uint_as_float(o32[4 * q4 + 1]) * inv_l;
          v.z = empty ? 0.f : __uint_as_float(o32[4 * q4 + 2]) * inv_l;
          v.w = empty ? 0.f : __uint_as_float(o32[4 * q4 + 3]) * inv_l;
          const uint32_t off = 16u * ((split * (DV / 4) + e) * rows_per + (slot ^ (e & 7)));
          dsmem_st4(dst + off, v);
        }
      }
    }
  }

  __syncwarp();
  if (p.cluster) {
    // Warps 0 and 1 take part in barrier A here; the softmax warps have
    // passed it above.  Barrier B: every row's partials are in its owner.
    if (warp < 2)
      asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    cluster_sync_all();
    if (warp >= 2) {
      // Step 2: merge this CTA's slice from its own shared memory, splits in
      // order; lanes across D (one float4 chunk per lane and step).
      const int S = p.splits;
      const int rows_per = kBM / S;
      const int w = warp - 2;
      const int sel = p.sel_row ? bars->sel : tp.n - 1;
      const long long* tab_row = reinterpret_cast<const long long*>(smem + SM::kTabRow);
      const int* tab_i = reinterpret_cast<const int*>(smem + SM::kTabI);
      const int* tab_bh = reinterpret_cast<const int*>(smem + SM::kTabBh);
      const float* rlse = reinterpret_cast<const float*>(smem + SM::kRecvLse);
      const int nch = DV / 4;                         // float4 chunks of this CTA's columns
      constexpr int CPL = D / 4 >= 32 ? D / 128 : 1;  // chunks per lane (at most)
      const int dcol = dh * DV;
      for (int j = w; j < rows_per; j += 4) {
        const int r = split * rows_per + j;
        const long long orow = tab_row[r];
        if (orow < 0) continue;
        float ls[kMaxClusterSplits];
        float lmax = -INFINITY;
#pragma unroll
        for (int s2 = 0; s2 < kMaxClusterSplits; ++s2) {
          ls[s2] = s2 < S ? rlse[s2 * rows_per + j] : -INFINITY;
          lmax = fmaxf(lmax, ls[s2]);
        }
        // Every split's chunks are loaded before any is used (the loads
        // overlap); splits without live keys are skipped in the sums, which
        // run in split order.
        float4 part[kMaxClusterSplits][CPL];
#pragma unroll
        for (int s2 = 0; s2 < kMaxClusterSplits; ++s2)
#pragma unroll
          for (int q = 0; q < CPL; ++q) {
            const int e = lane + 32 * q;
            part[s2][q] = (s2 < S && e < nch)
                              ? *reinterpret_cast<const float4*>(smem + 16u * ((s2 * nch + e) * rows_per + (j ^ (e & 7))))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        float4 acc[CPL];
#pragma unroll
        for (int q = 0; q < CPL; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        float wsum = 0.f;
        if (lmax != -INFINITY && lane < nch) {
#pragma unroll
          for (int s2 = 0; s2 < kMaxClusterSplits; ++s2) {
            if (s2 >= S || ls[s2] == -INFINITY) continue;
            const float wgt = fast_exp2(ls[s2] - lmax);
            wsum += wgt;
#pragma unroll
            for (int q = 0; q < CPL; ++q) {
              acc[q].x = __fmaf_rn(wgt, part[s2][q].x, acc[q].x);
              acc[q].y = __fmaf_rn(wgt, part[s2][q].y, acc[q].y);
              acc[q].z = __fmaf_rn(wgt, part[s2][q].z, acc[q].z);
              acc[q].w = __fmaf_rn(wgt, part[s2][q].w, acc[q].w);
            }
          }
        }
        if (lane >= nch) continue;
        if (!in_bounds(orow * D, D, n_qo(p), p.err)) continue;
        const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
        const bool is_sel = p.out_sel && tab_i[r] == sel && in_bounds(static_cast<long long>(tab_bh[r]) * D, D, n_sel(p), p.err);
#pragma unroll
        for (int q = 0; q < CPL; ++q) {
          const int e = lane + 32 * q;
          if (e >= nch) break;
          const float4 o = make_float4(acc[q].x * inv, acc[q].y * inv, acc[q].z * inv, acc[q].w * inv);
          *reinterpret_cast<uint2*>(p.out + static_cast<size_t>(orow) * D + dcol + 4 * e) =
              make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
          if (is_sel) *reinterpret_cast<float4*>(p.out_sel + static_cast<size_t>(tab_bh[r]) * D + dcol + 4 * e) = o;
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && bars->abort) set_err(p.err, CPA_EBIT_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Rotated chunk keys for the single-tile kernel: one thread per (row, 8-dim
// chunk pair), the append's fp32 arithmetic.  It lets the dependent attention
// grid start at once.
__global__ void __launch_bounds__(256) rope_chunk_k_kernel(const AttnParams p) {
  grid_launch_dependents();  // the attention grid touches no memory before its own wait
  grid_dependency_wait();    // launched as a dependent: whatever the launches before it wrote
  const int D = p.D;
  const int HP = D / 16;
  const int sh = __ffs(HP) - 1;  // HP is a power of two
  const unsigned k_items = static_cast<unsigned>(p.B) * p.Hkv * p.C * HP;
  const unsigned total = k_items + static_cast<unsigned>(p.B) * p.Hq * p.C * HP;  // < 2^31 (host)
  for (unsigned it = blockIdx.x * 256u + threadIdx.x; it < total; it += gridDim.x * 256u) {
    if (it >= k_items) {
      // a query row's chunk pair, rotated into the workspace (in half for an
      // fp16 cache: the products then run in fp16)
      const unsigned qi = it - k_items;
      const int kc = static_cast<int>(qi & (HP - 1));
      const unsigned qr = qi >> sh;  // row of [B, Hq, C]
      const long long r = qr;
      const int i = static_cast<int>(qr % static_cast<unsigned>(p.C));
      const int b = static_cast<int>(qr / static_cast<unsigned>(p.C) / static_cast<unsigned>(p.Hq));
      if (!in_bounds(r * D, D, n_qo(p), p.err) ||
          !in_bounds((static_cast<long long>(b) * p.C + i) * D, D, n_tab(p), p.err))
        continue;
      const uint16_t* src = p.q + r * D;
      uint4 lo = __ldg(reinterpret_cast<const uint4*>(src + kc * 8));
      uint4 hi = __ldg(reinterpret_cast<const uint4*>(src + D / 2 + kc * 8));
      const float* cr = p.cos + (static_cast<size_t>(b) * p.C + i) * D;
      const float* sr = p.sin + (static_cast<size_t>(b) * p.C + i) * D;
      if (p.f16) rope_pair<true>(lo, hi, cr + kc * 8, sr + kc * 8, cr + D / 2 + kc * 8, sr + D / 2 + kc * 8);
      else rope_pair(lo, hi, cr + kc * 8, sr + kc * 8, cr + D / 2 + kc * 8, sr + D / 2 + kc * 8);
      uint16_t* dst = p.q_rot + r * D;
      *reinterpret_cast<uint4*>(dst + kc * 8) = lo;
      *reinterpret_cast<uint4*>(dst + D / 2 + kc * 8) = hi;
      continue;
    }
    const int kc = static_cast<int>(it & (HP - 1));
    const unsigned rr = it >> sh;  // row of [B, Hkv, C]
    const long long r = rr;
    const int i = static_cast<int>(rr % static_cast<unsigned>(p.C));
    const int b = static_cast<int>(rr / static_cast<unsigned>(p.C) / static_cast<unsigned>(p.Hkv));
    if (!in_bounds(r * D, D, n_chunk(p), p.err) ||
        !in_bounds((static_cast<long long>(b) * p.C + i) * D, D, n_tab(p), p.err))
      continue;
    const uint16_t* src = p.k_new + r * D;
    uint4 lo = __ldg(reinterpret_cast<const uint4*>(src + kc * 8));
    uint4 hi = __ldg(reinterpret_cast<const uint4*>(src + D / 2 + kc * 8));
    const float* cr = p.cos + (static_cast<size_t>(b) * p.C + i) * D;
    const float* sr = p.sin + (static_cast<size_t>(b) * p.C + i) * D;
    if (p.f16) {
      rope_pair<true>(lo, hi, cr + kc * 8, sr + kc * 8, cr + D / 2 + kc * 8, sr + D / 2 + kc * 8);
      // the chunk's values in half, for the P V products
      const uint16_t* vs = p.v_new + r * D;
      uint16_t* vd = p.v_cvt + r * D;
      *reinterpret_cast<uint4*>(vd + kc * 8) = bf16x8_to_f16x8(__ldg(reinterpret_cast<const uint4*>(vs + kc * 8)));
      *reinterpret_cast<uint4*>(vd + D / 2 + kc * 8) =
          bf16x8_to_f16x8(__ldg(reinterpret_cast<const uint4*>(vs + D / 2 + kc * 8)));
    } else {
      rope_pair(lo, hi, cr + kc * 8, sr + kc * 8, cr + D / 2 + kc * 8, sr + D / 2 + kc * 8);
    }
    uint16_t* dst = p.k_rot + r * D;
    *reinterpret_cast<uint4*>(dst + kc * 8) = lo;
    *reinterpret_cast<uint4*>(dst + D / 2 + kc * 8) = hi;
    if (p.app_n) fused_append_pair(p, b, static_cast<int>((r / p.C) % p.Hkv), i, kc, lo, hi);
  }
}

// Fused append's length update, after the attention grid (and its merge).
__global__ void fused_len_kernel(const AttnParams p) {
  grid_dependency_wait();
  for (int b = threadIdx.x; b < p.B; b += blockDim.x) fused_append_len(p, b);
}

// Merge split-KV partials in fixed split order: one warp per output row.
__global__ void combine_kernel(const AttnParams p) {
  grid_dependency_wait();  // partials of the attention grid before it
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  const int rows = p.B * p.Hq * p.C;
  if (warp_global >= rows) return;
  const size_t row = warp_global;
  const int i = static_cast<int>(row % p.C);
  const int bh = static_cast<int>(row / p.C);
  const int b = bh / p.Hq;
  const int h = bh % p.Hq;
  const size_t stride = static_cast<size_t>(rows);
  if (!in_bounds((static_cast<long long>(p.splits - 1) * stride + row) * p.D, p.D, p.n_part, p.err) ||
      !in_bounds(static_cast<long long>(row) * p.D, p.D, n_qo(p), p.err) ||
      !in_bounds((static_cast<long long>(b) * p.Hq + h) * p.D, p.D, n_sel(p), p.err))
    return;
  // the splits' log2-sum-exps spread over the lanes, then the warp's maximum
  float lmax = -INFINITY;
  for (int s = lane; s < p.splits; s += 32) lmax = fmaxf(lmax, p.part_lse[s * stride + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
  const int D = p.D;
  const int per = D / 32;  // 2, 4 or 8 values per lane
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (lmax != -INFINITY) {
    // splits in order, four at a time with their loads issued before use
    constexpr int kB = 4;
    for (int s0 = 0; s0 < p.splits; s0 += kB) {
      float ls[kB], o[kB][8];
#pragma unroll
      for (int k = 0; k < kB; ++k) {
        ls[k] = -INFINITY;
        if (s0 + k < p.splits) {
          const size_t sr = (s0 + k) * stride + row;
          ls[k] = p.part_lse[sr];
          const float* src = p.part_o + sr * D + lane * per;
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            if (e < per) {
              const float2 v = *reinterpret_cast<const float2*>(src + e);
              o[k][e] = v.x;
              o[k][e + 1] = v.y;
            }
          }
        }
      }
#pragma unroll
      for (int k = 0; k < kB; ++k) {
        if (ls[k] == -INFINITY) continue;
        const float w = fast_exp2(ls[k] - lmax);
        wsum += w;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (e < per) acc[e] = __fmaf_rn(w, o[k][e], acc[e]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  int n = p.n_real ? min(max(p.n_real[b], 0), p.C) : p.C;
  const int sel = p.sel_row ? p.sel_row[b] : n - 1;
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    if (e < per) {
      const float o0 = acc[e] * inv, o1 = acc[e + 1] * inv;
      *reinterpret_cast<uint32_t*>(p.out + row * D + lane * per + e) = pack_bf16x2(o0, o1);
      if (p.out_sel && i == sel) {
        float* sd = p.out_sel + (static_cast<size_t>(b) * p.Hq + h) * D + lane * per + e;
        sd[0] = o0;
        sd[1] = o1;
      }
    }
  }
}

// ------------------------------------------------------------------ host side

template <int D, int BN, bool F16>
static cudaError_t launch_attn_t(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream) {
  using SM = AttnSmem<D, BN>;
  auto kern = attn_kernel<D, BN, F16>;
  static SmemAttr smem_attr;
  if (cudaError_t e = smem_attr.ensure(reinterpret_cast<const void*>(kern), SM::kAlloc, true); e != cudaSuccess)
    return e;
  dim3 grid(p.nq * p.splits * p.dsplit, p.Hkv, p.B);
  const long long items = static_cast<long long>(p.B) * (p.Hkv + p.Hq) * p.C * (D / 16);
  const int kblocks = static_cast<int>(max(1LL, min(static_cast<long long>(152) * 8, (items + 255) / 256)));
  cudaError_t e = launch_dependent(rope_chunk_k_kernel, dim3(kblocks), dim3(256), 0, stream, p);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SM::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (p.cluster) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = p.splits * p.dsplit;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], p);
}

// How many clusters of `size` CTAs of attn_kernel<D, BN> can be resident at
// once (the fp16 instantiation has the same resources; above 8 a cluster size
// is non-portable and must be allowed first); 0 when none fits.
template <int D, int BN>
static int cluster_count(int size) {
  using SM = AttnSmem<D, BN>;
  auto kern = attn_kernel<D, BN, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kAlloc) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(size);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SM::kAlloc;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = size;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n > 0 ? n : 0;
}

static cudaError_t launch_combine(const AttnParams& p, cudaStream_t stream) {
  const int rows = p.B * p.Hq * p.C;
  const int threads = 256;
  const int blocks = (rows * 32 + threads - 1) / threads;
  return launch_dependent(combine_kernel, dim3(blocks), dim3(threads), 0, stream, p);
}

int attn_block_n(int D) { return D == 256 ? 64 : 128; }

cudaError_t launch_fused_append_len(const AttnParams& p, cudaStream_t stream) {
  return launch_dependent(fused_len_kernel, dim3(1), dim3(256), 0, stream, p);
}

int attn_max_clusters(int D, int size) {
  if (size < 2 || size > kMaxClusterSize) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  // per device, head dim and cluster size: -1 unknown, else the count
  static int known[16][3][kMaxClusterSize + 1];
  static bool init = [] {
    for (auto& a : known)
      for (auto& b2 : a)
        for (int& k : b2) k = -1;
    return true;
  }();
  (void)init;
  const int di = D == 64 ? 0 : (D == 128 ? 1 : 2);
  if (dev < 0 || dev >= 16) return 0;
  int& k = known[dev][di][size];
  if (k < 0) {
    int n = 0;
    switch (D) {
      case 64: n = cluster_count<64, 128>(size); break;
      case 128: n = cluster_count<128, 128>(size); break;
      case 256: n = cluster_count<256, 64>(size); break;
      default: break;
    }
    k = n;
  }
  return k;
}

bool attn_cluster_ok(int D, int size) { return attn_max_clusters(D, size) > 0; }

cudaError_t launch_attn(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream) {
  cudaError_t e;
  if (attn_uses_decode(p.D, p.C, p.G)) {
    e = launch_attn_decode(maps, p, stream);
  } else {
    switch (p.D) {
      case 64:
        e = p.f16 ? launch_attn_t<64, 128, true>(maps, p, stream) : launch_attn_t<64, 128, false>(maps, p, stream);
        break;
      case 128:
        e = p.f16 ? launch_attn_t<128, 128, true>(maps, p, stream) : launch_attn_t<128, 128, false>(maps, p, stream);
        break;
      case 256:
        e = p.f16 ? launch_attn_t<256, 64, true>(maps, p, stream) : launch_attn_t<256, 64, false>(maps, p, stream);
        break;
      default: return cudaErrorInvalidValue;
    }
  }
  if (e != cudaSuccess || p.splits == 1 || p.cluster) return e;
  return launch_combine(p, stream);
}

}  // namespace cpa
