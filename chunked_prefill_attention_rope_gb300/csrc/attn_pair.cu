// Chunk-prefill attention for head dims 64 and 128 with two query tiles per CTA.
//
// Same computation as attn_kernel ("functiongemma: chunk prefill-with-past
// graph", Change: RoPE'd queries attend over past + chunk keys under an
// additive mask), organised so the tensor core never waits for softmax:
//
//   * A CTA owns 256 packed query rows of one (sequence, kv head), split into
//     query tiles Q0 and Q1 of 128 rows; both use every K/V tile the CTA loads.
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
// 32*(w%4)..+31), 8 TMA producer, 9 MMA issuer, 10-11 rotate raw chunk-K tiles
// in shared memory.
#include "tiles.cuh"

namespace cpa {

namespace {

constexpr int kBN = 128;
constexpr int kThreadsPair = 384;

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
};

struct __align__(8) PairBars {
  uint64_t k_full[4], v_full[4], kv_empty[4], k_rot[4];
  uint64_t s_full[2], p_full[2], o_done[2], q_ready[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

template <int D>
constexpr int pair_smem_bytes() {
  return PairCfg<D>::kBars + static_cast<int>(sizeof(PairBars)) + 1024;
}

}  // namespace

template <int D, bool EXPLICIT>
__global__ void __launch_bounds__(kThreadsPair, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap map_kc, const __grid_constant__ CUtensorMap map_vc,
                     const __grid_constant__ CUtensorMap map_kn, const __grid_constant__ CUtensorMap map_vn,
                     const AttnParams p) {
  using CF = PairCfg<D>;
  constexpr int NS = CF::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PairBars* bars = reinterpret_cast<PairBars*>(smem + CF::kBars);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int pair = blockIdx.x / p.splits;
  const int split = blockIdx.x % p.splits;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int i_min = pair * 2 * p.R;
  const int i_max = min(i_min + 2 * p.R, p.C) - 1;
  const TilePlan tp = plan_tiles<kBN>(p, b, i_min, i_max, split);
  const int nt = tp.count();

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
      mbar_init(&bars->k_rot[s], 64);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 128);
      mbar_init(&bars->o_done[s], 1);
      mbar_init(&bars->q_ready[s], 128);
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_barrier_init();
    if (kvh == 0 && blockIdx.x == 0) {
      if (p.past_len && (p.past_len[b] < 0 || p.past_len[b] > p.P)) set_err(p.err, CPA_EBIT_PAST_GT_SPAN);
      if (p.n_real && (p.n_real[b] < 0 || p.n_real[b] > p.C)) set_err(p.err, CPA_EBIT_NREAL_GT_C);
    }
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  uint8_t* sK = smem + CF::kK;
  uint8_t* sV = smem + CF::kV;

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && nt > 0) {
      prefetch_tensormap(&map_kc);
      prefetch_tensormap(&map_vc);
      prefetch_tensormap(&map_kn);
      prefetch_tensormap(&map_vn);
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int st = j % NS;
        if (!mbar_wait(&bars->kv_empty[st], ((j / NS) + 1) & 1, abort)) break;
        const int t = tp.index(j);
        const bool chunk = t < tp.Tc;
        const int base = (chunk ? t : t - tp.Tc) * kBN;
        const CUtensorMap* mk = chunk ? &map_kn : &map_kc;
        const CUtensorMap* mv = chunk ? &map_vn : &map_vc;
        mbar_arrive_expect_tx(&bars->k_full[st], CF::kKBytes);
#pragma unroll
        for (int blk = 0; blk < D / 64; ++blk)
          tma_load_4d(sK + st * CF::kKBytes + blk * kBN * 128, mk, &bars->k_full[st], blk * 64, base, kvh, b);
        mbar_arrive_expect_tx(&bars->v_full[st], CF::kVBytes);
#pragma unroll
        for (int blk = 0; blk < D / 64; ++blk)
          tma_load_4d(sV + st * CF::kVBytes + blk * kBN * 128, mv, &bars->v_full[st], blk * 64, base, kvh, b);
        issued = j + 1;
      }
      for (int j = max(0, issued - NS); j < issued; ++j) {  // let copies in flight land
        const int st = j % NS;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&bars->v_full[st], (j / NS) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
        while (!mbar_try_wait(&bars->k_full[st], (j / NS) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(128, kBN, false);
      constexpr uint32_t idesc_pv = idesc_bf16(128, D, true);
      const uint32_t q_addr = smem_u32(smem + CF::kQ);
      bool ok = nt > 0 && mbar_wait(&bars->q_ready[0], 0, abort) && mbar_wait(&bars->q_ready[1], 0, abort);
      auto k_ready = [&](int j) -> bool {
        const int st = j % NS;
        const bool chunk = tp.index(j) < tp.Tc;
        return mbar_wait(chunk ? &bars->k_rot[st] : &bars->k_full[st], (j / NS) & 1, abort);
      };
      auto issue_qk = [&](int i, int j) {
        const uint32_t k_addr = smem_u32(sK + (j % NS) * CF::kKBytes);
        const uint32_t qa = q_addr + i * CF::kQBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t a = sdesc_sw128(qa + (kk / 4) * (128 * 128) + (kk % 4) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(k_addr + (kk / 4) * (kBN * 128) + (kk % 4) * 32, 16, 1024);
          mma_bf16_ss(tmem + i * kBN, a, bd, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full[i]);
      };
      auto issue_pv = [&](int i, int j) {
        const uint32_t v_addr = smem_u32(sV + (j % NS) * CF::kVBytes);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t bd = sdesc_sw128(v_addr + kk * 2048, kBN * 128, 1024);
          mma_bf16_ts(tmem + CF::kOCol + i * D, tmem + i * kBN + kk * 8, bd, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
      };
      if (ok && (ok = k_ready(0))) {
        tc_fence_after();
        issue_qk(0, 0);
        issue_qk(1, 0);
      }
      for (int j = 0; ok && j < nt; ++j) {
        const int st = j % NS;
        if (!(ok = mbar_wait(&bars->p_full[0], j & 1, abort) && mbar_wait(&bars->v_full[st], (j / NS) & 1, abort)))
          break;
        tc_fence_after();
        issue_pv(0, j);
        if (j + 1 == nt) mma_commit(&bars->o_done[0]);
        if (j + 1 < nt) {
          if (!(ok = k_ready(j + 1))) break;
          tc_fence_after();
          issue_qk(0, j + 1);
        }
        if (!(ok = mbar_wait(&bars->p_full[1], j & 1, abort))) break;
        tc_fence_after();
        issue_pv(1, j);
        mma_commit(&bars->kv_empty[st]);
        if (j + 1 == nt) mma_commit(&bars->o_done[1]);
        if (j + 1 < nt) issue_qk(1, j + 1);
      }
      mma_commit(&bars->mma_done);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&bars->mma_done, 0) && global_timer_ns() - t0 < kWaitLimitNs) {}
    }
    __syncwarp();
  } else if (warp >= 10) {
    // ------------------------------------------------------------ chunk-K rotation
    const int tid = threadIdx.x - 320;  // 0..63
    for (int j = 0; j < nt; ++j) {
      const int t = tp.index(j);
      if (t >= tp.Tc) break;  // chunk tiles come first
      const int st = j % NS;
      if (!warp_all(mbar_wait(&bars->k_full[st], (j / NS) & 1, abort))) break;
      uint8_t* kt = sK + st * CF::kKBytes;
      const int base = t * kBN;
      for (int item = tid; item < kBN * (D / 16); item += 64) {
        const int r = item / (D / 16);
        const int kc = item % (D / 16);
        const int row = base + r;
        if (row >= p.C) continue;
        const int kh = kc + D / 16;
        uint4* plo = reinterpret_cast<uint4*>(kt + (kc / 8) * (kBN * 128) + sw128(r, kc % 8));
        uint4* phi = reinterpret_cast<uint4*>(kt + (kh / 8) * (kBN * 128) + sw128(r, kh % 8));
        uint4 lo = *plo, hi = *phi;
        const float* cr = p.cos + (static_cast<size_t>(b) * p.C + row) * D;
        const float* sr = p.sin + (static_cast<size_t>(b) * p.C + row) * D;
        rope_pair(lo, hi, cr + kc * 8, sr + kc * 8, cr + D / 2 + kc * 8, sr + D / 2 + kc * 8);
        *plo = lo;
        *phi = hi;
      }
      fence_async_smem();
      mbar_arrive(&bars->k_rot[st]);
    }
  } else {
    // ------------------------------------------------------------ softmax (query tile qi)
    const int qi = warp / 4;
    const int tid = threadIdx.x - qi * 128;
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lanes = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t s_col = tmem + lanes + qi * kBN;
    const uint32_t o_col = tmem + lanes + CF::kOCol + qi * D;
    const int qt = pair * 2 + qi;
    const int g = row / p.R;
    const int i = qt * p.R + row % p.R;
    const bool valid = g < p.G && i < p.C;
    const int h = kvh * p.G + (valid ? g : 0);

    // rotated Q rows into the swizzled K-major operand tile
    uint8_t* sQ = smem + CF::kQ + qi * CF::kQBytes;
    for (int item = tid; item < 128 * (D / 16); item += 128) {
      const int r = item / (D / 16);
      const int kc = item % (D / 16);
      const int rg = r / p.R;
      const int ri = qt * p.R + r % p.R;
      uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
      if (rg < p.G && ri < p.C) {
        const size_t off = ((static_cast<size_t>(b) * p.Hq + kvh * p.G + rg) * p.C + ri) * D;
        lo = *reinterpret_cast<const uint4*>(p.q + off + kc * 8);
        hi = *reinterpret_cast<const uint4*>(p.q + off + D / 2 + kc * 8);
        const float* cr = p.cos + (static_cast<size_t>(b) * p.C + ri) * D;
        const float* sr = p.sin + (static_cast<size_t>(b) * p.C + ri) * D;
        rope_pair(lo, hi, cr + kc * 8, sr + kc * 8, cr + D / 2 + kc * 8, sr + D / 2 + kc * 8);
      }
      const int kh = kc + D / 16;
      *reinterpret_cast<uint4*>(sQ + (kc / 8) * (128 * 128) + sw128(r, kc % 8)) = lo;
      *reinterpret_cast<uint4*>(sQ + (kh / 8) * (128 * 128) + sw128(r, kh % 8)) = hi;
    }
    fence_async_smem();
    mbar_arrive(&bars->q_ready[qi]);

    RowSpan span;
    span.init(p, tp, i, valid);
    const float* mrow = nullptr;
    if (EXPLICIT && valid)
      mrow = p.mask + ((static_cast<size_t>(b) * p.Hq + h) * p.C + i) * static_cast<size_t>(p.P + p.C);
    const float sl2 = p.sl2;
    float m_run = kMaskedLog2, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int t = tp.index(j);
      const bool chunk = t < tp.Tc;
      const int base = (chunk ? t : t - tp.Tc) * kBN;
      int lo, hi;
      span.tile(chunk, base, lo, hi);
      const float* mp = nullptr;
      int lim = 0;
      if (EXPLICIT) {
        lim = chunk ? p.C - base : p.P - base;
        if (mrow) mp = mrow + (chunk ? p.P + base : base);
      }
      if (!(ok = warp_all(mbar_wait(&bars->s_full[qi], j & 1, abort)))) break;
      tc_fence_after();

      // Scores of this row.  Implicit mask: one batch of TMEM loads, masked keys
      // set to -inf (they give exactly 0 below).  Explicit mask: the row max of
      // scale*s + mask (in log2 units), chunk by chunk.
      float sc[kBN];
      float m_tile;
      if (!EXPLICIT) {
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) tmem_ld32f(s_col + 32 * c, sc + 32 * c);
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) tmem_ld_waitf(sc + 32 * c);
        if (__any_sync(0xffffffffu, lo > 0 || hi < kBN)) {
#pragma unroll
          for (int e = 0; e < kBN; ++e) sc[e] = (e >= lo && e < hi) ? sc[e] : -INFINITY;
        }
        float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
        for (int e = 0; e < kBN; e += 8) {
          m0 = fmax3(m0, sc[e], sc[e + 1]);
          m1 = fmax3(m1, sc[e + 2], sc[e + 3]);
          m2 = fmax3(m2, sc[e + 4], sc[e + 5]);
          m3 = fmax3(m3, sc[e + 6], sc[e + 7]);
        }
        const float mt = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
        m_tile = (mt == -INFINITY) ? kMaskedLog2 : __fmul_rn(mt, sl2);
      } else {
        float mt = -INFINITY;
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(s_col + 32 * c, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int k = 32 * c + e;
            const float mv = (mp && k < lim) ? __ldg(mp + k) : -1e30f;
            mt = fmaxf(mt, __fmaf_rn(__uint_as_float(r[e]), sl2, __fmul_rn(mv, kLog2e)));
          }
        }
        m_tile = mt;
      }
      const float m_new = fmaxf(m_run, m_tile);
      const bool rescale = m_new > m_run + 8.f;
      float factor = 1.f;
      if (rescale) {
        factor = fast_exp2(m_run - m_new);
        m_run = m_new;
      }
      const bool live = m_run > kEmptyRow;
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
        // O holds every earlier P V (the S = Q K that signalled s_full was issued after them)
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(o_col + 32 * c, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
          tmem_st32(o_col + 32 * c, o);
        }
      }
      // P = 2^(scale*log2e*s - m), summed in one fixed order, written over S as bf16
      float2 accA = make_float2(0.f, 0.f), accB = accA;
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) {
        float* pv = sc + 32 * c;
        if (!EXPLICIT) {
          const float nm = live ? -m_run : -INFINITY;
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 x = ffma2(make_float2(pv[e], pv[e + 1]), make_float2(sl2, sl2), make_float2(nm, nm));
            pv[e] = fast_exp2(x.x);
            pv[e + 1] = fast_exp2(x.y);
          }
        } else {
          uint32_t r[32];
          tmem_ld32(s_col + 32 * c, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int k = 32 * c + e;
            const float mv = (mp && k < lim) ? __ldg(mp + k) : -1e30f;
            pv[e] = live ? fast_exp2(__fmaf_rn(__uint_as_float(r[e]), sl2, __fadd_rn(__fmul_rn(mv, kLog2e), -m_run)))
                         : 0.f;
          }
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          accA = fadd2(accA, make_float2(pv[e], pv[e + 1]));
          accB = fadd2(accB, make_float2(pv[e + 2], pv[e + 3]));
          w[e / 2] = pack_bf16x2(pv[e], pv[e + 1]);
          w[e / 2 + 1] = pack_bf16x2(pv[e + 2], pv[e + 3]);
        }
        tmem_st16(s_col + 16 * c, w);
      }
      const float sum = __fadd_rn(__fadd_rn(accA.x, accA.y), __fadd_rn(accB.x, accB.y));
      tmem_st_wait();
      l_run = __fmaf_rn(l_run, factor, sum);
      tc_fence_before();
      mbar_arrive(&bars->p_full[qi]);
    }

    // ---------------------------------------------------------- epilogue
    if (ok && nt > 0) ok = warp_all(mbar_wait(&bars->o_done[qi], 0, abort));
    tc_fence_after();
    const bool empty = !(nt > 0 && ok && m_run > kEmptyRow);
    const float inv_l = empty ? 0.f : 1.f / l_run;
    const int sel = valid ? (p.sel_row ? p.sel_row[b] : tp.n - 1) : -1;
    const size_t orow = (static_cast<size_t>(b) * p.Hq + h) * p.C + i;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o32[32];
      if (nt > 0) {
        tmem_ld32(o_col + 32 * c, o32);
        tmem_ld_wait(o32);
      }
      float o[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = empty ? 0.f : __uint_as_float(o32[e]) * inv_l;
      if (!valid) continue;
      if (p.part_o) {
        float* dst = p.part_o + (static_cast<size_t>(split) * p.B * p.Hq * p.C + orow) * D + 32 * c;
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(dst + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
      } else {
        uint16_t* dst = p.out + orow * D + 32 * c;
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 wv;
          wv.x = pack_bf16x2(o[e + 0], o[e + 1]);
          wv.y = pack_bf16x2(o[e + 2], o[e + 3]);
          wv.z = pack_bf16x2(o[e + 4], o[e + 5]);
          wv.w = pack_bf16x2(o[e + 6], o[e + 7]);
          *reinterpret_cast<uint4*>(dst + e) = wv;
        }
        if (p.out_sel && i == sel) {
          float* sd = p.out_sel + (static_cast<size_t>(b) * p.Hq + h) * D + 32 * c;
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(sd + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
        }
      }
    }
    if (valid && p.part_lse)
      p.part_lse[static_cast<size_t>(split) * p.B * p.Hq * p.C + orow] = empty ? -INFINITY : m_run + __log2f(l_run);
  }

  __syncthreads();
  if (threadIdx.x == 0 && bars->abort) set_err(p.err, CPA_EBIT_TIMEOUT);
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool EXPLICIT>
static cudaError_t launch_pair_t(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream) {
  constexpr int smem = pair_smem_bytes<D>();
  auto kern = attn_pair_kernel<D, EXPLICIT>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int pairs = (p.nq + 1) / 2;
  dim3 grid(pairs * p.splits, p.Hkv, p.B);
  kern<<<grid, kThreadsPair, smem, stream>>>(maps[0], maps[1], maps[2], maps[3], p);
  return cudaGetLastError();
}

cudaError_t launch_attn_pair(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream) {
  const bool ex = p.mask != nullptr;
  switch (p.D) {
    case 64: return ex ? launch_pair_t<64, true>(maps, p, stream) : launch_pair_t<64, false>(maps, p, stream);
    case 128: return ex ? launch_pair_t<128, true>(maps, p, stream) : launch_pair_t<128, false>(maps, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cpa
