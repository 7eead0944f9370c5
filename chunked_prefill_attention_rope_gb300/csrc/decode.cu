// One-token decode attention ("[quanization] Enable prefill-decode modeling",
// Runtime behavior / Mask/cache layout: a single new token attends over the
// valid past slots plus its own key; no causal mask is needed).
//
// Decode is bound by reading the KV cache once, and carries little arithmetic:
// the G query heads that share a kv head form G rows of a 16-row warp-level
// MMA tile, which is plenty of tensor throughput.  The kernel therefore spends
// its effort on keeping HBM busy:
//
//   * CTA = (sequence, kv head, split); the split owns a fixed range of the
//     key-tile index space (64-key tiles, tiles.cuh), so ~1-2k keys per CTA.
//   * Warp 4 streams K and V tiles with TMA into a 3-stage ring (96 KB at
//     D = 128, so two CTAs share an SM and keep ~190 KB of loads in flight).
//   * Warps 0-3 each take 16 keys of every tile: S = Q K^T and O += P V with
//     mma.sync m16n8k16 (bf16 in, or fp16 with an fp16 KV cache; fp32
//     accumulate), operands from the
//     swizzled tiles with ldmatrix.  Each warp keeps its own running max, sum
//     and O; the four are merged through shared memory at the end.
//
// Scores use the same arithmetic as the tcgen05 kernels (log2 domain, fused
// scale, rescale only when the max grows by more than 2^8, masked scores
// contribute exactly 0), so the explicit and implicit masks agree bitwise.
#include "tiles.cuh"

namespace cpa {

namespace {

constexpr int kDBN = 64;        // keys per tile
constexpr int kDThreads = 160;  // 4 MMA warps + 1 producer warp

template <int D>
struct DecCfg {
  static constexpr int kStages = D == 64 ? 6 : 3;
  static constexpr int kTile = kDBN * D * 2;  // bytes of one K (or V) tile
  static constexpr int kK = 0;
  static constexpr int kV = kStages * kTile;
  static constexpr int kBars = 2 * kStages * kTile;
  static constexpr int kSmem = kBars + 256 + 1024;
};

struct __align__(8) DecBars {
  uint64_t full[6], empty[6];
  int abort;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// C(16x8, fp32) += A(16x16, row) * B(16x8, col), A and B bf16 (or fp16 for
// an fp16 KV cache)
template <bool F16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (F16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Byte offset of (row, 16-byte chunk c along D) in a tile stored as D/64
// blocks of [64 rows x 128 B] with the 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_off(int row, int c) {
  return (c >> 3) * (kDBN * 128) + sw128(row, c & 7);
}

}  // namespace

template <int D, bool EXPLICIT, bool F16>
__global__ void __launch_bounds__(kDThreads, 2)
    attn_decode_kernel(const __grid_constant__ CUtensorMap map_kc, const __grid_constant__ CUtensorMap map_vc,
                       const __grid_constant__ CUtensorMap map_kn, const __grid_constant__ CUtensorMap map_vn,
                       const AttnParams p) {
  using CF = DecCfg<D>;
  constexpr int NS = CF::kStages;
  // combine_kernel may be scheduled now (on a partial SM budget, as this grid
  // ends); it waits for this grid
  if (!p.hold_dependents) grid_launch_dependents();
  grid_dependency_wait();  // launched as a dependent: whatever the launches before it wrote
  constexpr int KS = D / 16;  // k-steps of S = Q K^T
  constexpr int NB = D / 8;   // n-blocks of O
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  DecBars* bars = reinterpret_cast<DecBars*>(smem + CF::kBars);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const TilePlan tp = plan_tiles<kDBN>(p, b, 0, 0, split);
  const int nt = tp.count();

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 4);
    }
    bars->abort = 0;
    fence_barrier_init();
    if (kvh == 0 && split == 0) {
      if (p.past_len && (p.past_len[b] < 0 || p.past_len[b] > p.P)) set_err(p.err, CPA_EBIT_PAST_GT_SPAN);
      if (p.n_real && (p.n_real[b] < 0 || p.n_real[b] > p.C)) set_err(p.err, CPA_EBIT_NREAL_GT_C);
    }
  }
  __syncthreads();

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && nt > 0) {
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int st = j % NS;
        if (!mbar_wait(&bars->empty[st], ((j / NS) + 1) & 1, abort)) break;
        const int t = tp.index(j);
        const bool chunk = t < tp.Tc;
        const int base = (chunk ? t : t - tp.Tc) * kDBN;
        mbar_arrive_expect_tx(&bars->full[st], 2 * CF::kTile);
#pragma unroll
        for (int blk = 0; blk < D / 64; ++blk) {
          tma_load_4d(smem + CF::kK + st * CF::kTile + blk * kDBN * 128, chunk ? &map_kn : &map_kc, &bars->full[st],
                      blk * 64, base, kvh, b);
          tma_load_4d(smem + CF::kV + st * CF::kTile + blk * kDBN * 128, chunk ? &map_vn : &map_vc, &bars->full[st],
                      blk * 64, base, kvh, b);
        }
        issued = j + 1;
      }
      for (int j = max(0, issued - NS); j < issued; ++j) {  // let copies in flight land
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&bars->full[j % NS], (j / NS) & 1) && global_timer_ns() - t0 < kWaitLimitNs) {}
      }
    }
  }

  // -------------------------------------------------------------- MMA warps
  float o[D / 8][4];
  float m_run[2] = {kMaskedLog2, kMaskedLog2};
  float l_run[2] = {0.f, 0.f};
  bool ok = true;
  const int r0 = lane >> 2;        // fragment rows r0 and r0 + 8
  const int c2 = (lane & 3) * 2;   // fragment column pair
  if (warp < 4) {
  // Q fragments, rotated (rows >= G are zero).
  uint32_t qa[KS][4];
  {
    // checked builds: an out-of-range table row reads as zeros
    const bool tab_ok = in_bounds(static_cast<long long>(b) * D, D, n_tab(p), p.err);
    const float* cr = p.cos + (tab_ok ? static_cast<size_t>(b) * D : 0);
    const float* sr = p.sin + (tab_ok ? static_cast<size_t>(b) * D : 0);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int g = r0 + 8 * half;
      const bool ok = g < p.G && tab_ok &&
                      in_bounds((static_cast<long long>(b) * p.Hq + kvh * p.G + g) * D, D, n_qo(p), p.err);
      const uint16_t* qrow = p.q + (static_cast<size_t>(b) * p.Hq + kvh * p.G + (ok ? g : 0)) * D;
#pragma unroll
      for (int k = 0; k < KS / 2; ++k) {
#pragma unroll
        for (int hi8 = 0; hi8 < 2; ++hi8) {
          const int d = 16 * k + c2 + 8 * hi8;   // and d + 1; partners at d + D/2
          float x0 = 0.f, x1 = 0.f, z0 = 0.f, z1 = 0.f;
          if (ok) {
            const uint32_t lo = *reinterpret_cast<const uint32_t*>(qrow + d);
            const uint32_t hh = *reinterpret_cast<const uint32_t*>(qrow + d + D / 2);
            x0 = bf16_lo(lo); x1 = bf16_hi(lo); z0 = bf16_lo(hh); z1 = bf16_hi(hh);
          }
          const float y0 = __fsub_rn(__fmul_rn(x0, cr[d]), __fmul_rn(z0, sr[d]));
          const float y1 = __fsub_rn(__fmul_rn(x1, cr[d + 1]), __fmul_rn(z1, sr[d + 1]));
          const float u0 = __fadd_rn(__fmul_rn(z0, cr[d + D / 2]), __fmul_rn(x0, sr[d + D / 2]));
          const float u1 = __fadd_rn(__fmul_rn(z1, cr[d + D / 2 + 1]), __fmul_rn(x1, sr[d + D / 2 + 1]));
          // register slot: a0 (row r0, cols c2), a1 (row r0+8, c2), a2 (row r0, c2+8), a3 (row r0+8, c2+8)
          const int slot = half + 2 * hi8;
          qa[k][slot] = pack16x2<F16>(y0, y1);
          qa[k + KS / 2][slot] = pack16x2<F16>(u0, u1);
        }
      }
    }
  }

#pragma unroll
  for (int n = 0; n < NB; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  const float sl2 = p.sl2;
  const int W = p.window;
  const int L = tp.L;
  const int past_lo = W > 0 ? max(0, L - W + 1) : 0;
  const int sinkL = min(p.sink, L);  // pinned sink slots stay visible
  const float* mrow[2] = {nullptr, nullptr};
  if (EXPLICIT) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int g = r0 + 8 * half;
      const long long mo = (static_cast<long long>(b) * p.Hq + kvh * p.G + g) * (static_cast<long long>(p.P) + p.C);
      if (g < p.G && in_bounds(mo, static_cast<long long>(p.P) + p.C, n_mask(p), p.err)) mrow[half] = p.mask + mo;
    }
  }
  const uint32_t kbase = smem_u32(smem + CF::kK);
  const uint32_t vbase = smem_u32(smem + CF::kV);
  const int key0 = 16 * warp;  // this warp's keys inside a tile

  for (int j = 0; j < nt; ++j) {
    const int st = j % NS;
    if (!(ok = warp_all(mbar_wait(&bars->full[st], (j / NS) & 1, abort)))) break;
    const int t = tp.index(j);
    const bool chunk = t < tp.Tc;
    const int base = (chunk ? t : t - tp.Tc) * kDBN;
    const uint32_t kt = kbase + st * CF::kTile;
    const uint32_t vt = vbase + st * CF::kTile;
    if (chunk) {
      // rotate the chunk rows (the new token) in place before any warp reads them
      for (int item = threadIdx.x; item < kDBN * (D / 16); item += 128) {
        const int r = item / (D / 16);
        const int kc = item % (D / 16);
        if (base + r >= p.C) continue;
        const int kh = kc + D / 16;
        uint8_t* ktile = smem + CF::kK + st * CF::kTile;
        uint4* plo = reinterpret_cast<uint4*>(ktile + tile_off(r, kc));
        uint4* phi = reinterpret_cast<uint4*>(ktile + tile_off(r, kh));
        uint4 lo = *plo, hi = *phi;
        if (!in_bounds((static_cast<long long>(b) * p.C + base + r) * D, D, n_tab(p), p.err)) continue;
        const float* cr = p.cos + (static_cast<size_t>(b) * p.C + base + r) * D;
        const float* sr = p.sin + (static_cast<size_t>(b) * p.C + base + r) * D;
        rope_pair<F16>(lo, hi, cr + kc * 8, sr + kc * 8, cr + D / 2 + kc * 8, sr + D / 2 + kc * 8);
        *plo = lo;
        *phi = hi;
        if (F16) {  // the chunk's values, bf16 -> half, in place
          uint8_t* vtile = smem + CF::kV + st * CF::kTile;
          uint4* qlo = reinterpret_cast<uint4*>(vtile + tile_off(r, kc));
          uint4* qhi = reinterpret_cast<uint4*>(vtile + tile_off(r, kh));
          *qlo = bf16x8_to_f16x8(*qlo);
          *qhi = bf16x8_to_f16x8(*qhi);
        }
      }
      fence_async_smem();  // the ring slot is refilled by TMA later
      asm volatile("bar.sync 1, 128;" ::: "memory");
    }

    if (!EXPLICIT && !chunk) {
      // dead V rows among this warp's keys (cache slots past the length) are
      // cleared before its P V product reads them: P is zero there, but 0
      // times a non-finite value is not
      const int z0 = max(L - base, key0), z1 = min(min(p.P - base, kDBN), key0 + 16);
      if (z0 < z1) {
        zero_tile_rows<D>(smem + CF::kV + st * CF::kTile, kDBN, z0, z1, lane, 32);
        fence_async_smem();  // the ring slot is refilled by TMA later
        __syncwarp();
      }
    }

    // S = Q K^T for 16 keys: two n-blocks of 8 keys
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      const int mtx = lane >> 3;  // matrix: (keys 0-7 | 8-15) x (d chunk 2k | 2k+1)
      const int row = key0 + (mtx >> 1) * 8 + (lane & 7);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kt + tile_off(row, 2 * k + (mtx & 1)), b0, b1, b2, b3);
      mma16816<F16>(s[0], qa[k][0], qa[k][1], qa[k][2], qa[k][3], b0, b1);
      mma16816<F16>(s[1], qa[k][0], qa[k][1], qa[k][2], qa[k][3], b2, b3);
    }

    // scores -> masked log2-domain values; this thread holds rows r0 (idx 0,1) and r0+8 (idx 2,3)
    float mt[2];
    float x[2][4];   // [n-block][slot]
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      float m = -INFINITY;
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kk = key0 + nb * 8 + c2 + e;   // key inside the tile
          const int key = base + kk;
          const float sv = s[nb][2 * hf + e];
          float v;
          if (EXPLICIT) {
            const int lim = chunk ? p.C : p.P;
            const float mv = (mrow[hf] && key < lim) ? __ldg(mrow[hf] + (chunk ? p.P + key : key)) : -1e30f;
            v = __fmaf_rn(sv, sl2, __fmul_rn(mv, kLog2e));
            x[nb][2 * hf + e] = v;
          } else {
            const bool vis = chunk ? (key < tp.n) : ((key >= past_lo || key < sinkL) && key < L);
            v = vis ? sv : -INFINITY;
            x[nb][2 * hf + e] = v;
          }
          m = fmaxf(m, v);
        }
      }
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      mt[hf] = EXPLICIT ? m : (m == -INFINITY ? kMaskedLog2 : __fmul_rn(m, sl2));
    }
    float factor[2];
    bool live[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const float m_new = fmaxf(m_run[hf], mt[hf]);
      factor[hf] = 1.f;
      if (m_new > m_run[hf] + 8.f) {
        factor[hf] = fast_exp2(m_run[hf] - m_new);
        m_run[hf] = m_new;
      }
      live[hf] = m_run[hf] > kEmptyRow;
    }
    // P (bf16) as the A operand of O += P V; partial sums in a fixed order
    float psum[2] = {0.f, 0.f};
    uint32_t pa[4];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float pv[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float v = x[nb][2 * hf + e];
          if (EXPLICIT) {
            const int key = base + key0 + nb * 8 + c2 + e;
            const int lim = chunk ? p.C : p.P;
            const float mv = (mrow[hf] && key < lim) ? __ldg(mrow[hf] + (chunk ? p.P + key : key)) : -1e30f;
            pv[e] = live[hf] ? fast_exp2(__fmaf_rn(s[nb][2 * hf + e], sl2, __fadd_rn(__fmul_rn(mv, kLog2e), -m_run[hf])))
                             : 0.f;
          } else {
            pv[e] = live[hf] ? fast_exp2(__fmaf_rn(v, sl2, -m_run[hf])) : 0.f;
          }
        }
        psum[hf] = __fadd_rn(psum[hf], __fadd_rn(pv[0], pv[1]));
        pa[hf + 2 * nb] = pack16x2<F16>(pv[0], pv[1]);
      }
    }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) l_run[hf] = __fmaf_rn(l_run[hf], factor[hf], psum[hf]);
#pragma unroll
    for (int n = 0; n < NB; ++n) {
      o[n][0] *= factor[0];
      o[n][1] *= factor[0];
      o[n][2] *= factor[1];
      o[n][3] *= factor[1];
    }
    // O += P V: V^T fragments with ldmatrix.trans, two n-blocks of D per load
#pragma unroll
    for (int n2 = 0; n2 < NB / 2; ++n2) {
      const int mtx = lane >> 3;  // (keys 0-7 | 8-15) x (d chunk 2n2 | 2n2+1)
      const int row = key0 + (mtx & 1) * 8 + (lane & 7);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vt + tile_off(row, 2 * n2 + (mtx >> 1)), b0, b1, b2, b3);
      mma16816<F16>(o[2 * n2], pa[0], pa[1], pa[2], pa[3], b0, b1);
      mma16816<F16>(o[2 * n2 + 1], pa[0], pa[1], pa[2], pa[3], b2, b3);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->empty[st]);
  }
  }  // warp < 4

  // -------------------------------------------------------------- merge the four warps
  __syncthreads();  // all stages consumed and every copy landed: the ring is free
  float* red = reinterpret_cast<float*>(smem);           // [4 warps][16 rows][D] O
  float* ml = red + 4 * 16 * D;                          // [4 warps][16 rows][2] (m, l)
#pragma unroll
  for (int hf = 0; hf < 2 && warp < 4; ++hf) {
    float l = l_run[hf];
    l = __fadd_rn(l, __shfl_xor_sync(0xffffffffu, l, 1));
    l = __fadd_rn(l, __shfl_xor_sync(0xffffffffu, l, 2));
    const int row = r0 + 8 * hf;
    if ((lane & 3) == 0) {
      ml[(warp * 16 + row) * 2 + 0] = m_run[hf];
      ml[(warp * 16 + row) * 2 + 1] = l;
    }
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      red[(warp * 16 + row) * D + 8 * n + c2] = o[n][2 * hf];
      red[(warp * 16 + row) * D + 8 * n + c2 + 1] = o[n][2 * hf + 1];
    }
  }
  __syncthreads();
  // 128 threads: row g = threadIdx / 8 (16 rows), 8 threads per row over D
  if (warp < 4) {
    const int row = threadIdx.x / 8;
    const int part = threadIdx.x % 8;
    const int g = row;
    const bool valid = g < p.G && ok;
    float M = kMaskedLog2;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, ml[(w * 16 + row) * 2]);
    const bool empty = !(M > kEmptyRow) || nt == 0 || !ok;
    float wgt[4], lsum = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float mw = ml[(w * 16 + row) * 2];
      wgt[w] = (empty || !(mw > kEmptyRow)) ? 0.f : fast_exp2(mw - M);
      lsum = __fmaf_rn(wgt[w], ml[(w * 16 + row) * 2 + 1], lsum);
    }
    const float inv = empty ? 0.f : 1.f / lsum;
    const bool rows_ok =
        g < p.G && in_bounds(static_cast<long long>(b * p.Hq + kvh * p.G + g) * D, D, n_qo(p), p.err) &&
        (!p.part_o || in_bounds((static_cast<long long>(split) * p.B * p.Hq + b * p.Hq + kvh * p.G + g) * D, D,
                                p.n_part, p.err));
    if (rows_ok) {
      const int h = kvh * p.G + g;
      const size_t orow = static_cast<size_t>(b) * p.Hq + h;  // C == 1
      const int sel = p.sel_row ? p.sel_row[b] : tp.n - 1;
      for (int d0 = part * (D / 8); d0 < (part + 1) * (D / 8); d0 += 2) {
        float v0 = 0.f, v1 = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          v0 = __fmaf_rn(wgt[w], red[(w * 16 + row) * D + d0], v0);
          v1 = __fmaf_rn(wgt[w], red[(w * 16 + row) * D + d0 + 1], v1);
        }
        v0 *= inv;
        v1 *= inv;
        if (p.part_o) {
          float* dst = p.part_o + (static_cast<size_t>(split) * p.B * p.Hq + orow) * D + d0;
          dst[0] = v0;
          dst[1] = v1;
        } else {
          *reinterpret_cast<uint32_t*>(p.out + orow * D + d0) = pack_bf16x2(v0, v1);
          if (p.out_sel && sel == 0) {
            p.out_sel[orow * D + d0] = v0;
            p.out_sel[orow * D + d0 + 1] = v1;
          }
        }
      }
      if (p.part_lse && part == 0)
        p.part_lse[static_cast<size_t>(split) * p.B * p.Hq + orow] = empty ? -INFINITY : M + __log2f(lsum);
    }
    (void)valid;
  }
  if (threadIdx.x == 0 && bars->abort) set_err(p.err, CPA_EBIT_TIMEOUT);
}

template <int D, bool EXPLICIT, bool F16>
static cudaError_t launch_decode_t(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream) {
  using CF = DecCfg<D>;
  auto kern = attn_decode_kernel<D, EXPLICIT, F16>;
  static SmemAttr smem_attr;
  if (cudaError_t e = smem_attr.ensure(reinterpret_cast<const void*>(kern), CF::kSmem); e != cudaSuccess) return e;
  dim3 grid(p.splits, p.Hkv, p.B);
  return launch_dependent(kern, grid, dim3(kDThreads), CF::kSmem, stream, maps[0], maps[1], maps[2], maps[3], p);
}

template <int D>
static cudaError_t launch_decode_d(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream) {
  const bool ex = p.mask != nullptr;
  if (p.f16) return ex ? launch_decode_t<D, true, true>(maps, p, stream) : launch_decode_t<D, false, true>(maps, p, stream);
  return ex ? launch_decode_t<D, true, false>(maps, p, stream) : launch_decode_t<D, false, false>(maps, p, stream);
}

cudaError_t launch_attn_decode(const CUtensorMap* maps, const AttnParams& p, cudaStream_t stream) {
  switch (p.D) {
    case 64: return launch_decode_d<64>(maps, p, stream);
    case 128: return launch_decode_d<128>(maps, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cpa
