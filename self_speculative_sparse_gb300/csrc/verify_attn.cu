// Verification attention with fused logit aggregation.
//
// Vegas §2 step 1 (verification phase): the gamma+1 verify rows attend, with full
// attention, every prefix entry and the verify rows up to themselves; the same pass
// yields the pre-softmax logit of every prefix entry (Vegas §3, kernel
// instrumentation), summed over the rows of a mask and over all query heads — the
// per-entry objective of the selection formula (Vegas §2.A), on the Collect-2-Query
// rows (Vegas §2.B) or on all rows.
//
// GB300 design.  The work is the flattened list of (sequence, KV head, 64-key tile)
// items, split evenly over one persistent CTA per SM (ragged batches balance by
// construction).  In each CTA a producer warp streams K and V tiles with 2-D TMA
// (128-byte swizzled boxes) into a 5-stage shared-memory ring guarded by
// mbarriers; the consumer warps hold the G*(gamma+1) query rows of the current KV
// head as tensor-core fragments and run QK^T and PV on bf16 MMA with fp32
// accumulators and an online softmax.  The logit sums are taken from the same QK^T
// fragments, so the cache is read exactly once.  Each contiguous run of tiles of one
// (sequence, KV head) leaves one unnormalised partial (max, sum, O); a small
// combine kernel, launched as a programmatic dependent of this one, merges the
// partials with the verify rows' own causal keys, writes bf16 outputs, appends the
// verify rows' K/V to the cache and sums the per-KV-head partial scores in a fixed
// order (deterministic, no atomics).
#include <cooperative_groups.h>

#include "vg_common.cuh"
#include "vg_internal.h"

namespace vg {
namespace {

constexpr int TK = kVerifyTileKeys;
constexpr int kStages = 5;

template <int D, int MT>
struct VCfg {
  static constexpr int KGW = (MT == 4) ? 2 : 4;  // key-group warps per 16-row m-tile
  static constexpr int KPW = 4 / KGW;            // 16-key groups per warp per tile
  static constexpr int W = MT * KGW;             // consumer warps
  static constexpr int THREADS = (W + 1) * 32;   // + one producer warp
  static constexpr int MAXREG = (65536 / THREADS) / 8 * 8 > 255 ? 255 : (65536 / THREADS) / 8 * 8;
  static constexpr int HALVES = D / 64;          // 64-column (128-byte) swizzled boxes
  static constexpr int HALF_BYTES = TK * 128;
  static constexpr int TILE_BYTES = TK * D * 2;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int M = MT * 16;
  static constexpr int OFF_MERGE = kStages * STAGE_BYTES;   // float [M][D]
  static constexpr int OFF_MROW = OFF_MERGE + M * D * 4;    // float [KGW][M]
  static constexpr int OFF_LROW = OFF_MROW + KGW * M * 4;   // float [M]
  static constexpr int OFF_SC = OFF_LROW + M * 4;           // float [2 buf][2 mask][MT][TK]
  static constexpr int OFF_BAR = OFF_SC + 2 * 2 * MT * TK * 4;
  static constexpr int OFF_META = OFF_BAR + 2 * kStages * 8;  // int cum[B+1], nlen[B]
  static size_t smem(int B) { return 1024 + OFF_META + (size_t)(2 * B + 1) * 4; }
};

__device__ __forceinline__ float bf2f(__nv_bfloat16 v) { return __bfloat162float(v); }

// Per-sequence tile counts (one KV head) and checked lengths; warp 0 only.
// nlen[b] = -1 marks a sequence whose length or slots are out of range.
__device__ void seq_meta(const VerifyParams& p, int* cum, int* nlen) {
  const int lane = threadIdx.x & 31;
  int carry = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    int tiles = 0;
    if (b < p.B) {
      int n = p.prefix_len[b];
      const int64_t off = p.seq_offset[b];
      const bool ok = n >= 0 && n <= p.max_len && off >= 0 && off + (int64_t)n + p.R <= p.capacity;
      if (!ok) {
        report(p.status, VG_ERR_DEVICE_BOUNDS);
        n = -1;
      }
      nlen[b] = n;
      tiles = n > 0 ? (n + TK - 1) / TK : 0;
    }
    int v = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += t;
    }
    if (b < p.B) cum[b] = carry + v - tiles;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
  if (lane == 0) cum[p.B] = carry;
}

// Global tile x -> (sequence b, KV head g, tile j).  Order: b, then g, then j.
__device__ __forceinline__ void locate(int x, const int* cum, int B, int Hkv, int& b, int& g, int& j) {
  int lo = 0, hi = B;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (Hkv * cum[mid] <= x) lo = mid; else hi = mid - 1;
  }
  b = lo;
  const int tiles = cum[b + 1] - cum[b];
  const int off = x - Hkv * cum[b];
  g = off / tiles;
  j = off - g * tiles;
}

__device__ __forceinline__ void advance(int& b, int& g, int& j, const int* cum, int B, int Hkv) {
  if (++j == cum[b + 1] - cum[b]) {
    j = 0;
    if (++g == Hkv) {
      g = 0;
      ++b;
      while (b < B && cum[b + 1] == cum[b]) ++b;
    }
  }
}

template <int D, int MT>
__global__ void __launch_bounds__((VCfg<D, MT>::THREADS)) __maxnreg__((VCfg<D, MT>::MAXREG))
    verify_kernel(const VerifyParams p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  using C = VCfg<D, MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* merge = reinterpret_cast<float*>(smem + C::OFF_MERGE);
  float* mrow = reinterpret_cast<float*>(smem + C::OFF_MROW);
  float* lrow = reinterpret_cast<float*>(smem + C::OFF_LROW);
  float* sc = reinterpret_cast<float*>(smem + C::OFF_SC);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + kStages;
  int* cum = reinterpret_cast<int*>(smem + C::OFF_META);
  int* nlen = cum + p.B + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) seq_meta(p, cum, nlen);
  if (threadIdx.x == 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::W);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (blockIdx.x == 0) {  // the combine kernel reads these after this grid completes
    for (int i = threadIdx.x; i < 2 * p.B + 1; i += blockDim.x) p.meta[i] = cum[i];
  }
  pdl_launch_dependents();

  const int T = p.Hkv * cum[p.B];
  const int t0 = static_cast<int>(split_begin(blockIdx.x, T, p.nctas));
  const int t1 = static_cast<int>(split_begin(blockIdx.x + 1, T, p.nctas));
  if (t0 >= t1) return;

  // ------------------------------------------------------------ producer warp
  if (warp == C::W) {
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int b, g, j;
      locate(t0, cum, p.B, p.Hkv, b, g, j);
      int stage = 0;
      uint32_t phase = 0;
      for (int x = t0; x < t1; ++x) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, p.status)) break;
        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
        uint8_t* kdst = smem + stage * C::STAGE_BYTES;
        uint8_t* vdst = kdst + C::TILE_BYTES;
        const int y = static_cast<int>(p.seq_offset[b] + static_cast<int64_t>(j) * TK);
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          tma_load_2d(kdst + h * C::HALF_BYTES, &tmK, g * D + h * 64, y, &full[stage]);
          tma_load_2d(vdst + h * C::HALF_BYTES, &tmV, g * D + h * 64, y, &full[stage]);
        }
        if (x + 1 < t1) advance(b, g, j, cum, p.B, p.Hkv);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumer warps
  constexpr int NT = C::W * 32;
  const int mt = warp % MT, kgw = warp / MT;
  const int gid = lane >> 2, tig = lane & 3;
  const int row0 = mt * 16 + gid, row1 = row0 + 8;
  const int vt0 = row0 < p.M ? row0 / p.G : -1;  // verify row of each fragment row
  const int vt1 = row1 < p.M ? row1 / p.G : -1;
  const bool r0m0 = vt0 >= 0 && ((p.mask0 >> vt0) & 1u), r1m0 = vt1 >= 0 && ((p.mask0 >> vt1) & 1u);
  const bool r0m1 = vt0 >= 0 && ((p.mask1 >> vt0) & 1u), r1m1 = vt1 >= 0 && ((p.mask1 >> vt1) & 1u);
  const bool any_mask = (p.mask0 | p.mask1) != 0;
  const float NEG = neg_inf();

  int b, g, j;
  locate(t0, cum, p.B, p.Hkv, b, g, j);
  int stage = 0, it = 0;
  uint32_t phase = 0;
  bool lost = false;
  int x = t0;
  while (x < t1 && !lost) {
    const int tiles_b = cum[b + 1] - cum[b];
    const int seg_end = min(t1, x + (tiles_b - j));
    const int n_b = nlen[b];

    // query rows of this (sequence, KV head) as A fragments: row m -> (t = m / G, head g*G + m % G)
    uint32_t qf[D / 16][4];
    {
      const __nv_bfloat16* q0 = nullptr;
      const __nv_bfloat16* q1 = nullptr;
      if (row0 < p.M) q0 = p.q + ((static_cast<size_t>(b) * p.R + vt0) * p.Hq + g * p.G + row0 % p.G) * D;
      if (row1 < p.M) q1 = p.q + ((static_cast<size_t>(b) * p.R + vt1) * p.Hq + g * p.G + row1 % p.G) * D;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int c0 = ks * 16 + tig * 2;
        qf[ks][0] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + c0) : 0u;
        qf[ks][1] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + c0) : 0u;
        qf[ks][2] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + c0 + 8) : 0u;
        qf[ks][3] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + c0 + 8) : 0u;
      }
    }
    float m_run[2] = {NEG, NEG}, l_run[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;

    for (; x < seg_end; ++x, ++j, ++it) {
      if (!mbar_wait(&full[stage], phase, p.status)) {
        lost = true;
        break;
      }
      const uint32_t kb = smem_u32(smem + stage * C::STAGE_BYTES);
      const uint32_t vb = kb + C::TILE_BYTES;
      float* scb = sc + (it & 1) * (2 * MT * TK);
#pragma unroll
      for (int kp = 0; kp < C::KPW; ++kp) {
        const int kg = kgw * C::KPW + kp;
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const int mi = lane >> 3, rr = lane & 7;
          const int r = kg * 16 + (mi >> 1) * 8 + rr;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const int c16 = ks * 2 + (mi & 1);
            const uint32_t addr = kb + (c16 >> 3) * C::HALF_BYTES + r * 128 + (((c16 & 7) ^ (r & 7)) << 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(addr, b0, b1, b2, b3);
            mma_bf16(s[0], qf[ks], b0, b1);
            mma_bf16(s[1], qf[ks], b2, b3);
          }
        }
        const int key0 = j * TK + kg * 16;
        if (any_mask) {  // logit sums over this warp's rows of each mask, then over lanes sharing a key
          float v0[4], v1[4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const float a = s[nt][c], bq = s[nt][2 + c];
              v0[nt * 2 + c] = (r0m0 ? a : 0.f) + (r1m0 ? bq : 0.f);
              v1[nt * 2 + c] = (r0m1 ? a : 0.f) + (r1m1 ? bq : 0.f);
            }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
              v0[i] += __shfl_xor_sync(0xffffffffu, v0[i], off);
              v1[i] += __shfl_xor_sync(0xffffffffu, v1[i], off);
            }
          }
          if (gid == 0) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                const int col = kg * 16 + nt * 8 + tig * 2 + c;
                scb[(0 * MT + mt) * TK + col] = v0[nt * 2 + c] * p.scale;
                scb[(1 * MT + mt) * TK + col] = v1[nt * 2 + c] * p.scale;
              }
          }
        }
        // online softmax in log2 units; keys past the prefix end are masked
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const bool ok = key0 + nt * 8 + tig * 2 + c < n_b;
            s[nt][c] = ok ? s[nt][c] * p.scale_log2 : NEG;
            s[nt][2 + c] = ok ? s[nt][2 + c] * p.scale_log2 : NEG;
          }
        float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
        float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
        const float mu0 = mn0 == NEG ? 0.f : mn0, mu1 = mn1 == NEG ? 0.f : mn1;
        if (__any_sync(0xffffffffu, (mn0 > m_run[0]) || (mn1 > m_run[1]))) {
          const float a0 = ex2(m_run[0] - mu0), a1 = ex2(m_run[1] - mu1);
          l_run[0] *= a0;
          l_run[1] *= a1;
#pragma unroll
          for (int dn = 0; dn < D / 8; ++dn) {
            o[dn][0] *= a0;
            o[dn][1] *= a0;
            o[dn][2] *= a1;
            o[dn][3] *= a1;
          }
        }
        m_run[0] = mn0;
        m_run[1] = mn1;
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          pr[nt][0] = ex2(s[nt][0] - mu0);
          pr[nt][1] = ex2(s[nt][1] - mu0);
          pr[nt][2] = ex2(s[nt][2] - mu1);
          pr[nt][3] = ex2(s[nt][3] - mu1);
        }
        l_run[0] += pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1];
        l_run[1] += pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3];
        const uint32_t pa[4] = {pack_bf16(pr[0][0], pr[0][1]), pack_bf16(pr[0][2], pr[0][3]),
                                pack_bf16(pr[1][0], pr[1][1]), pack_bf16(pr[1][2], pr[1][3])};
        {
          const int mi = lane >> 3, rr = lane & 7;
          const int r = kg * 16 + (mi & 1) * 8 + rr;
#pragma unroll
          for (int dn2 = 0; dn2 < D / 16; ++dn2) {
            const int c16 = dn2 * 2 + (mi >> 1);
            const uint32_t addr = vb + (c16 >> 3) * C::HALF_BYTES + r * 128 + (((c16 & 7) ^ (r & 7)) << 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(addr, b0, b1, b2, b3);
            mma_bf16(o[2 * dn2], pa, b0, b1);
            mma_bf16(o[2 * dn2 + 1], pa, b2, b3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
      if (any_mask) {  // per-KV-head partial score of each key: sum over the m-tiles
        named_bar(1, NT);
        for (int e = threadIdx.x; e < 2 * TK; e += NT) {
          const int ms = e / TK, col = e - ms * TK;
          if ((ms ? p.mask1 : p.mask0) == 0u) continue;
          const int pos = j * TK + col;
          if (pos < n_b) {
            float v = 0.f;
#pragma unroll
            for (int m2 = 0; m2 < MT; ++m2) v += scb[(ms * MT + m2) * TK + col];
            p.part_s[((static_cast<size_t>(ms) * p.B + b) * p.Hkv + g) * p.max_len + pos] = v;
          }
        }
      }
    }

    // ---------------------------------------------------- segment partial
    l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 1);
    l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 2);
    l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 1);
    l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 2);
    if (tig == 0) {
      mrow[kgw * C::M + row0] = m_run[0];
      mrow[kgw * C::M + row1] = m_run[1];
    }
    named_bar(1, NT);
    float mf0 = NEG, mf1 = NEG;
#pragma unroll
    for (int w2 = 0; w2 < C::KGW; ++w2) {
      mf0 = fmaxf(mf0, mrow[w2 * C::M + row0]);
      mf1 = fmaxf(mf1, mrow[w2 * C::M + row1]);
    }
    {
      const float f0 = ex2(m_run[0] - (mf0 == NEG ? 0.f : mf0));
      const float f1 = ex2(m_run[1] - (mf1 == NEG ? 0.f : mf1));
      l_run[0] *= f0;
      l_run[1] *= f1;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        o[dn][0] *= f0;
        o[dn][1] *= f0;
        o[dn][2] *= f1;
        o[dn][3] *= f1;
      }
    }
    for (int w2 = 0; w2 < C::KGW; ++w2) {  // fixed order: deterministic sums
      if (kgw == w2) {
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
          float2* d0 = reinterpret_cast<float2*>(merge + row0 * D + dn * 8 + tig * 2);
          float2* d1 = reinterpret_cast<float2*>(merge + row1 * D + dn * 8 + tig * 2);
          if (w2 == 0) {
            *d0 = make_float2(o[dn][0], o[dn][1]);
            *d1 = make_float2(o[dn][2], o[dn][3]);
          } else {
            float2 a = *d0, c = *d1;
            *d0 = make_float2(a.x + o[dn][0], a.y + o[dn][1]);
            *d1 = make_float2(c.x + o[dn][2], c.y + o[dn][3]);
          }
        }
        if (tig == 0) {
          lrow[row0] = (w2 == 0 ? 0.f : lrow[row0]) + l_run[0];
          lrow[row1] = (w2 == 0 ? 0.f : lrow[row1]) + l_run[1];
        }
      }
      named_bar(1, NT);
    }
    {
      const size_t id = static_cast<size_t>(blockIdx.x) + static_cast<size_t>(b) * p.Hkv + g;
      float4* dst = reinterpret_cast<float4*>(p.part_o + id * C::M * D);
      const float4* src = reinterpret_cast<const float4*>(merge);
      for (int e = threadIdx.x; e < C::M * D / 4; e += NT) dst[e] = src[e];
      for (int r = threadIdx.x; r < C::M; r += NT) {
        float mf = NEG;
        for (int w2 = 0; w2 < C::KGW; ++w2) mf = fmaxf(mf, mrow[w2 * C::M + r]);
        p.part_ml[(id * C::M + r) * 2 + 0] = mf;
        p.part_ml[(id * C::M + r) * 2 + 1] = lrow[r];
      }
      named_bar(1, NT);
    }
    if (x < t1) {  // next (sequence, KV head)
      j = 0;
      if (++g == p.Hkv) {
        g = 0;
        ++b;
        while (b < p.B && cum[b + 1] == cum[b]) ++b;
      }
    }
  }
}

// Merge of the partials with the verify rows' causal keys, output, append, scores.
template <int D>
__global__ void __launch_bounds__(128) verify_combine_kernel(const VerifyParams p) {
  __shared__ float lg[16][16];  // [head in group][verify row u] logits, log2 units
  pdl_wait();
  const int* cum = p.meta;
  const int* nlen = p.meta + p.B + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float NEG = neg_inf();
  const int nO = p.B * p.Hkv * p.R;
  if (static_cast<int>(blockIdx.x) < nO) {
    const int t = blockIdx.x % p.R;
    const int bg = blockIdx.x / p.R;
    const int g = bg % p.Hkv, b = bg / p.Hkv;
    const int n = nlen[b];
    if (n < 0) return;
    const int64_t base = p.seq_offset[b];
    const __nv_bfloat16* kn = p.k_new ? p.k_new + (static_cast<size_t>(b) * p.R * p.Hkv + g) * D
                                      : p.K + ((base + n) * p.Hkv + g) * D;
    const __nv_bfloat16* vn = p.v_new ? p.v_new + (static_cast<size_t>(b) * p.R * p.Hkv + g) * D
                                      : p.V + ((base + n) * p.Hkv + g) * D;
    const size_t row_stride = static_cast<size_t>(p.Hkv) * D;  // between consecutive verify rows
    const int npairs = p.G * (t + 1);
    for (int pr = warp; pr < npairs; pr += 4) {
      const int jh = pr / (t + 1), u = pr - jh * (t + 1);
      const __nv_bfloat16* qr = p.q + ((static_cast<size_t>(b) * p.R + t) * p.Hq + g * p.G + jh) * D;
      const __nv_bfloat16* kr = kn + u * row_stride;
      float acc = 0.f;
      for (int e = lane; e < D; e += 32) acc += bf2f(qr[e]) * bf2f(kr[e]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0) lg[jh][u] = acc * p.scale_log2;
    }
    __syncthreads();
    const int tiles = cum[b + 1] - cum[b];
    int64_t cf = 0, cl = -1;
    if (tiles > 0) {
      const int64_t T = static_cast<int64_t>(p.Hkv) * cum[p.B];
      const int64_t S = static_cast<int64_t>(p.Hkv) * cum[b] + static_cast<int64_t>(g) * tiles;
      cf = owner_cta(S, T, p.nctas);
      cl = owner_cta(S + tiles - 1, T, p.nctas);
    }
    const size_t pair = static_cast<size_t>(b) * p.Hkv + g;
    if (tid < D) {
      const int e = tid;
      for (int jh = 0; jh < p.G; ++jh) {
        const int m = t * p.G + jh;
        float M = NEG, acc = 0.f, l = 0.f;
        for (int64_t c = cf; c <= cl; ++c) {
          const size_t id = static_cast<size_t>(c) + pair;
          const float ms = p.part_ml[(id * p.Mpad + m) * 2 + 0];
          const float ls = p.part_ml[(id * p.Mpad + m) * 2 + 1];
          const float os = p.part_o[(id * p.Mpad + m) * D + e];
          const float Mn = fmaxf(M, ms);
          const float a = ex2(M - Mn), w = ex2(ms - Mn);
          acc = acc * a + os * w;
          l = l * a + ls * w;
          M = Mn;
        }
        for (int u = 0; u <= t; ++u) {
          const float lu = lg[jh][u];
          const float Mn = fmaxf(M, lu);
          const float a = ex2(M - Mn), w = ex2(lu - Mn);
          acc = acc * a + w * bf2f(vn[u * row_stride + e]);
          l = l * a + w;
          M = Mn;
        }
        p.out[((static_cast<size_t>(b) * p.R + t) * p.Hq + g * p.G + jh) * D + e] = __float2bfloat16_rn(acc / l);
      }
      if (p.k_new) {  // append verify row t (Vegas §2 step 1: the chain enters the cache)
        const size_t dst = ((base + n + t) * p.Hkv + g) * D + e;
        p.K[dst] = kn[t * row_stride + e];
        p.V[dst] = vn[t * row_stride + e];
      }
    }
    return;
  }
  // score role: fixed-order sum of the per-KV-head partial scores
  const int nchunks = (p.max_len + kScoreChunk - 1) / kScoreChunk;
  const int sb = blockIdx.x - nO;
  const int b = sb / nchunks, ch = sb - b * nchunks;
  if (b >= p.B) return;
  const int n = nlen[b];
  const int lo = ch * kScoreChunk, hi = min(n, lo + kScoreChunk);
  for (int ms = 0; ms < 2; ++ms) {
    float* dst = ms ? p.scores1 : p.scores0;
    if ((ms ? p.mask1 : p.mask0) == 0u || dst == nullptr) continue;
    const float* src = p.part_s + (static_cast<size_t>(ms) * p.B + b) * p.Hkv * p.max_len;
    for (int pos = lo + tid; pos < hi; pos += 128) {
      float v = 0.f;
      for (int g = 0; g < p.Hkv; ++g) v += src[static_cast<size_t>(g) * p.max_len + pos];
      dst[static_cast<size_t>(b) * p.score_stride + pos] = v;
    }
  }
}

template <int D, int MT>
cudaError_t launch_verify_t(const VerifyParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            cudaStream_t stream) {
  using C = VCfg<D, MT>;
  const size_t smem = C::smem(p.B);
  cudaError_t e = cudaFuncSetAttribute(verify_kernel<D, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  verify_kernel<D, MT><<<p.nctas, C::THREADS, smem, stream>>>(p, tmK, tmV);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const int nO = p.B * p.Hkv * p.R;
  const int nS = ((p.mask0 | p.mask1) != 0u) ? p.B * ((p.max_len + kScoreChunk - 1) / kScoreChunk) : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nO + nS);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_combine_kernel<D>, p);
}

}  // namespace

size_t verify_smem_bytes(int D, int Mpad, int B) {
  const int MT = Mpad / 16;
#define VG_SMEM_CASE(DD, MM) \
  if (D == DD && MT == MM) return VCfg<DD, MM>::smem(B);
  VG_SMEM_CASE(64, 1) VG_SMEM_CASE(64, 2) VG_SMEM_CASE(64, 3) VG_SMEM_CASE(64, 4)
  VG_SMEM_CASE(128, 1) VG_SMEM_CASE(128, 2) VG_SMEM_CASE(128, 3) VG_SMEM_CASE(128, 4)
#undef VG_SMEM_CASE
  return 0;
}

cudaError_t launch_verify(const VerifyParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          cudaStream_t stream) {
  const int MT = p.Mpad / 16;
#define VG_LAUNCH_CASE(DD, MM) \
  if (p.D == DD && MT == MM) return launch_verify_t<DD, MM>(p, tmK, tmV, stream);
  VG_LAUNCH_CASE(64, 1) VG_LAUNCH_CASE(64, 2) VG_LAUNCH_CASE(64, 3) VG_LAUNCH_CASE(64, 4)
  VG_LAUNCH_CASE(128, 1) VG_LAUNCH_CASE(128, 2) VG_LAUNCH_CASE(128, 3) VG_LAUNCH_CASE(128, 4)
#undef VG_LAUNCH_CASE
  return cudaErrorInvalidValue;
}

}  // namespace vg
