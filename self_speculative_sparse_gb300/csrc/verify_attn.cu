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
// construction).  Thread 0 of each CTA streams K and V tiles with 2-D TMA
// (128-byte swizzled boxes) into a 5-stage shared-memory ring guarded by
// mbarriers; 8 or 12 warps hold the G*(gamma+1) query rows of the current KV head
// as tensor-core fragments and run QK^T and PV on bf16 MMA with fp32
// accumulators and an online softmax.  The logit sums are taken from the same
// QK^T fragments, so the cache is read exactly once.  Each contiguous run of tiles
// of one (sequence, KV head) leaves one unnormalised partial (max, sum, O); a
// combine kernel, launched as a programmatic dependent of this one, merges the
// partials with the verify rows' own causal keys, writes bf16 outputs, appends the
// verify rows' K/V to the cache and sums the per-KV-head partial scores in a fixed
// order (deterministic, no atomics).
#include <cstdio>

#include "attn_frag.cuh"
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
  static constexpr int W = MT * KGW;             // warps (a multiple of 4: one share per SM sub-partition)
  static constexpr int THREADS = W * 32;
  static constexpr int HALVES = D / 64;          // 64-column (128-byte) swizzled boxes
  static constexpr int HALF_BYTES = TK * 128;
  static constexpr int TILE_BYTES = TK * D * 2;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int M = MT * 16;
  static constexpr int MSTRIDE = D + 8;                        // padded merge rows: 2-way at most
  static constexpr int OFF_MERGE = kStages * STAGE_BYTES;      // float [M][MSTRIDE]
  static constexpr int OFF_MROW = OFF_MERGE + M * MSTRIDE * 4; // float [KGW][M]
  static constexpr int OFF_LROW = OFF_MROW + KGW * M * 4;      // float [M]
  static constexpr int OFF_BAR = (OFF_LROW + M * 4 + 7) & ~7;  // full[kStages], empty[kStages]
  static constexpr int OFF_META = OFF_BAR + 2 * kStages * 8;   // int cum[B+1], nlen[B]
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
__global__ void __launch_bounds__(VCfg<D, MT>::THREADS, 1)
    verify_kernel(const VerifyParams p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  using C = VCfg<D, MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* merge = reinterpret_cast<float*>(smem + C::OFF_MERGE);
  float* mrow = reinterpret_cast<float*>(smem + C::OFF_MROW);
  float* lrow = reinterpret_cast<float*>(smem + C::OFF_LROW);
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

  // The ring holds tiles x .. x + kStages - 1.  Thread 0 fills it first; every warp
  // arrives on a stage's empty barrier when done with its tile, and after finishing
  // tile x thread 0 refills the stage of tile x - 1 (normally released by then)
  // with tile x - 1 + kStages.  No warp waits for the others between tiles.
  auto issue = [&](int stage, int tile) {
    int ib, ig, ij;
    locate(tile, cum, p.B, p.Hkv, ib, ig, ij);
    fence_proxy_async_smem();  // the stage may hold zeros written by the generic proxy
    mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
    uint8_t* kdst = smem + stage * C::STAGE_BYTES;
    uint8_t* vdst = kdst + C::TILE_BYTES;
    const int y = static_cast<int>(p.seq_offset[ib] + static_cast<int64_t>(ij) * TK);
#pragma unroll
    for (int h = 0; h < C::HALVES; ++h) {
      tma_load_2d(kdst + h * C::HALF_BYTES, &tmK, ig * D + h * 64, y, &full[stage]);
      tma_load_2d(vdst + h * C::HALF_BYTES, &tmV, ig * D + h * 64, y, &full[stage]);
    }
  };
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int st = 0; st < kStages && t0 + st < t1; ++st) issue(st, t0 + st);
  }

  constexpr int NT = C::THREADS;
  const int mt = warp % MT, kgw = warp / MT;
  const int gid = lane >> 2, tig = lane & 3;
  const int row0 = mt * 16 + gid, row1 = row0 + 8;
  const int vt0 = row0 < p.M ? row0 / p.G : -1;  // verify row of each fragment row
  const int vt1 = row1 < p.M ? row1 / p.G : -1;
  const bool r0m0 = vt0 >= 0 && ((p.mask0 >> vt0) & 1u), r1m0 = vt1 >= 0 && ((p.mask0 >> vt1) & 1u);
  const bool r0m1 = vt0 >= 0 && ((p.mask1 >> vt0) & 1u), r1m1 = vt1 >= 0 && ((p.mask1 >> vt1) & 1u);
  const float NEG = neg_inf();

  int b, g, j;
  locate(t0, cum, p.B, p.Hkv, b, g, j);
  int stage = 0;
  uint32_t phase = 0;
  bool lost = false;
  int x = t0;
  while (x < t1 && !lost) {
    const int tiles_b = cum[b + 1] - cum[b];
    const int seg_end = min(t1, x + (tiles_b - j));
    const int n_b = nlen[b];

    // query rows of this (sequence, KV head): row m -> (t = m / G, head g*G + m % G)
    uint32_t qf[D / 16][4];
    load_q_frags<D>(qf,
                    row0 < p.M ? p.q + ((static_cast<size_t>(b) * p.R + vt0) * p.Hq + g * p.G + row0 % p.G) * D
                               : nullptr,
                    row1 < p.M ? p.q + ((static_cast<size_t>(b) * p.R + vt1) * p.Hq + g * p.G + row1 % p.G) * D
                               : nullptr,
                    tig);
    RowState<D> st;
    st.init();

    for (; x < seg_end; ++x, ++j) {
      if (!mbar_wait(&full[stage], phase, p.status)) {
        lost = true;
        break;
      }
      const int valid = n_b - j * TK;  // keys of this tile inside the prefix
      if (valid < TK) {  // (at most once per run of tiles, the only point where warps meet)
        // The rows past the prefix end hold whatever the cache has there; their
        // probabilities are zero, and zeroed values keep 0 * V exact even if the
        // slots hold non-finite garbage.
        uint4* vrows = reinterpret_cast<uint4*>(smem + stage * C::STAGE_BYTES + C::TILE_BYTES);
        const int per_half = TK * 8;  // 16-byte chunks in one 128-byte-wide box
        for (int e = threadIdx.x; e < C::HALVES * per_half; e += NT) {
          const int h = e / per_half, r = (e - h * per_half) >> 3;
          if (r >= valid) vrows[e] = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // before the next TMA write into this stage
        named_bar(2, NT);
      }
      const uint32_t kb = smem_u32(smem + stage * C::STAGE_BYTES);
      const uint32_t vb = kb + C::TILE_BYTES;
#pragma unroll
      for (int kp = 0; kp < C::KPW; ++kp) {
        const int kg = kgw * C::KPW + kp;
        // 128-byte swizzle of the TMA boxes: chunk c of row r sits at chunk c ^ (r & 7)
        auto kaddr = [&](int r, int c16) {
          const int rr = kg * 16 + r;
          return kb + (c16 >> 3) * C::HALF_BYTES + rr * 128 + (((c16 & 7) ^ (rr & 7)) << 4);
        };
        auto vaddr = [&](int r, int c16) {
          const int rr = kg * 16 + r;
          return vb + (c16 >> 3) * C::HALF_BYTES + rr * 128 + (((c16 & 7) ^ (rr & 7)) << 4);
        };
        float s[2][4];
        qk16<D>(qf, kaddr, s, lane);
        const int key0 = j * TK + kg * 16;
        // logit sums over this warp's rows of each mask (column sums of S), written
        // as this m-tile's share of the KV head's score of each key
        const int skey = key0 + ((lane >> 4) & 1) * 8 + tig * 2 + ((lane >> 3) & 1);
#pragma unroll
        for (int ms = 0; ms < 2; ++ms) {
          if ((ms ? p.mask1 : p.mask0) == 0u) continue;
          const bool m0 = ms ? r0m1 : r0m0, m1 = ms ? r1m1 : r1m0;
          float v[4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) v[nt * 2 + c] = (m0 ? s[nt][c] : 0.f) + (m1 ? s[nt][2 + c] : 0.f);
          const float sum = colsum16(v, lane);
          if ((lane & 4) == 0 && skey < n_b)
            p.part_s[(((static_cast<size_t>(ms) * p.B + b) * p.Hkv + g) * MT + mt) * p.max_len + skey] =
                sum * p.scale;
        }
        // softmax in log2 units; keys past the prefix end are masked
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const bool ok = key0 + nt * 8 + tig * 2 + c < n_b;
            s[nt][c] = ok ? s[nt][c] * p.scale_log2 : NEG;
            s[nt][2 + c] = ok ? s[nt][2 + c] * p.scale_log2 : NEG;
          }
        softmax_pv16<D>(st, s, vaddr, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (threadIdx.x == 0 && x > t0 && x - 1 + kStages < t1) {
        const int lp = x - 1 - t0;  // the previous tile's place in the ring
        if (mbar_wait(&empty[lp % kStages], static_cast<uint32_t>((lp / kStages) & 1), p.status))
          issue(lp % kStages, x - 1 + kStages);
      }
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }

    // segment partial: merge the key-group warps of each m-tile, then store
    merge_warps<D, C::KGW>(st, C::M, C::MSTRIDE, row0, kgw, merge, mrow, lrow, tig, 1, NT);
    const size_t id = static_cast<size_t>(blockIdx.x) + static_cast<size_t>(b) * p.Hkv + g;
    store_partial<D, C::KGW>(merge, C::MSTRIDE, mrow, lrow, C::M, p.part_o + id * C::M * D,
                             p.part_ml + id * C::M * 2, threadIdx.x, NT);
    named_bar(1, NT);
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
// Role A, one CTA per (sequence b, KV head g, verify row t): its G query rows.
//   phase 1: every (segment, row) max/sum into shared memory (one round trip);
//   phase 2: one warp per row, lanes across d, independent loads over segments.
// Role B, one CTA per (sequence, 1024 positions): fixed-order sum of the per-KV-head
// partial scores.
template <int D>
__global__ void __launch_bounds__(128) verify_combine_kernel(const VerifyParams p) {
  extern __shared__ float cs[];                  // [nctas][G] max, [nctas][G] sum
  __shared__ float lg[16][16];                   // [row in group][verify key u] logits, log2 units
  __shared__ __align__(16) __nv_bfloat16 qs[16][D];  // this verify row's G query rows
  __shared__ __align__(16) __nv_bfloat16 ks[16][D];  // the verify rows' own keys u <= t
  __shared__ __align__(16) __nv_bfloat16 vs[16][D];  // ... and values
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
    const int G = p.G;
    const int64_t base = p.seq_offset[b];
    const __nv_bfloat16* kn = p.k_new ? p.k_new + (static_cast<size_t>(b) * p.R * p.Hkv + g) * D
                                      : p.K + ((base + n) * p.Hkv + g) * D;
    const __nv_bfloat16* vn = p.v_new ? p.v_new + (static_cast<size_t>(b) * p.R * p.Hkv + g) * D
                                      : p.V + ((base + n) * p.Hkv + g) * D;
    const size_t row_stride = static_cast<size_t>(p.Hkv) * D;  // between consecutive verify rows
    // segments of this (sequence, KV head)
    const int tiles = cum[b + 1] - cum[b];
    const int64_t T = static_cast<int64_t>(p.Hkv) * cum[p.B];
    int64_t cf = 0, cl = -1;
    if (tiles > 0) {
      const int64_t S = static_cast<int64_t>(p.Hkv) * cum[b] + static_cast<int64_t>(g) * tiles;
      cf = owner_cta(S, T, p.nctas);
      cl = owner_cta(S + tiles - 1, T, p.nctas);
    }
    const int nseg = static_cast<int>(cl - cf + 1);
    const size_t pair = static_cast<size_t>(b) * p.Hkv + g;
    float* cm = cs;
    float* csum = cs + p.nctas * G;
    // phase 1: one round of independent loads - each warp's partial output rows into
    // registers, the verify rows' q/k/v and every partial's max/sum into shared memory
    constexpr int NB = 16;
    PartialRows<D, NB> pre;
    const int jw = warp < G ? warp : 0;  // the row this warp merges first
    auto orow = [&](int si) {
      return p.part_o + ((static_cast<size_t>(cf + si) + pair) * p.Mpad + t * G + jw) * D;
    };
    pre.load(orow, 0, 1, nseg, lane);
    constexpr int CH = D / 8;  // 16-byte chunks per row
    const __nv_bfloat16* qbase = p.q + ((static_cast<size_t>(b) * p.R + t) * p.Hq + g * G) * D;
    for (int e = tid; e < G * CH; e += 128)
      reinterpret_cast<uint4*>(&qs[0][0])[e] = reinterpret_cast<const uint4*>(qbase)[e];
    for (int e = tid; e < (t + 1) * CH; e += 128) {
      const int u = e / CH, c = e - u * CH;
      reinterpret_cast<uint4*>(&ks[u][0])[c] = reinterpret_cast<const uint4*>(kn + u * row_stride)[c];
      reinterpret_cast<uint4*>(&vs[u][0])[c] = reinterpret_cast<const uint4*>(vn + u * row_stride)[c];
    }
    for (int e = tid; e < nseg * G; e += 128) {
      const int si = e / G, jh = e - si * G;
      const int64_t c = cf + si;
      float ms = NEG, ls = 0.f;
      if (split_nonempty(c, T, p.nctas)) {  // CTAs with no items wrote no partial
        const size_t r = (static_cast<size_t>(c) + pair) * p.Mpad + t * G + jh;
        ms = p.part_ml[r * 2 + 0];
        ls = p.part_ml[r * 2 + 1];
      }
      cm[si * G + jh] = ms;
      csum[si * G + jh] = ls;
    }
    __syncthreads();
    // logits of the verify rows' own keys u <= t (causal), from shared memory
    for (int pr = warp; pr < G * (t + 1); pr += 4) {
      const int jh = pr / (t + 1), u = pr - jh * (t + 1);
      float acc = 0.f;
      for (int e = lane; e < D; e += 32) acc += bf2f(qs[jh][e]) * bf2f(ks[u][e]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0) lg[jh][u] = acc * p.scale_log2;
    }
    __syncthreads();
    // phase 2: one warp per query row, lanes across d
    constexpr int PER = D / 32;
    for (int jh = warp; jh < G; jh += 4) {
      float M = NEG;
      for (int si = lane; si < nseg; si += 32) M = fmaxf(M, cm[si * G + jh]);
      for (int u = lane; u <= t; u += 32) M = fmaxf(M, lg[jh][u]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
      float acc[PER];
#pragma unroll
      for (int q = 0; q < PER; ++q) acc[q] = 0.f;
      float l = 0.f;
      const int m = t * G + jh;
      auto orow_j = [&](int si) { return p.part_o + ((static_cast<size_t>(cf + si) + pair) * p.Mpad + m) * D; };
      if (jh == warp) {  // first row of this warp: most partials are already in registers
        pre.accumulate(cm + jh, csum + jh, G, 0, 1, nseg, M, acc, l);
        merge_partials<D>(cm + jh, csum + jh, G, nseg, M, orow_j, acc, l, lane, NB, 1);
      } else {
        merge_partials<D>(cm + jh, csum + jh, G, nseg, M, orow_j, acc, l, lane);
      }
      for (int u = 0; u <= t; ++u) {
        const float w = ex2(lg[jh][u] - M);
        l += w;
#pragma unroll
        for (int q = 0; q < PER; ++q) acc[q] += w * bf2f(vs[u][lane * PER + q]);
      }
      const float inv = 1.f / l;
      __nv_bfloat16* o = p.out + ((static_cast<size_t>(b) * p.R + t) * p.Hq + g * G + jh) * D + lane * PER;
#pragma unroll
      for (int q = 0; q < PER; ++q) o[q] = __float2bfloat16_rn(acc[q] * inv);
    }
    if (p.k_new) {  // append verify row t (the chain enters the cache)
      const size_t dst = ((base + n + t) * p.Hkv + g) * D;
      for (int c = tid; c < CH; c += 128) {
        reinterpret_cast<uint4*>(p.K + dst)[c] = reinterpret_cast<const uint4*>(&ks[t][0])[c];
        reinterpret_cast<uint4*>(p.V + dst)[c] = reinterpret_cast<const uint4*>(&vs[t][0])[c];
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
    const int parts = p.Hkv * (p.Mpad / 16);  // (KV head, m-tile) shares, in a fixed order
    const float* src = p.part_s + (static_cast<size_t>(ms) * p.B + b) * parts * p.max_len;
    for (int pos = lo + tid; pos < hi; pos += 128) {
      float v = 0.f;
#pragma unroll 8
      for (int q = 0; q < parts; ++q) v += src[static_cast<size_t>(q) * p.max_len + pos];
      dst[static_cast<size_t>(b) * p.score_stride + pos] = v;
    }
  }
}

template <int D, int MT>
cudaError_t launch_verify_t(const VerifyParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            cudaStream_t stream) {
  using C = VCfg<D, MT>;
  const size_t smem = C::smem(p.B);
  cudaError_t e = ensure_smem<verify_kernel<D, MT>>(smem);
  if (e != cudaSuccess) return e;
  verify_kernel<D, MT><<<p.nctas, C::THREADS, smem, stream>>>(p, tmK, tmV);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, verify_kernel<D, MT>) == cudaSuccess) {
      fprintf(stderr,
              "verify_kernel<%d,%d>: %s (regs=%d maxThreads=%d threads=%d staticSmem=%zu maxDynSmem=%d "
              "requestedSmem=%zu localBytes=%zu)\n",
              D, MT, cudaGetErrorString(e), fa.numRegs, fa.maxThreadsPerBlock, C::THREADS, fa.sharedSizeBytes,
              fa.maxDynamicSharedSizeBytes, smem, fa.localSizeBytes);
    }
    return e;
  }
  const int nO = p.B * p.Hkv * p.R;
  const int nS = ((p.mask0 | p.mask1) != 0u) ? p.B * ((p.max_len + kScoreChunk - 1) / kScoreChunk) : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nO + nS);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = static_cast<size_t>(p.nctas) * p.G * 2 * sizeof(float);
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
