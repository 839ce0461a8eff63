// Verification attention with fused logit aggregation, on 5th-generation tensor cores.
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
// construction).  Each CTA runs three roles:
//   warp 4   streams K and V tiles by 2-D TMA (128-byte swizzle) into a ring of
//            shared-memory stages;
//   warp 5   issues tcgen05.mma from one thread: S = Q K^T into a double-buffered
//            tensor-memory tile, then O += P V into a tensor-memory accumulator;
//   warps 0-3 own the 128 tensor-memory lanes, one A-operand row each: the G*(gamma+1)
//            query rows of the current KV head, then two rows per score mask that
//            hold the mask's summed query split into a bf16 high and low part.
// A row thread reads its row of S, runs the online softmax on it alone (max and sum
// are thread-local; the running max is raised only when a tile exceeds it by more
// than 2^8, after which the thread rescales its row of O in tensor memory), and
// writes its row of P (bf16) to shared memory for the P V product.  A score-row
// thread's S row is already the summed logit q_sum . k of each key of the tile
// (high part plus low part), so the aggregation costs two rows of the same MMA and
// no shuffles; the cache is read exactly once.  Each contiguous run of tiles of one
// (sequence, KV head) leaves one unnormalised partial (max, sum, O); a combine
// kernel, launched as a programmatic dependent of this one, merges the partials
// with the verify rows' own causal keys, writes bf16 outputs, appends the verify
// rows' K/V to the cache and sums the per-KV-head partial scores in a fixed order
// (deterministic, no atomics).
#include <cstdio>

#include "attn_frag.cuh"
#include "vg_common.cuh"
#include "vg_internal.h"

namespace vg {
namespace {

constexpr int TK = kVerifyTileKeys;
// A row's running max is raised only when a tile's max exceeds it by more than this
// (log2 units), so P stays below 2^8 and rescaling O is rare.
constexpr float kRescaleSlack = 8.f;

template <int D>
struct TCfg {
  static constexpr int kStages = (D == 128) ? 4 : 8;
  static constexpr int HALVES = D / 64;             // 64-column (128-byte) swizzled boxes
  static constexpr int HALF_BYTES = TK * 128;       // one box of a K or V tile
  static constexpr int TILE_BYTES = TK * D * 2;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile, then V tile
  static constexpr int QHALF = 128 * 128;           // A operand: 128 rows x 64 columns
  static constexpr int P_BYTES = 128 * TK * 2;      // P: 128 rows x 64 keys (one box wide)
  static constexpr int OFF_Q = kStages * STAGE_BYTES;
  static constexpr int OFF_P = OFF_Q + HALVES * QHALF;  // two P buffers
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  // full[S], empty[S], s_full[2], s_free[2], p_full[2], p_free[2], q_ready, fin
  static constexpr int NBAR = 2 * kStages + 10;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
  static constexpr int OFF_META = OFF_TMEM + 16;    // int cum[B+1], nlen[B]
  static constexpr int THREADS = 192;               // warps 0-3 rows, 4 TMA, 5 MMA
  static constexpr uint32_t TMEM_COLS = 256;        // O at columns [0, D), S buffers at 128 and 192
  static constexpr uint32_t COL_S = 128;
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


// A wait every lane of the warp takes together (so a lost wait cannot split the warp).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

template <int D>
__global__ void __launch_bounds__(TCfg<D>::THREADS, 1)
    verify_kernel(const VerifyParams p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  using C = TCfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sP = smem + C::OFF_P;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + S;
  uint64_t* s_full = full + 2 * S;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_full + 4;
  uint64_t* p_free = s_full + 6;
  uint64_t* q_ready = s_full + 8;
  uint64_t* fin = s_full + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM);
  int* cum = reinterpret_cast<int*>(smem + C::OFF_META);
  int* nlen = cum + p.B + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsc = 2 * ((p.mask0 ? 1 : 0) + (p.mask1 ? 1 : 0));  // score rows
  const int arows = p.M + nsc;                                   // A-operand rows in use

  if (warp == 0) seq_meta(p, cum, nlen);
  if (threadIdx.x == 32) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 4);
      mbar_init(&p_full[s], 4);
      mbar_init(&p_free[s], 1);
    }
    mbar_init(q_ready, 4);
    mbar_init(fin, 1);
    fence_mbar_init();
  }
  if (warp == 5) tc_alloc(tmem_slot, C::TMEM_COLS);
  // A-operand rows no segment writes stay zero: Q rows >= arows, P rows >= M
  {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const int qz = (128 - arows) * 8;
    for (int e = threadIdx.x; e < C::HALVES * qz; e += C::THREADS) {
      const int h = e / qz, r = arows + (e - h * qz) / 8, c = e & 7;
      *reinterpret_cast<uint4*>(sQ + h * C::QHALF + r * 128 + c * 16) = z;
    }
    const int pz = (128 - p.M) * 8;
    for (int e = threadIdx.x; e < 2 * pz; e += C::THREADS) {
      const int buf = e / pz, r = p.M + (e - buf * pz) / 8, c = e & 7;
      *reinterpret_cast<uint4*>(sP + buf * C::P_BYTES + r * 128 + c * 16) = z;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = *tmem_slot;
  if (blockIdx.x == 0) {  // the combine kernel reads these after this grid completes
    for (int i = threadIdx.x; i < 2 * p.B + 1; i += blockDim.x) p.meta[i] = cum[i];
  }
  pdl_launch_dependents();

  const int T = p.Hkv * cum[p.B];
  const int t0 = static_cast<int>(split_begin(blockIdx.x, T, p.nctas));
  const int ntiles = static_cast<int>(split_begin(blockIdx.x + 1, T, p.nctas)) - t0;

  if (ntiles > 0 && warp == 4 && lane == 0) {
    // ---------------------------------------------------------------- TMA producer
    int b, g, j;
    locate(t0, cum, p.B, p.Hkv, b, g, j);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    int issued = 0;
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % S;
      if (i >= S && !mbar_wait(&empty[st], ((i / S) - 1) & 1, p.status)) break;
      fence_proxy_async_smem();  // the stage may hold zeros written by the generic proxy
      mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
      uint8_t* kdst = smem + st * C::STAGE_BYTES;
      uint8_t* vdst = kdst + C::TILE_BYTES;
      const int y = static_cast<int>(p.seq_offset[b] + static_cast<int64_t>(j) * TK);
#pragma unroll
      for (int h = 0; h < C::HALVES; ++h) {
        tma_load_2d(kdst + h * C::HALF_BYTES, &tmK, g * D + h * 64, y, &full[st]);
        tma_load_2d(vdst + h * C::HALF_BYTES, &tmV, g * D + h * 64, y, &full[st]);
      }
      ++issued;
      advance(b, g, j, cum, p.B, p.Hkv);
    }
    // no copy may still be in flight when the CTA exits (normally all were consumed)
    for (int i = issued > S ? issued - S : 0; i < issued; ++i) mbar_wait(&full[i % S], (i / S) & 1, p.status);
  } else if (ntiles > 0 && warp == 5 && lane == 0) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idS = tc_idesc_bf16(128, TK, 0, 0);
    constexpr uint32_t idO = tc_idesc_bf16(128, D, 0, 1);
    const uint32_t base = smem_u32(smem), qaddr = smem_u32(sQ), paddr = smem_u32(sP);
    // O += P V for tile x (first: the first tile of its run, which overwrites O)
    auto pv = [&](int x, bool first) -> bool {
      if (!mbar_wait(&p_full[x & 1], (x >> 1) & 1, p.status)) return false;
      tc_fence_after();
      const int st = x % S;
      const uint32_t vaddr = base + st * C::STAGE_BYTES + C::TILE_BYTES;
#pragma unroll
      for (int kk = 0; kk < TK / 16; ++kk)
        tc_mma(tm, tc_desc_sw128(paddr + (x & 1) * C::P_BYTES + kk * 32, 16, 1024),
               tc_desc_sw128(vaddr + kk * 2048, C::HALF_BYTES, 1024), idO, (kk > 0 || !first) ? 1u : 0u);
      tc_commit(&empty[st]);
      tc_commit(&p_free[x & 1]);
      return true;
    };
    int b, g, j;
    locate(t0, cum, p.B, p.Hkv, b, g, j);
    int seg = 0;
    bool prev_first = false, ok = true;
    for (int i = 0; i < ntiles && ok; ++i) {
      const bool first = (i == 0) || (j == 0);
      // at a run boundary the row warps read O only after the previous run's last P V
      if (i > 0 && first && !pv(i - 1, prev_first)) { ok = false; break; }
      if (first) {
        if (!mbar_wait(q_ready, seg & 1, p.status)) { ok = false; break; }
        ++seg;
      }
      const int st = i % S;
      if (!mbar_wait(&full[st], (i / S) & 1, p.status)) { ok = false; break; }
      if (i >= 2 && !mbar_wait(&s_free[i & 1], ((i - 2) >> 1) & 1, p.status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t kaddr = base + st * C::STAGE_BYTES;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc_mma(tm + C::COL_S + (i & 1) * TK,
               tc_desc_sw128(qaddr + (kk >> 2) * C::QHALF + (kk & 3) * 32, 16, 1024),
               tc_desc_sw128(kaddr + (kk >> 2) * C::HALF_BYTES + (kk & 3) * 32, 16, 1024), idS,
               kk > 0 ? 1u : 0u);
      tc_commit(&s_full[i & 1]);
      // steady state: the previous tile's P V goes after this tile's Q K^T, so the
      // row warps find S ready as soon as they finish P
      if (i > 0 && !first && !pv(i - 1, prev_first)) { ok = false; break; }
      prev_first = first;
      advance(b, g, j, cum, p.B, p.Hkv);
    }
    if (ok) pv(ntiles - 1, prev_first);
    tc_commit(fin);  // every MMA of this thread complete before the CTA tears down
    mbar_wait(fin, 0, p.status);
  } else if (ntiles > 0 && warp < 4) {
    // ---------------------------------------------------------------- row warps
    const int tid = threadIdx.x;  // = tensor-memory lane = A-operand row
    const uint32_t tl = tm + (static_cast<uint32_t>(32 * warp) << 16);
    const bool wact = 32 * warp < arows;  // warp-uniform: lanes hold rows in use
    const bool is_row = tid < p.M;
    const int sci = tid - p.M;
    const bool is_sc = sci >= 0 && sci < nsc;
    const int sc_ms = (sci >> 1) == 0 && p.mask0 ? 0 : 1;  // score rows: mask0 first if in use
    const int sc_part = sci & 1;
    const float c2 = p.scale_log2;
    const float NEG = neg_inf();
    int b, g, j;
    locate(t0, cum, p.B, p.Hkv, b, g, j);
    bool ok = true;
    int i = 0;
    while (i < ntiles && ok) {
      const int n_b = nlen[b];
      const int seg_first = i;
      const int seg_end = min(ntiles, i + (cum[b + 1] - cum[b] - j));
      // query rows of this (sequence, KV head): row r -> (t = r / G, head g*G + r % G)
      for (int e = tid; e < p.M * (D / 8); e += 128) {
        const int r = e / (D / 8), c = e - r * (D / 8);
        const int t = r / p.G, hh = r - t * p.G;
        const uint4 v =
            *reinterpret_cast<const uint4*>(p.q + ((static_cast<size_t>(b) * p.R + t) * p.Hq + g * p.G + hh) * D + c * 8);
        *reinterpret_cast<uint4*>(sQ + (c >> 3) * C::QHALF + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
      }
      named_bar(1, 128);
      // score rows: column d of each mask's summed query, split into bf16 high + low
      if (nsc > 0 && tid < D) {
        const int cc = tid & 63;
        int a = 0;
        for (int ms = 0; ms < 2; ++ms) {
          const uint32_t mk = ms ? p.mask1 : p.mask0;
          if (mk == 0u) continue;
          float acc = 0.f;
          for (int r = 0; r < p.M; ++r) {
            if (((mk >> (r / p.G)) & 1u) == 0u) continue;
            acc += bf2f(*reinterpret_cast<const __nv_bfloat16*>(sQ + (tid >> 6) * C::QHALF + r * 128 +
                                                                 (((cc >> 3) ^ (r & 7)) << 4) + (cc & 7) * 2));
          }
          const __nv_bfloat16 hi = __float2bfloat16_rn(acc);
          const __nv_bfloat16 lo = __float2bfloat16_rn(acc - bf2f(hi));
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const int r = p.M + 2 * a + part;
            *reinterpret_cast<__nv_bfloat16*>(sQ + (tid >> 6) * C::QHALF + r * 128 + (((cc >> 3) ^ (r & 7)) << 4) +
                                              (cc & 7) * 2) = part ? lo : hi;
          }
          ++a;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_ready);

      float m = NEG, l = 0.f;
      for (; i < seg_end; ++i, ++j) {
        const int valid = min(TK, n_b - j * TK);  // keys of this tile inside the prefix (>= 1)
        if (!warp_wait(&s_full[i & 1], (i >> 1) & 1, p.status)) { ok = false; break; }
        tc_fence_after();
        float s[TK];
        if (wact) tc_ld64_sync(tl + C::COL_S + (i & 1) * TK, s);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[i & 1]);
        if (valid < TK) {
          // rows past the prefix end hold whatever the cache has there; their P is
          // zero, and zeroed V rows keep 0 * V exact even if the slots are not finite
          if (!warp_wait(&full[i % S], (i / S) & 1, p.status)) { ok = false; break; }
          uint8_t* vt = smem + (i % S) * C::STAGE_BYTES + C::TILE_BYTES;
          for (int e = tid; e < C::HALVES * TK * 8; e += 128) {
            const int h = e / (TK * 8), r = (e >> 3) & (TK - 1);
            if (r >= valid)
              *reinterpret_cast<uint4*>(vt + h * C::HALF_BYTES + r * 128 + (e & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        if (wact) {
          float mx = NEG;
          if (valid == TK) {
#pragma unroll
            for (int c = 0; c < TK; ++c) mx = fmaxf(mx, s[c]);
          } else {
#pragma unroll
            for (int c = 0; c < TK; ++c) mx = fmaxf(mx, c < valid ? s[c] : NEG);
          }
          mx *= c2;
          const bool first = (i == seg_first);
          const float mn = (is_row && (first || mx > m + kRescaleSlack)) ? fmaxf(m, mx) : m;
          const bool resc = is_row && !first && mn != m;
          if (__any_sync(0xffffffffu, resc)) {
            // rare: the running max rises; rescale l and this row of O once P V of
            // the previous tile has landed in tensor memory
            const float alpha = resc ? ex2(m - mn) : 1.f;
            l *= alpha;
            if (!warp_wait(&p_free[(i - 1) & 1], ((i - 1) >> 1) & 1, p.status)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              float o[32];
              tc_ld32_sync(tl + c0, o);
#pragma unroll
              for (int q = 0; q < 32; ++q) o[q] *= alpha;
              tc_st32(tl + c0, o);
            }
            tc_wait_st();
          }
          m = mn;
          // P of this tile goes to the buffer P V of tile i - 2 read
          if (i >= 2 && !warp_wait(&p_free[i & 1], ((i - 2) >> 1) & 1, p.status)) { ok = false; break; }
          if (is_row) {
            uint32_t pk[TK / 2];
            float ls = 0.f;
#pragma unroll
            for (int c = 0; c < TK; c += 2) {
              float p0 = ex2(fmaf(s[c], c2, -m)), p1 = ex2(fmaf(s[c + 1], c2, -m));
              if (valid < TK) {
                p0 = c < valid ? p0 : 0.f;
                p1 = c + 1 < valid ? p1 : 0.f;
              }
              ls += p0 + p1;
              pk[c / 2] = pack_bf16(p0, p1);
            }
            l += ls;
            uint8_t* prow = sP + (i & 1) * C::P_BYTES + tid * 128;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
              *reinterpret_cast<uint4*>(prow + ((cc ^ (tid & 7)) << 4)) =
                  make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
          } else if (is_sc) {
            float* dst = p.part_s +
                         (((static_cast<size_t>(sc_ms) * p.B + b) * p.Hkv + g) * 2 + sc_part) * p.s_stride + j * TK;
            if (valid == TK) {
#pragma unroll
              for (int c = 0; c < TK; c += 4)
                *reinterpret_cast<float4*>(dst + c) =
                    make_float4(s[c] * p.scale, s[c + 1] * p.scale, s[c + 2] * p.scale, s[c + 3] * p.scale);
            } else {
#pragma unroll
              for (int c = 0; c < TK; ++c)
                if (c < valid) dst[c] = s[c] * p.scale;
            }
          }
        }
        fence_proxy_async_smem();  // P (and zeroed V rows) before the async proxy reads them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[i & 1]);
      }
      if (!ok) break;
      // run partial: (O, max, sum) of each query row once P V of its last tile landed
      const int last = i - 1;
      if (!warp_wait(&p_free[last & 1], (last >> 1) & 1, p.status)) break;
      tc_fence_after();
      if (32 * warp < p.M) {
        const size_t prow = (static_cast<size_t>(blockIdx.x) + static_cast<size_t>(b) * p.Hkv + g) * p.Mpad + tid;
        float* orow = p.part_o + prow * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          tc_ld32_sync(tl + c0, o);
          if (is_row) {
#pragma unroll
            for (int q = 0; q < 32; q += 4)
              *reinterpret_cast<float4*>(orow + c0 + q) = make_float4(o[q], o[q + 1], o[q + 2], o[q + 3]);
          }
        }
        if (is_row) {
          p.part_ml[prow * 2 + 0] = m;
          p.part_ml[prow * 2 + 1] = l;
        }
      }
      tc_fence_before();
      // next (sequence, KV head)
      j = 0;
      if (++g == p.Hkv) {
        g = 0;
        ++b;
        while (b < p.B && cum[b + 1] == cum[b]) ++b;
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tc_dealloc(tm, C::TMEM_COLS);
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
    const int parts = p.Hkv * 2;  // (KV head, high / low part) shares, in a fixed order
    const float* src = p.part_s + (static_cast<size_t>(ms) * p.B + b) * parts * p.s_stride;
    for (int pos = lo + tid; pos < hi; pos += 128) {
      float v = 0.f;
#pragma unroll 8
      for (int q = 0; q < parts; ++q) v += src[static_cast<size_t>(q) * p.s_stride + pos];
      dst[static_cast<size_t>(b) * p.score_stride + pos] = v;
    }
  }
}

template <int D>
cudaError_t launch_verify_t(const VerifyParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            cudaStream_t stream) {
  using C = TCfg<D>;
  const size_t smem = C::smem(p.B);
  cudaError_t e = ensure_smem<verify_kernel<D>>(smem);
  if (e != cudaSuccess) return e;
  verify_kernel<D><<<p.nctas, C::THREADS, smem, stream>>>(p, tmK, tmV);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, verify_kernel<D>) == cudaSuccess) {
      fprintf(stderr,
              "verify_kernel<%d>: %s (regs=%d maxThreads=%d threads=%d staticSmem=%zu maxDynSmem=%d "
              "requestedSmem=%zu localBytes=%zu)\n",
              D, cudaGetErrorString(e), fa.numRegs, fa.maxThreadsPerBlock, C::THREADS, fa.sharedSizeBytes,
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

size_t verify_smem_bytes(int D, int B) {
  if (D == 64) return TCfg<64>::smem(B);
  if (D == 128) return TCfg<128>::smem(B);
  return 0;
}

cudaError_t launch_verify(const VerifyParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          cudaStream_t stream) {
  if (p.D == 64) return launch_verify_t<64>(p, tmK, tmV, stream);
  if (p.D == 128) return launch_verify_t<128>(p, tmK, tmV, stream);
  return cudaErrorInvalidValue;
}

}  // namespace vg
