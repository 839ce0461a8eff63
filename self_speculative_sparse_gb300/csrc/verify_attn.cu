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
// construction).  Each CTA runs four roles:
//   warp 8   streams K and V tiles by 2-D TMA (128-byte swizzle) into a ring of
//            shared-memory stages;
//   warp 9   issues tcgen05.mma from one thread: S = Q K^T into a double-buffered
//            tensor-memory tile;
//   warp 10  issues O += P V from one thread into a tensor-memory accumulator, as
//            soon as a tile's P is written;
//   warps 0-7 own the 128 tensor-memory lanes, one A-operand row per lane: the
//            G*(gamma+1) query rows of the current KV head, then two rows per score
//            mask that hold the mask's summed query split into a bf16 high and low
//            part.  Warps w and w + 4 share lane quadrant w and take the low and high
//            32 keys of each tile.
// A row thread reads its half row of S and runs the online softmax on it (max and
// sum are per thread; the two halves of a row agree on the tile max through shared
// memory; the running max is raised only when a tile exceeds it by more than 2^8,
// after which the row's O is rescaled in tensor memory), and writes its half row of
// P (bf16) to shared memory for the P V product; in runs of a short prefix it also
// writes P's low part, P - bf16(P), which a second P V product adds in.  When the
// query and score rows fit in 64, the MMAs use M = 64, which halves the Q and P
// buffers and leaves room for more stages.  A score-row
// thread's S row is already the summed logit q_sum . k of each key of the tile
// (high part plus low part), so the aggregation costs two rows of the same MMA and
// no shuffles; the cache is read exactly once.  Each contiguous run of tiles of one
// (sequence, KV head) leaves one unnormalised partial (max, sum, O); a combine
// kernel, launched as a programmatic dependent of this one, merges the partials
// with the verify rows' own causal keys, writes bf16 outputs, appends the verify
// rows' K/V to the cache and sums the per-KV-head partial scores in a fixed order
// (deterministic, no atomics).
#include <cstdio>

#include "vg_common.cuh"
#include "vg_internal.h"

namespace vg {
namespace {

constexpr int TK = kVerifyTileKeys;
// A row's running max is raised only when a tile's max exceeds it by more than this
// (log2 units), so P stays below 2^8 and rescaling O is rare.
constexpr float kRescaleSlack = 8.f;
// Runs of a sequence with at most this many prefix keys carry P as a bf16 high part
// plus a bf16 low part (P - bf16(P)), so their weights are exact to about 2^-17.  With
// round-to-nearest the output's error from rounding P to bf16 alone is about
// 2^-9 * sqrt(sum_i w_i^2 v_i^2), which only rows whose weight sits on a few keys bring
// near the 2e-3 asked of the outputs; few keys make that likely.  A second P V product
// adds the low part in; longer runs, whose weights spread, go without it.
constexpr int kLowRunKeys = 1024;

// MR: rows of the MMA (64 when the query and score rows fit, else 128).  With
// M = 64 the accumulator's row r sits in lane 16 (r / 16) + r % 16 of quadrant r / 16.
template <int D, int MR>
struct TCfg {
  static constexpr int STAGE_BYTES_ = 2 * kVerifyTileKeys * D * 2;
  static constexpr int kStages =  // as many stages as 208 KB leave beside Q and four P buffers
      (212992 - (D / 64) * MR * 128 - 4 * MR * kVerifyTileKeys * 2) / STAGE_BYTES_ > 12
          ? 12
          : (212992 - (D / 64) * MR * 128 - 4 * MR * kVerifyTileKeys * 2) / STAGE_BYTES_;
  static constexpr int HALVES = D / 64;             // 64-column (128-byte) swizzled boxes
  static constexpr int HALF_BYTES = TK * 128;       // one box of a K or V tile
  static constexpr int TILE_BYTES = TK * D * 2;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile, then V tile
  static constexpr int QHALF = MR * 128;            // A operand: MR rows x 64 columns
  static constexpr int P_BYTES = MR * TK * 2;       // P: MR rows x 64 keys (one box wide)
  static constexpr int OFF_Q = kStages * STAGE_BYTES;
  static constexpr int OFF_P = OFF_Q + HALVES * QHALF;  // P high part [2], then low part [2]
  static constexpr int OFF_BAR = OFF_P + 4 * P_BYTES;
  // full[S], empty[S], s_full[2], s_free[2], p_full[2], p_free[2], q_ready, fin[2], q_landed
  static constexpr int NBAR = 2 * kStages + 12;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;  // tensor-memory base, abort flag
  static constexpr int OFF_X = OFF_TMEM + 16;       // float xm[2][2][128] tile maxima, xl[128] sums
  static constexpr int OFF_META = OFF_X + 5 * 128 * 4;  // int cum[B+1], nlen[B]
  static constexpr int RWARPS = 8;                  // row warps: two per tensor-memory lane quadrant
  static constexpr int THREADS = (RWARPS + 3) * 32; // + TMA producer, Q K^T issuer, P V issuer
  static constexpr uint32_t TMEM_COLS = 256;        // O at columns [0, D), S buffers at 128 and 192
  static constexpr uint32_t COL_S = 128;
  static constexpr size_t smem(int B) { return 1024 + OFF_META + (size_t)(2 * B + 1) * 4; }
};
// every configuration fits the 227 KB a CTA may hold at the largest batch
static_assert(TCfg<64, 64>::smem(kMaxBatch) <= 232448 && TCfg<64, 128>::smem(kMaxBatch) <= 232448 &&
                  TCfg<128, 64>::smem(kMaxBatch) <= 232448 && TCfg<128, 128>::smem(kMaxBatch) <= 232448,
              "verify shared memory exceeds the per-CTA limit");


__device__ __forceinline__ float bf2f(__nv_bfloat16 v) { return __bfloat162float(v); }

// A prefix length the cache can hold with the gamma+1 verify rows after it: the slot
// pool from seq_offset[b] on, or the sequence's pages in the page table (page entries
// are checked where they are read).
__device__ __forceinline__ bool seq_len_ok(const VerifyParams& p, int b, int n) {
  if (n < 0 || n > p.max_len) return false;
  if (p.ptab) return static_cast<int64_t>(n) + p.R <= static_cast<int64_t>(p.pstride) * p.psize;
  const int64_t off = p.seq_offset[b];
  return off >= 0 && off + static_cast<int64_t>(n) + p.R <= p.capacity;
}

// The key / value row of verify row u of sequence b (prefix length n), KV head g: from
// the inputs when given, else from the cache slot after the prefix (null if that slot
// is outside the cache).
template <int D>
__device__ __forceinline__ const __nv_bfloat16* verify_row(const VerifyParams& p, const __nv_bfloat16* fresh,
                                                           const __nv_bfloat16* cache, int b, int n, int u, int g) {
  if (fresh) return fresh + ((static_cast<size_t>(b) * p.R + u) * p.Hkv + g) * D;
  const int64_t slot = kv_slot(p.seq_offset, p.ptab, p.psize, p.pstride, p.capacity, b, n + u);
  return slot >= 0 ? cache + (slot * p.Hkv + g) * D : nullptr;
}

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
      if (!seq_len_ok(p, b, n)) {
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
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int32_t* status, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait_ab(bar, parity, status, abort));
}

// PAGED: the cache is read through a page table (a separate instantiation, so that the
// slot pool's kernel keeps its lean producer).
template <int D, int MR, bool PAGED>
__global__ void __launch_bounds__(TCfg<D, MR>::THREADS, 1)
    verify_kernel(const VerifyParams p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  using C = TCfg<D, MR>;
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
  uint64_t* q_landed = s_full + 11;  // the first run's query rows are in shared memory
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM);
  // Raised by the first wait that runs out; every later wait then gives up at once.
  // The TMA producer and the two issuers stop and drain what they started; the row
  // warps run their loops to the end without waiting, so that the warp pairs' named
  // barriers still match and no thread is left behind at one.
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::OFF_TMEM + 4);
  int* cum = reinterpret_cast<int*>(smem + C::OFF_META);
  int* nlen = cum + p.B + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsc = 2 * ((p.mask0 ? 1 : 0) + (p.mask1 ? 1 : 0));  // score rows
  const int arows = nsc ? p.sc_row0 + nsc : p.M;                 // A-operand rows in use

  // Launched as a programmatic dependent: shared and tensor memory are set up while
  // the previous kernel in the stream finishes; nothing in global memory (the
  // lengths, the inputs, the cache, the workspace) is read or written before the wait.
  if (threadIdx.x == 32) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], C::RWARPS);
      mbar_init(&p_full[s], C::RWARPS);
      mbar_init(&p_free[s], 1);
    }
    mbar_init(q_ready, C::RWARPS);
    mbar_init(&fin[0], 1);
    mbar_init(&fin[1], 1);
    mbar_init(q_landed, C::RWARPS);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == C::RWARPS + 1) tc_alloc(tmem_slot, C::TMEM_COLS);  // (and frees it at the end)
  // A-operand rows no segment writes stay zero: Q rows in [M, sc_row0) and >= arows,
  // P rows >= M
  {
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    const int gap = nsc ? p.sc_row0 - p.M : 0;  // rows between the query rows and the score rows
    const int qz = (MR - arows + gap) * 8;
    for (int e = threadIdx.x; e < C::HALVES * qz; e += C::THREADS) {
      const int h = e / qz, k = (e - h * qz) / 8, c = e & 7;
      const int r = k < gap ? p.M + k : arows + (k - gap);
      *reinterpret_cast<uint4*>(sQ + h * C::QHALF + r * 128 + c * 16) = z;
    }
    const int pz = (MR - p.M) * 8;
    for (int e = threadIdx.x; e < 2 * pz; e += C::THREADS) {
      const int buf = e / pz, r = p.M + (e - buf * pz) / 8, c = e & 7;
      *reinterpret_cast<uint4*>(sP + buf * C::P_BYTES + r * 128 + c * 16) = z;
    }
    for (int e = threadIdx.x; e < 2 * C::P_BYTES / 16; e += C::THREADS)  // (low-part rows >= M stay zero)
      reinterpret_cast<uint4*>(sP + 2 * C::P_BYTES)[e] = z;
  }
  fence_proxy_async_smem();
  pdl_wait();
  if (warp == 0) seq_meta(p, cum, nlen);
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

  if (!PAGED && ntiles > 0 && warp == C::RWARPS) {
    // ---------------------------------------------------------------- TMA producer (slot pool)
    // one thread: a tile of 64 keys is one box per half of K and of V
    if (lane == 0) {
      int b, g, j;
      locate(t0, cum, p.B, p.Hkv, b, g, j);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int issued = 0;
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % S;
        // after the first stage, the first run's query rows go first: issued together
        // with the whole ring, their loads would queue behind it (about 3 us at the start)
        if (i == 1 && !mbar_wait_ab(q_landed, 0, p.status, abort)) break;
        if (i >= S && !mbar_wait_ab(&empty[st], ((i / S) - 1) & 1, p.status, abort)) break;
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
    }
    __syncwarp();
  } else if (PAGED && ntiles > 0 && warp == C::RWARPS) {
    // ---------------------------------------------------------------- TMA producer (paged)
    // A tile of 64 keys is WPT = 64 / box_rows boxes (page pieces; pages of 8, 16, 32
    // tokens or a multiple of 64, so WPT <= 8), each at its page's physical rows; lane s
    // issues box s.  The page-table words are loaded a batch ahead, one a lane (tile
    // base + lane / WPT, box lane % WPT) with an unconditional, clamped load, and reach
    // the issuing lanes by shuffle when their tile is issued: no load's latency sits
    // between two tiles' copies.  Boxes wholly past the prefix are not loaded (their rows
    // are masked, and the row warps zero such value rows).  Lane 0 takes the waits and
    // the byte count.
    int b, g, j;
    locate(t0, cum, p.B, p.Hkv, b, g, j);
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    const int BR = p.box_rows;
    const int WPT = TK / BR;   // page words a tile
    const int TPB = 32 / WPT;  // tiles a batch of words
    // word and kind (0: no box, 1: past the sequence's table, 2: a table word) of this
    // lane's box in the batch starting at tile `base`
    auto load_words = [&](int base, int& w, int& kind) {
      const int ti = base + lane / WPT, sb = lane % WPT;
      int bb = 0, gg = 0, jj = 0;
      if (ti < ntiles) locate(t0 + ti, cum, p.B, p.Hkv, bb, gg, jj);
      const int keys = ti < ntiles ? min(TK, nlen[bb] - jj * TK) : 0;
      const int pos = jj * TK + sb * BR;
      const int lim = p.pstride * p.psize;
      kind = sb * BR >= keys ? 0 : (pos < lim ? 2 : 1);
      const int pi = min(pos, lim - 1) / p.psize;  // (always inside the table: the load is unconditional)
      w = p.ptab[static_cast<size_t>(bb) * p.pstride + pi];
    };
    int cw, ck, nw, nk;
    load_words(0, cw, ck);
    load_words(TPB, nw, nk);
    int base = 0, issued = 0;
    for (int i = 0; i < ntiles; ++i) {
      if (i - base == TPB) {  // the next batch (loaded a batch ago), and the one after it
        cw = nw;
        ck = nk;
        base += TPB;
        load_words(base + TPB, nw, nk);
      }
      const int st = i % S;
      // after the first stage, the first run's query rows go first: issued together
      // with the whole ring, their loads would queue behind it (about 3 us at the start)
      bool ok = true;
      if (lane == 0) {
        if (i == 1) ok = mbar_wait_ab(q_landed, 0, p.status, abort);
        if (ok && i >= S) ok = mbar_wait_ab(&empty[st], ((i / S) - 1) & 1, p.status, abort);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const int src = (i - base) * WPT + (lane < WPT ? lane : 0);
      const int w = __shfl_sync(0xffffffffu, cw, src), kind = __shfl_sync(0xffffffffu, ck, src);
      int y = -1;
      if (lane < WPT && kind != 0) {
        if (kind == 1 || w < 0 || (static_cast<int64_t>(w) + 1) * p.psize > p.capacity)
          report(p.status, VG_ERR_DEVICE_BOUNDS);
        else
          y = w * p.psize + (j * TK + lane * BR) % p.psize;
      }
      const int nload = __popc(__ballot_sync(0xffffffffu, y >= 0));
      if (lane == 0) {
        fence_proxy_async_smem();  // the stage may hold zeros written by the generic proxy
        mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(nload * BR * 128 * C::HALVES * 2));
      }
      __syncwarp();
      if (y >= 0) {
        uint8_t* kdst = smem + st * C::STAGE_BYTES + lane * BR * 128;
        uint8_t* vdst = kdst + C::TILE_BYTES;
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          tma_load_2d(kdst + h * C::HALF_BYTES, &tmK, g * D + h * 64, y, &full[st]);
          tma_load_2d(vdst + h * C::HALF_BYTES, &tmV, g * D + h * 64, y, &full[st]);
        }
      }
      ++issued;
      advance(b, g, j, cum, p.B, p.Hkv);
    }
    // no copy may still be in flight when the CTA exits (normally all were consumed)
    if (lane == 0)
      for (int i = issued > S ? issued - S : 0; i < issued; ++i) mbar_wait(&full[i % S], (i / S) & 1, p.status);
    __syncwarp();
  } else if (ntiles > 0 && warp == C::RWARPS + 1 && lane == 0) {
    // ---------------------------------------------------------------- Q K^T issuer
    constexpr uint32_t idS = tc_idesc_bf16(MR, TK, 0, 0);
    const uint32_t base = smem_u32(smem), qaddr = smem_u32(sQ);
    int b, g, j;
    locate(t0, cum, p.B, p.Hkv, b, g, j);
    int seg = 0;
    for (int i = 0; i < ntiles; ++i) {
      if (i == 0 || j == 0) {  // a new run: its query rows must be in shared memory
        if (!mbar_wait_ab(q_ready, seg & 1, p.status, abort)) break;
        ++seg;
      }
      const int st = i % S;
      if (!mbar_wait_ab(&full[st], (i / S) & 1, p.status, abort)) break;
      if (i >= 2 && !mbar_wait_ab(&s_free[i & 1], ((i - 2) >> 1) & 1, p.status, abort)) break;
      tc_fence_after();
      const uint32_t kaddr = base + st * C::STAGE_BYTES;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        tc_mma(tm + C::COL_S + (i & 1) * TK,
               tc_desc_sw128(qaddr + (kk >> 2) * C::QHALF + (kk & 3) * 32, 16, 1024),
               tc_desc_sw128(kaddr + (kk >> 2) * C::HALF_BYTES + (kk & 3) * 32, 16, 1024), idS,
               kk > 0 ? 1u : 0u);
      tc_commit(&s_full[i & 1]);
      advance(b, g, j, cum, p.B, p.Hkv);
    }
    tc_commit(&fin[0]);  // every MMA of this thread complete before the CTA tears down
    mbar_wait(&fin[0], 0, p.status);
  } else if (ntiles > 0 && warp == C::RWARPS + 2 && lane == 0) {
    // ---------------------------------------------------------------- P V issuer
    // (its own thread, so P V of a tile starts as soon as P is written, not after the
    // next tile's Q K^T has been issued)
    constexpr uint32_t idO = tc_idesc_bf16(MR, D, 0, 1);
    const uint32_t base = smem_u32(smem), paddr = smem_u32(sP);
    int b, g, j;
    locate(t0, cum, p.B, p.Hkv, b, g, j);
    bool lo = nlen[b] <= kLowRunKeys;  // a short run: its P's low part too
    for (int i = 0; i < ntiles; ++i) {
      const bool first = (i == 0) || (j == 0);  // the first tile of a run overwrites O
      if (!mbar_wait_ab(&p_full[i & 1], (i >> 1) & 1, p.status, abort)) break;
      tc_fence_after();
      const int st = i % S;
      const uint32_t vaddr = base + st * C::STAGE_BYTES + C::TILE_BYTES;
#pragma unroll
      for (int kk = 0; kk < TK / 16; ++kk)
        tc_mma(tm, tc_desc_sw128(paddr + (i & 1) * C::P_BYTES + kk * 32, 16, 1024),
               tc_desc_sw128(vaddr + kk * 2048, C::HALF_BYTES, 1024), idO, (kk > 0 || !first) ? 1u : 0u);
      if (lo) {
#pragma unroll
        for (int kk = 0; kk < TK / 16; ++kk)
          tc_mma(tm, tc_desc_sw128(paddr + (2 + (i & 1)) * C::P_BYTES + kk * 32, 16, 1024),
                 tc_desc_sw128(vaddr + kk * 2048, C::HALF_BYTES, 1024), idO, 1u);
      }
      tc_commit(&empty[st]);
      tc_commit(&p_free[i & 1]);
      advance(b, g, j, cum, p.B, p.Hkv);
      if (j == 0) lo = b < p.B && nlen[b] <= kLowRunKeys;
    }
    tc_commit(&fin[1]);
    mbar_wait(&fin[1], 0, p.status);
  } else if (ntiles > 0 && warp < C::RWARPS) {
    // ---------------------------------------------------------------- row warps
    constexpr int NR = C::RWARPS * 32;
    constexpr int HK = TK / 2;            // keys of a tile per half
    const int rtid = threadIdx.x;         // 0 .. NR-1, for cooperative loops
    const int quad = warp & 3, half = warp >> 2;
    constexpr int QR = MR / 4;            // accumulator rows per lane quadrant
    const int row = lane < QR ? QR * quad + lane : 128;  // A-operand row of this lane (128: none)
    const bool has_row = row < 128;
    const uint32_t tl = tm + (static_cast<uint32_t>(32 * quad) << 16);
    const bool wact = QR * quad < arows;  // warp-uniform: lanes hold rows in use
    const bool is_row = row < p.M;
    const int sci = row - p.sc_row0;
    const bool is_sc = sci >= 0 && sci < nsc;
    const int sc_ms = (sci >> 1) == 0 && p.mask0 ? 0 : 1;  // score rows: mask0 first if in use
    const int sc_part = sci & 1;
    const float c2 = p.scale_log2;
    const float NEG = neg_inf();
    float* xm = reinterpret_cast<float*>(smem + C::OFF_X);  // [tile parity][half][row]
    float* xl = xm + 4 * 128;                               // [row]
    int b, g, j;
    locate(t0, cum, p.B, p.Hkv, b, g, j);
    int i = 0;
    while (i < ntiles) {
      const int n_b = nlen[b];
      const bool lo_run = n_b <= kLowRunKeys;  // (uniform over the CTA)
      const int seg_first = i;
      const int seg_end = min(ntiles, i + (cum[b + 1] - cum[b] - j));
      // query rows of this (sequence, KV head): row r -> (t = r / G, head g*G + r % G)
      for (int e = rtid; e < p.M * (D / 8); e += NR) {
        const int r = e / (D / 8), c = e - r * (D / 8);
        const int t = r / p.G, hh = r - t * p.G;
        const uint4 v =
            *reinterpret_cast<const uint4*>(p.q + ((static_cast<size_t>(b) * p.R + t) * p.Hq + g * p.G + hh) * D + c * 8);
        *reinterpret_cast<uint4*>(sQ + (c >> 3) * C::QHALF + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
      }
      named_bar(1, NR);
      if (seg_first == 0) {  // (the TMA producer holds back the ring until then)
        __syncwarp();
        if (lane == 0) mbar_arrive(q_landed);
      }
      // score rows: column d of each mask's summed query, split into bf16 high + low
      if (nsc > 0 && rtid < D) {
        const int cc = rtid & 63;
        int a = 0;
        for (int ms = 0; ms < 2; ++ms) {
          const uint32_t mk = ms ? p.mask1 : p.mask0;
          if (mk == 0u) continue;
          float acc = 0.f;
          for (uint32_t bits = mk; bits != 0u; bits &= bits - 1u) {  // the mask's rows t, then heads
            const int r0 = (__ffs(bits) - 1) * p.G;
            for (int r = r0; r < r0 + p.G; ++r)
              acc += bf2f(*reinterpret_cast<const __nv_bfloat16*>(sQ + (rtid >> 6) * C::QHALF + r * 128 +
                                                                   (((cc >> 3) ^ (r & 7)) << 4) + (cc & 7) * 2));
          }
          const __nv_bfloat16 hi = __float2bfloat16_rn(acc);
          const __nv_bfloat16 lo = __float2bfloat16_rn(acc - bf2f(hi));
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const int r = p.sc_row0 + 2 * a + part;
            *reinterpret_cast<__nv_bfloat16*>(sQ + (rtid >> 6) * C::QHALF + r * 128 + (((cc >> 3) ^ (r & 7)) << 4) +
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
        const int valid = min(TK, n_b - j * TK) - half * HK;  // keys of this half inside the prefix
        warp_wait(&s_full[i & 1], (i >> 1) & 1, p.status, abort);
        tc_fence_after();
        float s[HK];
        if (wact) tc_ld32_sync(tl + C::COL_S + (i & 1) * TK + half * HK, s);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[i & 1]);
        const int vt_keys = min(TK, n_b - j * TK);
        if (vt_keys < TK) {
          // rows past the prefix end hold whatever the cache has there; their P is
          // zero, and zeroed V rows keep 0 * V exact even if the slots are not finite
          warp_wait(&full[i % S], (i / S) & 1, p.status, abort);
          uint8_t* vt = smem + (i % S) * C::STAGE_BYTES + C::TILE_BYTES;
          for (int e = rtid; e < C::HALVES * TK * 8; e += NR) {
            const int h = e / (TK * 8), r = (e >> 3) & (TK - 1);
            if (r >= vt_keys)
              *reinterpret_cast<uint4*>(vt + h * C::HALF_BYTES + r * 128 + (e & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        if (wact) {
          float mx = NEG;
          if (valid >= HK) {
#pragma unroll
            for (int c = 0; c < HK; ++c) mx = fmaxf(mx, s[c]);
          } else {
#pragma unroll
            for (int c = 0; c < HK; ++c) mx = fmaxf(mx, c < valid ? s[c] : NEG);
          }
          mx *= c2;
          // both halves of the row take the max of the whole tile
          if (has_row) xm[((i & 1) * 2 + half) * 128 + row] = mx;
          named_bar(2 + quad, 64);
          if (has_row) mx = fmaxf(mx, xm[((i & 1) * 2 + (half ^ 1)) * 128 + row]);
          const bool first = (i == seg_first);
          const float mn = (is_row && (first || mx > m + kRescaleSlack)) ? fmaxf(m, mx) : m;
          const bool resc = is_row && !first && mn != m;
          if (__any_sync(0xffffffffu, resc)) {
            // rare: the running max rises; rescale l, and (low half) this row of O
            // once P V of the previous tile has landed in tensor memory
            const float alpha = resc ? ex2(m - mn) : 1.f;
            l *= alpha;
            if (half == 0) {
              warp_wait(&p_free[(i - 1) & 1], ((i - 1) >> 1) & 1, p.status, abort);
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
          }
          m = mn;
        }
        // P of this tile goes to the buffer P V of tile i - 2 read.  Every row warp waits,
        // also one whose lanes hold no row in use: its arrival on p_full must not run
        // ahead into the phase of tile i - 2 (its own S wait only bounds it by the
        // s_free phase of that tile), or P V of tile i - 2 could start before an active
        // warp has written its P rows.
        if (i >= 2) warp_wait(&p_free[i & 1], ((i - 2) >> 1) & 1, p.status, abort);
        if (wact) {
          if (is_row) {
            if (!lo_run) {
              uint32_t pk[HK / 2];
              float ls = 0.f;
#pragma unroll
              for (int c = 0; c < HK; c += 2) {
                float p0 = ex2(fmaf(s[c], c2, -m)), p1 = ex2(fmaf(s[c + 1], c2, -m));
                if (valid < HK) {
                  p0 = c < valid ? p0 : 0.f;
                  p1 = c + 1 < valid ? p1 : 0.f;
                }
                // the sum takes the bf16 values P V multiplies, so a row's weights sum to one
                // up to fp32 rounding (with the lazily raised max a dominant P is not a
                // power of two, and its bf16 rounding would otherwise shift the row)
                pk[c / 2] = pack_bf16(p0, p1);
                ls = add_bf16x2_f32(pk[c / 2], ls);
              }
              l += ls;
              uint8_t* prow = sP + (i & 1) * C::P_BYTES + row * 128;
#pragma unroll
              for (int cc = 0; cc < HK / 8; ++cc)
                *reinterpret_cast<uint4*>(prow + (((half * (HK / 8) + cc) ^ (row & 7)) << 4)) =
                    make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
            } else {
              // a short run: P = high + low, both bf16, eight keys at a time
              float ls = 0.f;
              uint8_t* prow = sP + (i & 1) * C::P_BYTES + row * 128;
#pragma unroll
              for (int cc = 0; cc < HK / 8; ++cc) {
                uint32_t hk[4], lk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int c = 8 * cc + 2 * e;
                  float p0 = ex2(fmaf(s[c], c2, -m)), p1 = ex2(fmaf(s[c + 1], c2, -m));
                  p0 = c < valid ? p0 : 0.f;
                  p1 = c + 1 < valid ? p1 : 0.f;
                  hk[e] = pack_bf16(p0, p1);
                  lk[e] = pack_bf16(p0 - __uint_as_float(hk[e] << 16), p1 - __uint_as_float(hk[e] & 0xffff0000u));
                  ls = add_bf16x2_f32(lk[e], add_bf16x2_f32(hk[e], ls));
                }
                const int off = ((half * (HK / 8) + cc) ^ (row & 7)) << 4;
                *reinterpret_cast<uint4*>(prow + off) = make_uint4(hk[0], hk[1], hk[2], hk[3]);
                *reinterpret_cast<uint4*>(prow + 2 * C::P_BYTES + off) = make_uint4(lk[0], lk[1], lk[2], lk[3]);
              }
              l += ls;
            }
          } else if (is_sc && valid > 0) {
            float* dst = p.part_s +
                         (((static_cast<size_t>(sc_ms) * p.B + b) * p.Hkv + g) * 2 + sc_part) * p.s_stride + j * TK +
                         half * HK;
            if (valid >= HK) {
#pragma unroll
              for (int c = 0; c < HK; c += 4)
                *reinterpret_cast<float4*>(dst + c) =
                    make_float4(s[c] * p.scale, s[c + 1] * p.scale, s[c + 2] * p.scale, s[c + 3] * p.scale);
            } else {
#pragma unroll
              for (int c = 0; c < HK; ++c)
                if (c < valid) dst[c] = s[c] * p.scale;
            }
          }
        }
        fence_proxy_async_smem();  // P (and zeroed V rows) before the async proxy reads them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[i & 1]);
      }
      // run partial: (O, max, sum) of each query row once P V of its last tile landed
      const int last = i - 1;
      if (QR * quad < p.M) {  // the two halves' sums meet in the low half
        if (half == 1 && has_row) xl[row] = l;
        named_bar(2 + quad, 64);
      }
      if (half == 0) {
        warp_wait(&p_free[last & 1], (last >> 1) & 1, p.status, abort);
        tc_fence_after();
        if (QR * quad < p.M) {
          const size_t prow = (static_cast<size_t>(blockIdx.x) + static_cast<size_t>(b) * p.Hkv + g) * p.Mpad + row;
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
            p.part_ml[prow * 2 + 1] = l + xl[row];
          }
        }
        tc_fence_before();
      }
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
  if (warp == C::RWARPS + 1) {
    tc_fence_after();
    tc_dealloc(tm, C::TMEM_COLS);
  }
}

// Merge of the partials with the verify rows' causal keys, output, append, scores.
// Role A, CTAs over (sequence b, KV head g, 8 consecutive rows r = t*G + jh of the
// head's G*(gamma+1) query rows), one warp per row, lanes across d.  A warp issues
// every load it needs in one round (the partials' max/sum, the first partial rows,
// its query row and the verify rows' own keys and values u <= t), then merges in a
// fixed order: partials by CTA, then the causal keys u = 0..t.
// Role B, CTAs of 1024 prefix positions (4 per thread): fixed-order sum of the
// per-(KV head, high / low part) partial scores.
constexpr int kCombineWarps = 8;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32, 2) verify_combine_kernel(const VerifyParams p) {
  constexpr int PER = D / 32;  // elements of a row per lane
  constexpr int NB = D == 128 ? 4 : 8;  // partial rows per round of loads (two rounds in registers)
  __shared__ float lgs[kCombineWarps][16];               // a warp's causal logits (log2 units)
  __shared__ __align__(16) __nv_bfloat16 kvs[2][16][D];  // the verify rows' keys and values
  pdl_launch_dependents();  // the selection kernel may start its prologue
  pdl_wait();
  const int* cum = p.meta;
  const int* nlen = p.meta + p.B + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float NEG = neg_inf();
  const int rblocks = (p.M + kCombineWarps - 1) / kCombineWarps;  // CTAs per (sequence, KV head)
  const int nA = p.B * p.Hkv * rblocks;
  if (static_cast<int>(blockIdx.x) < nA) {
    const int bg = blockIdx.x / rblocks;
    const int r0 = (blockIdx.x - bg * rblocks) * kCombineWarps;
    const int r = r0 + warp;  // row t*G + jh
    const int g = bg % p.Hkv, b = bg / p.Hkv;
    const int n = nlen[b];
    if (n < 0) return;  // the whole CTA
    const int G = p.G;
    const bool active = r < p.M;
    const int t = active ? r / G : 0, jh = r - t * G;
    const int tmax = min(p.M - 1, r0 + kCombineWarps - 1) / G;  // last verify row of this CTA
    // partials of this (sequence, KV head): CTAs cf..cl of the verify split
    const int tiles = cum[b + 1] - cum[b];
    const int64_t T = static_cast<int64_t>(p.Hkv) * cum[p.B];
    int64_t cf = 0, cl = -1;
    if (tiles > 0) {
      const int64_t S = static_cast<int64_t>(p.Hkv) * cum[b] + static_cast<int64_t>(g) * tiles;
      cf = owner_cta(S, T, p.nctas);
      cl = owner_cta(S + tiles - 1, T, p.nctas);
    }
    const int nseg = active ? static_cast<int>(cl - cf + 1) : 0;
    const size_t pair = static_cast<size_t>(b) * p.Hkv + g;
    auto prow = [&](int si) { return (static_cast<size_t>(cf + si) + pair) * p.Mpad + r; };
    auto load_ml = [&](int si, float& ms, float& ls) {
      ms = NEG;
      ls = 0.f;
      if (si < nseg && split_nonempty(cf + si, T, p.nctas)) {  // CTAs with no items wrote no partial
        const float2 v = *reinterpret_cast<const float2*>(p.part_ml + prow(si) * 2);
        ms = v.x;
        ls = v.y;
      }
    };
    // (rows past nseg, or of a CTA with no items, read as zeros: their weight is zero
    // and the row holds whatever was there)
    auto load_rows = [&](int s0, float (&v)[NB][PER]) {
#pragma unroll
      for (int q = 0; q < NB; ++q) {
        const bool ok = s0 + q < nseg && split_nonempty(cf + s0 + q, T, p.nctas);
        const float* src = p.part_o + prow(ok ? s0 + q : 0) * D + lane * PER;
        if constexpr (PER == 4) {
          const float4 x = ok ? *reinterpret_cast<const float4*>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[q][0] = x.x; v[q][1] = x.y; v[q][2] = x.z; v[q][3] = x.w;
        } else {
          const float2 x = ok ? *reinterpret_cast<const float2*>(src) : make_float2(0.f, 0.f);
          v[q][0] = x.x; v[q][1] = x.y;
        }
      }
    };
    // ---- one round of loads: the verify rows' keys/values (the CTA, into shared
    // memory), this warp's partial max/sum, first two batches of partial rows, query
    constexpr int CH = D / 8;  // 16-byte chunks of a row
    for (int e = tid; e < 2 * (tmax + 1) * CH; e += kCombineWarps * 32) {
      const int which = e / ((tmax + 1) * CH), rem = e - which * (tmax + 1) * CH;
      const int u = rem / CH, c = rem - u * CH;
      const __nv_bfloat16* row = which ? verify_row<D>(p, p.v_new, p.V, b, n, u, g) : verify_row<D>(p, p.k_new, p.K, b, n, u, g);
      reinterpret_cast<uint4*>(&kvs[which][u][0])[c] =
          row ? reinterpret_cast<const uint4*>(row)[c] : make_uint4(0u, 0u, 0u, 0u);
    }
    float pm = NEG, pl = 0.f;
    float va[NB][PER], vb[NB][PER];
    float qv[PER];
    if (active) {
      load_ml(lane, pm, pl);
      load_rows(0, va);
      load_rows(NB, vb);
      const __nv_bfloat16* qrow = p.q + ((static_cast<size_t>(b) * p.R + t) * p.Hq + g * G + jh) * D + lane * PER;
#pragma unroll
      for (int e = 0; e < PER; ++e) qv[e] = bf2f(qrow[e]);
    }
    __syncthreads();
    if (!active) return;
    // ---- causal logits of the verify rows' own keys u <= t
    float* lg = lgs[warp];
    float mc = NEG;
    for (int u = 0; u <= t; ++u) {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc += qv[e] * bf2f(kvs[0][u][lane * PER + e]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      acc *= p.scale_log2;
      mc = fmaxf(mc, acc);
      if (lane == 0) lg[u] = acc;
    }
    __syncwarp();
    // ---- global max over the partials and the causal keys
    float M = pm;
    for (int s0 = 32; s0 < nseg; s0 += 32) {  // more than 32 partials: further rounds
      float ms, ls;
      load_ml(s0 + lane, ms, ls);
      M = fmaxf(M, ms);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    M = fmaxf(M, mc);
    // ---- merge, in the order of the partials, then the causal keys; two batches of
    // partial rows in flight (the next is loaded while this one is added)
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float l = 0.f, w = 0.f;
    for (int s0 = 0; s0 < nseg; s0 += NB) {
      if ((s0 & 31) == 0) {  // weights of the next 32 partials
        float ms = pm, ls = pl;
        if (s0 > 0) load_ml(s0 + lane, ms, ls);
        w = (ms != NEG) ? ex2(ms - M) : 0.f;
        float wl = w * ls;  // fixed-order butterfly
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) wl += __shfl_xor_sync(0xffffffffu, wl, off);
        l += wl;
      }
#pragma unroll
      for (int q = 0; q < NB; ++q) {
        const float wq = __shfl_sync(0xffffffffu, w, (s0 + q) & 31);
        if (s0 + q < nseg) {
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[e] += wq * va[q][e];
        }
      }
#pragma unroll
      for (int q = 0; q < NB; ++q)
#pragma unroll
        for (int e = 0; e < PER; ++e) va[q][e] = vb[q][e];
      if (s0 + 2 * NB < nseg) load_rows(s0 + 2 * NB, vb);
    }
    for (int u = 0; u <= t; ++u) {
      const float wu = ex2(lg[u] - M);
      l += wu;
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] += wu * bf2f(kvs[1][u][lane * PER + e]);
    }
    const float inv = 1.f / l;
    __nv_bfloat16* o = p.out + ((static_cast<size_t>(b) * p.R + t) * p.Hq + g * G + jh) * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) o[e] = __float2bfloat16_rn(acc[e] * inv);
    if (p.k_new && jh == 0) {  // append verify row t (the chain enters the cache)
      const int64_t slot = kv_slot(p.seq_offset, p.ptab, p.psize, p.pstride, p.capacity, b, n + t);
      if (slot >= 0) {
        const size_t dst = (slot * p.Hkv + g) * D + lane * PER;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
          p.K[dst + e] = kvs[0][t][lane * PER + e];
          p.V[dst + e] = kvs[1][t][lane * PER + e];
        }
      }
    }
    return;
  }
  // score role: fixed-order sum of the per-(KV head, part) partial scores
  constexpr int CH = kCombineWarps * 32 * 4;
  const int nchunks = (p.max_len + CH - 1) / CH;
  const int sb = blockIdx.x - nA;
  const int b = sb / nchunks, ch = sb - b * nchunks;
  if (b >= p.B) return;
  const int n = nlen[b];
  const int pos = ch * CH + tid * 4;
  if (pos >= n) return;
  const int parts = p.Hkv * 2;
  for (int ms = 0; ms < 2; ++ms) {
    float* dst = ms ? p.scores1 : p.scores0;
    if ((ms ? p.mask1 : p.mask0) == 0u || dst == nullptr) continue;
    const float* src = p.part_s + (static_cast<size_t>(ms) * p.B + b) * parts * p.s_stride + pos;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q0 = 0; q0 < parts; q0 += 16) {  // one round of loads up to H_kv = 8
      float4 v[16];  // rows are s_stride (a multiple of 64) apart: in bounds
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (q0 + q < parts) v[q] = *reinterpret_cast<const float4*>(src + static_cast<size_t>(q0 + q) * p.s_stride);
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (q0 + q < parts) {
          a.x += v[q].x;
          a.y += v[q].y;
          a.z += v[q].z;
          a.w += v[q].w;
        }
    }
    float* d = dst + static_cast<size_t>(b) * p.score_stride + pos;
    d[0] = a.x;
    if (pos + 1 < n) d[1] = a.y;
    if (pos + 2 < n) d[2] = a.z;
    if (pos + 3 < n) d[3] = a.w;
  }
}

// The same merge for a grid with few (sequence, KV head) pairs: spread over many
// small CTAs, so that each SM moves little.  128-thread CTAs; a row's D outputs are
// split over D/32 warps, one element per lane (RPC rows per CTA).  Everything that
// needs only the call's inputs happens before the dependency wait: the sequence's tile
// counts (from the lengths), the query and verify-row K/V staged in shared memory,
// and the row's causal part (max, sum and output over its own keys u <= t).  After
// the wait, one round of loads (up to kNarrowRound partials a lane) and a merge in a
// fixed order: the causal part, then the partials by CTA.  Role B: CTAs of 256 prefix
// positions, 2 per thread.
constexpr int kNarrowThreads = 128;
constexpr int kNarrowRound = 32;  // partial rows a lane loads in one round
constexpr int kMaxR = 16;         // verify rows (gamma + 1 <= 16)

// Tiles of one KV head before sequence b and of b, the total, and b's checked length
// (-1 if its length or slots are out of range: the verify kernel reports that).  One
// warp; the same checks and counts as the verify kernel's own.
__device__ void combine_seq_meta(const VerifyParams& p, int b, int* out4) {
  const int lane = threadIdx.x & 31;
  int before = 0, total = 0, mine = 0, nb = -1;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int bb = b0 + lane;
    int tiles = 0, n = -1;
    if (bb < p.B) {
      n = p.prefix_len[bb];
      if (!seq_len_ok(p, bb, n)) n = -1;
      tiles = n > 0 ? (n + TK - 1) / TK : 0;
    }
    int tb = bb < b ? tiles : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tb += __shfl_xor_sync(0xffffffffu, tb, o);
      tiles += __shfl_xor_sync(0xffffffffu, tiles, o);
    }
    before += tb;
    total += tiles;
    const bool here = b >= b0 && b < b0 + 32;
    const int nsh = __shfl_sync(0xffffffffu, n, here ? b - b0 : 0);
    if (here) {
      nb = nsh;
      mine = nsh > 0 ? (nsh + TK - 1) / TK : 0;
    }
  }
  if (lane == 0) {
    out4[0] = before;
    out4[1] = mine;
    out4[2] = total;
    out4[3] = nb;
  }
}

template <int D>
__global__ void __launch_bounds__(kNarrowThreads, 4) verify_combine_narrow_kernel(const VerifyParams p) {
  constexpr int WPR = D / 32;                       // warps per row
  constexpr int RPC = (kNarrowThreads / 32) / WPR;  // rows per CTA
  constexpr int PD = D / 32;                        // elements of a dot product per lane
  __shared__ __align__(16) __nv_bfloat16 sq[RPC][D];        // this CTA's query rows
  __shared__ __align__(16) __nv_bfloat16 skv[2][kMaxR][D];  // the verify rows' keys and values
  __shared__ int smeta[4];
  pdl_launch_dependents();  // the selection kernel may start its prologue
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float NEG = neg_inf();
  const int rblocks = (p.M + RPC - 1) / RPC;  // CTAs per (sequence, KV head)
  const int nA = p.B * p.Hkv * rblocks;
  if (static_cast<int>(blockIdx.x) < nA) {
    const int bg = blockIdx.x / rblocks;
    const int r0 = (blockIdx.x - bg * rblocks) * RPC;
    const int g = bg % p.Hkv, b = bg / p.Hkv;
    const int G = p.G;
    const int rw = warp / WPR;                 // this warp's row within the CTA
    const int r = r0 + rw;
    const int d = (warp % WPR) * 32 + lane;    // this lane's output element
    const bool active = r < p.M;
    const int t = active ? r / G : 0, jh = r - t * G;
    const int tmax = min(p.M - 1, r0 + RPC - 1) / G;  // last verify row of this CTA
    // ---- before the dependency wait: the call's inputs only
    if (warp == 0) combine_seq_meta(p, b, smeta);
    __syncthreads();
    const int n = smeta[3];
    if (n < 0) return;  // the whole CTA
    constexpr int CH = D / 8;  // 16-byte chunks of a row
    for (int e = tid; e < 2 * (tmax + 1) * CH; e += kNarrowThreads) {
      const int which = e / ((tmax + 1) * CH), rem = e - which * (tmax + 1) * CH;
      const int u = rem / CH, c = rem - u * CH;
      const __nv_bfloat16* row = which ? verify_row<D>(p, p.v_new, p.V, b, n, u, g) : verify_row<D>(p, p.k_new, p.K, b, n, u, g);
      reinterpret_cast<uint4*>(&skv[which][u][0])[c] =
          row ? reinterpret_cast<const uint4*>(row)[c] : make_uint4(0u, 0u, 0u, 0u);
    }
    for (int e = tid; e < RPC * CH; e += kNarrowThreads) {
      const int rr = e / CH, c = e - rr * CH;
      const int r2 = r0 + rr;
      if (r2 < p.M) {
        const int t2 = r2 / G, j2 = r2 - t2 * G;
        reinterpret_cast<uint4*>(&sq[rr][0])[c] = reinterpret_cast<const uint4*>(
            p.q + ((static_cast<size_t>(b) * p.R + t2) * p.Hq + g * G + j2) * D)[c];
      }
    }
    __syncthreads();
    if (!active) return;
    // causal part of this row: its own keys u = 0..t (at least itself)
    float mc = NEG, lc = 0.f, oc = 0.f;
    {
      float qv[PD];
#pragma unroll
      for (int e = 0; e < PD; ++e) qv[e] = bf2f(sq[rw][lane * PD + e]);
      float lg[kMaxR];
#pragma unroll
      for (int u = 0; u < kMaxR; ++u) {
        lg[u] = NEG;
        if (u <= t) {
          float acc = 0.f;
#pragma unroll
          for (int e = 0; e < PD; ++e) acc += qv[e] * bf2f(skv[0][u][lane * PD + e]);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
          lg[u] = acc * p.scale_log2;
          mc = fmaxf(mc, lg[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < kMaxR; ++u) {
        if (u <= t) {
          const float w = ex2(lg[u] - mc);
          lc += w;
          oc += w * bf2f(skv[1][u][d]);
        }
      }
    }
    // ---- after the wait: the verify kernel's partials of this (sequence, KV head),
    // written by CTAs cf..cl of its split
    pdl_wait();
    const int tiles = smeta[1];
    const int64_t T = static_cast<int64_t>(p.Hkv) * smeta[2];
    int64_t cf = 0, cl = -1;
    if (tiles > 0) {
      const int64_t S = static_cast<int64_t>(p.Hkv) * smeta[0] + static_cast<int64_t>(g) * tiles;
      cf = owner_cta(S, T, p.nctas);
      cl = owner_cta(S + tiles - 1, T, p.nctas);
    }
    const int nseg = static_cast<int>(cl - cf + 1);
    const size_t pair = static_cast<size_t>(b) * p.Hkv + g;
    float Mr = mc, lr = lc, acc = oc;  // running merge, starting with the causal part
    for (int s0 = 0; s0 < nseg; s0 += kNarrowRound) {
      const int ns = min(kNarrowRound, nseg - s0);
      float mv = NEG, lv = 0.f;
      if (lane < ns && split_nonempty(cf + s0 + lane, T, p.nctas)) {  // CTAs with no items wrote none
        const float2 v = *reinterpret_cast<const float2*>(
            p.part_ml + ((static_cast<size_t>(cf + s0 + lane) + pair) * p.Mpad + r) * 2);
        mv = v.x;
        lv = v.y;
      }
      float ov[kNarrowRound];  // (0 for a CTA with no items: its row holds whatever was there)
#pragma unroll
      for (int q = 0; q < kNarrowRound; ++q)
        ov[q] = q < ns && split_nonempty(cf + s0 + q, T, p.nctas)
                    ? p.part_o[((static_cast<size_t>(cf + s0 + q) + pair) * p.Mpad + r) * D + d]
                    : 0.f;
      float mx = mv;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float Mn = fmaxf(Mr, mx);
      const float sc = ex2(Mr - Mn);  // Mr is finite: the causal part has at least one key
      acc *= sc;
      lr *= sc;
      Mr = Mn;
      const float w = mv != NEG ? ex2(mv - Mr) : 0.f;
      float wl = w * lv;  // fixed-order butterfly
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) wl += __shfl_xor_sync(0xffffffffu, wl, off);
      lr += wl;
#pragma unroll
      for (int q = 0; q < kNarrowRound; ++q) {
        const float wq = __shfl_sync(0xffffffffu, w, q);
        if (q < ns) acc += wq * ov[q];
      }
    }
    p.out[((static_cast<size_t>(b) * p.R + t) * p.Hq + g * G + jh) * D + d] = __float2bfloat16_rn(acc / lr);
    if (p.k_new && jh == 0) {  // append verify row t (the chain enters the cache)
      const int64_t slot = kv_slot(p.seq_offset, p.ptab, p.psize, p.pstride, p.capacity, b, n + t);
      if (slot >= 0) {
        const size_t dst = (slot * p.Hkv + g) * D + d;
        p.K[dst] = skv[0][t][d];
        p.V[dst] = skv[1][t][d];
      }
    }
    return;
  }
  // score role: fixed-order sum of the per-(KV head, part) partial scores, 2 positions a
  // thread, each mask's parts loaded in one round (up to H_kv = 8)
  constexpr int CHS = kNarrowThreads * 2;
  const int nchunks = (p.max_len + CHS - 1) / CHS;
  const int sb = blockIdx.x - nA;
  const int b = sb / nchunks, ch = sb - b * nchunks;
  if (b >= p.B) return;
  const int n = p.prefix_len[b];
  if (!seq_len_ok(p, b, n)) return;
  const int pos = ch * CHS + tid * 2;
  if (pos >= n) return;
  pdl_wait();
  const int parts = p.Hkv * 2;
  for (int ms = 0; ms < 2; ++ms) {
    float* dst = ms ? p.scores1 : p.scores0;
    if ((ms ? p.mask1 : p.mask0) == 0u || dst == nullptr) continue;
    const float* src = p.part_s + (static_cast<size_t>(ms) * p.B + b) * parts * p.s_stride + pos;
    float2 a = make_float2(0.f, 0.f);
    for (int q0 = 0; q0 < parts; q0 += 16) {
      float2 v[16];  // rows are s_stride (a multiple of 64) apart: in bounds
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (q0 + q < parts) v[q] = *reinterpret_cast<const float2*>(src + static_cast<size_t>(q0 + q) * p.s_stride);
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (q0 + q < parts) {
          a.x += v[q].x;
          a.y += v[q].y;
        }
    }
    float* dd = dst + static_cast<size_t>(b) * p.score_stride + pos;
    dd[0] = a.x;
    if (pos + 1 < n) dd[1] = a.y;
  }
}

template <int D, int MR, bool PAGED>
cudaError_t launch_verify_t(const VerifyParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            cudaStream_t stream) {
  using C = TCfg<D, MR>;
  const size_t smem = C::smem(p.B);
  cudaError_t e = ensure_smem<verify_kernel<D, MR, PAGED>>(smem);
  if (e != cudaSuccess) return e;
  {
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.nctas);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, verify_kernel<D, MR, PAGED>, p, tmK, tmV);
  }
  if (e != cudaSuccess) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, verify_kernel<D, MR, PAGED>) == cudaSuccess) {
      fprintf(stderr,
              "verify_kernel<%d,%d>: %s (regs=%d maxThreads=%d threads=%d staticSmem=%zu maxDynSmem=%d "
              "requestedSmem=%zu localBytes=%zu)\n",
              D, MR, cudaGetErrorString(e), fa.numRegs, fa.maxThreadsPerBlock, C::THREADS, fa.sharedSizeBytes,
              fa.maxDynamicSharedSizeBytes, smem, fa.localSizeBytes);
    }
    return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  const bool scores = (p.mask0 | p.mask1) != 0u;
  // few (sequence, KV head) pairs: the narrow combine spreads the merge over many SMs
  constexpr int RPCN = (kNarrowThreads / 32) / (D / 32);
  const int nAn = p.B * p.Hkv * ((p.M + RPCN - 1) / RPCN);
  if (nAn <= 8 * p.nctas) {  // (measured: 8 x the grid is no slower on any workload)
    constexpr int CHS = kNarrowThreads * 2;
    const int nSn = scores ? p.B * ((p.max_len + CHS - 1) / CHS) : 0;
    cfg.gridDim = dim3(nAn + nSn);
    cfg.blockDim = dim3(kNarrowThreads);
    return cudaLaunchKernelEx(&cfg, verify_combine_narrow_kernel<D>, p);
  }
  const int nA = p.B * p.Hkv * ((p.M + kCombineWarps - 1) / kCombineWarps);
  constexpr int CH = kCombineWarps * 32 * 4;
  const int nS = scores ? p.B * ((p.max_len + CH - 1) / CH) : 0;
  cfg.gridDim = dim3(nA + nS);
  cfg.blockDim = dim3(kCombineWarps * 32);
  return cudaLaunchKernelEx(&cfg, verify_combine_kernel<D>, p);
}

}  // namespace

int verify_sc_row0(int M, int nsc) {
  if (nsc == 0) return M;
  const int MR = M + nsc <= 64 ? 64 : 128;  // the MMA shape the packed rows need
  const int QR = MR / 4;                    // rows a lane quadrant holds
  const int r0 = (M + QR - 1) / QR * QR;
  return r0 + nsc <= MR ? r0 : M;
}

size_t verify_smem_bytes(int D, int B) {
  auto mx = [](size_t a, size_t b) { return a > b ? a : b; };
  if (D == 64) return mx(TCfg<64, 64>::smem(B), TCfg<64, 128>::smem(B));
  if (D == 128) return mx(TCfg<128, 64>::smem(B), TCfg<128, 128>::smem(B));
  return 0;
}

cudaError_t launch_verify(const VerifyParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                          cudaStream_t stream) {
  // A-operand rows: the query rows, then a high and a low row per score mask
  const int nsc = 2 * ((p.mask0 ? 1 : 0) + (p.mask1 ? 1 : 0));
  const int arows = nsc ? p.sc_row0 + nsc : p.M;
  const bool paged = p.ptab != nullptr;
  if (arows <= 64) {
    if (p.D == 64) return paged ? launch_verify_t<64, 64, true>(p, tmK, tmV, stream)
                                : launch_verify_t<64, 64, false>(p, tmK, tmV, stream);
    if (p.D == 128) return paged ? launch_verify_t<128, 64, true>(p, tmK, tmV, stream)
                                 : launch_verify_t<128, 64, false>(p, tmK, tmV, stream);
  } else {
    if (p.D == 64) return paged ? launch_verify_t<64, 128, true>(p, tmK, tmV, stream)
                                : launch_verify_t<64, 128, false>(p, tmK, tmV, stream);
    if (p.D == 128) return paged ? launch_verify_t<128, 128, true>(p, tmK, tmV, stream)
                                 : launch_verify_t<128, 128, false>(p, tmK, tmV, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace vg
