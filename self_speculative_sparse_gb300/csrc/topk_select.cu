// Per-sequence top-k selection of prefix entries by aggregated logit.
//
// Vegas §2 step 2 / §2.A: the selected set maximises the summed logits over the
// prefix; since the objective is a sum of per-entry scores, that set is the k
// largest scores.  Equal scores prefer the lower position (so the set is unique)
// and the output lists the positions in ascending order, ready to serve as the
// page indices of the draft's page-size-one attention (Vegas §3).
//
// GB300 design.  One thread-block cluster of up to 16 CTAs per sequence; each CTA
// keeps its contiguous slice of the scores in shared memory as order-preserving
// 32-bit keys.  An exact MSB-first radix select (4 passes of 8 bits) finds the
// k-th largest key: every pass builds per-warp histograms, eight steps in flight and
// no contention between warps (the first pass, whose top-byte digits pile onto a few
// sign/exponent values, aggregates equal digits of a warp into one increment; later
// passes digit inside one top-byte class and increment directly); each CTA pushes its histogram into every CTA of the
// cluster through distributed shared memory (stores before the cluster barrier, so
// that after it every CTA sums the cluster's counts from its own shared memory with
// no remote round trip), and a scan over the digits by the 256 digit threads lets
// every CTA pick the same digit.  After two passes the keys still matching the 16-bit
// prefix are usually few; each CTA then pushes its own into every CTA, and after one
// cluster barrier every CTA finds the threshold among them itself instead of running
// the last two passes (too many of them, as with many equal scores, and the passes run).
// A final cluster-wide exclusive scan in position order (the CTAs'
// counts pushed the same way) writes the selected positions, taking the needed
// number of threshold-equal keys from the lowest positions.
// Everything is integer work: the result is bit-exact and deterministic.
#include <atomic>

#include <cooperative_groups.h>

#include "vg_common.cuh"
#include "vg_internal.h"

namespace cg = cooperative_groups;

namespace vg {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 256;  // radix digit: 8 bits
constexpr int kListPerWarp = 256;  // candidate-list capacity of a warp for the last two passes
constexpr int kMaxCluster = 16;    // CTAs per sequence (more than 8 needs the non-portable cluster size)
// After two passes the keys still matching the 16-bit prefix are usually few: when no
// CTA holds more than kCandPerCta of them and the cluster holds at most kThreads, every
// CTA receives them all and finds the threshold among them itself, in place of the last
// two passes (one cluster barrier instead of two, and no histograms).  Slices long
// enough for the warps' candidate lists keep the two list passes, which cost less there.
constexpr int kCandPerCta = 64;

// fp32 -> key with the same order; -0.0 is mapped to the key of +0.0.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkParams p) {
  extern __shared__ uint32_t tk_smem[];
  uint32_t* keys = tk_smem;                          // [per_cta]
  uint32_t* hist = keys + p.per_cta;                 // [kWarps][kBins] per-warp digit histograms
  // [2][kMaxCluster][kBins]: every CTA of the cluster pushes its histogram of a pass into
  // slot (pass parity, its rank) of every CTA, so the sums are read locally
  uint32_t* hall = hist + kWarps * kBins;
  int* call = reinterpret_cast<int*>(hall + 2 * kMaxCluster * kBins);  // [kMaxCluster][2] (#greater, #equal), pushed
  int* wsum = call + 2 * kMaxCluster;                // [32]
  int* misc = wsum + 32;                             // [48]
  // per-warp lists of the keys still in the running after two passes (passes 3 and 4
  // scan only these; a warp with more candidates than its list holds scans its keys)
  uint32_t* clist = reinterpret_cast<uint32_t*>(misc + 48);  // [kWarps][kListPerWarp]
  uint32_t* cown = clist + kWarps * kListPerWarp;     // [kCandPerCta] this CTA's candidates
  int* ccnt = reinterpret_cast<int*>(cown + kCandPerCta);  // [kMaxCluster] candidates of each CTA, pushed
  uint32_t* cpush = reinterpret_cast<uint32_t*>(ccnt + kMaxCluster);  // [kMaxCluster][kCandPerCta], pushed

  cg::cluster_group cluster = cg::this_cluster();
  const int r = static_cast<int>(cluster.block_rank());
  const int C = static_cast<int>(cluster.num_blocks());
  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31;

  pdl_launch_dependents();  // the draft step may start its prologue
  pdl_wait();
  int n = p.len[b];
  if (n < 0 || n > p.max_len || n > C * p.per_cta) {
    report(p.status, VG_ERR_DEVICE_BOUNDS);
    n = 0;
  }
  const int k = p.k;
  const int cnt = min(k, n);
  int32_t* out = p.idx + static_cast<size_t>(b) * k;
  // trailing -1 slots and the count (spread over the cluster)
  for (int i = cnt + r * kThreads + tid; i < k; i += C * kThreads) out[i] = -1;
  if (r == 0 && tid == 0) p.count[b] = cnt;
  if (cnt == 0) return;

  const int L = (n + C - 1) / C;
  const int start = min(n, r * L);
  const int mine = min(n, start + L) - start;
  const float* src = p.scores + static_cast<size_t>(b) * p.score_stride + start;

  if (cnt == n) {  // every entry is selected
    for (int i = tid; i < mine; i += kThreads) out[start + i] = start + i;
    return;
  }
  // every CTA of the cluster must be running before the first push into its shared
  // memory: arrive now, wait once the keys are loaded (the returns above are taken by
  // the whole cluster, which shares the sequence)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  {
    // batched loads: up to 8 independent loads in flight per thread per round
    // (start is a multiple of 4 unless this is the ragged last CTA: then scalar)
    const bool vec = (start & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
    if (vec) {
      const int n4 = mine >> 2;
      const float4* s4 = reinterpret_cast<const float4*>(src);
      for (int base = 0; base < n4; base += 8 * kThreads) {
        float4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i4 = base + q * kThreads + tid;
          v[q] = i4 < n4 ? s4[i4] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i4 = base + q * kThreads + tid;
          if (i4 < n4) {
            keys[4 * i4 + 0] = order_key(v[q].x);
            keys[4 * i4 + 1] = order_key(v[q].y);
            keys[4 * i4 + 2] = order_key(v[q].z);
            keys[4 * i4 + 3] = order_key(v[q].w);
          }
        }
      }
      for (int i = (n4 << 2) + tid; i < mine; i += kThreads) keys[i] = order_key(src[i]);
    } else {
      for (int base = 0; base < mine; base += 8 * kThreads) {
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i = base + q * kThreads + tid;
          v[q] = i < mine ? src[i] : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i = base + q * kThreads + tid;
          if (i < mine) keys[i] = order_key(v[q]);
        }
      }
    }
  }

  __syncthreads();  // the passes read keys that other threads stored
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

  // ---------------------------------------------------------------- radix select
  uint32_t prefix = 0u, pmask = 0u;
  int remaining = cnt;  // how many keys >= the threshold are still to be taken inside the prefix class
  const int rounds = (mine + kThreads - 1) / kThreads;
  const int warp_id = tid >> 5;
  uint32_t* wlist = clist + warp_id * kListPerWarp;
  int wcnt = 0;  // candidates of this warp after two passes (warp-uniform)
  const bool lists = rounds > 8;  // on short slices the list costs more than the scans it saves
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    uint32_t* hw = hist + (tid >> 5) * kBins;
    for (int i = lane; i < kBins; i += 32) hw[i] = 0u;  // this warp's own histogram
    __syncwarp();
    // counting into the warp's own histogram, eight independent steps at a time.
    // Passes 1-2 scan every key of the slice; passes 3-4 only the warp's list of
    // remaining candidates.
    const bool from_list = lists && pass >= 2 && wcnt <= kListPerWarp;
    const int steps = from_list ? (wcnt + 31) / 32 : rounds;
    for (int rb = 0; rb < steps; rb += 8) {
      uint32_t dg[8];
      bool cand[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        bool in;
        uint32_t key;
        if (from_list) {
          const int e = (rb + q) * 32 + lane;
          in = e < wcnt;
          key = in ? wlist[e] : 0u;
        } else {
          const int i = (rb + q) * kThreads + tid;
          in = i < mine;
          key = in ? keys[i] : 0u;
        }
        cand[q] = in && (key & pmask) == prefix;
        dg[q] = cand[q] ? ((key >> shift) & 255u) : 0xffffffffu;
      }
      if (pass == 0) {  // top byte (sign, high exponent bits): few distinct digits, aggregate
        unsigned peers[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) peers[q] = __match_any_sync(0xffffffffu, dg[q]);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (cand[q] && lane == __ffs(peers[q]) - 1) atomicAdd(&hw[dg[q]], static_cast<uint32_t>(__popc(peers[q])));
      } else {  // inside one top-byte class the digits spread: plain increments
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (cand[q]) atomicAdd(&hw[dg[q]], 1u);
      }
    }
    __syncthreads();
    uint32_t* hb = hall + (pass & 1) * kMaxCluster * kBins;  // [source rank][digit]
    if (tid < kBins) {  // this CTA's count of digit tid, pushed to every CTA of the cluster
      uint32_t sum = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) sum += hist[w * kBins + tid];
      for (int rr = 0; rr < C; ++rr) *cluster.map_shared_rank(hb + r * kBins + tid, rr) = sum;
    }
    cluster.sync();  // the pushes have landed (a buffer is reused two passes on, after
                     // the next pass's sync, so no CTA still reads it)
    // cluster-wide counts, highest digit first: thread t (< 256) owns digit 255 - t.
    // The eight warps of digit threads scan their counts, meet once, and each adds the
    // totals of the warps before it; the thread whose digit holds the remaining-th
    // largest key of the prefix class publishes it (double-buffered by pass parity, so
    // a thread still reading one pass's result is never overwritten by the next).
    int* res = misc + 2 * (pass & 1);
    if (tid < kBins) {
      int c = 0;
#pragma unroll
      for (int rr = 0; rr < kMaxCluster; ++rr)
        if (rr < C) c += static_cast<int>(hb[rr * kBins + (kBins - 1 - tid)]);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (lane == 31) wsum[tid >> 5] = incl;
      asm volatile("bar.sync 1, %0;" ::"n"(kBins) : "memory");
      int before = 0;
      for (int w = 0; w < (tid >> 5); ++w) before += wsum[w];
      const int run = before + incl - c;
      if (run < remaining && remaining <= run + c) {
        res[0] = kBins - 1 - tid;
        res[1] = run;
      }
    }
    __syncthreads();
    const int digit = res[0];
    remaining -= res[1];
    prefix |= static_cast<uint32_t>(digit) << shift;
    pmask |= 255u << shift;
    if (lists && pass == 1) {  // the keys still matching the 16-bit prefix, in this warp's list
      const unsigned lt = (1u << lane) - 1u;
      for (int rr = 0; rr < rounds; ++rr) {
        const int i = rr * kThreads + tid;
        const uint32_t key = i < mine ? keys[i] : 0u;
        const bool c = i < mine && (key & pmask) == prefix;
        const unsigned m = __ballot_sync(0xffffffffu, c);
        if (c && wcnt + __popc(m & lt) < kListPerWarp) wlist[wcnt + __popc(m & lt)] = key;
        wcnt += __popc(m);
      }
      __syncwarp();
    }
    if (pass == 1 && !lists) {  // the keys matching the 16-bit prefix, to every CTA (see kCandPerCta)
      int* nloc = misc + 4;
      if (tid == 0) {
        *nloc = 0;
        misc[6] = -1;  // (set below by the thread holding the threshold)
      }
      __syncthreads();
      for (int i = tid; i < mine; i += kThreads) {
        const uint32_t key = keys[i];
        if ((key & pmask) == prefix) {
          const int slot = atomicAdd(nloc, 1);  // (any order: only the multiset matters)
          if (slot < kCandPerCta) cown[slot] = key;
        }
      }
      __syncthreads();
      const int nc = *nloc;
      for (int e = tid; e < C * (kCandPerCta + 1); e += kThreads) {
        const int rr = e / (kCandPerCta + 1), q = e - rr * (kCandPerCta + 1);
        if (q == kCandPerCta)
          *cluster.map_shared_rank(ccnt + r, rr) = nc;
        else if (q < nc && nc <= kCandPerCta)
          *cluster.map_shared_rank(cpush + r * kCandPerCta + q, rr) = cown[q];
      }
      cluster.sync();  // (these buffers are written once a launch)
      int total = 0;
      bool fits = true;
      for (int rr = 0; rr < C; ++rr) {
        total += ccnt[rr];
        fits = fits && ccnt[rr] <= kCandPerCta;
      }
      if (fits && total <= kThreads) {
        // the remaining-th largest candidate: thread t takes candidate t and counts the
        // candidates above it and equal to it (the same decision in every CTA)
        if (tid < total) {
          int rr = 0, q = tid;
          while (q >= ccnt[rr]) q -= ccnt[rr++];
          const uint32_t x = cpush[rr * kCandPerCta + q];
          int above = 0, same = 0;
          for (int r2 = 0; r2 < C; ++r2)
            for (int q2 = 0; q2 < ccnt[r2]; ++q2) {
              const uint32_t y = cpush[r2 * kCandPerCta + q2];
              above += y > x;
              same += y == x;
            }
          if (above < remaining && remaining <= above + same) {  // (threads holding equal keys agree)
            misc[5] = static_cast<int>(x);
            misc[6] = remaining - above;
          }
        }
        __syncthreads();
        if (misc[6] > 0) {  // (always, for consistent counts; otherwise the last two passes run)
          prefix = static_cast<uint32_t>(misc[5]);
          remaining = misc[6];
          break;
        }
      }
    }
  }
  const uint32_t thr = prefix;  // k-th largest key; `remaining` keys equal to it are taken

  // ---------------------------------------------------------------- compaction
  // Warp w owns the contiguous run [w0, w1) of this CTA's slice; within a run, 32
  // consecutive keys are handled per step (conflict-free shared reads) and ballots
  // give each selected position its output slot in position order.
  const int warp = tid >> 5;
  const int WR = ((mine + kWarps - 1) / kWarps + 31) & ~31;
  const int w0 = min(mine, warp * WR), w1 = min(mine, w0 + WR);
  int ngt = 0, neq = 0;
  for (int i = w0 + lane; i < w1; i += 32) {
    const uint32_t key = keys[i];
    ngt += key > thr;
    neq += key == thr;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ngt += __shfl_xor_sync(0xffffffffu, ngt, o);
    neq += __shfl_xor_sync(0xffffffffu, neq, o);
  }
  if (lane == 0) {
    wsum[warp] = ngt;
    wsum[kWarps + warp] = neq;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scans over the warps' runs, and this CTA's totals
    const int g = lane < kWarps ? wsum[lane] : 0;
    const int e = lane < kWarps ? wsum[kWarps + lane] : 0;
    int gi = g, ei = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int tg = __shfl_up_sync(0xffffffffu, gi, o);
      const int te = __shfl_up_sync(0xffffffffu, ei, o);
      if (lane >= o) {
        gi += tg;
        ei += te;
      }
    }
    if (lane < kWarps) {
      misc[8 + lane] = gi - g;   // greater keys before warp `lane`'s run
      misc[24 + lane] = ei - e;  // equal keys before it
    }
    if (lane == kWarps - 1) {  // this CTA's totals, pushed to every CTA of the cluster
      for (int rr = 0; rr < C; ++rr) {
        int* dst = cluster.map_shared_rank(call + 2 * r, rr);
        dst[0] = gi;
        dst[1] = ei;
      }
    }
  }
  cluster.sync();  // (the last access to another CTA's shared memory precedes it)
  int off = 0, eq_prev = 0, take_mine = 0;
  for (int rr = 0; rr < C; ++rr) {
    const int g_r = call[2 * rr], e_r = call[2 * rr + 1];
    const int take_r = max(0, min(e_r, remaining - eq_prev));
    if (rr < r) off += g_r + take_r;
    if (rr == r) take_mine = take_r;
    eq_prev += e_r;
  }
  const int gt_before = misc[8 + warp], eq_before = misc[24 + warp];
  int sel_base = off + gt_before + min(eq_before, take_mine);
  int eq_rank = eq_before;
  const unsigned lt = (1u << lane) - 1u;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const bool valid = i < w1;
    const uint32_t key = valid ? keys[i] : 0u;
    const bool gt = valid && key > thr;
    const bool eq = valid && key == thr;
    const unsigned eqm = __ballot_sync(0xffffffffu, eq);
    const bool sel = gt || (eq && eq_rank + __popc(eqm & lt) < take_mine);
    const unsigned selm = __ballot_sync(0xffffffffu, sel);
    const int slot = sel_base + __popc(selm & lt);
    if (sel && slot < cnt) out[slot] = start + i;  // (slot < cnt always holds for consistent counts)
    sel_base += __popc(selm);
    eq_rank += __popc(eqm);
  }
}

// The query-agnostic comparison policy (Vegas §1, problem statement: simple
// query-agnostic selections such as sliding windows cost little to select but draft
// poorly): the last k prefix positions of each sequence, in the same output form as
// the score-based selection.  Grid (ceil(k / 256), B).
__global__ void __launch_bounds__(256) window_kernel(const int32_t* len, int B, int max_len, int k, int32_t* idx,
                                                     int32_t* count, int32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.y;
  int n = len[b];
  if (n < 0 || n > max_len) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(status, VG_ERR_DEVICE_BOUNDS);
    n = 0;
  }
  const int cnt = min(k, n);
  const int i = blockIdx.x * 256 + threadIdx.x;
  if (i < k) idx[static_cast<size_t>(b) * k + i] = i < cnt ? n - cnt + i : -1;
  if (i == 0) count[b] = cnt;
}

}  // namespace

cudaError_t launch_window(const int32_t* len, int B, int max_len, int k, int32_t* idx, int32_t* count,
                          int32_t* status, cudaStream_t stream) {
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((k + 255) / 256, B);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, window_kernel, len, B, max_len, k, idx, count, status);
}

size_t topk_smem_bytes(int per_cta) {
  return static_cast<size_t>(per_cta) * 4 + static_cast<size_t>(kWarps + 2 * kMaxCluster) * kBins * 4 +
         (2 * kMaxCluster + 32 + 48) * 4 + static_cast<size_t>(kWarps) * kListPerWarp * 4 +
         static_cast<size_t>(kCandPerCta + kMaxCluster + kMaxCluster * kCandPerCta) * 4;
}

cudaError_t launch_topk(const TopkParams& p, int cluster, cudaStream_t stream, bool pdl) {
  const size_t smem = topk_smem_bytes(p.per_cta);
  cudaError_t e = ensure_smem<topk_kernel>(smem);
  if (e != cudaSuccess) return e;
  if (cluster > 8) {
    static std::atomic<int> nonportable[64] = {};  // (set once per device; any thread)
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!nonportable[dev].load(std::memory_order_acquire)) {
      e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      nonportable[dev].store(1, std::memory_order_release);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, p.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel, p);
}

}  // namespace vg
