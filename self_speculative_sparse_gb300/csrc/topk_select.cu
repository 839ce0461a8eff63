// Per-sequence top-k selection of prefix entries by aggregated logit.
//
// Vegas §2 step 2 / §2.A: the selected set maximises the summed logits over the
// prefix; since the objective is a sum of per-entry scores, that set is the k
// largest scores.  Equal scores prefer the lower position (so the set is unique)
// and the output lists the positions in ascending order, ready to serve as the
// page indices of the draft's page-size-one attention (Vegas §3).
//
// GB300 design.  One thread-block cluster of up to 8 CTAs per sequence; each CTA
// keeps its contiguous slice of the scores in shared memory as order-preserving
// 32-bit keys.  An exact MSB-first radix select (4 passes of 8 bits) finds the
// k-th largest key: every pass builds per-warp histograms with warp-aggregated
// increments (no same-bin atomic conflicts), the cluster sums them through
// distributed shared memory, and every CTA picks the same digit.  A final
// cluster-wide exclusive scan in position order writes the selected positions,
// taking the needed number of threshold-equal keys from the lowest positions.
// Everything is integer work: the result is bit-exact and deterministic.
#include <cooperative_groups.h>

#include "vg_common.cuh"
#include "vg_internal.h"

namespace cg = cooperative_groups;

namespace vg {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

// fp32 -> key with the same order; -0.0 is mapped to the key of +0.0.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkParams p) {
  extern __shared__ uint32_t tk_smem[];
  uint32_t* keys = tk_smem;                          // [per_cta]
  uint32_t* hist = keys + p.per_cta;                 // [2][kWarps][256] per-warp histograms
  uint32_t* hsum = hist + 2 * kWarps * 256;          // [2][256]
  int* wsum = reinterpret_cast<int*>(hsum + 2 * 256);  // [32]
  int* misc = wsum + 32;                             // [48]
  int* cnts = misc + 48;                             // [2]: this CTA's (#greater, #equal)
  uint32_t* revc = reinterpret_cast<uint32_t*>(cnts + 2);  // [256] digit counts, highest first

  cg::cluster_group cluster = cg::this_cluster();
  const int r = static_cast<int>(cluster.block_rank());
  const int C = static_cast<int>(cluster.num_blocks());
  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31;

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

  // ---------------------------------------------------------------- radix select
  uint32_t prefix = 0u, pmask = 0u;
  int remaining = cnt;  // how many keys >= the threshold are still to be taken inside the prefix class
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const int hb = pass & 1;
    uint32_t* h = hist + hb * kWarps * 256;
    for (int i = tid; i < kWarps * 256; i += kThreads) h[i] = 0u;
    __syncthreads();
    // warp-aggregated counting: lanes with the same digit add once, into their
    // warp's own histogram, so concentrated digits cause no atomic conflicts
    uint32_t* hw = h + (tid >> 5) * 256;
    const int rounds = (mine + kThreads - 1) / kThreads;
    for (int rd = 0; rd < rounds; ++rd) {
      const int i = rd * kThreads + tid;
      const uint32_t key = i < mine ? keys[i] : 0u;
      const bool cand = i < mine && (key & pmask) == prefix;
      const uint32_t dg = cand ? ((key >> shift) & 255u) : 256u;
      const unsigned peers = __match_any_sync(0xffffffffu, dg);
      if (cand && lane == __ffs(peers) - 1) atomicAdd(&hw[dg], static_cast<uint32_t>(__popc(peers)));
    }
    __syncthreads();
    if (tid < 256) {
      uint32_t s = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) s += h[w * 256 + tid];
      hsum[hb * 256 + tid] = s;
    }
    cluster.sync();
    // cluster-wide count of each digit, stored highest digit first
    if (tid < 256) {
      uint32_t tot = 0;
      for (int rr = 0; rr < C; ++rr) tot += *cluster.map_shared_rank(&hsum[hb * 256 + tid], rr);
      revc[255 - tid] = tot;
    }
    __syncthreads();
    // warp 0 walks the digits from the top, 32 at a time, to the one holding the
    // remaining-th largest key of the current prefix class
    if (tid < 32) {
      int above = 0, found = -1, found_above = 0;
      for (int base = 0; base < 256 && found < 0; base += 32) {
        const int c = static_cast<int>(revc[base + lane]);  // digit 255 - (base + lane)
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const int excl = above + incl - c;  // keys of this class in higher digits
        const bool hit = excl < remaining && remaining <= excl + c;
        const unsigned ball = __ballot_sync(0xffffffffu, hit);
        if (ball) {
          const int src_lane = __ffs(ball) - 1;
          found = 255 - (base + src_lane);
          found_above = __shfl_sync(0xffffffffu, excl, src_lane);
        }
        above += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        misc[0] = found;
        misc[1] = found_above;
      }
    }
    __syncthreads();
    const int digit = misc[0];
    if (digit < 0) {  // cannot happen with consistent counts; stay safe
      report(p.status, VG_ERR_DEVICE_BOUNDS);
    }
    remaining -= misc[1];
    prefix |= static_cast<uint32_t>(digit & 255) << shift;
    pmask |= 255u << shift;
    __syncthreads();
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
    if (lane == kWarps - 1) {
      cnts[0] = gi;
      cnts[1] = ei;
    }
  }
  cluster.sync();
  int off = 0, eq_prev = 0, take_mine = 0;
  for (int rr = 0; rr < C; ++rr) {
    const int g_r = *cluster.map_shared_rank(&cnts[0], rr);
    const int e_r = *cluster.map_shared_rank(&cnts[1], rr);
    const int take_r = max(0, min(e_r, remaining - eq_prev));
    if (rr < r) off += g_r + take_r;
    if (rr == r) take_mine = take_r;
    eq_prev += e_r;
  }
  cluster.sync();  // no CTA leaves while its counters may still be read
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
    if (sel) out[sel_base + __popc(selm & lt)] = start + i;
    sel_base += __popc(selm);
    eq_rank += __popc(eqm);
  }
}

}  // namespace

size_t topk_smem_bytes(int per_cta) {
  return static_cast<size_t>(per_cta) * 4 + (2 * kWarps * 256 + 2 * 256) * 4 + (32 + 48 + 2 + 256) * 4;
}

cudaError_t launch_topk(const TopkParams& p, int cluster, cudaStream_t stream, bool pdl) {
  const size_t smem = topk_smem_bytes(p.per_cta);
  cudaError_t e = ensure_smem<topk_kernel>(smem);
  if (e != cudaSuccess) return e;
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
