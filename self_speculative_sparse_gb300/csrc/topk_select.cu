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
// k-th largest key: every pass builds a CTA histogram (replicated 8x across banks
// to tame same-bin conflicts), the cluster sums the histograms through
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
constexpr int kRep = 8;  // histogram replicas (by lane % 8)

// fp32 -> key with the same order; -0.0 is mapped to the key of +0.0.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread; returns the total in *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += t;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? warp_sums[lane] : 0;
    const int wv = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    if (lane < kWarps) warp_sums[lane] = w - wv;
    if (lane == 31) *total = w;
  }
  __syncthreads();
  const int r = warp_sums[warp] + x - v;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkParams p) {
  extern __shared__ uint32_t tk_smem[];
  uint32_t* keys = tk_smem;                          // [per_cta]
  uint32_t* hist = keys + p.per_cta;                 // [2][256 * kRep]
  uint32_t* hsum = hist + 2 * 256 * kRep;            // [2][256]
  int* wsum = reinterpret_cast<int*>(hsum + 2 * 256);  // [32]
  int* misc = wsum + 32;                             // [8]
  int* cnts = misc + 8;                              // [2]: this CTA's (#greater, #equal)
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
  for (int i = tid; i < mine; i += kThreads) keys[i] = order_key(src[i]);

  // ---------------------------------------------------------------- radix select
  uint32_t prefix = 0u, pmask = 0u;
  int remaining = cnt;  // how many keys >= the threshold are still to be taken inside the prefix class
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const int hb = pass & 1;
    uint32_t* h = hist + hb * 256 * kRep;
    for (int i = tid; i < 256 * kRep; i += kThreads) h[i] = 0u;
    __syncthreads();
    for (int i = tid; i < mine; i += kThreads) {
      const uint32_t key = keys[i];
      if ((key & pmask) == prefix) atomicAdd(&h[((key >> shift) & 255u) * kRep + (lane & (kRep - 1))], 1u);
    }
    __syncthreads();
    if (tid < 256) {
      uint32_t s = 0;
#pragma unroll
      for (int c = 0; c < kRep; ++c) s += h[tid * kRep + c];
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
  // thread t owns the contiguous run [t*E, (t+1)*E) of this CTA's slice
  const int E = (mine + kThreads - 1) / kThreads;
  const int i0 = min(mine, tid * E), i1 = min(mine, i0 + E);
  int ngt = 0, neq = 0;
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = keys[i];
    ngt += key > thr;
    neq += key == thr;
  }
  int cta_gt = 0, cta_eq = 0;
  const int gt_before = block_exclusive_scan(ngt, wsum, &misc[2]);
  cta_gt = misc[2];
  __syncthreads();
  const int eq_before = block_exclusive_scan(neq, wsum, &misc[3]);
  cta_eq = misc[3];
  if (tid == 0) {
    cnts[0] = cta_gt;
    cnts[1] = cta_eq;
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
  (void)gt_before;
  // selected count before my run: greater keys before + equal keys taken before
  const int sel_before = gt_before + min(eq_before, take_mine);
  int pos = off + sel_before;
  int eq_rank = eq_before;
  for (int i = i0; i < i1; ++i) {
    const uint32_t key = keys[i];
    bool sel = key > thr;
    if (key == thr) {
      sel = eq_rank < take_mine;
      ++eq_rank;
    }
    if (sel) out[pos++] = start + i;
  }
}

}  // namespace

size_t topk_smem_bytes(int per_cta) {
  return static_cast<size_t>(per_cta) * 4 + (2 * 256 * kRep + 2 * 256) * 4 + (32 + 8 + 2 + 256) * 4;
}

cudaError_t launch_topk(const TopkParams& p, int cluster, cudaStream_t stream, bool pdl) {
  const size_t smem = topk_smem_bytes(p.per_cta);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
