// Acceptance of the draft chain after verification.
//
// Vegas §2 step 1 (verification phase): the target's full-attention pass accepts or
// rejects the draft tokens; Vegas §5 (lossless quality): what is committed follows the
// target model's distribution.  The page leaves the rule to standard speculative
// decoding; this is that rule on given logits:
//   greedy   draft t survives while it is the target's most likely token at row t
//            (ties: lowest token); the next token is the most likely token at row a;
//   sampling draft t survives iff u_t q_t(x_t) < p_t(x_t) (p, q the softmax of the target
//            and draft logits); at the first rejection a the next token is drawn from
//            max(0, p_a - q_a) (from p_a if that is zero everywhere), after gamma
//            acceptances from p_gamma; a draw takes the smallest v whose running sum of
//            weights exceeds u_res times their total.
//
// GB300 design.  HBM-bound reductions over the vocabulary, in PDL-chained kernels.
//   accept_stats_kernel: one CTA per (row, 8192-entry chunk) of the target rows (and the
//     draft rows when sampling): the chunk's max, sum of exp2 relative to it and argmax
//     (lowest index), in a fixed reduction order.
//   accept_decide_kernel: one CTA per sequence merges the chunks' statistics (in chunk
//     order) and takes the gamma decisions at once (one round of loads).  Greedy: it
//     writes the results.  Sampling: it leaves the accepted count and row a's statistics.
//   accept_tiles_kernel (sampling): one CTA per (tile of 4096 entries, sequence) sums
//     the tile's weights of row a, max(0, p - q) and p itself (the fallback when the
//     excess is zero everywhere), with a fixed-order block reduction.
//   accept_pick_kernel (sampling): one CTA per sequence adds the tile totals in order,
//     finds the tile where the running sum passes the target and scans that tile alone,
//     with the same reduction as the tile totals, so the two agree.
// Logits are read as log2-scaled values (l * log2 e), so every exponential is one ex2.
#include "vg_common.cuh"
#include "vg_internal.h"

namespace vg {
namespace {

constexpr int kChunk = 8192;      // vocabulary entries per statistics CTA
constexpr int kStatThreads = 256;
constexpr int kDecThreads = 1024;  // threads of a tile-sum or pick CTA (4 entries each)
constexpr int kDecideThreads = 512;  // threads of a decision CTA (a warp a row's merge: 2 gamma + 1 <= 31 rows)
constexpr int kTile = kDecThreads * 4;  // vocabulary entries per tile of the draw
constexpr float kLog2e = 1.4426950408889634f;

struct Stat {
  float m;   // max of l * log2 e
  float s;   // sum of exp2(l * log2 e - m)
  float av;  // the max's logit (for the argmax)
  int ai;    // argmax, lowest index
};

__device__ __forceinline__ void merge(Stat& a, const Stat& b) {
  const float NEG = neg_inf();
  const float m = fmaxf(a.m, b.m);
  const float sa = a.m == NEG ? 0.f : a.s * ex2(a.m - m);
  const float sb = b.m == NEG ? 0.f : b.s * ex2(b.m - m);
  a.s = sa + sb;
  a.m = m;
  if (b.av > a.av || (b.av == a.av && b.ai < a.ai)) {
    a.av = b.av;
    a.ai = b.ai;
  }
}

__device__ __forceinline__ Stat warp_merge(Stat v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Stat w;
    w.m = __shfl_xor_sync(0xffffffffu, v.m, o);
    w.s = __shfl_xor_sync(0xffffffffu, v.s, o);
    w.av = __shfl_xor_sync(0xffffffffu, v.av, o);
    w.ai = __shfl_xor_sync(0xffffffffu, v.ai, o);
    // fixed order: the lower lane's value first, so both lanes compute the same merge
    const bool low = (threadIdx.x & o) == 0;
    Stat a = low ? v : w, b = low ? w : v;
    merge(a, b);
    v = a;
  }
  return v;
}

// Logit row r of the call: target rows (b, t) for t <= gamma first, then draft rows.
__device__ __forceinline__ const float* row_ptr(const AcceptParams& p, int r) {
  const int np = p.B * (p.gamma + 1);
  if (r < np) return p.p_logits + static_cast<size_t>(r) * p.V;
  return p.q_logits + static_cast<size_t>(r - np) * p.V;
}

__global__ void __launch_bounds__(kStatThreads) accept_stats_kernel(const AcceptParams p) {
  __shared__ Stat red[kStatThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int c = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
  const float* row = row_ptr(p, r);
  const int v0 = c * kChunk, v1 = min(p.V, v0 + kChunk);
  const float NEG = neg_inf();
  // the thread's kPer entries, all loaded before any is used (16-byte loads when the
  // rows are 16-byte aligned: float4 k * kStatThreads + tid of the chunk), in
  // increasing index order; entries past the row read as -inf
  constexpr int kPer = kChunk / kStatThreads;
  float l[kPer];
  const bool vec = (p.V & 3) == 0;
  if (vec) {
#pragma unroll
    for (int k = 0; k < kPer / 4; ++k) {
      const int v = v0 + (k * kStatThreads + tid) * 4;
      const float4 f = v < v1 ? *reinterpret_cast<const float4*>(row + v) : make_float4(NEG, NEG, NEG, NEG);
      l[4 * k] = f.x;
      l[4 * k + 1] = f.y;
      l[4 * k + 2] = f.z;
      l[4 * k + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int v = v0 + k * kStatThreads + tid;
      l[k] = v < v1 ? row[v] : NEG;
    }
  }
  auto index = [&](int k) { return vec ? v0 + ((k >> 2) * kStatThreads + tid) * 4 + (k & 3) : v0 + k * kStatThreads + tid; };
  // max (and the first index holding it), then the sum of exp2 relative to it
  Stat st{NEG, 0.f, NEG, 0x7fffffff};
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    if (l[k] > st.av) {  // strictly greater: the first (lowest) index of a tie stays
      st.av = l[k];
      st.ai = index(k);
    }
  }
  st.m = st.av * kLog2e;
  if (st.av != NEG) {
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) sum += ex2(l[k] * kLog2e - st.m);  // (-inf entries add 0)
    st.s = sum;
  }
  st = warp_merge(st);
  if ((tid & 31) == 0) red[tid >> 5] = st;
  __syncthreads();
  if (tid == 0) {
    Stat a = red[0];
    for (int w = 1; w < kStatThreads / 32; ++w) merge(a, red[w]);
    reinterpret_cast<float4*>(p.stats)[static_cast<size_t>(r) * p.nchunk + c] =
        make_float4(a.m, a.s, a.av, __int_as_float(a.ai));
  }
}

// Sum of the block's values in position order: an inclusive scan inside each warp, then
// the warps' totals in order.  Returns the total (to every thread) and, through
// `before`, the sum of the values of the threads before this one.  The search for a
// draw uses the same arithmetic as the tile totals, so the two agree.
__device__ __forceinline__ float block_scan(float v, float* red, float& before) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  float s = 0.f, pre = 0.f;
#pragma unroll
  for (int w = 0; w < kDecThreads / 32; ++w) {
    if (w == warp) pre = s;
    s += red[w];
  }
  before = pre + (incl - v);
  return s;
}

// Per-sequence decision record (workspace): a, the next token (greedy), and row a's
// statistics of p and q (max and sum in log2 units).
struct Decision {
  int a, next;
  float pm, ps, qm, qs;
  int pad[2];
};

__global__ void __launch_bounds__(kDecideThreads) accept_decide_kernel(const AcceptParams p) {
  __shared__ Stat rs[32];  // merged statistics of this sequence's rows: p rows, then q rows
  __shared__ int sh[2];
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.gamma;
  const int nrows = p.sample ? 2 * G + 1 : G + 1;
  const float NEG = neg_inf();
  // ---- each warp merges one row's chunks (lanes over chunks, then chunk order)
  for (int i = warp; i < nrows; i += kDecideThreads / 32) {
    const int r = i <= G ? b * (G + 1) + i : p.B * (G + 1) + b * G + (i - G - 1);
    Stat acc{NEG, 0.f, NEG, 0x7fffffff};
    for (int c0 = 0; c0 < p.nchunk; c0 += 32) {
      Stat v{NEG, 0.f, NEG, 0x7fffffff};
      if (c0 + lane < p.nchunk) {
        const float4 f = reinterpret_cast<const float4*>(p.stats)[static_cast<size_t>(r) * p.nchunk + c0 + lane];
        v = Stat{f.x, f.y, f.z, __float_as_int(f.w)};
      }
      v = warp_merge(v);
      merge(acc, v);
    }
    if (lane == 0) rs[i] = acc;
  }
  __syncthreads();
  // ---- the decisions, lane t for draft t (all loads in one round); a = the first failure
  if (warp == 0) {
    const int t = lane;
    bool ok = true, oob = false;
    if (t < G) {
      const int x = p.draft[static_cast<size_t>(b) * G + t];
      if (x < 0 || x >= p.V) {
        ok = false;
        oob = true;
      } else if (!p.sample) {
        ok = x == rs[t].ai;
      } else {
        const float lp = p.p_logits[(static_cast<size_t>(b) * (G + 1) + t) * p.V + x];
        const float lq = p.q_logits[(static_cast<size_t>(b) * G + t) * p.V + x];
        const float pt = ex2(lp * kLog2e - rs[t].m) / rs[t].s;
        const float qt = ex2(lq * kLog2e - rs[G + 1 + t].m) / rs[G + 1 + t].s;
        ok = p.u[static_cast<size_t>(b) * G + t] * qt < pt;
      }
    }
    const unsigned fail = __ballot_sync(0xffffffffu, t < G && !ok);
    const int a = fail ? __ffs(fail) - 1 : G;
    if (t == a && oob) report(p.status, VG_ERR_DEVICE_BOUNDS);  // (as the first rejection)
    if (lane == 0) {
      sh[0] = a;
      sh[1] = rs[a].ai;  // (greedy: the next token)
    }
  }
  __syncthreads();
  if (tid != 0) return;
  const int a = sh[0];
  if (!p.sample) {
    p.n_accept[b] = a;
    p.next_token[b] = sh[1];
    if (p.advance_len) p.advance_len[b] += a + 1;
    return;
  }
  const bool rej = a < G;
  Decision d{};
  d.a = a;
  d.next = sh[1];
  d.pm = rs[a].m;
  d.ps = rs[a].s;
  d.qm = rej ? rs[G + 1 + a].m : 0.f;
  d.qs = rej ? rs[G + 1 + a].s : 1.f;
  reinterpret_cast<Decision*>(p.dec)[b] = d;
}

// The four weights of thread tid in tile `tile` of row a: max(0, p - q) after a
// rejection (excess), else p; p, q the softmax of the rows.
struct DrawRow {
  const float* lp;
  const float* lq;
  float pm, ip, qm, iq;
  int V;
};

__device__ __forceinline__ DrawRow draw_row(const AcceptParams& p, int b, const Decision& d) {
  const int G = p.gamma;
  DrawRow r;
  r.lp = p.p_logits + (static_cast<size_t>(b) * (G + 1) + d.a) * p.V;
  r.lq = d.a < G ? p.q_logits + (static_cast<size_t>(b) * G + d.a) * p.V : nullptr;
  r.pm = d.pm;
  r.ip = 1.f / d.ps;
  r.qm = d.qm;
  r.iq = 1.f / d.qs;
  r.V = p.V;
  return r;
}

// p's weight and the excess weight of the tid's four entries of a tile (zeros past V).
__device__ __forceinline__ void tile_weights(const DrawRow& r, int tile, int tid, float (&wp)[4], float (&wx)[4]) {
  const int v = tile * kTile + tid * 4;
  float lp[4], lq[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    lp[e] = 0.f;
    lq[e] = 0.f;
  }
  if (v + 3 < r.V && (r.V & 3) == 0) {
    const float4 fp = *reinterpret_cast<const float4*>(r.lp + v);
    lp[0] = fp.x; lp[1] = fp.y; lp[2] = fp.z; lp[3] = fp.w;
    if (r.lq) {
      const float4 fq = *reinterpret_cast<const float4*>(r.lq + v);
      lq[0] = fq.x; lq[1] = fq.y; lq[2] = fq.z; lq[3] = fq.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (v + e < r.V) {
        lp[e] = r.lp[v + e];
        if (r.lq) lq[e] = r.lq[v + e];
      }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const bool in = v + e < r.V;
    const float pv = in ? ex2(lp[e] * kLog2e - r.pm) * r.ip : 0.f;
    wp[e] = pv;
    wx[e] = (in && r.lq) ? fmaxf(0.f, pv - ex2(lq[e] * kLog2e - r.qm) * r.iq) : 0.f;
  }
}

__global__ void __launch_bounds__(kDecThreads) accept_tiles_kernel(const AcceptParams p) {
  __shared__ float red[kDecThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int tile = blockIdx.x, b = blockIdx.y;
  const Decision d = reinterpret_cast<const Decision*>(p.dec)[b];
  const DrawRow r = draw_row(p, b, d);
  float wp[4], wx[4], bef;
  tile_weights(r, tile, threadIdx.x, wp, wx);
  const float tx = block_scan(((wx[0] + wx[1]) + wx[2]) + wx[3], red, bef);
  const float tp = block_scan(((wp[0] + wp[1]) + wp[2]) + wp[3], red, bef);
  if (threadIdx.x == 0) {
    p.tiles[(static_cast<size_t>(b) * 2 + 0) * p.ntiles + tile] = tx;
    p.tiles[(static_cast<size_t>(b) * 2 + 1) * p.ntiles + tile] = tp;
  }
}

__global__ void __launch_bounds__(kDecThreads) accept_pick_kernel(const AcceptParams p) {
  __shared__ float red[kDecThreads / 32];
  __shared__ int sh[4];
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x, tid = threadIdx.x;
  const Decision d = reinterpret_cast<const Decision*>(p.dec)[b];
  const DrawRow r = draw_row(p, b, d);
  const int ntiles = p.ntiles;
  // the weights: the excess after a rejection, unless it is zero everywhere; then p
  if (tid == 0) {
    const float* tx = p.tiles + (static_cast<size_t>(b) * 2 + 0) * ntiles;
    const float* tp = tx + ntiles;
    bool excess = d.a < p.gamma;
    float total = 0.f;
    if (excess) {
      for (int t = 0; t < ntiles; ++t) total += tx[t];  // (fixed order)
      if (total <= 0.f) excess = false;
    }
    if (!excess) {
      total = 0.f;
      for (int t = 0; t < ntiles; ++t) total += tp[t];
    }
    // the tile where the running sum passes u_res * total
    const float* ts = excess ? tx : tp;
    const float target = p.u_res[b] * total;
    float run = 0.f;
    int t = 0;
    for (; t < ntiles - 1; ++t) {
      if (run + ts[t] > target) break;
      run += ts[t];
    }
    sh[0] = t;
    reinterpret_cast<float*>(sh)[1] = run;
    reinterpret_cast<float*>(sh)[2] = target;
    sh[3] = excess ? 1 : 0;
  }
  __syncthreads();
  const int tile = sh[0];
  const float base = reinterpret_cast<float*>(sh)[1], target = reinterpret_cast<float*>(sh)[2];
  const bool excess = sh[3] != 0;
  float wp[4], wx[4], bef;
  tile_weights(r, tile, tid, wp, wx);
  float w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) w[e] = excess ? wx[e] : wp[e];
  block_scan(((w[0] + w[1]) + w[2]) + w[3], red, bef);  // the entries of the tile in order
  __syncthreads();
  if (tid == 0) sh[0] = 0x7fffffff;
  __syncthreads();
  // the first entry whose running sum exceeds the target (last positive entry if
  // rounding leaves the target at or above the total)
  float run = base + bef;
  const int v0 = tile * kTile + tid * 4;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    run += w[e];
    if (w[e] > 0.f && run > target && v0 + e < p.V) {
      atomicMin(&sh[0], v0 + e);
      break;
    }
  }
  __syncthreads();
  int next = sh[0];
  if (next == 0x7fffffff) {  // (the target reached the total through rounding)
    __syncthreads();
    if (tid == 0) sh[1] = -1;
    __syncthreads();
    for (int tt = ntiles - 1; tt >= 0 && sh[1] < 0; --tt) {
      float wp2[4], wx2[4];
      tile_weights(r, tt, tid, wp2, wx2);
      int last = -1;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((excess ? wx2[e] : wp2[e]) > 0.f) last = tt * kTile + tid * 4 + e;
      if (last >= 0) atomicMax(&sh[1], last);
      __syncthreads();
    }
    next = sh[1];
  }
  if (tid == 0) {
    p.n_accept[b] = d.a;
    p.next_token[b] = next;
    if (p.advance_len) p.advance_len[b] += d.a + 1;
  }
}

}  // namespace

cudaError_t launch_accept(const AcceptParams& p, cudaStream_t stream) {
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  const int nrows = p.B * (p.gamma + 1) + (p.sample ? p.B * p.gamma : 0);
  cfg.gridDim = dim3(p.nchunk, nrows);
  cfg.blockDim = dim3(kStatThreads);
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, accept_stats_kernel, p);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(p.B);
  cfg.blockDim = dim3(kDecideThreads);
  if ((e = cudaLaunchKernelEx(&cfg, accept_decide_kernel, p)) != cudaSuccess || !p.sample) return e;
  cfg.gridDim = dim3(p.ntiles, p.B);
  cfg.blockDim = dim3(kDecThreads);
  if ((e = cudaLaunchKernelEx(&cfg, accept_tiles_kernel, p)) != cudaSuccess) return e;
  cfg.gridDim = dim3(p.B);
  return cudaLaunchKernelEx(&cfg, accept_pick_kernel, p);
}

int accept_chunks(int V) { return (V + kChunk - 1) / kChunk; }
int accept_tiles(int V) { return (V + kTile - 1) / kTile; }

}  // namespace vg
