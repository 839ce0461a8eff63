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
// GB300 design.  Two kernels, both HBM-bound reductions over the vocabulary.
//   accept_stats_kernel: one CTA per (row, 8192-entry chunk) of the target rows (and the
//     draft rows when sampling): the chunk's max, sum of exp2 relative to it and argmax
//     (lowest index), in a fixed reduction order.
//   accept_decide_kernel: one CTA per sequence merges the chunks' statistics (in chunk
//     order), takes the decisions, and for a draw sums the weights in tiles of 4096
//     entries (float4 loads, a fixed-order block reduction per tile), finds the tile
//     where the running sum passes the target and scans that tile alone.  It writes the
//     accepted count and the next token, and advances the prefix length if asked.
// Logits are read as log2-scaled values (l * log2 e), so every exponential is one ex2.
#include "vg_common.cuh"
#include "vg_internal.h"

namespace vg {
namespace {

constexpr int kChunk = 8192;      // vocabulary entries per statistics CTA
constexpr int kStatThreads = 256;
constexpr int kDecThreads = 1024;
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
  const int c = blockIdx.x, r = blockIdx.y;
  const float* row = row_ptr(p, r);
  const int v0 = c * kChunk, v1 = min(p.V, v0 + kChunk);
  const float NEG = neg_inf();
  Stat st{NEG, 0.f, NEG, 0x7fffffff};
  // each thread walks its entries in increasing order (online max and sum)
  for (int v = v0 + threadIdx.x; v < v1; v += kStatThreads) {
    const float l = row[v];
    const float x = l * kLog2e;
    if (x > st.m) {
      st.s = (st.m == NEG ? 0.f : st.s * ex2(st.m - x)) + 1.f;
      st.m = x;
    } else {
      st.s += ex2(x - st.m);
    }
    if (l > st.av) {  // strictly greater: the first (lowest) index of a tie stays
      st.av = l;
      st.ai = v;
    }
  }
  st = warp_merge(st);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = st;
  __syncthreads();
  if (threadIdx.x == 0) {
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

__global__ void __launch_bounds__(kDecThreads) accept_decide_kernel(const AcceptParams p) {
  __shared__ Stat rs[64];        // merged statistics of this sequence's rows: p rows, then q rows
  __shared__ float red[kDecThreads / 32];
  __shared__ float tiles[kMaxAcceptTiles];
  __shared__ int sh[4];
  pdl_wait();
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.gamma;
  const int nrows = p.sample ? 2 * G + 1 : G + 1;
  const float NEG = neg_inf();
  // ---- each warp merges one row's chunks (lanes over chunks, then chunk order)
  for (int i = warp; i < nrows; i += kDecThreads / 32) {
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
  // ---- decisions (one thread; at most gamma dependent loads)
  if (tid == 0) {
    int a = G;
    for (int t = 0; t < G; ++t) {
      const int x = p.draft[static_cast<size_t>(b) * G + t];
      bool ok;
      if (x < 0 || x >= p.V) {
        report(p.status, VG_ERR_DEVICE_BOUNDS);
        ok = false;
      } else if (!p.sample) {
        ok = x == rs[t].ai;
      } else {
        const Stat& sp = rs[t];
        const Stat& sq = rs[G + 1 + t];
        const float pt = ex2(p.p_logits[(static_cast<size_t>(b) * (G + 1) + t) * p.V + x] * kLog2e - sp.m) / sp.s;
        const float qt = ex2(p.q_logits[(static_cast<size_t>(b) * G + t) * p.V + x] * kLog2e - sq.m) / sq.s;
        ok = p.u[static_cast<size_t>(b) * G + t] * qt < pt;
      }
      if (!ok) {
        a = t;
        break;
      }
    }
    sh[0] = a;
    sh[1] = rs[a].ai;  // (greedy: the next token)
  }
  __syncthreads();
  const int a = sh[0];
  int next = sh[1];
  if (p.sample) {
    // ---- the draw: weights of row a (excess over the draft after a rejection)
    const bool rej = a < G;
    const Stat sp = rs[a];
    const Stat sq = rej ? rs[G + 1 + a] : Stat{0.f, 1.f, 0.f, 0};
    const float* lp = p.p_logits + (static_cast<size_t>(b) * (G + 1) + a) * p.V;
    const float* lq = rej ? p.q_logits + (static_cast<size_t>(b) * G + a) * p.V : nullptr;
    const float ip = 1.f / sp.s, iq = 1.f / sq.s;
    const int ntiles = (p.V + kTile - 1) / kTile;
    auto weight = [&](int v, float l_p, float l_q, bool excess) {
      const float pv = ex2(l_p * kLog2e - sp.m) * ip;
      if (!excess) return pv;
      return fmaxf(0.f, pv - ex2(l_q * kLog2e - sq.m) * iq);
    };
    auto tile_weights = [&](int tile, bool excess, float (&w)[4]) {
      const int v = tile * kTile + tid * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) w[e] = 0.f;
      if (v + 3 < p.V && (p.V & 3) == 0) {
        const float4 fp = *reinterpret_cast<const float4*>(lp + v);
        const float4 fq = excess ? *reinterpret_cast<const float4*>(lq + v) : make_float4(0.f, 0.f, 0.f, 0.f);
        w[0] = weight(v, fp.x, fq.x, excess);
        w[1] = weight(v + 1, fp.y, fq.y, excess);
        w[2] = weight(v + 2, fp.z, fq.z, excess);
        w[3] = weight(v + 3, fp.w, fq.w, excess);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (v + e < p.V) w[e] = weight(v + e, lp[v + e], excess ? lq[v + e] : 0.f, excess);
      }
    };
    bool excess = rej;
    float total = 0.f;
    for (int pass = 0; pass < 2; ++pass) {  // (a second pass only if the excess is zero everywhere)
      total = 0.f;
      for (int tile = 0; tile < ntiles; ++tile) {
        float w[4], bef;
        tile_weights(tile, excess, w);
        const float ts = block_scan(((w[0] + w[1]) + w[2]) + w[3], red, bef);
        if (tid == 0) tiles[tile] = ts;
        total += ts;  // (every thread: the same values in the same order)
      }
      if (!(excess && total <= 0.f)) break;
      excess = false;
    }
    __syncthreads();
    // the tile where the running sum passes u_res * total, then the entry inside it
    const float target = p.u_res[b] * total;
    if (tid == 0) {
      float run = 0.f;
      int t = 0;
      for (; t < ntiles - 1; ++t) {
        if (run + tiles[t] > target) break;
        run += tiles[t];
      }
      sh[2] = t;
      reinterpret_cast<float*>(sh)[3] = run;
    }
    __syncthreads();
    const int tile = sh[2];
    const float base = reinterpret_cast<float*>(sh)[3];
    float w[4], bef;
    tile_weights(tile, excess, w);
    block_scan(((w[0] + w[1]) + w[2]) + w[3], red, bef);  // the entries of the tile in order
    const float before = base + bef;
    // the first entry whose running sum exceeds the target (last positive entry if
    // rounding leaves the target at or above the total)
    if (tid == 0) sh[0] = 0x7fffffff;
    __syncthreads();
    float run = before;
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
    next = sh[0];
    if (next == 0x7fffffff) {  // (the target reached the total through rounding)
      __syncthreads();
      if (tid == 0) sh[1] = -1;
      __syncthreads();
      for (int tt = ntiles - 1; tt >= 0 && sh[1] < 0; --tt) {
        float w2[4];
        tile_weights(tt, excess, w2);
        int last = -1;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (w2[e] > 0.f) last = tt * kTile + tid * 4 + e;
        if (last >= 0) atomicMax(&sh[1], last);
        __syncthreads();
      }
      next = sh[1];
    }
  }
  if (tid == 0) {
    p.n_accept[b] = a;
    p.next_token[b] = next;
    if (p.advance_len) p.advance_len[b] += a + 1;
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
  cfg.blockDim = dim3(kDecThreads);
  return cudaLaunchKernelEx(&cfg, accept_decide_kernel, p);
}

int accept_chunks(int V) { return (V + kChunk - 1) / kChunk; }

}  // namespace vg
