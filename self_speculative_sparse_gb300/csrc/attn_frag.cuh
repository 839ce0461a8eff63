// Warp-level flash-attention steps on bf16 tensor cores (mma.sync m16n8k16),
// shared by the verify and sparse-draft kernels.
//
// A warp owns a 16-row m-tile of query rows (held as A fragments) and consumes
// keys 16 at a time from shared memory.  Logits stay in log2 units so the
// softmax uses MUFU.EX2 directly; the running max / sum / output are the usual
// online-softmax state, rescaled only when some row's max moves.
#pragma once

#include "vg_common.cuh"

namespace vg {

template <int D>
struct RowState {
  float m[2];          // running max of rows gid and gid + 8 (log2 units)
  float l[2];          // this thread's share of the running sum
  float o[D / 8][4];   // unnormalised output, C-fragment layout
  __device__ __forceinline__ void init() {
    m[0] = m[1] = neg_inf();
    l[0] = l[1] = 0.f;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
  }
};

// A fragments of 16 query rows: row0 / row1 point at rows gid and gid + 8 (or are null).
template <int D>
__device__ __forceinline__ void load_q_frags(uint32_t (&qf)[D / 16][4], const __nv_bfloat16* row0,
                                             const __nv_bfloat16* row1, int tig) {
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int c0 = ks * 16 + tig * 2;
    qf[ks][0] = row0 ? *reinterpret_cast<const uint32_t*>(row0 + c0) : 0u;
    qf[ks][1] = row1 ? *reinterpret_cast<const uint32_t*>(row1 + c0) : 0u;
    qf[ks][2] = row0 ? *reinterpret_cast<const uint32_t*>(row0 + c0 + 8) : 0u;
    qf[ks][3] = row1 ? *reinterpret_cast<const uint32_t*>(row1 + c0 + 8) : 0u;
  }
}

// s = Q K^T for 16 keys.  kaddr(r, c16) is the shared address of key r (0..15),
// 16-byte chunk c16 of its d values.
// (Even and odd k-steps accumulate separately: four independent MMA chains.)
template <int D, typename KAddr>
__device__ __forceinline__ void qk16(const uint32_t (&qf)[D / 16][4], KAddr kaddr, float (&s)[2][4], int lane) {
  float t[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    t[nt][0] = t[nt][1] = t[nt][2] = t[nt][3] = 0.f;
  }
  const int mi = lane >> 3, rr = lane & 7;
  const int r = (mi >> 1) * 8 + rr;
#pragma unroll
  for (int ks = 0; ks < D / 16; ks += 2) {
    uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
    ldsm_x4(kaddr(r, ks * 2 + (mi & 1)), b0, b1, b2, b3);
    ldsm_x4(kaddr(r, (ks + 1) * 2 + (mi & 1)), c0, c1, c2, c3);
    mma_bf16(s[0], qf[ks], b0, b1);
    mma_bf16(s[1], qf[ks], b2, b3);
    mma_bf16(t[0], qf[ks + 1], c0, c1);
    mma_bf16(t[1], qf[ks + 1], c2, c3);
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) s[nt][c] += t[nt][c];
}

// Column sums of a 16x16 S tile over the warp's 16 rows, in 4 shuffles: v[nt*2+c]
// holds this thread's (row-masked) contribution to key nt*8 + tig*2 + c.  A
// transposing butterfly halves the values carried at each step; the result is the
// sum for key ((lane >> 4) & 1) * 8 + tig * 2 + ((lane >> 3) & 1), and lanes that
// differ only in bit 2 hold the same sum.
__device__ __forceinline__ float colsum16(const float (&v)[4], int lane) {
  const bool h2 = (lane & 16) != 0;
  float k0 = h2 ? v[2] : v[0];
  float k1 = h2 ? v[3] : v[1];
  k0 += __shfl_xor_sync(0xffffffffu, h2 ? v[0] : v[2], 16);
  k1 += __shfl_xor_sync(0xffffffffu, h2 ? v[1] : v[3], 16);
  const bool h1 = (lane & 8) != 0;
  float keep = h1 ? k1 : k0;
  keep += __shfl_xor_sync(0xffffffffu, h1 ? k0 : k1, 8);
  keep += __shfl_xor_sync(0xffffffffu, keep, 4);
  return keep;
}

// Online-softmax update with 16 logits per row already in log2 units (masked
// keys at -inf), then O += P V.  vaddr(r, c16) as kaddr, for the value rows.
template <int D, typename VAddr>
__device__ __forceinline__ void softmax_pv16(RowState<D>& st, float (&s)[2][4], VAddr vaddr, int lane) {
  const float NEG = neg_inf();
  float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
  float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
  const float mu0 = mn0 == NEG ? 0.f : mn0, mu1 = mn1 == NEG ? 0.f : mn1;
  if (__any_sync(0xffffffffu, (mn0 > st.m[0]) || (mn1 > st.m[1]))) {
    const float a0 = ex2(st.m[0] - mu0), a1 = ex2(st.m[1] - mu1);
    st.l[0] *= a0;
    st.l[1] *= a1;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      st.o[dn][0] *= a0;
      st.o[dn][1] *= a0;
      st.o[dn][2] *= a1;
      st.o[dn][3] *= a1;
    }
  }
  st.m[0] = mn0;
  st.m[1] = mn1;
  float pr[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    pr[nt][0] = ex2(s[nt][0] - mu0);
    pr[nt][1] = ex2(s[nt][1] - mu0);
    pr[nt][2] = ex2(s[nt][2] - mu1);
    pr[nt][3] = ex2(s[nt][3] - mu1);
  }
  st.l[0] += pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1];
  st.l[1] += pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3];
  const uint32_t pa[4] = {pack_bf16(pr[0][0], pr[0][1]), pack_bf16(pr[0][2], pr[0][3]),
                          pack_bf16(pr[1][0], pr[1][1]), pack_bf16(pr[1][2], pr[1][3])};
  const int mi = lane >> 3, rr = lane & 7;
  const int r = (mi & 1) * 8 + rr;
#pragma unroll
  for (int dn2 = 0; dn2 < D / 16; ++dn2) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(vaddr(r, dn2 * 2 + (mi >> 1)), b0, b1, b2, b3);
    mma_bf16(st.o[2 * dn2], pa, b0, b1);
    mma_bf16(st.o[2 * dn2 + 1], pa, b2, b3);
  }
}

// Merge the states of the KGW warps that share an m-tile (warp index kgw within
// it) into shared memory, in a fixed order: merge[M][ms] holds the unnormalised
// output rebased to the merged max, lrow[M] the sum and mrow[0][*] ... the maxima.
// All NT consumer threads call it; bar_id is a named barrier for them.
template <int D, int KGW>
__device__ __forceinline__ void merge_warps(RowState<D>& st, int M, int ms, int row0, int kgw, float* merge,
                                            float* mrow, float* lrow, int tig, int bar_id, int nthreads) {
  const float NEG = neg_inf();
  const int row1 = row0 + 8;
  st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], 1);
  st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], 2);
  st.l[1] += __shfl_xor_sync(0xffffffffu, st.l[1], 1);
  st.l[1] += __shfl_xor_sync(0xffffffffu, st.l[1], 2);
  if (tig == 0) {
    mrow[kgw * M + row0] = st.m[0];
    mrow[kgw * M + row1] = st.m[1];
  }
  named_bar(bar_id, nthreads);
  float mf0 = NEG, mf1 = NEG;
#pragma unroll
  for (int w2 = 0; w2 < KGW; ++w2) {
    mf0 = fmaxf(mf0, mrow[w2 * M + row0]);
    mf1 = fmaxf(mf1, mrow[w2 * M + row1]);
  }
  const float f0 = ex2(st.m[0] - (mf0 == NEG ? 0.f : mf0));
  const float f1 = ex2(st.m[1] - (mf1 == NEG ? 0.f : mf1));
  st.l[0] *= f0;
  st.l[1] *= f1;
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) {
    st.o[dn][0] *= f0;
    st.o[dn][1] *= f0;
    st.o[dn][2] *= f1;
    st.o[dn][3] *= f1;
  }
  for (int w2 = 0; w2 < KGW; ++w2) {
    if (kgw == w2) {
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        float2* d0 = reinterpret_cast<float2*>(merge + row0 * ms + dn * 8 + tig * 2);
        float2* d1 = reinterpret_cast<float2*>(merge + row1 * ms + dn * 8 + tig * 2);
        if (w2 == 0) {
          *d0 = make_float2(st.o[dn][0], st.o[dn][1]);
          *d1 = make_float2(st.o[dn][2], st.o[dn][3]);
        } else {
          const float2 a = *d0, c = *d1;
          *d0 = make_float2(a.x + st.o[dn][0], a.y + st.o[dn][1]);
          *d1 = make_float2(c.x + st.o[dn][2], c.y + st.o[dn][3]);
        }
      }
      if (tig == 0) {
        lrow[row0] = (w2 == 0 ? 0.f : lrow[row0]) + st.l[0];
        lrow[row1] = (w2 == 0 ? 0.f : lrow[row1]) + st.l[1];
      }
    }
    named_bar(bar_id, nthreads);
  }
}

// Copies a merged m-tile group (rows [0, M)) to a partial slot in global memory:
// out_o[M][D] and out_ml[M][2] = (max over the KGW warps, sum).
template <int D, int KGW>
__device__ __forceinline__ void store_partial(const float* merge, int ms, const float* mrow, const float* lrow,
                                              int M, float* out_o, float* out_ml, int tid, int nthreads) {
  const float NEG = neg_inf();
  float4* dst = reinterpret_cast<float4*>(out_o);
  for (int e = tid; e < M * D / 4; e += nthreads) {
    const int r = e / (D / 4), c = e - r * (D / 4);
    dst[e] = *reinterpret_cast<const float4*>(merge + r * ms + c * 4);
  }
  for (int r = tid; r < M; r += nthreads) {
    float mf = NEG;
#pragma unroll
    for (int w2 = 0; w2 < KGW; ++w2) mf = fmaxf(mf, mrow[w2 * M + r]);
    out_ml[r * 2 + 0] = mf;
    out_ml[r * 2 + 1] = lrow[r];
  }
}

// Register prefetch of up to NB partial output rows for one warp (partials first,
// first + step, ...): the loads are issued before their weights are known, so they
// overlap the loads of the maxima and sums.  Out-of-range slots read partial
// `first` again (a readable address) and are never used.
template <int D, int NB>
struct PartialRows {
  float v[NB][D / 32];
  template <typename ORow>
  __device__ __forceinline__ void load(ORow orow, int first, int step, int nseg, int lane) {
    constexpr int PER = D / 32;
#pragma unroll
    for (int q = 0; q < NB; ++q) {
      const int si = first + q * step < nseg ? first + q * step : first;
      const float* src = orow(si) + lane * PER;
      if constexpr (PER == 4) {
        const float4 t = *reinterpret_cast<const float4*>(src);
        v[q][0] = t.x;
        v[q][1] = t.y;
        v[q][2] = t.z;
        v[q][3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(src);
        v[q][0] = t.x;
        v[q][1] = t.y;
      }
    }
  }
  // acc += sum w_s O_s, l += sum w_s l_s over the prefetched partials
  __device__ __forceinline__ void accumulate(const float* cm, const float* csum, int cstride, int first, int step,
                                             int nseg, float M, float (&acc)[D / 32], float& l) const {
    const float NEG = neg_inf();
#pragma unroll
    for (int q = 0; q < NB; ++q) {
      const int si = first + q * step;
      if (si < nseg) {
        const float ms = cm[si * cstride];
        if (ms != NEG) {
          const float w = ex2(ms - M);
          l += w * csum[si * cstride];
#pragma unroll
          for (int c = 0; c < D / 32; ++c) acc[c] += w * v[q][c];
        }
      }
    }
  }
};

// One warp merges the partials of one query row: acc[lane's d values] and l get
// sum_s w_s * O_s and sum_s w_s * l_s with w_s = 2^(m_s - M).  Partial s has its
// (max, sum) at cm[s * cstride], csum[s * cstride] (max = -inf: no partial) and its
// output row at orow(s) (a float pointer, always a readable address).  Loads are
// issued 8 at a time, unconditionally, so each batch costs one memory round trip;
// absent partials are dropped with a select (their memory may hold anything).
// The warp visits partials first, first + step, ... (several warps can split them).
template <int D, typename ORow>
__device__ __forceinline__ void merge_partials(const float* cm, const float* csum, int cstride, int nseg, float M,
                                               ORow orow, float (&acc)[D / 32], float& l, int lane, int first = 0,
                                               int step = 1) {
  constexpr int PER = D / 32;
  const float NEG = neg_inf();
  for (int s0 = first; s0 < nseg; s0 += 8 * step) {
    float w[8];
    float v[8][PER];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const bool in = s0 + q * step < nseg;
      const int si = in ? s0 + q * step : s0;
      const float ms = cm[si * cstride];
      w[q] = (in && ms != NEG) ? ex2(ms - M) : 0.f;
      const float* src = orow(si) + lane * PER;
      if constexpr (PER == 4) {
        const float4 t = *reinterpret_cast<const float4*>(src);
        v[q][0] = t.x;
        v[q][1] = t.y;
        v[q][2] = t.z;
        v[q][3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(src);
        v[q][0] = t.x;
        v[q][1] = t.y;
      }
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (w[q] > 0.f) {
        l += w[q] * csum[(s0 + q * step) * cstride];
#pragma unroll
        for (int c = 0; c < PER; ++c) acc[c] += w[q] * v[q][c];
      }
    }
  }
}

}  // namespace vg
