// Warp-level flash-attention steps on bf16 tensor cores (mma.sync m16n8k16),
// used by the sparse-draft kernel.
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

// Online-softmax update with 16 logits per row already in log2 units (masked
// keys at -inf), then O += P V.  vaddr(r, c16) as kaddr, for the value rows.
// P goes to the tensor cores as a bf16 high part plus a bf16 low part, P - bf16(P),
// each multiplied with the same value fragments, so the weights carry about 16 bits
// (relative error near 2^-17) and agree with the fp32 row sum l: rounding P to bf16
// alone would move a row whose weight sits on a few keys by up to 2^-9 of its values.
//
// PACK (at most 8 query rows, so rows 8..15 hold no query): the low part of row r
// takes the A-operand row r + 8, and one MMA per value block yields both products,
// the high part's in accumulator rows 0..7 and the low part's in rows 8..15; the
// output of row r is then o[.][0..1] + o[.][2..3] (fold_packed).
template <int D, bool PACK = false, typename VAddr>
__device__ __forceinline__ void softmax_pv16(RowState<D>& st, float (&s)[2][4], VAddr vaddr, int lane) {
  const float NEG = neg_inf();
  if constexpr (PACK) {
    float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    const float mn0 = fmaxf(st.m[0], mx0);
    const float mu0 = mn0 == NEG ? 0.f : mn0;
    if (__any_sync(0xffffffffu, mn0 > st.m[0])) {
      const float a0 = ex2(st.m[0] - mu0);
      st.l[0] *= a0;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        st.o[dn][0] *= a0;
        st.o[dn][1] *= a0;
        st.o[dn][2] *= a0;
        st.o[dn][3] *= a0;
      }
    }
    st.m[0] = mn0;
    const float p00 = ex2(s[0][0] - mu0), p01 = ex2(s[0][1] - mu0);
    const float p10 = ex2(s[1][0] - mu0), p11 = ex2(s[1][1] - mu0);
    st.l[0] += p00 + p01 + p10 + p11;
    uint32_t a[4];  // rows r: high part, rows r + 8: low part (keys 0..7, then 8..15)
    split_bf16(p00, p01, a[0], a[1]);
    split_bf16(p10, p11, a[2], a[3]);
    const int mi = lane >> 3, rr = lane & 7;
    const int r = (mi & 1) * 8 + rr;
#pragma unroll
    for (int dn2 = 0; dn2 < D / 16; ++dn2) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vaddr(r, dn2 * 2 + (mi >> 1)), b0, b1, b2, b3);
      mma_bf16(st.o[2 * dn2], a, b0, b1);
      mma_bf16(st.o[2 * dn2 + 1], a, b2, b3);
    }
    return;
  }
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
  uint32_t ph[4], pl[4];
  split_bf16(pr[0][0], pr[0][1], ph[0], pl[0]);
  split_bf16(pr[0][2], pr[0][3], ph[1], pl[1]);
  split_bf16(pr[1][0], pr[1][1], ph[2], pl[2]);
  split_bf16(pr[1][2], pr[1][3], ph[3], pl[3]);
  const int mi = lane >> 3, rr = lane & 7;
  const int r = (mi & 1) * 8 + rr;
#pragma unroll
  for (int dn2 = 0; dn2 < D / 16; ++dn2) {
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(vaddr(r, dn2 * 2 + (mi >> 1)), b0, b1, b2, b3);
    mma_bf16(st.o[2 * dn2], ph, b0, b1);
    mma_bf16(st.o[2 * dn2 + 1], ph, b2, b3);
    mma_bf16(st.o[2 * dn2], pl, b0, b1);
    mma_bf16(st.o[2 * dn2 + 1], pl, b2, b3);
  }
}

// Output rows of a PACK state: adds the low part's products (rows 8..15) to the high
// part's (rows 0..7).
template <int D>
__device__ __forceinline__ void fold_packed(RowState<D>& st) {
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) {
    st.o[dn][0] += st.o[dn][2];
    st.o[dn][1] += st.o[dn][3];
  }
}

}  // namespace vg
