// Sparse draft attention over the verification-selected entries.
//
// Vegas §2 step 3 (draft phase): each draft token attends only the critical KV
// entries chosen from the previous verification, plus the draft tokens appended
// since; Vegas §3 (sparse execution) runs this as a paged attention with a page
// of one token, the selected positions serving as page indices.
//
// GB300 design.  The gathered entries of all sequences form one flattened list,
// split evenly over one persistent CTA per SM.  A producer warp turns each selected
// position into two TMA bulk copies (the token's K row and V row, all KV heads
// contiguous: H_kv*d*2 bytes each) landing in a padded shared-memory ring guarded by
// mbarriers; one consumer warp per KV head runs QK^T and PV on bf16 tensor cores with
// fp32 online softmax and leaves one unnormalised partial per run of entries.  A
// combine kernel (programmatic dependent launch) adds the short tail of draft
// tokens, merges the partials, writes bf16 outputs and appends the current draft
// token's K/V.
#include "vg_common.cuh"
#include "vg_internal.h"

namespace vg {
namespace {

constexpr int TKD = kDraftStageKeys;
constexpr int kMaxTail = 256;
constexpr int kMaxKvHeads = 16;

__device__ __forceinline__ float bf2f(__nv_bfloat16 v) { return __bfloat162float(v); }

struct DLayout {
  int row_stride;  // bytes per gathered token row in shared memory (padded by 16)
  int half;        // K (or V) rows of one stage
  int stage;
  int off_pos, off_bar, off_cum, total;
  __host__ __device__ DLayout(int Hkv, int D, int stages, int B) {
    row_stride = Hkv * D * 2 + 16;
    half = TKD * row_stride;
    stage = 2 * half;
    off_pos = stages * stage;
    off_bar = off_pos + stages * TKD * 4;
    off_bar = (off_bar + 7) & ~7;
    off_cum = off_bar + 2 * stages * 8;
    total = off_cum + (B + 1) * 4;
  }
};

__device__ __forceinline__ int tail_len_of(const DraftParams& p, int b) {
  return p.tail_len ? p.tail_len[b] : p.tail_len_const;
}

// Entries per sequence (checked) and their prefix sums; warp 0 only.
__device__ void draft_meta(const DraftParams& p, int* cum) {
  const int lane = threadIdx.x & 31;
  int carry = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    int e = 0;
    if (b < p.B) {
      e = p.count[b];
      const int64_t off = p.seq_offset[b];
      const int ts = p.tail_start[b];
      const bool ok = e >= 0 && e <= p.k_stride && off >= 0 && ts >= 0 && off + ts <= p.capacity;
      if (!ok) {
        report(p.status, VG_ERR_DEVICE_BOUNDS);
        e = 0;
      }
    }
    int v = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += t;
    }
    if (b < p.B) cum[b] = carry + v - e;
    carry += __shfl_sync(0xffffffffu, v, 31);
  }
  if (lane == 0) cum[p.B] = carry;
}

__device__ __forceinline__ void locate_entry(int x, const int* cum, int B, int& b, int& j) {
  int lo = 0, hi = B;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cum[mid] <= x) lo = mid; else hi = mid - 1;
  }
  b = lo;
  j = x - cum[b];
}

// MAXW: the most KV heads (consumer warps) this instantiation serves.
template <int D, int MAXW>
__global__ void __launch_bounds__((MAXW + 1) * 32) __maxnreg__((65536 / ((MAXW + 1) * 32)) / 8 * 8 > 255 ? 255 : (65536 / ((MAXW + 1) * 32)) / 8 * 8)
    draft_kernel(const DraftParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const DLayout L(p.Hkv, D, p.stages, p.B);
  int* posb = reinterpret_cast<int*>(smem + L.off_pos);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_bar);
  uint64_t* empty = full + p.stages;
  int* cum = reinterpret_cast<int*>(smem + L.off_cum);
  const int W = p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float NEG = neg_inf();

  pdl_wait();  // idx / count come from the selection kernel
  if (warp == 0) draft_meta(p, cum);
  if (threadIdx.x == 32) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], W);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < p.B + 1; i += blockDim.x) p.meta[i] = cum[i];
  }
  pdl_launch_dependents();

  const int E = cum[p.B];
  const int x0 = static_cast<int>(split_begin(blockIdx.x, E, p.nctas));
  const int x1 = static_cast<int>(split_begin(blockIdx.x + 1, E, p.nctas));
  if (x0 >= x1) return;
  const int rowbytes = p.Hkv * D * 2;

  // ------------------------------------------------------------ producer warp
  if (warp == W) {
    int b, j;
    locate_entry(x0, cum, p.B, b, j);
    int stage = 0;
    uint32_t phase = 0;
    for (int x = x0; x < x1;) {
      const int nvalid = min(TKD, min(x1 - x, (cum[b + 1] - cum[b]) - j));
      bool ok_wait = true;
      if (lane == 0) ok_wait = mbar_wait(&empty[stage], phase ^ 1u, p.status);
      ok_wait = __shfl_sync(0xffffffffu, ok_wait, 0);
      if (!ok_wait) break;
      int pos = -1;
      bool ok = false;
      if (lane < nvalid) {
        pos = p.idx[static_cast<size_t>(b) * p.k_stride + j + lane];
        ok = pos >= 0 && pos < p.tail_start[b];
        if (!ok) report(p.status, VG_ERR_DEVICE_BOUNDS);
      }
      if (lane < TKD) posb[stage * TKD + lane] = ok ? pos : -1;
      const int nload = __popc(__ballot_sync(0xffffffffu, ok));
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(nload * 2 * rowbytes));
      __syncwarp();
      if (ok) {
        const size_t slot = static_cast<size_t>(p.seq_offset[b] + pos);
        uint8_t* kd = smem + stage * L.stage + lane * L.row_stride;
        bulk_load(kd, p.K + slot * p.Hkv * D, rowbytes, &full[stage]);
        bulk_load(kd + L.half, p.V + slot * p.Hkv * D, rowbytes, &full[stage]);
      }
      x += nvalid;
      j += nvalid;
      if (x < x1 && j == cum[b + 1] - cum[b]) {
        j = 0;
        ++b;
        while (b < p.B && cum[b + 1] == cum[b]) ++b;
      }
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    return;
  }
  if (warp > W) return;

  // ------------------------------------------------------------ consumer warp g
  const int g = warp;
  const int gid = lane >> 2, tig = lane & 3;
  int b, j;
  locate_entry(x0, cum, p.B, b, j);
  int stage = 0;
  uint32_t phase = 0;
  bool lost = false;
  for (int x = x0; x < x1 && !lost;) {
    const int seg_end = min(x1, x + (cum[b + 1] - cum[b]) - j);
    uint32_t qf[D / 16][4];
    {
      const __nv_bfloat16* q0 = gid < p.G ? p.q + (static_cast<size_t>(b) * p.Hq + g * p.G + gid) * D : nullptr;
      const __nv_bfloat16* q1 =
          gid + 8 < p.G ? p.q + (static_cast<size_t>(b) * p.Hq + g * p.G + gid + 8) * D : nullptr;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int c0 = ks * 16 + tig * 2;
        qf[ks][0] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + c0) : 0u;
        qf[ks][1] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + c0) : 0u;
        qf[ks][2] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + c0 + 8) : 0u;
        qf[ks][3] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + c0 + 8) : 0u;
      }
    }
    float m_run[2] = {NEG, NEG}, l_run[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;

    while (x < seg_end) {
      const int nvalid = min(TKD, seg_end - x);
      if (!mbar_wait(&full[stage], phase, p.status)) {
        lost = true;
        break;
      }
      const uint32_t kb = smem_u32(smem + stage * L.stage) + g * D * 2;
      const uint32_t vb = kb + L.half;
      const int* ps = posb + stage * TKD;
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      {
        const int mi = lane >> 3, rr = lane & 7;
        const int r = (mi >> 1) * 8 + rr;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int c16 = ks * 2 + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + r * L.row_stride + c16 * 16, b0, b1, b2, b3);
          mma_bf16(s[0], qf[ks], b0, b1);
          mma_bf16(s[1], qf[ks], b2, b3);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const bool ok = ps[nt * 8 + tig * 2 + c] >= 0;  // stage rows past nvalid hold -1
          s[nt][c] = ok ? s[nt][c] * p.scale_log2 : NEG;
          s[nt][2 + c] = ok ? s[nt][2 + c] * p.scale_log2 : NEG;
        }
      float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
      float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
      const float mu0 = mn0 == NEG ? 0.f : mn0, mu1 = mn1 == NEG ? 0.f : mn1;
      if (__any_sync(0xffffffffu, (mn0 > m_run[0]) || (mn1 > m_run[1]))) {
        const float a0 = ex2(m_run[0] - mu0), a1 = ex2(m_run[1] - mu1);
        l_run[0] *= a0;
        l_run[1] *= a1;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
          o[dn][0] *= a0;
          o[dn][1] *= a0;
          o[dn][2] *= a1;
          o[dn][3] *= a1;
        }
      }
      m_run[0] = mn0;
      m_run[1] = mn1;
      float pr[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        pr[nt][0] = ex2(s[nt][0] - mu0);
        pr[nt][1] = ex2(s[nt][1] - mu0);
        pr[nt][2] = ex2(s[nt][2] - mu1);
        pr[nt][3] = ex2(s[nt][3] - mu1);
      }
      l_run[0] += pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1];
      l_run[1] += pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3];
      const uint32_t pa[4] = {pack_bf16(pr[0][0], pr[0][1]), pack_bf16(pr[0][2], pr[0][3]),
                              pack_bf16(pr[1][0], pr[1][1]), pack_bf16(pr[1][2], pr[1][3])};
      {
        const int mi = lane >> 3, rr = lane & 7;
        const int r = (mi & 1) * 8 + rr;
#pragma unroll
        for (int dn2 = 0; dn2 < D / 16; ++dn2) {
          const int c16 = dn2 * 2 + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + r * L.row_stride + c16 * 16, b0, b1, b2, b3);
          mma_bf16(o[2 * dn2], pa, b0, b1);
          mma_bf16(o[2 * dn2 + 1], pa, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
      }
      x += nvalid;
      j += nvalid;
    }
    // partial of this run of entries, rows = the G query heads of KV head g
    l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 1);
    l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], 2);
    l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 1);
    l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], 2);
    const size_t id = static_cast<size_t>(blockIdx.x) + b;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int jh = gid + half * 8;
      if (jh < p.G) {
        const size_t row = id * p.Hq + g * p.G + jh;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn)
          *reinterpret_cast<float2*>(p.part_o + row * D + dn * 8 + tig * 2) =
              make_float2(o[dn][half * 2], o[dn][half * 2 + 1]);
        if (tig == 0) {
          p.part_ml[row * 2 + 0] = m_run[half];
          p.part_ml[row * 2 + 1] = l_run[half];
        }
      }
    }
    if (x < x1) {
      j = 0;
      ++b;
      while (b < p.B && cum[b + 1] == cum[b]) ++b;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(128) draft_combine_kernel(const DraftParams p) {
  __shared__ float lg[kMaxTail];
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y;
  const int g = h / p.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float NEG = neg_inf();
  const int* cum = p.meta;
  const int64_t off = p.seq_offset[b];
  const int ts = p.tail_start[b];
  const int tl = tail_len_of(p, b);
  const bool ok = off >= 0 && ts >= 0 && tl >= 0 && tl <= kMaxTail && off + ts + tl <= p.capacity &&
                  (p.k_new == nullptr || tl >= 1);
  if (!ok) {
    if (tid == 0) report(p.status, VG_ERR_DEVICE_BOUNDS);
    return;
  }
  const __nv_bfloat16* qh = p.q + (static_cast<size_t>(b) * p.Hq + h) * D;
  auto key_row = [&](int u) -> const __nv_bfloat16* {
    if (p.k_new && u == tl - 1) return p.k_new + (static_cast<size_t>(b) * p.Hkv + g) * D;
    return p.K + ((off + ts + u) * p.Hkv + g) * D;
  };
  auto val_row = [&](int u) -> const __nv_bfloat16* {
    if (p.v_new && u == tl - 1) return p.v_new + (static_cast<size_t>(b) * p.Hkv + g) * D;
    return p.V + ((off + ts + u) * p.Hkv + g) * D;
  };
  for (int u = warp; u < tl; u += 4) {
    const __nv_bfloat16* kr = key_row(u);
    float acc = 0.f;
    for (int e = lane; e < D; e += 32) acc += bf2f(qh[e]) * bf2f(kr[e]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) lg[u] = acc * p.scale_log2;
  }
  __syncthreads();
  const int Eb = cum[b + 1] - cum[b];
  int64_t cf = 0, cl = -1;
  if (Eb > 0) {
    const int64_t E = cum[p.B];
    cf = owner_cta(cum[b], E, p.nctas);
    cl = owner_cta(cum[b] + Eb - 1, E, p.nctas);
  }
  if (tid < D) {
    const int e = tid;
    float M = NEG, acc = 0.f, l = 0.f;
    for (int64_t c = cf; c <= cl; ++c) {
      const size_t row = (static_cast<size_t>(c) + b) * p.Hq + h;
      const float ms = p.part_ml[row * 2 + 0], ls = p.part_ml[row * 2 + 1];
      const float os = p.part_o[row * D + e];
      const float Mn = fmaxf(M, ms);
      const float a = ex2(M - Mn), w = ex2(ms - Mn);
      acc = acc * a + os * w;
      l = l * a + ls * w;
      M = Mn;
    }
    for (int u = 0; u < tl; ++u) {
      const float lu = lg[u];
      const float Mn = fmaxf(M, lu);
      const float a = ex2(M - Mn), w = ex2(lu - Mn);
      acc = acc * a + w * bf2f(val_row(u)[e]);
      l = l * a + w;
      M = Mn;
    }
    p.out[(static_cast<size_t>(b) * p.Hq + h) * D + e] = __float2bfloat16_rn(l > 0.f ? acc / l : 0.f);
    if (p.k_new && h % p.G == 0) {  // append the current draft token (one CTA per KV head)
      const size_t dst = ((off + ts + tl - 1) * p.Hkv + g) * D + e;
      p.K[dst] = p.k_new[(static_cast<size_t>(b) * p.Hkv + g) * D + e];
      p.V[dst] = p.v_new[(static_cast<size_t>(b) * p.Hkv + g) * D + e];
    }
  }
}

template <int D, int MAXW>
cudaError_t launch_draft_t(const DraftParams& p, cudaStream_t stream, bool pdl) {
  const DLayout L(p.Hkv, D, p.stages, p.B);
  const size_t smem = static_cast<size_t>(L.total) + 128;
  cudaError_t e = cudaFuncSetAttribute(draft_kernel<D, MAXW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nctas);
  cfg.blockDim = dim3((p.Hkv + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, draft_kernel<D, MAXW>, p);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg2 = {};
  cfg2.gridDim = dim3(p.Hq, p.B);
  cfg2.blockDim = dim3(128);
  cfg2.dynamicSmemBytes = 0;
  cfg2.stream = stream;
  cfg2.attrs = at;
  cfg2.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg2, draft_combine_kernel<D>, p);
}

}  // namespace

int draft_stages(int Hkv, int D) {
  const DLayout L(Hkv, D, 1, 1);
  int s = (200 * 1024) / L.stage;
  return s < 1 ? 1 : (s > 4 ? 4 : s);
}

size_t draft_smem_bytes(int Hkv, int D, int stages, int B) {
  const DLayout L(Hkv, D, stages, B);
  return static_cast<size_t>(L.total) + 128;
}

cudaError_t launch_draft(const DraftParams& p, cudaStream_t stream, bool pdl) {
  if (p.Hkv <= 8) {
    if (p.D == 64) return launch_draft_t<64, 8>(p, stream, pdl);
    if (p.D == 128) return launch_draft_t<128, 8>(p, stream, pdl);
  } else {
    if (p.D == 64) return launch_draft_t<64, kMaxKvHeads>(p, stream, pdl);
    if (p.D == 128) return launch_draft_t<128, kMaxKvHeads>(p, stream, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace vg
