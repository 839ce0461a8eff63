// Sparse draft attention over the verification-selected entries.
//
// Vegas §2 step 3 (draft phase): each draft token attends only the critical KV
// entries chosen from the previous verification, plus the draft tokens appended
// since; Vegas §3 (sparse execution) runs this as a paged attention with a page
// of one token, the selected positions serving as page indices.
//
// GB300 design.  A token's page is its cache slot: all KV heads contiguous, H_kv*d*2
// bytes of K and as many of V.  Each sequence's attended entries are its selected
// positions followed by the tail of draft-token slots.  The work is the fixed grid
// of (sequence, entry slot) items, k_stride + a tail bound slots per sequence (slots
// past the sequence's entries are masked), split evenly over one persistent CTA per
// SM: the split needs no device data, so each CTA's first memory round trip already
// fetches its positions, and the combine kernel knows where the partials are.  A
// producer warp turns each entry into two TMA bulk copies of a whole page (large
// requests keep the copy engine efficient; the current draft token comes straight
// from the inputs) landing in a padded, bank-conflict-free shared-memory ring
// guarded by mbarriers; one consumer warp per KV head runs QK^T and PV on bf16
// tensor cores with fp32 online softmax and writes one unnormalised partial per
// (run, head).  A combine kernel (programmatic dependent launch) merges the
// partials with 8 warps splitting them, writes bf16 outputs and appends the
// current draft token's K/V to the cache.
#include "attn_frag.cuh"
#include "vg_common.cuh"
#include "vg_internal.h"

namespace vg {
namespace {

constexpr int kKeys = 16;  // entries per pipeline stage
constexpr int kStages = 2;
constexpr int kCombineRows = 12;  // partial rows a combine warp loads in its first round

struct DLayout {
  int row;  // bytes per gathered page in shared memory (padded by 16: ldmatrix rows hit distinct banks)
  int half, stage, off_pos, off_bar, total;
  __host__ __device__ DLayout(int Hkv, int D) {
    row = Hkv * D * 2 + 16;
    half = kKeys * row;
    stage = 2 * half;
    off_pos = kStages * stage;                           // int [kStages][kKeys]
    off_bar = (off_pos + kStages * kKeys * 4 + 7) & ~7;  // full[kStages], empty[kStages]
    total = off_bar + 2 * kStages * 8;
  }
};

__device__ __forceinline__ int tail_len_of(const DraftParams& p, int b) {
  return p.tail_len ? p.tail_len[b] : p.tail_len_const;
}

// Entry slots per sequence in the static work split.
__host__ __device__ __forceinline__ int draft_slots(const DraftParams& p) {
  return p.k_stride + (p.tail_len ? kDraftMaxTail : p.tail_len_const);
}

// MAXW: the most KV heads (consumer warps) this instantiation serves.
template <int D, int MAXW>
__global__ void __launch_bounds__((MAXW + 1) * 32, 1) draft_kernel(const DraftParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const DLayout L(p.Hkv, D);
  int* posb = reinterpret_cast<int*>(smem + L.off_pos);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_bar);
  uint64_t* empty = full + kStages;
  const int W = p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float NEG = neg_inf();

  if (threadIdx.x == 32) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], W);
    }
    fence_mbar_init();
  }
  // The value rows of every stage start zeroed (shared memory only, so before the
  // dependency wait): a slot of a chunk that loads no page keeps either these zeros or
  // a value row an earlier chunk attended, so 0 * V stays exact without zeroing rows on
  // the producer's critical path.
  for (int st = 0; st < kStages; ++st) {
    uint4* vr = reinterpret_cast<uint4*>(smem + st * L.stage + L.half);
    for (int q = threadIdx.x; q < L.half / 16; q += blockDim.x) vr[q] = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();  // the zeros precede the bulk copies into the same stages
  __syncthreads();
  const int S = draft_slots(p);
  const int64_t E = static_cast<int64_t>(p.B) * S;
  const int x0 = static_cast<int>(split_begin(blockIdx.x, E, p.nctas));
  const int x1 = static_cast<int>(split_begin(blockIdx.x + 1, E, p.nctas));
  pdl_launch_dependents();
  if (x0 >= x1) return;
  // idx / count come from the selection kernel, the tail pages from the previous step.
  // Kernels of this library trigger their dependents early, so several may be in
  // flight: nothing an earlier kernel writes is read before this wait.
  pdl_wait();
  const int page = p.Hkv * D * 2;  // bytes of one token's K (or V), all heads

  // ------------------------------------------------------------ producer warp
  if (warp == W) {
    int b = x0 / S, j = x0 - b * S;
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;  // chunks whose copies were started
    for (int x = x0; x < x1;) {
      const int nvalid = min(kKeys, min(x1 - x, S - j));
      bool ok_wait = true;
      if (lane == 0) ok_wait = mbar_wait(&empty[stage], phase ^ 1u, p.status);
      if (!__shfl_sync(0xffffffffu, ok_wait, 0)) break;
      // one round of independent loads: this sequence's counts and the chunk's positions
      const int jj = j + lane;  // selected entries first, then the draft-token tail
      const int cnt_raw = p.count[b];
      const int tl = tail_len_of(p, b);
      const int ts = p.tail_start[b];
      const int64_t off = p.seq_offset[b];
      const int sel = (lane < nvalid && jj < p.k_stride) ? p.idx[static_cast<size_t>(b) * p.k_stride + jj] : 0;
      const bool seq_ok = cnt_raw >= 0 && cnt_raw <= p.k_stride && tl >= 0 && tl <= kDraftMaxTail && off >= 0 &&
                          ts >= 0 && off + ts + tl <= p.capacity && (p.k_new == nullptr || tl >= 1);
      if (!seq_ok && lane == 0 && j == 0) report(p.status, VG_ERR_DEVICE_BOUNDS);
      const int nsel = seq_ok ? cnt_raw : 0;
      uint8_t* kst = smem + stage * L.stage;
      int pos = -1;
      if (seq_ok && lane < nvalid) {
        if (jj < nsel) {
          pos = sel;
          if (pos < 0 || pos >= ts) {
            report(p.status, VG_ERR_DEVICE_BOUNDS);
            pos = -1;
          }
        } else if (jj < nsel + tl) {
          pos = ts + (jj - nsel);
        }
      }
      if (lane < kKeys) posb[stage * kKeys + lane] = pos;
      const int nload = __popc(__ballot_sync(0xffffffffu, pos >= 0));
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(nload * 2 * page));
      __syncwarp();
      if (pos >= 0) {
        const __nv_bfloat16* ksrc;
        const __nv_bfloat16* vsrc;
        if (p.k_new && pos == ts + tl - 1) {  // the current draft token, straight from the inputs
          ksrc = p.k_new + static_cast<size_t>(b) * p.Hkv * D;
          vsrc = p.v_new + static_cast<size_t>(b) * p.Hkv * D;
        } else {
          ksrc = p.K + static_cast<size_t>(off + pos) * p.Hkv * D;
          vsrc = p.V + static_cast<size_t>(off + pos) * p.Hkv * D;
        }
        bulk_load(kst + lane * L.row, ksrc, page, &full[stage]);
        bulk_load(kst + L.half + lane * L.row, vsrc, page, &full[stage]);
      }
      ++issued;
      x += nvalid;
      j += nvalid;
      if (j == S) {
        j = 0;
        ++b;
      }
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // no copy may still be in flight when the CTA exits, also when a consumer gave up
    // (normally the consumers have already seen every chunk land)
    if (lane == 0)
      for (int c = issued > kStages ? issued - kStages : 0; c < issued; ++c)
        mbar_wait(&full[c % kStages], static_cast<uint32_t>((c / kStages) & 1), p.status);
    __syncwarp();
    return;
  }

  // ------------------------------------------------------------ consumer warp: KV head g
  const int g = warp;
  const int gid = lane >> 2, tig = lane & 3;
  int b = x0 / S, j = x0 - b * S;
  int stage = 0;
  uint32_t phase = 0;
  bool lost = false;
  for (int x = x0; x < x1 && !lost;) {
    const int seg_end = min(x1, x + (S - j));
    uint32_t qf[D / 16][4];
    load_q_frags<D>(qf, gid < p.G ? p.q + (static_cast<size_t>(b) * p.Hq + g * p.G + gid) * D : nullptr,
                    gid + 8 < p.G ? p.q + (static_cast<size_t>(b) * p.Hq + g * p.G + gid + 8) * D : nullptr, tig);
    RowState<D> st;
    st.init();
    while (x < seg_end) {
      const int nvalid = min(kKeys, seg_end - x);
      if (!mbar_wait(&full[stage], phase, p.status)) {
        lost = true;
        break;
      }
      const uint32_t kb = smem_u32(smem + stage * L.stage) + g * D * 2;
      const uint32_t vb = kb + L.half;
      const int row = L.row;
      auto kaddr = [&](int r, int c16) { return kb + r * row + c16 * 16; };
      auto vaddr = [&](int r, int c16) { return vb + r * row + c16 * 16; };
      float s[2][4];
      qk16<D>(qf, kaddr, s, lane);
      const int* ps = posb + stage * kKeys;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int e = nt * 8 + tig * 2 + c;
          const bool ok = e < nvalid && ps[e] >= 0;
          s[nt][c] = ok ? s[nt][c] * p.scale_log2 : NEG;
          s[nt][2 + c] = ok ? s[nt][2 + c] * p.scale_log2 : NEG;
        }
      softmax_pv16<D>(st, s, vaddr, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
      x += nvalid;
      j += nvalid;
    }
    // partial of this run for the G query heads of KV head g
    st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], 1);
    st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], 2);
    st.l[1] += __shfl_xor_sync(0xffffffffu, st.l[1], 1);
    st.l[1] += __shfl_xor_sync(0xffffffffu, st.l[1], 2);
    const size_t id = static_cast<size_t>(blockIdx.x) + b;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int jh = gid + half * 8;
      if (jh < p.G) {
        const size_t r = id * p.Hq + g * p.G + jh;
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn)
          *reinterpret_cast<float2*>(p.part_o + r * D + dn * 8 + tig * 2) =
              make_float2(st.o[dn][half * 2], st.o[dn][half * 2 + 1]);
        if (tig == 0) {
          p.part_ml[r * 2 + 0] = st.m[half];
          p.part_ml[r * 2 + 1] = st.l[half];
        }
      }
    }
    if (x < x1) {
      j = 0;
      ++b;
    }
  }
}

// One CTA per (query head h, sequence b), NW warps (enough that each holds at most
// kCombineRows partials).  Warp w owns partials w, w + NW, ...: it loads their (max, sum) one per lane and their output rows (lanes across d)
// in a single round, the CTA agrees on the global max through shared memory, and the
// warps' weighted sums are added in a fixed order (deterministic).  The CTA of each
// KV head's first query head then appends the current draft token.
template <int D, int NW>
__global__ void __launch_bounds__(NW * 32) draft_combine_kernel(const DraftParams p) {
  constexpr int kCombineWarps = NW;
  constexpr int PER = D / 32;  // elements of a row per lane
  __shared__ float red[kCombineWarps][D];
  __shared__ float redl[kCombineWarps];
  __shared__ float redm[kCombineWarps];
  const int h = blockIdx.x, b = blockIdx.y;
  const int g = h / p.G;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float NEG = neg_inf();
  // the partials of sequence b come from the CTAs whose static ranges meet its slots
  const int S = draft_slots(p);
  const int64_t E = static_cast<int64_t>(p.B) * S;
  const int64_t cf = owner_cta(static_cast<int64_t>(b) * S, E, p.nctas);
  const int64_t cl = owner_cta(static_cast<int64_t>(b + 1) * S - 1, E, p.nctas);
  const int nseg = static_cast<int>(cl - cf + 1);  // <= 32 * kCombineWarps (host choice)
  auto prow = [&](int si) { return (static_cast<size_t>(cf + si) + b) * p.Hq + h; };
  pdl_launch_dependents();  // the next draft step may start its prologue
  pdl_wait();
  // ---- one round of loads: lane q holds (max, sum) of partial warp + NW q; the first
  // kCombineRows output rows of the warp's partials go to registers
  float pm = NEG, pl = 0.f;
  {
    const int si = warp + kCombineWarps * lane;
    if (si < nseg && split_nonempty(cf + si, E, p.nctas)) {  // CTAs with no entries wrote no partial
      const float2 v = *reinterpret_cast<const float2*>(p.part_ml + prow(si) * 2);
      pm = v.x;
      pl = v.y;
    }
  }
  // (rows past nseg, or of a CTA with no entries, read as zeros: their weight is zero
  // and the row holds whatever was there)
  float v[kCombineRows][PER];
#pragma unroll
  for (int q = 0; q < kCombineRows; ++q) {
    const int si = warp + kCombineWarps * q;
    const bool ok = si < nseg && split_nonempty(cf + si, E, p.nctas);
    const float* src = p.part_o + prow(ok ? si : 0) * D + lane * PER;
    if constexpr (PER == 4) {
      const float4 x = ok ? *reinterpret_cast<const float4*>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
      v[q][0] = x.x; v[q][1] = x.y; v[q][2] = x.z; v[q][3] = x.w;
    } else {
      const float2 x = ok ? *reinterpret_cast<const float2*>(src) : make_float2(0.f, 0.f);
      v[q][0] = x.x; v[q][1] = x.y;
    }
  }
  // ---- global max
  float mx = pm;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) redm[warp] = mx;
  __syncthreads();
  float M = NEG;
#pragma unroll
  for (int w = 0; w < kCombineWarps; ++w) M = fmaxf(M, redm[w]);
  // ---- this warp's weighted sum, partials in order
  const float wt = (pm != NEG) ? ex2(pm - M) : 0.f;
  float l = wt * pl;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
#pragma unroll
  for (int q = 0; q < kCombineRows; ++q) {
    const float wq = __shfl_sync(0xffffffffu, wt, q);
    if (warp + kCombineWarps * q < nseg) {
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] += wq * v[q][e];
    }
  }
  for (int q = kCombineRows; warp + kCombineWarps * q < nseg; ++q) {  // rare: more partials per warp
    const float wq = __shfl_sync(0xffffffffu, wt, q);
    if (!split_nonempty(cf + warp + kCombineWarps * q, E, p.nctas)) continue;  // (warp-uniform)
    const float* src = p.part_o + prow(warp + kCombineWarps * q) * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] += wq * src[e];
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) red[warp][lane * PER + e] = acc[e];
  if (lane == 0) redl[warp] = l;
  __syncthreads();
  if (tid < D) {
    float a = 0.f, lt = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {  // fixed order: deterministic
      a += red[w][tid];
      lt += redl[w];
    }
    p.out[(static_cast<size_t>(b) * p.Hq + h) * D + tid] = __float2bfloat16_rn(lt > 0.f ? a / lt : 0.f);
  }
  if (p.k_new && h % p.G == 0) {  // append the current draft token at tail_start + tail_len - 1
    const int64_t off = p.seq_offset[b];
    const int ts = p.tail_start[b];
    const int tl = tail_len_of(p, b);
    if (off >= 0 && ts >= 0 && tl >= 1 && tl <= kDraftMaxTail && off + ts + tl <= p.capacity) {
      const size_t dst = ((off + ts + tl - 1) * p.Hkv + g) * D;
      const size_t src = (static_cast<size_t>(b) * p.Hkv + g) * D;
      for (int c = tid; c < D / 8; c += kCombineWarps * 32) {
        reinterpret_cast<uint4*>(p.K + dst)[c] = reinterpret_cast<const uint4*>(p.k_new + src)[c];
        reinterpret_cast<uint4*>(p.V + dst)[c] = reinterpret_cast<const uint4*>(p.v_new + src)[c];
      }
    }
  }
}

template <int D, int MAXW>
cudaError_t launch_draft_t(const DraftParams& p, cudaStream_t stream, bool pdl) {
  const size_t smem = static_cast<size_t>(DLayout(p.Hkv, D).total) + 128;
  cudaError_t e = ensure_smem<draft_kernel<D, MAXW>>(smem);
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
  // partials per sequence: the CTAs whose static ranges meet its slots
  const int64_t E = static_cast<int64_t>(p.B) * draft_slots(p);
  int nseg_max = 0;
  for (int b = 0; b < p.B; ++b) {
    const int64_t cf = owner_cta(static_cast<int64_t>(b) * draft_slots(p), E, p.nctas);
    const int64_t cl = owner_cta(static_cast<int64_t>(b + 1) * draft_slots(p) - 1, E, p.nctas);
    nseg_max = max(nseg_max, static_cast<int>(cl - cf + 1));
  }
  cudaLaunchConfig_t cfg2 = {};
  cfg2.gridDim = dim3(p.Hq, p.B);
  cfg2.dynamicSmemBytes = 0;
  cfg2.stream = stream;
  cfg2.attrs = at;
  cfg2.numAttrs = 1;
  if (nseg_max <= 4 * kCombineRows) {
    cfg2.blockDim = dim3(4 * 32);
    return cudaLaunchKernelEx(&cfg2, draft_combine_kernel<D, 4>, p);
  }
  if (nseg_max <= 8 * kCombineRows) {
    cfg2.blockDim = dim3(8 * 32);
    return cudaLaunchKernelEx(&cfg2, draft_combine_kernel<D, 8>, p);
  }
  cfg2.blockDim = dim3(16 * 32);
  return cudaLaunchKernelEx(&cfg2, draft_combine_kernel<D, 16>, p);
}

}  // namespace

size_t draft_smem_bytes(int D, int Hkv) { return static_cast<size_t>(DLayout(Hkv, D).total) + 128; }

cudaError_t launch_draft(const DraftParams& p, cudaStream_t stream, bool pdl) {
  if (p.Hkv <= 8) {
    if (p.D == 64) return launch_draft_t<64, 8>(p, stream, pdl);
    if (p.D == 128) return launch_draft_t<128, 8>(p, stream, pdl);
  } else if (p.D == 64) {  // (more than 8 KV heads at d = 128 exceed a 1024-element page)
    return launch_draft_t<64, 16>(p, stream, pdl);
  }
  return cudaErrorInvalidValue;
}

}  // namespace vg
