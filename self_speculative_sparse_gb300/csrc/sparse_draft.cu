// Sparse draft attention over the verification-selected entries.
//
// Vegas §2 step 3 (draft phase): each draft token attends only the critical KV
// entries chosen from the previous verification, plus the draft tokens appended
// since; Vegas §3 (sparse execution) runs this as a paged attention with a page
// of one token, the selected positions serving as page indices.
//
// GB300 design.
//   * A token's page is its cache slot: all KV heads contiguous, H_kv*d*2 bytes of K
//     and as many of V.  Each sequence's attended entries are its selected positions
//     followed by the tail of draft-token slots.  The work is the fixed list of
//     (sequence, entry slot) items - k_stride + a tail bound per sequence, slots past
//     the sequence's entries masked - split evenly over the step's CTAs (one a SM for a
//     large step; fewer, of at least two chunks, for a small one), so the split needs no
//     device data and each CTA's first round trip fetches its positions.
//   * Every thread resolves one of the CTA's first entries (position, cache slot) into
//     a shared-memory table during the set-up; each producer warp resolves later
//     entries a batch ahead into its own ring, so no position round trip sits on the
//     per-chunk path.
//   * Two producer warps turn each entry into a bulk copy of a whole page each, one the
//     key page, the other the value page (large requests keep the copy engine
//     efficient, and a warp issues copies at a bounded rate; the current draft token
//     comes straight from the inputs) into a padded shared-memory ring guarded by
//     mbarriers; one
//     consumer warp per KV head runs Q K^T and P V on bf16 tensor cores with fp32
//     online softmax, P carried as a bf16 high and low part.
//   * Within a draft phase the selection does not change between steps.  When the
//     caller says so (VG_DRAFT_SELECTION_SETTLED), the CTA resolves its first entries
//     and the producer warps start their page copies before the dependency wait, so the
//     gather overlaps the end of the previous step; only the draft-token tail, which
//     the previous step appended, waits for it.  The draft kernel releases its
//     dependents only after its own dependency wait, the combine at entry (its set-up
//     then overlaps the merge): when a draft step starts, the selection kernel and
//     every step before the previous one have completed.
//   * A sequence whose entries one CTA holds entirely is finished by that CTA.  Every
//     other (CTA, sequence) run leaves an unnormalised partial (O, max, sum), and a
//     combine kernel (programmatic dependent launch) merges each (sequence, query
//     head) in a fixed order.  No atomics: results are deterministic.
//   * Whoever finishes a sequence's first query head of a KV head appends the current
//     draft token's K/V row of that head to the cache.
#include "attn_frag.cuh"
#include "vg_common.cuh"
#include "vg_internal.h"

namespace vg {
namespace {

constexpr int kKeys = kDraftChunk;  // entries per pipeline stage (one MMA key block)
constexpr int kMinStages = 2;  // ring stages: 2, or 3 for CTAs with many chunks (the host picks)
constexpr int kMaxStages = 3;
constexpr int kCombineRows = 12;  // partial rows a combine warp loads in one round

constexpr int kBatch = 128;  // entries a producer warp resolves in one round of loads (4 a lane)
constexpr int kTab = 256;    // ring of resolved entries (two batches)

// One resolved entry: its position (-1: masked), whether it is a draft-token slot
// (appended by earlier steps, or the current token, read from the inputs), and where
// its K and V pages are.
struct Entry {
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int pos;
  int tail;
};

struct DLayout {
  int row;  // bytes per gathered page in shared memory (padded by 16: ldmatrix rows hit distinct banks)
  int half, stage, off_pos, off_tab, off_bar, total;
  __host__ __device__ DLayout(int Hkv, int D, int NS) {
    row = Hkv * D * 2 + 16;
    half = kKeys * row;
    stage = 2 * half;
    off_pos = NS * stage;                             // int [NS][kKeys]
    off_tab = (off_pos + NS * kKeys * 4 + 15) & ~15;  // Entry [2][kTab]: each producer warp's own ring
    off_bar = off_tab + 2 * kTab * static_cast<int>(sizeof(Entry));  // full[NS], empty[NS]
    total = off_bar + 2 * NS * 8;
  }
};

__device__ __forceinline__ int tail_len_of(const DraftParams& p, int b) {
  return p.tail_len ? p.tail_len[b] : p.tail_len_const;
}

// Appends the current draft token's key and value of KV head g of sequence b at slot
// tail_start + tail_len - 1 (threads t, t + nt, ... of a group; skipped, never
// faulted, if out of range).
template <int D>
__device__ __forceinline__ void append_token(const DraftParams& p, int b, int g, int t, int nt) {
  const int ts = p.tail_start[b];
  const int tl = tail_len_of(p, b);
  if (!(ts >= 0 && tl >= 1 && tl <= kDraftMaxTail)) return;
  const int64_t slot = kv_slot<true>(p.seq_offset, p.ptab, p.psize, p.pstride, p.capacity, b, ts + tl - 1);
  if (slot < 0) return;
  const size_t dst = (slot * p.Hkv + g) * D;
  const size_t src = (static_cast<size_t>(b) * p.Hkv + g) * D;
  for (int c = t; c < D / 8; c += nt) {
    reinterpret_cast<uint4*>(p.K + dst)[c] = reinterpret_cast<const uint4*>(p.k_new + src)[c];
    reinterpret_cast<uint4*>(p.V + dst)[c] = reinterpret_cast<const uint4*>(p.v_new + src)[c];
  }
}

// The CTAs holding items of sequence b (first and last: the split is contiguous).
struct SeqSpan {
  int cf, cl;
};
__host__ __device__ __forceinline__ SeqSpan seq_span(int b, int S, int64_t E, int nctas) {
  return SeqSpan{static_cast<int>(owner_cta(static_cast<int64_t>(b) * S, E, nctas)),
                 static_cast<int>(owner_cta(static_cast<int64_t>(b + 1) * S - 1, E, nctas))};
}

// The loads behind entry e of the CTA's items, all independent, so one round trip
// serves every entry a warp resolves at once.  (They bypass L1, cached at L2 only: with
// a settled selection they run before the dependency wait, and must see what kernels
// that completed earlier wrote.)
struct RawEntry {
  int sel, cnt, tl, ts;
  int64_t so;  // seq_offset of the entry's sequence (flat caches)
};

__device__ __forceinline__ RawEntry load_entry(const DraftParams& p, int e, int x1, int S) {
  RawEntry r{0, 0, 0, 0, 0};
  if (e < x1) {
    const int b = e / S, jj = e - b * S;
    r.cnt = __ldcg(p.count + b);
    r.tl = p.tail_len ? __ldcg(p.tail_len + b) : p.tail_len_const;
    r.ts = __ldcg(p.tail_start + b);
    if (jj < p.k_stride) r.sel = __ldcg(p.idx + static_cast<size_t>(b) * p.k_stride + jj);
    if (p.ptab == nullptr) r.so = __ldcg(p.seq_offset + b);
  }
  return r;
}

// Entry slot jj of sequence b: its selected entries first, then the draft-token tail.
// A paged cache looks the position's page up (a second round trip: the page number
// depends on the position).
template <int D>
__device__ __forceinline__ Entry finish_entry(const DraftParams& p, const RawEntry& r, int e, int S) {
  Entry t{nullptr, nullptr, -1, 0};
  const int b = e / S, jj = e - b * S;
  const bool seq_ok = r.cnt >= 0 && r.cnt <= p.k_stride && r.tl >= 0 && r.tl <= kDraftMaxTail && r.cnt + r.tl <= S &&
                      r.ts >= 0 && (p.k_new == nullptr || r.tl >= 1);
  if (!seq_ok) {
    if (jj == 0) report(p.status, VG_ERR_DEVICE_BOUNDS);
    return t;
  }
  if (jj < r.cnt) {
    t.pos = r.sel;
    if (t.pos < 0 || t.pos >= r.ts) {
      report(p.status, VG_ERR_DEVICE_BOUNDS);
      t.pos = -1;
      return t;
    }
  } else if (jj < r.cnt + r.tl) {
    t.pos = r.ts + (jj - r.cnt);
    t.tail = 1;
  } else {
    return t;
  }
  if (p.k_new && t.tail && t.pos == r.ts + r.tl - 1) {  // the current draft token, from the inputs
    t.k = p.k_new + static_cast<size_t>(b) * p.Hkv * D;
    t.v = p.v_new + static_cast<size_t>(b) * p.Hkv * D;
    return t;
  }
  int64_t slot;
  if (p.ptab == nullptr) {
    const int64_t s2 = r.so + t.pos;
    slot = s2 >= 0 && s2 < p.capacity ? s2 : -1;
  } else {
    slot = kv_slot<true>(p.seq_offset, p.ptab, p.psize, p.pstride, p.capacity, b, t.pos);
  }
  if (slot < 0) {  // outside the cache (or the page table): skipped, reported
    report(p.status, VG_ERR_DEVICE_BOUNDS);
    t.pos = -1;
  } else {
    t.k = p.K + static_cast<size_t>(slot) * p.Hkv * D;
    t.v = p.V + static_cast<size_t>(slot) * p.Hkv * D;
  }
  return t;
}

// A batch of kBatch entries for a producer warp: entry xb + lane + 32 i.
__device__ __forceinline__ void load_batch(const DraftParams& p, RawEntry (&r)[kBatch / 32], int xb, int x1, int S,
                                           int lane) {
#pragma unroll
  for (int i = 0; i < kBatch / 32; ++i) r[i] = load_entry(p, xb + lane + 32 * i, x1, S);
}

// Its table entries, ring slot (e - x0) mod kTab (all resolved before any is stored, so
// a paged cache's page lookups overlap).
template <int D>
__device__ __forceinline__ void finish_batch(const DraftParams& p, const RawEntry (&r)[kBatch / 32], Entry* tab,
                                             int x0, int xb, int x1, int S, int lane) {
  Entry t[kBatch / 32];
#pragma unroll
  for (int i = 0; i < kBatch / 32; ++i) {
    const int e = xb + lane + 32 * i;
    t[i] = e < x1 ? finish_entry<D>(p, r[i], e, S) : Entry{nullptr, nullptr, -1, 0};
  }
#pragma unroll
  for (int i = 0; i < kBatch / 32; ++i) {
    const int e = xb + lane + 32 * i;
    if (e < x1) tab[(e - x0) & (kTab - 1)] = t[i];
  }
}

// MAXW: the most KV heads (consumer warps) this instantiation serves; PACK: at most 8
// query heads a KV head (their P high and low parts share one MMA); NS: ring stages.
template <int D, int MAXW, bool PACK, int NS>
__global__ void __launch_bounds__((MAXW + 2) * 32, 1) draft_kernel(const DraftParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const DLayout L(p.Hkv, D, NS);
  int* posb = reinterpret_cast<int*>(smem + L.off_pos);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.off_bar);
  uint64_t* empty = full + NS;
  const int W = p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float NEG = neg_inf();

  const int S = p.slots;
  const int64_t E = static_cast<int64_t>(p.B) * S;
  const int x0 = static_cast<int>(split_begin(blockIdx.x, E, p.nctas));
  const int x1 = static_cast<int>(split_begin(blockIdx.x + 1, E, p.nctas));
  Entry* tab = reinterpret_cast<Entry*>(smem + L.off_tab);
  // The first entries of the CTA (one a thread, up to the table's size) are resolved
  // during the set-up, by every thread at once: with a settled selection their loads
  // are issued first and land while the stages are zeroed; otherwise after the
  // dependency wait.
  const int n0 = min(static_cast<int>(blockDim.x), kTab);
  const int e0 = x0 + static_cast<int>(threadIdx.x);
  const bool mine = static_cast<int>(threadIdx.x) < n0 && e0 < x1;
  RawEntry r0{0, 0, 0, 0, 0};
  if (p.settled && mine) r0 = load_entry(p, e0, x1, S);
  if (threadIdx.x == 32) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], W);
    }
    fence_mbar_init();
  }
  // The value rows of every stage start zeroed (shared memory only, so before the
  // dependency wait): a slot of a chunk that loads no page keeps either these zeros or
  // a value row an earlier chunk attended, so 0 * V stays exact without zeroing rows on
  // the producers' critical path.
  for (int st = 0; st < NS; ++st) {
    uint4* vr = reinterpret_cast<uint4*>(smem + st * L.stage + L.half);
    for (int i = threadIdx.x; i < L.half / 16; i += blockDim.x) vr[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (!p.settled) {
    pdl_wait();
    if (mine) r0 = load_entry(p, e0, x1, S);
  }
  if (mine) tab[threadIdx.x] = finish_entry<D>(p, r0, e0, S);
  fence_proxy_async_smem();  // the zeros precede the bulk copies into the same stages
  __syncthreads();
  if (x0 >= x1) return;
  const int page = p.Hkv * D * 2;  // bytes of one token's K (or V), all heads

  // ------------------------------------------------------------------ producer warps
  // Warp W issues the key pages (and keeps the positions and the byte counts), warp W + 1
  // the value pages: a warp issues bulk copies at a bounded rate, and two halve the time
  // to start a chunk's copies.  The two walk the same chunks and wait on the same
  // barriers, each from its own ring of resolved entries (no exchange between them).
  if (warp >= W) {
    const int role = warp - W;  // 0: keys, 1: values
    Entry* ring = tab + role * kTab;
    if (role == 1) {  // the set-up's entries, into this warp's own ring
      for (int i = lane; i < n0; i += 32) ring[i] = tab[i];
      __syncwarp();
    }
    // Later entries are resolved a batch ahead: a batch's table entries are written
    // when the chunks reach it, while the next batch's loads are already in flight.
    RawEntry raw[kBatch / 32];
    int res_end = min(x1, x0 + n0);  // entries [x0, res_end) are in the ring
    if (res_end < x1) load_batch(p, raw, res_end, x1, S, lane);
    auto advance_tables = [&]() {
      finish_batch<D>(p, raw, ring, x0, res_end, x1, S, lane);
      res_end = min(x1, res_end + kBatch);
      if (res_end < x1) load_batch(p, raw, res_end, x1, S, lane);
      __syncwarp();
    };
    // Chunk [x, x + nvalid) into stage st: (keys) its positions for the consumers and
    // the byte count on the stage's barrier, and this warp's copies.  part: 0 all
    // pages, 1 all but the draft-token slots, 2 only those (a chunk whose part 1 is
    // already issued).
    auto issue_chunk = [&](int st, int x, int nvalid, int part) {
      const Entry t = lane < nvalid ? ring[(x + lane - x0) & (kTab - 1)] : Entry{nullptr, nullptr, -1, 0};
      if (role == 0 && part != 2) {
        if (lane < kKeys) posb[st * kKeys + lane] = t.pos;
        const int nload = __popc(__ballot_sync(0xffffffffu, t.pos >= 0));
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(nload * 2 * page));
        __syncwarp();
      }
      if (t.pos >= 0 && (part == 0 || (part == 1) == !t.tail)) {
        uint8_t* kst = smem + st * L.stage;
        if (role == 0)
          bulk_load(kst + lane * L.row, t.k, page, &full[st]);
        else
          bulk_load(kst + L.half + lane * L.row, t.v, page, &full[st]);
      }
    };
    int b = x0 / S, j = x0 - b * S;
    int x = x0;
    int stage = 0;
    uint32_t phase = 0;
    int issued;  // chunks whose copies were started
    // With a settled selection the first chunks' selected pages (as many chunks as the
    // ring holds) are requested before the dependency wait; their draft-token pages (the
    // previous step appended the last of them) and every later chunk wait for it.
    int ex[NS], en[NS];
    int nearly = 0;
    if (p.settled) {
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        if (x < x1) {
          const int nvalid = min(kKeys, min(x1 - x, S - j));
          issue_chunk(i, x, nvalid, 1);
          ex[i] = x;
          en[i] = nvalid;
          nearly = i + 1;
          x += nvalid;
          j += nvalid;
          if (j == S) {
            j = 0;
            ++b;
          }
        }
      }
    }
    // idx / count come from the selection kernel, the tail pages from the previous step:
    // nothing an earlier kernel writes is read before this wait (but for the settled
    // selection above, which the caller vouches for).  Dependents are released only
    // after it, so when a later step starts its settled gather, every kernel before
    // this one has completed (the selection kernel triggers at entry, and without this
    // order a chain of early triggers could run a later step ahead of it).
    pdl_wait();
    pdl_launch_dependents();
#pragma unroll
    for (int i = 0; i < NS; ++i)
      if (i < nearly) issue_chunk(i, ex[i], en[i], 2);
    issued = nearly;
    stage = nearly % NS;
    phase = static_cast<uint32_t>((nearly / NS) & 1);
    while (x < x1) {
      const int nvalid = min(kKeys, min(x1 - x, S - j));
      if (x + nvalid > res_end) advance_tables();
      bool ok_wait = true;
      if (lane == 0 && issued >= NS) ok_wait = mbar_wait(&empty[stage], phase ^ 1u, p.status);
      if (!__shfl_sync(0xffffffffu, ok_wait, 0)) break;
      issue_chunk(stage, x, nvalid, 0);
      ++issued;
      x += nvalid;
      j += nvalid;
      if (j == S) {
        j = 0;
        ++b;
      }
      if (++stage == NS) {
        stage = 0;
        phase ^= 1u;
      }
    }
    // no copy may still be in flight when the CTA exits, also when a consumer gave up
    // (normally the consumers have already seen every chunk land)
    if (lane == 0)
      for (int c = issued > NS ? issued - NS : 0; c < issued; ++c)
        mbar_wait(&full[c % NS], static_cast<uint32_t>((c / NS) & 1), p.status);
    __syncwarp();
    return;
  }

  // ------------------------------------------------------------------ consumer warp: KV head g
  pdl_wait();  // (the queries are the call's inputs: read once the dependency resolved)
  pdl_launch_dependents();
  const int g = warp;
  const int gid = lane >> 2, tig = lane & 3;
  int b = x0 / S, j = x0 - b * S;
  int stage = 0;
  uint32_t phase = 0;
  bool lost = false;
  for (int x = x0; x < x1;) {
    const int run_x0 = x, run_j0 = j;
    const int seg_end = min(x1, x + (S - j));
    uint32_t qf[D / 16][4];
    load_q_frags<D>(qf, gid < p.G ? p.q + (static_cast<size_t>(b) * p.Hq + g * p.G + gid) * D : nullptr,
                    gid + 8 < p.G ? p.q + (static_cast<size_t>(b) * p.Hq + g * p.G + gid + 8) * D : nullptr, tig);
    RowState<D> st;
    st.init();
    while (x < seg_end && !lost) {
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
      softmax_pv16<D, PACK>(st, s, vaddr, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == NS) {
        stage = 0;
        phase ^= 1u;
      }
      x += nvalid;
      j += nvalid;
    }
    if (lost) x = seg_end;  // (results of a lost wait are unspecified; the status says so)
    if constexpr (PACK) fold_packed<D>(st);
    st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], 1);
    st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], 2);
    st.l[1] += __shfl_xor_sync(0xffffffffu, st.l[1], 1);
    st.l[1] += __shfl_xor_sync(0xffffffffu, st.l[1], 2);
    const bool complete = run_j0 == 0 && seg_end - run_x0 == S;  // this CTA holds every entry of b
    const size_t id = static_cast<size_t>(blockIdx.x) + b;       // (unique per (CTA, sequence) run)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int jh = gid + half * 8;
      if (jh < p.G) {
        const int h = g * p.G + jh;
        if (complete) {
          const float inv = st.l[half] > 0.f ? 1.f / st.l[half] : 0.f;
          __nv_bfloat16* o = p.out + (static_cast<size_t>(b) * p.Hq + h) * D;
#pragma unroll
          for (int dn = 0; dn < D / 8; ++dn)
            *reinterpret_cast<__nv_bfloat162*>(o + dn * 8 + tig * 2) =
                __floats2bfloat162_rn(st.o[dn][half * 2] * inv, st.o[dn][half * 2 + 1] * inv);
        } else {
          const size_t r = id * p.Hq + h;
#pragma unroll
          for (int dn = 0; dn < D / 8; ++dn)
            *reinterpret_cast<float2*>(p.part_o + r * D + dn * 8 + tig * 2) =
                make_float2(st.o[dn][half * 2], st.o[dn][half * 2 + 1]);
          if (tig == 0) *reinterpret_cast<float2*>(p.part_ml + r * 2) = make_float2(st.m[half], st.l[half]);
        }
      }
    }
    if (complete && p.k_new) append_token<D>(p, b, g, lane, 32);
    if (x < x1) {
      j = 0;
      ++b;
    }
  }
}

// Merge of the partials of (query head h, sequence b) = (blockIdx.x, blockIdx.y),
// written by the CTAs cf..cl that hold some of b's entries (row c + b); nothing to do
// when one CTA held all of them.  NW warps (4, 8 or 16, from the partial count): warp w
// loads partials w, w + NW, ... in one round, the CTA agrees on their max and adds the
// warps in a fixed order, then writes the bf16 output.  The CTA of each KV head's first
// query head also appends the current draft token: the draft kernel writes none of
// what that append reads (the token's row, the sequence's offsets), and every kernel
// before the draft kernel completed before it released this one, so those loads are
// issued before the dependency wait and leave the merge's critical path.
template <int D, int NW>
__global__ void __launch_bounds__(NW * 32) draft_combine_kernel(const DraftParams p) {
  constexpr int PER = D / 32;
  __shared__ float red[NW][D];
  __shared__ float redl[NW], redm[NW];
  const int h = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float NEG = neg_inf();
  const int S = p.slots;
  const int64_t E = static_cast<int64_t>(p.B) * S;
  const SeqSpan sp = seq_span(b, S, E, p.nctas);
  const int nseg = sp.cl - sp.cf + 1;
  // the append (first query head of a KV head): the token's row and its slot, early
  const bool app = p.k_new && h % p.G == 0 && nseg > 1 && tid < D / 8;
  uint4 kr = make_uint4(0u, 0u, 0u, 0u), vr = kr;
  int64_t adst = -1;
  if (app) {
    const int g = h / p.G;
    const int ts = p.tail_start[b];
    const int tl = tail_len_of(p, b);
    const size_t src = (static_cast<size_t>(b) * p.Hkv + g) * D;
    kr = reinterpret_cast<const uint4*>(p.k_new + src)[tid];
    vr = reinterpret_cast<const uint4*>(p.v_new + src)[tid];
    if (ts >= 0 && tl >= 1 && tl <= kDraftMaxTail) {
      const int64_t slot = kv_slot<true>(p.seq_offset, p.ptab, p.psize, p.pstride, p.capacity, b, ts + tl - 1);
      if (slot >= 0) adst = (slot * p.Hkv + g) * D;
    }
  }
  // The next draft step may start its prologue now.  A step with a settled selection
  // reads the selection and gathers selected pages before its dependency wait: no
  // kernel still running writes either (this step's appends go to draft-token slots),
  // and the selection kernel has completed, since every draft kernel releases its
  // dependents only after its own dependency wait.
  pdl_launch_dependents();
  pdl_wait();
  if (nseg == 1) return;  // the one CTA holding b finished it
  auto prow = [&](int si) { return (static_cast<size_t>(sp.cf + si) + b) * p.Hq + h; };
  // ---- one round of loads: lane q holds (max, sum) of partial warp + NW q; the first
  // kCombineRows output rows of the warp's partials go to registers
  float pm = NEG, pl = 0.f;
  {
    const int si = warp + NW * lane;
    if (si < nseg && split_nonempty(sp.cf + si, E, p.nctas)) {  // CTAs without entries wrote no partial
      const float2 v = *reinterpret_cast<const float2*>(p.part_ml + prow(si) * 2);
      pm = v.x;
      pl = v.y;
    }
  }
  // (rows past nseg, or of a CTA without entries, read as zeros: their weight is zero)
  float v[kCombineRows][PER];
#pragma unroll
  for (int q = 0; q < kCombineRows; ++q) {
    const int si = warp + NW * q;
    const bool ok = si < nseg && split_nonempty(sp.cf + si, E, p.nctas);
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
  for (int w = 0; w < NW; ++w) M = fmaxf(M, redm[w]);
  // ---- this warp's weighted sum, partials in order
  const float wt = (pm != NEG) ? ex2(pm - M) : 0.f;
  float l = wt * pl;  // fixed-order butterfly
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
#pragma unroll
  for (int q = 0; q < kCombineRows; ++q) {
    const float wq = __shfl_sync(0xffffffffu, wt, q);
    if (warp + NW * q < nseg) {
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] += wq * v[q][e];
    }
  }
  for (int q = kCombineRows; warp + NW * q < nseg; ++q) {  // rare: more partials a warp
    const float wq = __shfl_sync(0xffffffffu, wt, q);
    if (!split_nonempty(sp.cf + warp + NW * q, E, p.nctas)) continue;  // (warp-uniform)
    const float* src = p.part_o + prow(warp + NW * q) * D + lane * PER;
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
    for (int w = 0; w < NW; ++w) {  // fixed order: deterministic
      a += red[w][tid];
      lt += redl[w];
    }
    p.out[(static_cast<size_t>(b) * p.Hq + h) * D + tid] = __float2bfloat16_rn(lt > 0.f ? a / lt : 0.f);
  }
  if (app && adst >= 0) {
    reinterpret_cast<uint4*>(p.K + adst)[tid] = kr;
    reinterpret_cast<uint4*>(p.V + adst)[tid] = vr;
  }
}

template <int D, int MAXW, bool PACK, int NS>
cudaError_t launch_draft_t(const DraftParams& p, cudaStream_t stream, bool pdl) {
  const size_t smem = draft_smem_bytes(D, p.Hkv, NS);
  cudaError_t e = ensure_smem<draft_kernel<D, MAXW, PACK, NS>>(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nctas);
  cfg.blockDim = dim3((p.Hkv + 2) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  if ((e = cudaLaunchKernelEx(&cfg, draft_kernel<D, MAXW, PACK, NS>, p)) != cudaSuccess) return e;
  const int nw = draft_combine_warps(p.B, p.slots, p.nctas);
  if (nw == 0) return cudaSuccess;  // every sequence was finished by the CTA holding it
  cudaLaunchConfig_t cfg2 = {};
  cfg2.gridDim = dim3(p.Hq, p.B);
  cfg2.blockDim = dim3(nw * 32);
  cfg2.stream = stream;
  cfg2.attrs = at;
  cfg2.numAttrs = 1;
  if (nw == 4) return cudaLaunchKernelEx(&cfg2, draft_combine_kernel<D, 4>, p);
  if (nw == 8) return cudaLaunchKernelEx(&cfg2, draft_combine_kernel<D, 8>, p);
  return cudaLaunchKernelEx(&cfg2, draft_combine_kernel<D, 16>, p);
}

}  // namespace

size_t draft_smem_bytes(int D, int Hkv, int nstage) {
  return static_cast<size_t>(DLayout(Hkv, D, nstage).total) + 128;
}

// Three stages pay off when a CTA has three chunks or more to stream (more bytes in
// flight, and with a settled selection all three requested before the dependency wait);
// with one or two chunks a CTA the deeper ring only lengthens the set-up.
int draft_stages(int D, int Hkv, int B, int slots, int nctas, size_t smem_optin) {
  const int64_t per_cta = (static_cast<int64_t>(B) * slots + nctas - 1) / nctas;
  if (per_cta > 2 * kKeys && draft_smem_bytes(D, Hkv, kMaxStages) <= smem_optin) return kMaxStages;
  return kMinStages;
}

// CTAs of a draft step.  A step with at least three chunks for every SM streams at the
// HBM rate and takes every SM (each one's copies in flight count).  A smaller step is
// bound by latency: it takes about 60% of the SMs, with at least two chunks a CTA, so
// that the next step's CTAs start their set-up and early gather on the SMs this one
// leaves free, and the merge has fewer partials.  (Measured on one-sequence steps of
// 2055 and 4112 entries: 6.7 -> 5.3 us and 8.1 -> 6.8 us against one CTA per SM.)
int draft_grid(int B, int slots, int sms) {
  const int all = sms < 512 ? sms : 512;
  const int64_t e = static_cast<int64_t>(B) * slots;
  if (e >= static_cast<int64_t>(3) * kKeys * all) return all;
  int64_t per = (e * 5 + 3 * all - 1) / (3 * all);  // e / (0.6 all), rounded up
  if (per < 2 * kKeys) per = 2 * kKeys;
  per = (per + kKeys - 1) / kKeys * kKeys;  // whole chunks
  const int64_t n = (e + per - 1) / per;
  return n < 1 ? 1 : (n > all ? all : static_cast<int>(n));
}

int draft_combine_warps(int B, int slots, int nctas) {
  const int64_t E = static_cast<int64_t>(B) * slots;
  int nseg_max = 0;
  for (int b = 0; b < B; ++b) {
    const SeqSpan sp = seq_span(b, slots, E, nctas);
    nseg_max = max(nseg_max, sp.cl - sp.cf + 1);
  }
  if (nseg_max <= 1) return 0;
  if (nseg_max <= 4 * kCombineRows) return 4;
  if (nseg_max <= 8 * kCombineRows) return 8;
  return 16;
}

cudaError_t launch_draft(const DraftParams& p, cudaStream_t stream, bool pdl) {
  const bool pack = p.G <= 8, deep = p.nstage == 3;
#define VG_DRAFT_FORMS(D_, W_)                                                          \
  return pack ? (deep ? launch_draft_t<D_, W_, true, 3>(p, stream, pdl)                  \
                      : launch_draft_t<D_, W_, true, 2>(p, stream, pdl))                 \
              : (deep ? launch_draft_t<D_, W_, false, 3>(p, stream, pdl)                 \
                      : launch_draft_t<D_, W_, false, 2>(p, stream, pdl))
  if (p.Hkv <= 8) {
    if (p.D == 64) VG_DRAFT_FORMS(64, 8);
    if (p.D == 128) VG_DRAFT_FORMS(128, 8);
  } else if (p.D == 64) {  // (more than 8 KV heads at d = 128 exceed a 1024-element page)
    VG_DRAFT_FORMS(64, 16);
  }
#undef VG_DRAFT_FORMS
  return cudaErrorInvalidValue;
}

}  // namespace vg
