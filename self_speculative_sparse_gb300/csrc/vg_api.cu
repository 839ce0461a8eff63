// Host side of the C ABI declared in include/vg.h: argument validation (before
// any CUDA call, so bad arguments never touch the device), workspace carving,
// TMA descriptor encoding and the launch sequence of each entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "vg.h"
#include "vg_common.cuh"
#include "vg_internal.h"

namespace vg {
namespace {

thread_local std::string g_err;

vg_status fail(vg_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

vg_status cuda_fail(cudaError_t e, const char* what) {
  return fail(VG_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- device info
struct DevInfo {
  bool ok = false;
  int sms = 0;
  size_t smem_optin = 0;
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

vg_status device_info(DevInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(VG_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_dev[dev].ok) {
    int sms = 0, optin = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    g_dev[dev].sms = sms;
    g_dev[dev].smem_optin = static_cast<size_t>(optin);
    g_dev[dev].ok = true;
  }
  *out = g_dev[dev];
  return VG_OK;
}

// ---------------------------------------------------------------- TMA encode
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

vg_status get_encoder(EncodeTiledFn* fn) {
  static std::once_flag once;
  static EncodeTiledFn f = nullptr;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) f = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!f) return fail(VG_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
  *fn = f;
  return VG_OK;
}

// [capacity][Hkv*D] bf16 viewed as a 2-D tensor; boxes of 64 columns x box_rows rows
// (64 for the slot pool, the page's rows for a paged cache), 128-byte swizzle.
vg_status encode_cache_map(CUtensorMap* map, void* base, int64_t capacity, int Hkv, int D, int box_rows) {
  EncodeTiledFn enc;
  vg_status st = get_encoder(&enc);
  if (st != VG_OK) return st;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(Hkv) * D, static_cast<cuuint64_t>(capacity)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(Hkv) * D * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(VG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return VG_OK;
}

// ---------------------------------------------------------------- shapes
struct Shape {
  int B, Hq, Hkv, G, D, gamma, R, M, Mpad, max_len;
  float scale;
};

vg_status check_dims(const vg_dims* d, Shape* s) {
  if (!d) return fail(VG_ERR_INVALID_ARG, "dims is NULL");
  if (d->B < 1 || d->B > kMaxBatch) return fail(VG_ERR_UNSUPPORTED_SHAPE, "B=%d outside [1, %d]", d->B, kMaxBatch);
  if (d->H_kv < 1 || d->H_kv > 16) return fail(VG_ERR_UNSUPPORTED_SHAPE, "H_kv=%d outside [1, 16]", d->H_kv);
  if (d->H_q < d->H_kv || d->H_q % d->H_kv != 0)
    return fail(VG_ERR_INVALID_ARG, "H_q=%d is not a multiple of H_kv=%d", d->H_q, d->H_kv);
  const int G = d->H_q / d->H_kv;
  if (G > 16) return fail(VG_ERR_UNSUPPORTED_SHAPE, "group size %d > 16", G);
  if (d->d != 64 && d->d != 128) return fail(VG_ERR_UNSUPPORTED_SHAPE, "head dim %d not in {64, 128}", d->d);
  if (d->gamma < 0 || d->gamma > 15) return fail(VG_ERR_UNSUPPORTED_SHAPE, "gamma=%d outside [0, 15]", d->gamma);
  const int R = d->gamma + 1;
  if (G * R > 64) return fail(VG_ERR_UNSUPPORTED_SHAPE, "G*(gamma+1)=%d > 64", G * R);
  if (d->max_len < 0) return fail(VG_ERR_INVALID_ARG, "max_len=%d < 0", d->max_len);
  if (!(d->scale >= 0.f) || !std::isfinite(d->scale)) return fail(VG_ERR_INVALID_ARG, "scale must be finite and >= 0");
  s->B = d->B;
  s->Hq = d->H_q;
  s->Hkv = d->H_kv;
  s->G = G;
  s->D = d->d;
  s->gamma = d->gamma;
  s->R = R;
  s->M = G * R;
  s->Mpad = ((G * R + 15) / 16) * 16;
  s->max_len = d->max_len;
  s->scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt(static_cast<float>(d->d));
  return VG_OK;
}

vg_status check_cache(const vg_kv_cache* c) {
  if (!c) return fail(VG_ERR_INVALID_ARG, "cache is NULL");
  if (!c->K || !c->V) return fail(VG_ERR_INVALID_ARG, "cache K and V must be non-NULL");
  if (!c->page_table && !c->seq_offset) return fail(VG_ERR_INVALID_ARG, "seq_offset must be non-NULL without a page table");
  if (!aligned16(c->K) || !aligned16(c->V) || !aligned16(c->seq_offset) || !aligned16(c->page_table))
    return fail(VG_ERR_INVALID_ARG, "cache pointers must be 16-byte aligned");
  if (c->capacity_slots < 1 || c->capacity_slots > 0x7fffffffLL)
    return fail(VG_ERR_INVALID_ARG, "capacity_slots=%lld outside [1, 2^31)", static_cast<long long>(c->capacity_slots));
  if (c->page_table) {
    if (c->page_size < 1 || c->page_size > (1 << 20) || c->page_size > c->capacity_slots)
      return fail(VG_ERR_INVALID_ARG, "page_size=%d outside [1, min(2^20, capacity_slots)]", c->page_size);
    if (c->pages_per_seq < 1) return fail(VG_ERR_INVALID_ARG, "pages_per_seq=%d < 1", c->pages_per_seq);
  }
  return VG_OK;
}

// The verify pass reads a paged cache as TMA boxes of a page's rows, which keeps each
// box's shared-memory destination on the swizzle pattern's 1024-byte period for pages of
// 8, 16 or 32 tokens or a multiple of 64; the draft step reads any page size.
vg_status check_verify_pages(const vg_kv_cache* c) {
  if (!c->page_table) return VG_OK;
  const int P = c->page_size;
  if (P == 8 || P == 16 || P == 32 || P % 64 == 0) return VG_OK;
  return fail(VG_ERR_UNSUPPORTED_SHAPE, "verify reads pages of 8, 16, 32 or a multiple of 64 tokens (page_size=%d)", P);
}

int verify_box_rows(const vg_kv_cache* c) {
  return c->page_table ? (c->page_size < kVerifyTileKeys ? c->page_size : kVerifyTileKeys) : kVerifyTileKeys;
}

vg_status check_mask(uint32_t mask, int R, const char* name) {
  const uint32_t allowed = (R >= 32) ? 0xffffffffu : ((1u << R) - 1u);
  if (mask & ~allowed) return fail(VG_ERR_INVALID_ARG, "%s=0x%x names a row beyond gamma", name, mask);
  return VG_OK;
}

// ---------------------------------------------------------------- workspace
inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Most CTAs of a draft step (one per SM, up to 512): sizes the draft partials of the
// workspace (draft_grid picks the step's grid, at most this many).
inline int draft_ctas(int sms) { return sms < 512 ? sms : 512; }

struct WsLayout {
  size_t meta = 0, part_o = 0, part_ml = 0, part_s = 0;
  size_t dpart_o = 0, dpart_ml = 0, dend = 0;
  size_t total = 0;
};

// Row stride of the per-KV-head partial scores: 16-byte-aligned rows for vector stores.
inline int score_stride(const Shape& s) { return (s.max_len + 63) & ~63; }

// Workspace: the verify call's scratch; the draft step's partials reuse the same bytes
// (the calls are stream-ordered).
WsLayout ws_layout(const Shape& s, int sms) {
  WsLayout w;
  const size_t segs = static_cast<size_t>(sms) + static_cast<size_t>(s.B) * s.Hkv;
  size_t off = 0;
  w.meta = off;
  off = up256(off + (2 * static_cast<size_t>(s.B) + 1) * 4);
  w.part_o = off;
  off = up256(off + segs * s.Mpad * s.D * 4);
  w.part_ml = off;
  off = up256(off + segs * s.Mpad * 2 * 4);
  w.part_s = off;
  off = up256(off + 2 * static_cast<size_t>(s.B) * s.Hkv * 2 * static_cast<size_t>(score_stride(s)) * 4);
  const size_t verify_total = off;
  const size_t dsegs = static_cast<size_t>(draft_ctas(sms)) + s.B;  // (CTA, sequence) runs of a draft step
  off = 0;
  w.dpart_o = off;
  off = up256(off + dsegs * s.Hq * s.D * 4);
  w.dpart_ml = off;
  off = up256(off + dsegs * s.Hq * 2 * 4);
  w.dend = off;
  w.total = verify_total > w.dend ? verify_total : w.dend;
  return w;
}

vg_status check_ws(const Shape& s, const DevInfo& di, void* ws, size_t ws_bytes, WsLayout* w) {
  *w = ws_layout(s, di.sms);
  if (!ws) return fail(VG_ERR_WORKSPACE, "workspace is NULL (need %zu bytes)", w->total);
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return fail(VG_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < w->total) return fail(VG_ERR_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, w->total);
  return VG_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// ---------------------------------------------------------------- verify
struct VerifyArgs {
  const void *q, *k_new, *v_new;
  const int32_t* prefix_len;
  uint32_t mask0, mask1;
  float *scores0, *scores1;
  int64_t score_stride;
  void* out;
};

vg_status check_verify_args(const Shape& s, const VerifyArgs& a) {
  if (!a.q || !a.prefix_len || !a.out) return fail(VG_ERR_INVALID_ARG, "q, prefix_len and out must be non-NULL");
  if ((a.k_new == nullptr) != (a.v_new == nullptr)) return fail(VG_ERR_INVALID_ARG, "k_new and v_new: both or neither");
  if (!aligned16(a.q) || !aligned16(a.k_new) || !aligned16(a.v_new) || !aligned16(a.prefix_len) || !aligned16(a.out))
    return fail(VG_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  vg_status st = check_mask(a.mask0, s.R, "row_mask0");
  if (st != VG_OK) return st;
  st = check_mask(a.mask1, s.R, "row_mask1");
  if (st != VG_OK) return st;
  if ((a.mask0 != 0) != (a.scores0 != nullptr)) return fail(VG_ERR_INVALID_ARG, "scores0 must be given iff row_mask0 != 0");
  if ((a.mask1 != 0) != (a.scores1 != nullptr)) return fail(VG_ERR_INVALID_ARG, "scores1 must be given iff row_mask1 != 0");
  if ((a.mask0 | a.mask1) && a.score_stride < s.max_len)
    return fail(VG_ERR_INVALID_ARG, "score_stride=%lld < max_len=%d", static_cast<long long>(a.score_stride), s.max_len);
  if (!aligned16(a.scores0) || !aligned16(a.scores1)) return fail(VG_ERR_INVALID_ARG, "scores must be 16-byte aligned");
  return VG_OK;
}

vg_status run_verify(const Shape& s, const vg_kv_cache* c, const VerifyArgs& a, void* ws, const WsLayout& w,
                     const DevInfo& di, int32_t* dev_status, cudaStream_t stream) {
  if (verify_smem_bytes(s.D, s.B) > di.smem_optin)
    return fail(VG_ERR_UNSUPPORTED_SHAPE, "verify needs %zu bytes of shared memory", verify_smem_bytes(s.D, s.B));
  CUtensorMap tmK, tmV;
  vg_status st = encode_cache_map(&tmK, c->K, c->capacity_slots, s.Hkv, s.D, verify_box_rows(c));
  if (st != VG_OK) return st;
  st = encode_cache_map(&tmV, c->V, c->capacity_slots, s.Hkv, s.D, verify_box_rows(c));
  if (st != VG_OK) return st;
  VerifyParams p = {};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k_new = static_cast<const __nv_bfloat16*>(a.k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(a.v_new);
  p.K = static_cast<__nv_bfloat16*>(c->K);
  p.V = static_cast<__nv_bfloat16*>(c->V);
  p.seq_offset = c->seq_offset;
  p.ptab = c->page_table;
  p.psize = c->page_table ? c->page_size : 1;
  p.pstride = c->page_table ? c->pages_per_seq : 0;
  p.box_rows = verify_box_rows(c);
  p.prefix_len = a.prefix_len;
  p.capacity = c->capacity_slots;
  p.B = s.B;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.G = s.G;
  p.R = s.R;
  p.D = s.D;
  p.M = s.M;
  p.Mpad = s.Mpad;
  p.sc_row0 = verify_sc_row0(s.M, 2 * ((a.mask0 ? 1 : 0) + (a.mask1 ? 1 : 0)));
  p.max_len = s.max_len;
  p.scale = s.scale;
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.mask0 = a.mask0;
  p.mask1 = a.mask1;
  p.nctas = di.sms;
  p.meta = at<int32_t>(ws, w.meta);
  p.part_o = at<float>(ws, w.part_o);
  p.part_ml = at<float>(ws, w.part_ml);
  p.part_s = at<float>(ws, w.part_s);
  p.s_stride = score_stride(s);
  p.scores0 = a.scores0;
  p.scores1 = a.scores1;
  p.score_stride = a.score_stride;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.status = dev_status;
  cudaError_t e = launch_verify(p, tmK, tmV, stream);
  if (e != cudaSuccess) return cuda_fail(e, "verify launch");
  return VG_OK;
}

// ---------------------------------------------------------------- top-k
vg_status check_topk_args(const float* scores, int64_t stride, const int32_t* len, int B, int max_len, int k,
                          const int32_t* idx, const int32_t* count) {
  if (!scores || !len || !idx || !count) return fail(VG_ERR_INVALID_ARG, "scores, len, idx and count must be non-NULL");
  if (!aligned16(scores) || !aligned16(len) || !aligned16(idx) || !aligned16(count))
    return fail(VG_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  if (B < 1 || B > kMaxBatch) return fail(VG_ERR_UNSUPPORTED_SHAPE, "B=%d outside [1, %d]", B, kMaxBatch);
  if (max_len < 0 || max_len > kTopkMaxLen)
    return fail(VG_ERR_UNSUPPORTED_SHAPE, "max_len=%d outside [0, %d]", max_len, kTopkMaxLen);
  if (k < 1) return fail(VG_ERR_INVALID_ARG, "k=%d < 1", k);
  if (stride < max_len) return fail(VG_ERR_INVALID_ARG, "score_stride < max_len");
  return VG_OK;
}

vg_status run_topk(const float* scores, int64_t stride, const int32_t* len, int B, int max_len, int k, int32_t* idx,
                   int32_t* count, int32_t* dev_status, cudaStream_t stream, bool pdl) {
  // one CTA per 4096 positions, up to a cluster of 16: the radix passes are
  // latency-bound, so shorter slices per CTA finish sooner
  int C = (max_len + 4095) / 4096;
  C = C < 1 ? 1 : (C > 16 ? 16 : C);
  int per = (max_len + C - 1) / C;
  per = ((per + 3) / 4) * 4;
  if (per < 4) per = 4;
  TopkParams p = {};
  p.scores = scores;
  p.score_stride = stride;
  p.len = len;
  p.B = B;
  p.max_len = max_len;
  p.k = k;
  p.per_cta = per;
  p.idx = idx;
  p.count = count;
  p.status = dev_status;
  cudaError_t e = launch_topk(p, C, stream, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  return VG_OK;
}

// ---------------------------------------------------------------- draft
struct DraftArgs {
  const void *q, *k_new, *v_new;
  const int32_t *idx, *count;
  int k_stride;
  const int32_t *tail_start, *tail_len;
  int tail_len_const;
  void* out;
  bool settled;
};

vg_status check_draft_args(const DraftArgs& a) {
  if (!a.q || !a.idx || !a.count || !a.tail_start || !a.out)
    return fail(VG_ERR_INVALID_ARG, "q, idx, count, tail_start and out must be non-NULL");
  if ((a.k_new == nullptr) != (a.v_new == nullptr)) return fail(VG_ERR_INVALID_ARG, "k_new and v_new: both or neither");
  if (!aligned16(a.q) || !aligned16(a.k_new) || !aligned16(a.v_new) || !aligned16(a.idx) || !aligned16(a.count) ||
      !aligned16(a.tail_start) || !aligned16(a.tail_len) || !aligned16(a.out))
    return fail(VG_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  if (a.k_stride < 1 || a.k_stride > (1 << 24)) return fail(VG_ERR_INVALID_ARG, "k_stride=%d outside [1, 2^24]", a.k_stride);
  return VG_OK;
}

// One token's K and V pages of every KV head are staged whole in shared memory, which
// the draft kernels are built for up to 1024 elements a page (checked on the host,
// before any device query, so an unsupported shape never gets as far as a launch).
vg_status check_draft_page(const Shape& s) {
  if (s.Hkv * s.D > 1024)
    return fail(VG_ERR_UNSUPPORTED_SHAPE, "sparse draft: H_kv * d = %d > 1024 (one token's page is staged whole)",
                s.Hkv * s.D);
  return VG_OK;
}

// Pipeline stages of the draft kernel: two when they fit beside the run partials.
vg_status check_draft_smem(const Shape& s, const DevInfo& di) {
  if (const vg_status st = check_draft_page(s); st != VG_OK) return st;
  if (draft_smem_bytes(s.D, s.Hkv, 2) > di.smem_optin)
    return fail(VG_ERR_UNSUPPORTED_SHAPE, "sparse draft: H_kv * d = %d needs more shared memory than a CTA has",
                s.Hkv * s.D);
  return VG_OK;
}

vg_status run_draft(const Shape& s, const vg_kv_cache* c, const DraftArgs& a, void* ws, const WsLayout& w,
                    const DevInfo& di, int32_t* dev_status, cudaStream_t stream, bool pdl) {
  if (const vg_status st = check_draft_smem(s, di); st != VG_OK) return st;
  DraftParams p = {};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k_new = static_cast<const __nv_bfloat16*>(a.k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(a.v_new);
  p.K = static_cast<__nv_bfloat16*>(c->K);
  p.V = static_cast<__nv_bfloat16*>(c->V);
  p.seq_offset = c->seq_offset;
  p.ptab = c->page_table;
  p.psize = c->page_table ? c->page_size : 1;
  p.pstride = c->page_table ? c->pages_per_seq : 0;
  p.capacity = c->capacity_slots;
  p.idx = a.idx;
  p.count = a.count;
  p.k_stride = a.k_stride;
  p.tail_start = a.tail_start;
  p.tail_len = a.tail_len;
  p.tail_len_const = a.tail_len_const;
  p.slots = a.k_stride + (a.tail_len ? kDraftMaxTail : a.tail_len_const);
  p.B = s.B;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.G = s.G;
  p.D = s.D;
  p.scale = s.scale;
  p.scale_log2 = s.scale * 1.4426950408889634f;
  p.settled = a.settled ? 1 : 0;
  p.nctas = draft_grid(s.B, p.slots, di.sms);
  p.nstage = draft_stages(s.D, s.Hkv, s.B, p.slots, p.nctas, di.smem_optin);
  p.part_o = at<float>(ws, w.dpart_o);
  p.part_ml = at<float>(ws, w.dpart_ml);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.status = dev_status;
  cudaError_t e = launch_draft(p, stream, pdl);
  if (e != cudaSuccess) return cuda_fail(e, "draft launch");
  return VG_OK;
}

// Self-test of the bounded waits (vg_selftest_lost_wait): warp 0 waits, with a limit
// of limit_ns, on an mbarrier that nothing arrives on; warp 1 waits on another with the
// full limit.  The first wait runs out, reports VG_ERR_DEVICE_TIMEOUT and raises the
// CTA's abort flag; the second must then give up at once.  No copy or MMA is tracked
// by either mbarrier, so nothing is in flight when the CTA exits.
__global__ void __launch_bounds__(64) lost_wait_kernel(int32_t* status, unsigned long long limit_ns,
                                                       unsigned long long* elapsed_ns) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const unsigned long long t0 = globaltimer();
  if ((threadIdx.x & 31) == 0) {
    volatile int* ab = &abort_flag;
    if (threadIdx.x == 0)
      mbar_wait_ab(&bars[0], 0, status, ab, limit_ns);
    else
      mbar_wait_ab(&bars[1], 0, status, ab);
  }
  __syncthreads();
  if (threadIdx.x == 0 && elapsed_ns) *elapsed_ns = globaltimer() - t0;
}

}  // namespace
}  // namespace vg

using namespace vg;

namespace vg {
namespace {

// One vg_iteration call, validated: everything its launch sequence needs.
struct IterCall {
  Shape s;
  const vg_kv_cache* cache;
  const vg_iter_inputs* in;
  vg_iter_outputs out;
  int32_t k;
  VerifyArgs va;
  void* ws;
  WsLayout w;
  DevInfo di;
};

vg_status iteration_prepare(const vg_dims* dims, const vg_kv_cache* cache, const vg_iter_inputs* in, int32_t k,
                            uint32_t row_mask0, uint32_t row_mask1, const vg_iter_outputs* out, void* ws,
                            size_t ws_bytes, IterCall* c) {
  vg_status st = check_dims(dims, &c->s);
  if (st != VG_OK) return st;
  const Shape& s = c->s;
  if ((st = check_cache(cache)) != VG_OK) return st;
  if ((st = check_verify_pages(cache)) != VG_OK) return st;
  if (!in || !out) return fail(VG_ERR_INVALID_ARG, "inputs and outputs must be non-NULL");
  if (k < 1) return fail(VG_ERR_INVALID_ARG, "k=%d < 1", k);
  if (row_mask0 == 0) return fail(VG_ERR_INVALID_ARG, "row_mask0 (the selection rows) must be non-zero");
  if (s.max_len > kTopkMaxLen) return fail(VG_ERR_UNSUPPORTED_SHAPE, "max_len=%d > %d", s.max_len, kTopkMaxLen);
  c->va = VerifyArgs{in->q_verify, in->k_verify, in->v_verify, in->prefix_len, row_mask0, row_mask1,
                     out->scores0,  out->scores1,  out->score_stride, out->out_verify};
  if ((st = check_verify_args(s, c->va)) != VG_OK) return st;
  if (!out->idx || !out->count || !aligned16(out->idx) || !aligned16(out->count))
    return fail(VG_ERR_INVALID_ARG, "idx and count must be non-NULL and 16-byte aligned");
  if ((out->idx1 == nullptr) != (out->count1 == nullptr)) return fail(VG_ERR_INVALID_ARG, "idx1 and count1: both or neither");
  if (out->idx1 && (!out->scores1 || !aligned16(out->idx1) || !aligned16(out->count1)))
    return fail(VG_ERR_INVALID_ARG, "idx1 needs scores1 and 16-byte aligned idx1/count1");
  if (s.gamma > 0) {
    DraftArgs da{in->q_draft, in->k_draft, in->v_draft, out->idx, out->count, k, in->prefix_len, nullptr, 1,
                 out->out_draft, false};
    if (!in->k_draft || !in->v_draft) return fail(VG_ERR_INVALID_ARG, "k_draft and v_draft must be non-NULL");
    if ((st = check_draft_args(da)) != VG_OK) return st;
    if ((st = check_draft_page(s)) != VG_OK) return st;
  }
  if ((st = device_info(&c->di)) != VG_OK) return st;
  // (checked here, not first in the draft launches: an error must leave nothing enqueued)
  if (s.gamma > 0 && (st = check_draft_smem(s, c->di)) != VG_OK) return st;
  if ((st = check_ws(s, c->di, ws, ws_bytes, &c->w)) != VG_OK) return st;
  c->cache = cache;
  c->in = in;
  c->out = *out;
  c->k = k;
  c->ws = ws;
  return VG_OK;
}

// The launch sequence: verify (kernel + combine), the selection(s), gamma draft steps.
vg_status iteration_enqueue(const IterCall& c, int32_t* dev_status, cudaStream_t strm) {
  const Shape& s = c.s;
  const vg_iter_inputs* in = c.in;
  const vg_iter_outputs& out = c.out;
  vg_status st = run_verify(s, c.cache, c.va, c.ws, c.w, c.di, dev_status, strm);
  if (st != VG_OK) return st;
  if ((st = run_topk(out.scores0, out.score_stride, in->prefix_len, s.B, s.max_len, c.k, out.idx, out.count,
                     dev_status, strm, true)) != VG_OK)
    return st;
  if (out.idx1 && (st = run_topk(out.scores1, out.score_stride, in->prefix_len, s.B, s.max_len, c.k, out.idx1,
                                 out.count1, dev_status, strm, true)) != VG_OK)
    return st;
  const size_t qstep = static_cast<size_t>(s.B) * s.Hq * s.D * 2;
  const size_t kvstep = static_cast<size_t>(s.B) * s.Hkv * s.D * 2;
  for (int step = 0; step < s.gamma; ++step) {
    DraftArgs da{static_cast<const char*>(in->q_draft) + step * qstep,
                 static_cast<const char*>(in->k_draft) + step * kvstep,
                 static_cast<const char*>(in->v_draft) + step * kvstep,
                 out.idx,
                 out.count,
                 c.k,
                 in->prefix_len,
                 nullptr,
                 step + 1,
                 static_cast<char*>(out.out_draft) + step * qstep,
                 step > 0};  // (the selection was made before the previous step's kernels)
    if ((st = run_draft(s, c.cache, da, c.ws, c.w, c.di, dev_status, strm, true)) != VG_OK) return st;
  }
  return VG_OK;
}

}  // namespace
}  // namespace vg

// A captured vg_iteration: the launch sequence of one argument set, as a CUDA graph.
struct vg_iteration_plan {
  int device;
  cudaGraphExec_t exec;
};


extern "C" {

int32_t vg_version(void) { return 100; }

vg_status vg_selftest_lost_wait(uint32_t limit_us, int32_t* dev_status, uint64_t* elapsed_ns, void* stream) {
  g_err.clear();
  if (limit_us < 1 || limit_us > 1000000) return fail(VG_ERR_INVALID_ARG, "limit_us=%u outside [1, 1000000]", limit_us);
  if (!dev_status) return fail(VG_ERR_INVALID_ARG, "dev_status must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(dev_status) & 3u) != 0 || (reinterpret_cast<uintptr_t>(elapsed_ns) & 7u) != 0)
    return fail(VG_ERR_INVALID_ARG, "dev_status must be 4-byte and elapsed_ns 8-byte aligned");
  lost_wait_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(
      dev_status, static_cast<unsigned long long>(limit_us) * 1000ull, reinterpret_cast<unsigned long long*>(elapsed_ns));
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return VG_OK;
}

const char* vg_last_error(void) { return g_err.c_str(); }

int32_t vg_sparse_draft_launches(const vg_dims* dims, int32_t k_stride, int32_t tail_len_max) {
  g_err.clear();
  Shape s;
  if (check_dims(dims, &s) != VG_OK) return 0;
  if (k_stride < 1 || k_stride > (1 << 24) || tail_len_max < 0 || tail_len_max > kDraftMaxTail) {
    fail(VG_ERR_INVALID_ARG, "k_stride=%d or tail_len_max=%d out of range", k_stride, tail_len_max);
    return 0;
  }
  if (check_draft_page(s) != VG_OK) return 0;
  DevInfo di;
  if (device_info(&di) != VG_OK) return 0;
  if (check_draft_smem(s, di) != VG_OK) return 0;
  const int slots = k_stride + (tail_len_max ? tail_len_max : kDraftMaxTail);
  return draft_combine_warps(s.B, slots, draft_grid(s.B, slots, di.sms)) > 0 ? 2 : 1;
}

size_t vg_workspace_size(const vg_dims* dims, int32_t k) {
  Shape s;
  if (check_dims(dims, &s) != VG_OK) return 0;
  if (k < 1) {
    fail(VG_ERR_INVALID_ARG, "k=%d < 1", k);
    return 0;
  }
  DevInfo di;
  if (device_info(&di) != VG_OK) return 0;
  g_err.clear();
  return ws_layout(s, di.sms).total;
}

vg_status vg_verify_attn(const vg_dims* dims, const vg_kv_cache* cache, const void* q, const void* k_new,
                         const void* v_new, const int32_t* prefix_len, uint32_t row_mask0, uint32_t row_mask1,
                         float* scores0, float* scores1, int64_t score_stride, void* out, void* ws, size_t ws_bytes,
                         int32_t* dev_status, void* stream) {
  g_err.clear();
  Shape s;
  vg_status st = check_dims(dims, &s);
  if (st != VG_OK) return st;
  if ((st = check_cache(cache)) != VG_OK) return st;
  if ((st = check_verify_pages(cache)) != VG_OK) return st;
  VerifyArgs a{q, k_new, v_new, prefix_len, row_mask0, row_mask1, scores0, scores1, score_stride, out};
  if ((st = check_verify_args(s, a)) != VG_OK) return st;
  if ((reinterpret_cast<uintptr_t>(dev_status) & 3u) != 0) return fail(VG_ERR_INVALID_ARG, "dev_status must be 4-byte aligned");
  DevInfo di;
  if ((st = device_info(&di)) != VG_OK) return st;
  WsLayout w;
  if ((st = check_ws(s, di, ws, ws_bytes, &w)) != VG_OK) return st;
  return run_verify(s, cache, a, ws, w, di, dev_status, static_cast<cudaStream_t>(stream));
}

vg_status vg_topk_select(const float* scores, int64_t score_stride, const int32_t* len, int32_t B, int32_t max_len,
                         int32_t k, int32_t* idx, int32_t* count, void* ws, size_t ws_bytes, int32_t* dev_status,
                         void* stream) {
  (void)ws;
  (void)ws_bytes;
  g_err.clear();
  vg_status st = check_topk_args(scores, score_stride, len, B, max_len, k, idx, count);
  if (st != VG_OK) return st;
  return run_topk(scores, score_stride, len, B, max_len, k, idx, count, dev_status,
                  static_cast<cudaStream_t>(stream), true);
}

size_t vg_accept_workspace_size(int32_t B, int32_t gamma, int32_t V) {
  g_err.clear();
  if (B < 1 || B > kMaxBatch || gamma < 0 || gamma > 15 || V < 1 || V > kMaxAcceptTiles * 4096) {
    fail(VG_ERR_UNSUPPORTED_SHAPE, "B=%d, gamma=%d or V=%d out of range", B, gamma, V);
    return 0;
  }
  const size_t rows = static_cast<size_t>(B) * (2 * gamma + 1);
  // per-chunk statistics, per-sequence decision records (32 B), per-tile sums
  return up256(rows * accept_chunks(V) * 16) + up256(static_cast<size_t>(B) * 32) +
         up256(static_cast<size_t>(B) * 2 * accept_tiles(V) * 4);
}

vg_status vg_accept(int32_t B, int32_t gamma, int32_t V, const float* p_logits, const float* q_logits,
                    const int32_t* draft_tokens, const float* u_accept, const float* u_resample, uint32_t mode,
                    int32_t* n_accept, int32_t* next_token, int32_t* advance_len, void* ws, size_t ws_bytes,
                    int32_t* dev_status, void* stream) {
  g_err.clear();
  if (mode != VG_ACCEPT_GREEDY && mode != VG_ACCEPT_SAMPLE) return fail(VG_ERR_INVALID_ARG, "mode=%u unknown", mode);
  const bool sample = mode == VG_ACCEPT_SAMPLE;
  const size_t need = vg_accept_workspace_size(B, gamma, V);
  if (need == 0) return VG_ERR_UNSUPPORTED_SHAPE;
  if (!p_logits || !n_accept || !next_token || (gamma > 0 && !draft_tokens))
    return fail(VG_ERR_INVALID_ARG, "p_logits, draft_tokens, n_accept and next_token must be non-NULL");
  if (sample && (!u_resample || (gamma > 0 && (!q_logits || !u_accept))))
    return fail(VG_ERR_INVALID_ARG, "sampling needs q_logits, u_accept and u_resample");
  if (!aligned16(p_logits) || !aligned16(q_logits) || !aligned16(draft_tokens) || !aligned16(u_accept) ||
      !aligned16(u_resample) || !aligned16(n_accept) || !aligned16(next_token) || !aligned16(advance_len))
    return fail(VG_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(dev_status) & 3u) != 0) return fail(VG_ERR_INVALID_ARG, "dev_status must be 4-byte aligned");
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < need)
    return fail(VG_ERR_WORKSPACE, "workspace must be 256-byte aligned and hold %zu bytes", need);
  AcceptParams p = {};
  p.p_logits = p_logits;
  p.q_logits = q_logits;
  p.draft = draft_tokens;
  p.u = u_accept;
  p.u_res = u_resample;
  p.B = B;
  p.gamma = gamma;
  p.V = V;
  p.nchunk = accept_chunks(V);
  p.sample = sample ? 1 : 0;
  const size_t rows = static_cast<size_t>(B) * (2 * gamma + 1);
  const size_t off_dec = up256(rows * accept_chunks(V) * 16);
  p.stats = static_cast<float*>(ws);
  p.dec = reinterpret_cast<float*>(static_cast<char*>(ws) + off_dec);
  p.tiles = reinterpret_cast<float*>(static_cast<char*>(ws) + off_dec + up256(static_cast<size_t>(B) * 32));
  p.ntiles = accept_tiles(V);
  p.n_accept = n_accept;
  p.next_token = next_token;
  p.advance_len = advance_len;
  p.status = dev_status;
  const cudaError_t e = launch_accept(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "accept launch");
  return VG_OK;
}

vg_status vg_window_select(const int32_t* len, int32_t B, int32_t max_len, int32_t k, int32_t* idx, int32_t* count,
                           int32_t* dev_status, void* stream) {
  g_err.clear();
  if (!len || !idx || !count) return fail(VG_ERR_INVALID_ARG, "len, idx and count must be non-NULL");
  if (!aligned16(len) || !aligned16(idx) || !aligned16(count))
    return fail(VG_ERR_INVALID_ARG, "device pointers must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(dev_status) & 3u) != 0) return fail(VG_ERR_INVALID_ARG, "dev_status must be 4-byte aligned");
  if (B < 1 || B > kMaxBatch) return fail(VG_ERR_UNSUPPORTED_SHAPE, "B=%d outside [1, %d]", B, kMaxBatch);
  if (max_len < 0) return fail(VG_ERR_INVALID_ARG, "max_len=%d < 0", max_len);
  if (k < 1 || k > (1 << 24)) return fail(VG_ERR_INVALID_ARG, "k=%d outside [1, 2^24]", k);
  const cudaError_t e = launch_window(len, B, max_len, k, idx, count, dev_status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "window selection launch");
  return VG_OK;
}

vg_status vg_sparse_draft_attn(const vg_dims* dims, const vg_kv_cache* cache, const void* q, const void* k_new,
                               const void* v_new, const int32_t* idx, const int32_t* count, int32_t k_stride,
                               const int32_t* tail_start, const int32_t* tail_len, uint32_t flags, void* out,
                               void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  g_err.clear();
  Shape s;
  vg_status st = check_dims(dims, &s);
  if (st != VG_OK) return st;
  if ((st = check_cache(cache)) != VG_OK) return st;
  if (!tail_len) return fail(VG_ERR_INVALID_ARG, "tail_len must be non-NULL");
  if (flags & ~VG_DRAFT_SELECTION_SETTLED) return fail(VG_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  DraftArgs a{q, k_new, v_new, idx, count, k_stride, tail_start, tail_len, 0, out,
              (flags & VG_DRAFT_SELECTION_SETTLED) != 0};
  if ((st = check_draft_args(a)) != VG_OK) return st;
  if ((st = check_draft_page(s)) != VG_OK) return st;
  DevInfo di;
  if ((st = device_info(&di)) != VG_OK) return st;
  WsLayout w;
  if ((st = check_ws(s, di, ws, ws_bytes, &w)) != VG_OK) return st;
  return run_draft(s, cache, a, ws, w, di, dev_status, static_cast<cudaStream_t>(stream), true);
}

vg_status vg_iteration(const vg_dims* dims, const vg_kv_cache* cache, const vg_iter_inputs* in, int32_t k,
                       uint32_t row_mask0, uint32_t row_mask1, vg_iter_outputs* out, void* ws, size_t ws_bytes,
                       int32_t* dev_status, void* stream) {
  g_err.clear();
  IterCall c;
  vg_status st = iteration_prepare(dims, cache, in, k, row_mask0, row_mask1, out, ws, ws_bytes, &c);
  if (st != VG_OK) return st;
  return iteration_enqueue(c, dev_status, static_cast<cudaStream_t>(stream));
}

vg_status vg_iteration_plan_create(const vg_dims* dims, const vg_kv_cache* cache, const vg_iter_inputs* in,
                                   int32_t k, uint32_t row_mask0, uint32_t row_mask1, const vg_iter_outputs* out,
                                   void* ws, size_t ws_bytes, int32_t* dev_status, vg_iteration_plan** plan) {
  g_err.clear();
  if (!plan) return fail(VG_ERR_INVALID_ARG, "plan is NULL");
  *plan = nullptr;
  IterCall c;
  vg_status st = iteration_prepare(dims, cache, in, k, row_mask0, row_mask1, out, ws, ws_bytes, &c);
  if (st != VG_OK) return st;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  // The sequence is recorded on a private stream.  Relaxed mode: the first launch of a
  // kernel may raise its shared-memory limit (cudaFuncSetAttribute), which enqueues
  // nothing and needs no capture.
  cudaStream_t cs = nullptr;
  if ((e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking)) != cudaSuccess)
    return cuda_fail(e, "cudaStreamCreateWithFlags");
  if ((e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed)) != cudaSuccess) {
    cudaStreamDestroy(cs);
    return cuda_fail(e, "cudaStreamBeginCapture");
  }
  st = iteration_enqueue(c, dev_status, cs);
  std::string enqueue_err = g_err;
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(cs, &graph);
  cudaStreamDestroy(cs);
  if (st != VG_OK || e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    if (st != VG_OK) {
      g_err = enqueue_err;
      return st;
    }
    return cuda_fail(e, "cudaStreamEndCapture");
  }
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphInstantiate");
  vg_iteration_plan* p = new (std::nothrow) vg_iteration_plan{dev, exec};
  if (!p) {
    cudaGraphExecDestroy(exec);
    return fail(VG_ERR_CUDA, "out of host memory for the plan");
  }
  *plan = p;
  return VG_OK;
}

vg_status vg_iteration_plan_launch(const vg_iteration_plan* plan, void* stream) {
  g_err.clear();
  if (!plan) return fail(VG_ERR_INVALID_ARG, "plan is NULL");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != plan->device)
    return fail(VG_ERR_INVALID_ARG, "plan was made on device %d, the current device is %d", plan->device, dev);
  e = cudaGraphLaunch(plan->exec, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch");
  return VG_OK;
}

vg_status vg_iteration_plan_destroy(vg_iteration_plan* plan) {
  g_err.clear();
  if (!plan) return VG_OK;
  const cudaError_t e = cudaGraphExecDestroy(plan->exec);
  delete plan;
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphExecDestroy");
  return VG_OK;
}

// ---------------------------------------------------------------- no-allocation draft step
// Some callers cannot give this library device memory: a host that runs the
// draft step from a context where it must not call cudaMalloc (the call can
// synchronise the device and stall other streams), or one that has no workspace
// to hand over.  vg_sparse_draft_attn_noalloc serves them from a fixed scratch
// area that lives in the library itself.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB per device, held until the process exits
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {nullptr};

// Device address of g_noalloc_scratch on the current device (the host-side
// symbol is only a stand-in).  Looked up once per device, on that device.
vg_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(VG_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return VG_OK;
}

}  // namespace

vg_status vg_sparse_draft_attn_noalloc(const vg_dims* dims, const vg_kv_cache* cache, const void* q,
                                       const void* k_new, const void* v_new, const int32_t* idx,
                                       const int32_t* count, int32_t k_stride, const int32_t* tail_start,
                                       const int32_t* tail_len, void* out, int32_t* dev_status, void* stream) {
  g_err.clear();
  Shape s;
  vg_status st = check_dims(dims, &s);
  if (st != VG_OK) return st;
  if ((st = check_cache(cache)) != VG_OK) return st;
  if (!tail_len) return fail(VG_ERR_INVALID_ARG, "tail_len must be non-NULL");
  DraftArgs a{q, k_new, v_new, idx, count, k_stride, tail_start, tail_len, 0, out, false};
  if ((st = check_draft_args(a)) != VG_OK) return st;
  if ((st = check_draft_page(s)) != VG_OK) return st;
  DevInfo di;
  if ((st = device_info(&di)) != VG_OK) return st;
  const WsLayout w = ws_layout(s, di.sms);
  const size_t need = w.dend;  // end of the draft step's scratch
  if (need > kNoAllocScratchBytes)
    return fail(VG_ERR_WORKSPACE,
                "no-allocation draft step needs %zu bytes of scratch for these dims; its built-in area holds %zu "
                "(use vg_sparse_draft_attn with a workspace)",
                need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != VG_OK) return st;
  return run_draft(s, cache, a, scratch, w, di, dev_status, static_cast<cudaStream_t>(stream), true);
}

}  // extern "C"
