// Device helpers shared by the Vegas kernels: inline PTX for mbarriers, TMA /
// bulk copies, ldmatrix, bf16 tensor-core MMA, PDL, bounded waits and status
// reporting.  Written for sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "vg.h"

namespace vg {

// A wait that has not completed after this long is treated as lost.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// First device-side error wins; the caller zeroes *status before the call.
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of `bar` to complete, for at most kWaitLimitNs.
// Returns false (and reports VG_ERR_DEVICE_TIMEOUT) if the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && globaltimer() - t0 > kWaitLimitNs) {
      report(status, VG_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

// As mbar_wait, for kernels whose roles wait on one another: the first wait that runs
// out raises the CTA's abort flag (shared memory), and every wait of the CTA then
// gives up at once, so a broken wait costs one limit, not one per remaining wait.
__device__ __forceinline__ bool mbar_wait_ab(uint64_t* bar, uint32_t parity, int32_t* status, volatile int* abort,
                                             unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > limit_ns) {
        *abort = 1;
        report(status, VG_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

// ------------------------------------------------------------------ bulk copies
// 2-D tiled TMA load of box (x, y) into shared memory; completion is counted on bar.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// Orders this thread's earlier generic-proxy shared-memory accesses before its later
// async-proxy (TMA / bulk copy) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Contiguous global -> shared copy by the TMA engine (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ tensor cores
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Two fp32 -> packed bf16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// Two fp32 -> their bf16 high parts (hi, packed) and the bf16 rounding of what the high
// parts leave out (lo, packed): a + b = hi + lo to about 2^-17 relative.
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(a, b);
  lo = pack_bf16(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xffff0000u));
}
// acc + lo + hi for a packed bf16 pair, each half widened exactly to fp32 (the
// mixed-precision add of sm_100 and later: one instruction per element).
__device__ __forceinline__ float add_bf16x2_f32(uint32_t w, float acc) {
  float d;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tadd.rn.f32.bf16 %0, lo, %2;\n\tadd.rn.f32.bf16 %0, hi, %0;\n\t}"
      : "=f"(d)
      : "r"(w), "f"(acc));
  return d;
}
// 2^x on the special-function unit (MUFU.EX2), flushing subnormal results.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ tcgen05 (5th-gen tensor cores)
// Shared-memory matrix descriptor of a 128-byte-swizzled operand (the layout a TMA
// box with a 128-byte inner extent and CU_TENSOR_MAP_SWIZZLE_128B produces: rows of
// 128 bytes, 16-byte chunk c of row r stored at chunk c ^ (r & 7), 8-row groups of
// 1024 bytes).  addr must lie in a 1024-byte-aligned tile.  For a K-major operand
// sbo is the stride between 8-row groups and lbo is unused; for an MN-major operand
// lbo is the stride between 64-element column blocks and sbo the stride between
// 8-row groups along K.  Bits 46-47 hold the descriptor version (1), bits 61-63 the
// layout (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of a dense bf16 x bf16 -> fp32 MMA of shape M x N (K = 16);
// a_mn / b_mn select an MN-major (instead of K-major) A / B operand.
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread; accumulate selects D += .
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on bar when every earlier tcgen05 operation of this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// Whole-warp tensor-memory allocation; the base address is written to *slot.
__device__ __forceinline__ void tc_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// N consecutive fp32 columns of this thread's tensor-memory lane, loaded and waited
// for in one statement (so no use of the registers can be scheduled before the
// wait).  Warp-collective; warp w reaches lanes 32 (w % 4) .. 32 (w % 4) + 31.
__device__ __forceinline__ void tc_ld32_sync(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ sync
__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Programmatic dependent launch: let the next kernel in the stream start its
// prologue now / wait until the previous kernel's results are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Physical slot of logical token i of sequence b in the KV cache, or -1 when it falls
// outside the cache.  Without a page table the slot pool holds sequence b from slot
// seq_offset[b] on; with one, token i lives at row i mod page_size of physical page
// page_table[b][i / page_size] (pages of page_size slots: page p spans slots
// p * page_size .. p * page_size + page_size - 1).  L2_ONLY loads bypass L1 (the draft
// step resolves slots before its dependency wait when its selection is settled, and must
// see what kernels that completed earlier wrote).
template <bool L2_ONLY = false>
__device__ __forceinline__ int64_t kv_slot(const int64_t* seq_offset, const int32_t* ptab, int psize, int pstride,
                                           int64_t capacity, int b, int64_t i) {
  if (i < 0) return -1;
  if (ptab == nullptr) {
    const int64_t s = (L2_ONLY ? __ldcg(seq_offset + b) : seq_offset[b]) + i;
    return s >= 0 && s < capacity ? s : -1;
  }
  if (i >= static_cast<int64_t>(pstride) * psize) return -1;
  // (32-bit arithmetic: i < 2^31; a shift for the usual power-of-two page sizes)
  const int ii = static_cast<int>(i);
  int pi, row;
  if ((psize & (psize - 1)) == 0) {
    const int sh = __ffs(psize) - 1;
    pi = ii >> sh;
    row = ii & (psize - 1);
  } else {
    pi = ii / psize;
    row = ii - pi * psize;
  }
  const int32_t* e = ptab + static_cast<int64_t>(b) * pstride + pi;
  const int64_t pg = L2_ONLY ? __ldcg(e) : *e;
  return pg >= 0 && (pg + 1) * psize <= capacity ? pg * psize + row : -1;
}

// CTA of a balanced contiguous split of T items over N CTAs that owns item x:
// CTA c owns [floor(c T / N), floor((c+1) T / N)).  (A 64-bit division is a long
// instruction sequence on the GPU: when the products fit in 32 bits, as they do for
// T < 2^22 items over at most 512 CTAs, the division is done in 32 bits.)
__host__ __device__ __forceinline__ int64_t owner_cta(int64_t x, int64_t T, int64_t N) {
  if (T < (int64_t{1} << 22) && N <= 512)
    return static_cast<int64_t>((static_cast<uint32_t>(x + 1) * static_cast<uint32_t>(N) - 1u) / static_cast<uint32_t>(T));
  return ((x + 1) * N - 1) / T;
}
__host__ __device__ __forceinline__ int64_t split_begin(int64_t c, int64_t T, int64_t N) {
  if (T < (int64_t{1} << 22) && N <= 512 && c <= N)
    return static_cast<int64_t>(static_cast<uint32_t>(c) * static_cast<uint32_t>(T) / static_cast<uint32_t>(N));
  return (c * T) / N;
}
// True if CTA c (0 <= c < N) of that split owns at least one item.  Every CTA does when
// T >= N; otherwise (c + 1) * T < N * N, so 32-bit arithmetic is exact (and cheap:
// a 64-bit division is a long instruction sequence, and callers test many CTAs).
__host__ __device__ __forceinline__ bool split_nonempty(int64_t c, int64_t T, int64_t N) {
  if (T >= N) return true;
  const int ci = static_cast<int>(c), ti = static_cast<int>(T), ni = static_cast<int>(N);
  return (ci * ti) / ni < ((ci + 1) * ti) / ni;
}

// Sets a kernel's dynamic shared-memory limit once per device (and again only if a
// larger size is asked for), so repeated launches - and launches under stream
// capture - make no attribute calls.  Host threads may launch concurrently: the
// limit already set is read atomically, and setting a new one (attribute call and
// cache update together) holds the kernel's lock, so the cache never runs ahead of
// the attribute.
template <auto Kernel>
inline cudaError_t ensure_smem(size_t bytes) {
  static std::atomic<int> done[64] = {};  // one table per kernel (the template argument is the kernel itself)
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire) >= static_cast<int>(bytes)) return cudaSuccess;
  std::lock_guard<std::mutex> lk(mu);
  if (done[dev].load(std::memory_order_relaxed) >= static_cast<int>(bytes)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) done[dev].store(static_cast<int>(bytes), std::memory_order_release);
  return e;
}

}  // namespace vg
