// gdn_common.cuh - device helpers shared by the GDN kernels (sm_103a).
//
// Warp-level tensor-core fragments (mma.sync m16n8k16) and ldmatrix loads,
// swizzled 16-bit tiles, cp.async, bulk copies and bounded mbarrier waits, and
// the fp32 blocked unit-lower-triangular inverse of the fp32 path's #3 Solve
// ("Empowering Hybrid Attention Models on NPUs", §2.1, Figure 1(b); the UT
// transform (I + A)^-1 of "Exp 2026-07-13 — Linear-Attention Scans on the NPU",
// §1).  The 5th-generation tensor-core and TMA primitives are in gdn_tc.cuh.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

// Optional phase timing (compile with -DGDN_PROFILE): thread 0 of every CTA adds
// the clock64() cycles spent since the previous mark to g_gdn_phase[id].  Off in
// the library build, where the marks compile to nothing.
#ifdef GDN_PROFILE
extern __device__ unsigned long long g_gdn_phase[64];  // defined in gdn_abi.cu; needs -rdc
#define GDN_PHASE_INIT \
  long long gdn_phase_t = clock64(); \
  const long long gdn_phase_start = gdn_phase_t; \
  (void)gdn_phase_start
// cycles since the CTA started, added to g_gdn_phase[id] by thread t only
#define GDN_STAMP(id, t)                                                            \
  do {                                                                             \
    if (threadIdx.x == (t))                                                        \
      atomicAdd(&g_gdn_phase[(id)], (unsigned long long)(clock64() - gdn_phase_start)); \
  } while (0)
#define GDN_PHASE(id)                                                              \
  do {                                                                             \
    if (threadIdx.x == 0) {                                                        \
      const long long now = clock64();                                             \
      atomicAdd(&g_gdn_phase[(id)], (unsigned long long)(now - gdn_phase_t));      \
      gdn_phase_t = now;                                                           \
    }                                                                              \
  } while (0)
#else
#define GDN_PHASE_INIT
#define GDN_STAMP(id, t) \
  do {                   \
  } while (0)
#define GDN_PHASE(id) \
  do {                \
  } while (0)
#endif

namespace gdn {

// Device error word (read by gdn_device_status): a bounded wait gave up, or a KDA
// log-decay lay outside the range the KDA forward is exact for.  The first non-zero
// code written stays until it is read.
// kErrOperandRange: an on-chip fp16 operand (V_new or the state) left fp16's finite range,
// so that call's result is not exact; kErrInput: the input check of an _ex call found a
// gate outside its domain or an unordered cu_seqlens.
enum : unsigned {
  kErrNone = 0u,
  kErrWaitTimeout = 1u,
  kErrGateRange = 2u,
  kErrOperandRange = 3u,
  kErrInput = 4u
};

// Record `code` in the error word unless an earlier code is already there.
__device__ __forceinline__ void record_error(unsigned* err, unsigned code) {
  if (err) atomicCAS(err, kErrNone, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- cp.async (16-byte, zero-fill when src_bytes == 0) ----------------------
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src, bool valid) {
  const uint32_t d = smem_u32(smem_dst);
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(gmem_src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// ---- bulk copies (TMA engine, untiled) and mbarriers --------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// Arrive once and add `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// One test of whether phase `parity` of `bar` has completed.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Wait for phase `parity` of `bar` to complete, giving up after `limit` cycles:
// returns false then, and records kErrWaitTimeout in *err.  The phase is tested once
// before the clock is read, so a completed phase costs one test and no clock read.
__device__ __forceinline__ bool mbar_wait_limit(uint64_t* bar, unsigned parity, unsigned* err,
                                                long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit) {
      record_error(err, kErrWaitTimeout);
      return false;
    }
  }
}
// The kernels' wait: gives up after ~2^31 cycles (about a second).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, unsigned* err) {
  return mbar_wait_limit(bar, parity, err, 1ll << 31);
}
// global -> shared, `bytes` a multiple of 16, both addresses 16-byte aligned;
// completion is counted on `bar` (its transaction count must expect the bytes).
// Programmatic dependent launch: a kernel lets the next launch on its stream (made with
// launch_after) start early; that kernel's griddep_wait() returns once this grid has
// completed and its memory operations are visible.  Both are no-ops otherwise.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, unsigned bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
// Wait until at most N committed bulk stores still read their shared source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;\n" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;\n" ::"n"(N) : "memory");
}
// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy / tensor core) reads.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// ---- swizzled 16-bit tiles ---------------------------------------------------
// Dense row-major tiles whose 16-byte chunks are XOR-permuted so that 8
// consecutive rows read at one column chunk hit 8 different bank groups
// (ldmatrix without padding, and the layout survives a verbatim bulk copy).
//   W = 64 or 128 halves per row: chunk c of row r sits at chunk
//       (c & ~7) | ((c ^ r) & 7)          (XOR inside each 128-byte segment)
//   W = 32 halves per row (64-byte rows): chunk c sits at c ^ ((r >> 1) & 3)
//   W = 16 halves per row (32-byte rows): chunk c sits at c ^ ((r >> 2) & 1)
template <int W>
__device__ __forceinline__ int swz(int r, int col) {
  static_assert(W == 16 || W == 32 || W == 64 || W == 128, "tile width");
  const int c = col >> 3;
  int pc;
  if (W == 16) pc = c ^ ((r >> 2) & 1);
  else if (W == 32) pc = c ^ ((r >> 1) & 3);
  else pc = (c & ~7) | ((c ^ r) & 7);
  return r * W + (pc << 3) + (col & 7);
}

// Blocked 128-byte swizzle for tiles wider than 64 halves: 64-column blocks of
// ROWS rows each, stored one after another, every block laid out as swz<64>.
// This is the tensor cores' 128-byte-swizzled operand layout, for K-major and
// MN-major use alike.
template <int ROWS>
__host__ __device__ __forceinline__ int swzb(int r, int col) {
  return (col >> 6) * (ROWS * 64) + r * 64 + (((((col & 63) >> 3) ^ r) & 7) << 3) + (col & 7);
}

// mbarrier arrive (release), one count.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// Barrier among the first `nthreads` threads of the block (id 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- ldmatrix ---------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

// D = A * B + D, fp16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Fragment loads from swizzled tiles (tile width W halves, see swz): A fragments
// (16x16) of [m][k] tiles, or of tiles stored transposed as [k][m]; pairs of B
// fragments (k16 x n8, n tiles n0 and n0 + 8) of tiles stored as [k][n].
template <int W>
__device__ __forceinline__ void load_a_sw(uint32_t (&a)[4], const __half* base, int m0, int k0,
                                          int lane) {
  ldsm_x4(a[0], a[1], a[2], a[3], base + swz<W>(m0 + (lane & 15), k0 + ((lane >> 4) << 3)));
}
template <int W>
__device__ __forceinline__ void load_a_trans_sw(uint32_t (&a)[4], const __half* base, int m0,
                                                int k0, int lane) {
  const int g = lane >> 3;
  ldsm_x4_t(a[0], a[1], a[2], a[3],
            base + swz<W>(k0 + (lane & 7) + ((g >> 1) << 3), m0 + ((g & 1) << 3)));
}
template <int W>
__device__ __forceinline__ void load_b_kn_sw(uint32_t (&b)[4], const __half* base, int n0, int k0,
                                             int lane) {
  const int g = lane >> 3;
  ldsm_x4_t(b[0], b[1], b[2], b[3],
            base + swz<W>(k0 + (lane & 7) + ((g & 1) << 3), n0 + ((g >> 1) << 3)));
}

// A fragment of a tile stored transposed ([k][m], m contiguous) in the blocked
// layout swzb<ROWS> (ROWS = number of k rows).
template <int ROWS>
__device__ __forceinline__ void load_a_trans_blk(uint32_t (&a)[4], const __half* base, int m0,
                                                 int k0, int lane) {
  const int g = lane >> 3;
  ldsm_x4_t(a[0], a[1], a[2], a[3],
            base + swzb<ROWS>(k0 + (lane & 7) + ((g >> 1) << 3), m0 + ((g & 1) << 3)));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Eight bf16 values at p (16-byte aligned, shared memory) rewritten in place as
// fp16.  Exact for |x| in [2^-14, 65504]; smaller magnitudes keep an absolute
// error below 2^-25.
__device__ __forceinline__ void bf16x8_to_f16x8(void* p) {
  uint4 raw = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
  uint4 out;
  __half2* h = reinterpret_cast<__half2*>(&out);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(b[i]);
    h[i] = __floats2half2_rn(f.x, f.y);
  }
  *reinterpret_cast<uint4*>(p) = out;
}


// Non-zero if either fp16 half of `w` is an infinity or a NaN (exponent field all
// ones): adding 1 to a full 5-bit exponent field carries into the half's sign bit.
__device__ __forceinline__ uint32_t f16_inf_or_nan(uint32_t w) {
  return ((w & 0x7c007c00u) + 0x04000400u) & 0x80008000u;
}

// C fragments of two adjacent n8 tiles -> the A fragment of one k16 step (fp16).
__device__ __forceinline__ void c_to_a(uint32_t (&a)[4], const float (&c0)[4], const float (&c1)[4]) {
  a[0] = pack_f16(c0[0], c0[1]);
  a[1] = pack_f16(c0[2], c0[3]);
  a[2] = pack_f16(c1[0], c1[1]);
  a[3] = pack_f16(c1[2], c1[3]);
}


// Launch `kernel` as a programmatic dependent of the previous work on `stream`: its
// CTAs may become resident before that work completes, and must call griddep_wait()
// before reading anything it wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                         cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace gdn
