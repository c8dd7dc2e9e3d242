// Internal helpers shared by the libpseq translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pseq.h"

namespace pseq {

// ----------------------------------------------------------------------------
// Host side (runtime.cu)
// ----------------------------------------------------------------------------
pseq_status fail(pseq_status st, const char* fmt, ...);
pseq_status check_launch(const char* what);
void clear_error();
void count_launches(int n);
// Resident CTAs per SM of `kernel` at `threads` and `smem` bytes of dynamic
// shared memory (cached per device).
int occupancy(const void* kernel, int threads, size_t smem);
// Raise `kernel`'s dynamic shared memory limit to `bytes` on the current
// device, once per (device, kernel); safe to call from several host threads.
cudaError_t allow_dynamic_smem(const void* kernel, size_t bytes);
int sm_count();
int64_t wait_limit_ns();
int64_t withhold_tile();

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launch `kernel` with programmatic dependent launch enabled, so its CTAs
// may start while the previous kernel on the stream finishes; the kernel
// must call pdl_wait() before reading what that kernel wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ----------------------------------------------------------------------------
// Device side
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Acquire side of a release/acquire pair whose flag was read with ld_relaxed.
__device__ __forceinline__ void fence_acquire() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Relaxed 64-bit accesses at GPU scope, for self-validating summary words
// that other CTAs poll.
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
// The same on two adjacent words (16-byte aligned): each word is read or
// written whole, the pair is not.
__device__ __forceinline__ void ld_relaxed_v2_u64(const unsigned long long* p, unsigned long long& x,
                                                  unsigned long long& y) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(x), "=l"(y) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_relaxed_v2_u64(unsigned long long* p, unsigned long long x, unsigned long long y) {
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(x), "l"(y) : "memory");
}
// Four adjacent words (32-byte aligned) in one access of 256 bits; each word
// is read or written whole, the four together are not.
__device__ __forceinline__ void ld_relaxed_v4_u64(const unsigned long long* p, unsigned long long& x,
                                                  unsigned long long& y, unsigned long long& z,
                                                  unsigned long long& w) {
  asm volatile("ld.relaxed.gpu.global.v4.u64 {%0, %1, %2, %3}, [%4];"
               : "=l"(x), "=l"(y), "=l"(z), "=l"(w)
               : "l"(p)
               : "memory");
}
__device__ __forceinline__ void st_relaxed_v4_u64(unsigned long long* p, unsigned long long x, unsigned long long y,
                                                  unsigned long long z, unsigned long long w) {
  asm volatile("st.relaxed.gpu.global.v4.u64 [%0], {%1, %2, %3, %4};" ::"l"(p), "l"(x), "l"(y), "l"(z), "l"(w)
               : "memory");
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Wrapping counter of finished CTAs (acq_rel): returns the old value; the
// value after `limit` is 0, so the last of limit+1 arrivals leaves it zero.
__device__ __forceinline__ unsigned inc_acq_rel(unsigned* p, unsigned limit) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(limit) : "memory");
  return old;
}

// 64-bit add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ unsigned long long add_acq_rel_u64(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}

// 64-bit add with release semantics at GPU scope; no value comes back, so
// the issuing thread does not wait for the round trip.
__device__ __forceinline__ void red_release_add_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait until the grid this one depends on (programmatic dependent launch)
// has completed and its writes are visible.  A no-op without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Let the dependent grid be scheduled now (its pdl_wait still waits for us).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// First statement of every kernel of this library.  Every launch carries the
// programmatic-dependent-launch attribute, so a kernel may become resident
// while the previous kernel on the stream is still running: wait until that
// kernel has finished and its writes are visible before touching memory,
// then let the next kernel on the stream be scheduled.  This hides the launch
// latency between back-to-back calls without reordering any memory access.
__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_launch_dependents();
}

__device__ __forceinline__ int4 ld_stream(const int4* p) {
  int4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(int4* p, int4 v) {
  asm volatile("st.global.cs.v4.s32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Copy `bytes` bytes from src to dst with every thread of the block.
// Raw bytes: no element is interpreted.  Uses 16-byte accesses when src and
// dst share their alignment modulo 16, else 8-, 4- or 1-byte accesses.
template <typename V, int UNROLL>
__device__ __forceinline__ void block_copy_vec(unsigned char* dst, const unsigned char* src,
                                               int64_t bytes) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const uintptr_t s = reinterpret_cast<uintptr_t>(src);
  int64_t head = (int64_t)((sizeof(V) - (s & (sizeof(V) - 1))) & (sizeof(V) - 1));
  if (head > bytes) head = bytes;
  for (int64_t i = tid; i < head; i += nt) dst[i] = src[i];
  const int64_t nvec = (bytes - head) / (int64_t)sizeof(V);
  const V* vs = reinterpret_cast<const V*>(src + head);
  V* vd = reinterpret_cast<V*>(dst + head);
  int64_t i = tid;
  const int64_t step = (int64_t)nt * UNROLL;
  for (; i + (int64_t)(UNROLL - 1) * nt < nvec; i += step) {
    V r[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) r[u] = vs[i + (int64_t)u * nt];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) vd[i + (int64_t)u * nt] = r[u];
  }
  for (; i < nvec; i += nt) vd[i] = vs[i];
  const int64_t done = head + nvec * (int64_t)sizeof(V);
  for (int64_t j = done + tid; j < bytes; j += nt) dst[j] = src[j];
}

template <int UNROLL>
__device__ __forceinline__ void block_copy_16(unsigned char* dst, const unsigned char* src,
                                              int64_t bytes) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const uintptr_t s = reinterpret_cast<uintptr_t>(src);
  int64_t head = (int64_t)((16 - (s & 15)) & 15);
  if (head > bytes) head = bytes;
  for (int64_t i = tid; i < head; i += nt) dst[i] = src[i];
  const int64_t nvec = (bytes - head) >> 4;
  const int4* vs = reinterpret_cast<const int4*>(src + head);
  int4* vd = reinterpret_cast<int4*>(dst + head);
  int64_t i = tid;
  const int64_t step = (int64_t)nt * UNROLL;
  for (; i + (int64_t)(UNROLL - 1) * nt < nvec; i += step) {
    int4 r[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) r[u] = ld_stream(vs + i + (int64_t)u * nt);
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) st_stream(vd + i + (int64_t)u * nt, r[u]);
  }
  for (; i < nvec; i += nt) st_stream(vd + i, ld_stream(vs + i));
  const int64_t done = head + (nvec << 4);
  for (int64_t j = done + tid; j < bytes; j += nt) dst[j] = src[j];
}

__device__ __forceinline__ void block_copy(void* dst_, const void* src_, int64_t bytes) {
  unsigned char* dst = static_cast<unsigned char*>(dst_);
  const unsigned char* src = static_cast<const unsigned char*>(src_);
  if (bytes <= 0) return;
  const uintptr_t x = reinterpret_cast<uintptr_t>(dst) ^ reinterpret_cast<uintptr_t>(src);
  if ((x & 15) == 0) block_copy_16<4>(dst, src, bytes);
  else if ((x & 7) == 0) block_copy_vec<uint2, 4>(dst, src, bytes);
  else if ((x & 3) == 0) block_copy_vec<uint32_t, 4>(dst, src, bytes);
  else block_copy_vec<unsigned char, 4>(dst, src, bytes);
}

// Fill `count` elements of EB bytes (1, 2, 4 or 8) at dst with the low EB
// bytes of `value` (little-endian), with every thread of the block.  dst
// must start on an element boundary.  Byte j of the region holds byte
// j mod EB of the element; EB is a power of two, so that is a mask.
template <int EB>
__device__ __forceinline__ void block_fill(void* dst_, int64_t count, int64_t value) {
  static_assert(EB == 1 || EB == 2 || EB == 4 || EB == 8, "element of 1, 2, 4 or 8 bytes");
  unsigned char* dst = static_cast<unsigned char*>(dst_);
  if (count <= 0) return;
  const int tid = threadIdx.x, nt = blockDim.x;
  const uint64_t v = (uint64_t)value;
  const int64_t bytes = count * EB;
  const unsigned head = (unsigned)min((int64_t)((16 - (reinterpret_cast<uintptr_t>(dst) & 15)) & 15), bytes);
  auto byte_at = [&](int64_t j) { return (unsigned char)(v >> (8 * ((unsigned)j & (EB - 1)))); };
  for (unsigned i = tid; i < head; i += nt) dst[i] = byte_at(i);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int k = 0; k < 16; ++k) w[k >> 2] |= (uint32_t)byte_at(head + k) << (8 * (k & 3));
  const int4 q = make_int4((int)w[0], (int)w[1], (int)w[2], (int)w[3]);
  const int64_t nvec = (bytes - head) >> 4;
  int4* vd = reinterpret_cast<int4*>(dst + head);
  for (int64_t i = tid; i < nvec; i += nt) st_stream(vd + i, q);
  const int64_t done = head + (nvec << 4);
  for (int64_t j = done + tid; j < bytes; j += nt) dst[j] = byte_at(j);
}

// Fill `count` bytes with `b` using every thread of the block.
__device__ __forceinline__ void block_fill_bytes(uint8_t* dst, int64_t count, uint8_t b) {
  block_fill<1>(dst, count, b);
}

// ----------------------------------------------------------------------------
// block-wide scans of small tables
// ----------------------------------------------------------------------------
struct Triple {
  int count;
  long long real, padded;
};

__device__ __forceinline__ Triple add(const Triple& a, const Triple& b) {
  return {a.count + b.count, a.real + b.real, a.padded + b.padded};
}

__device__ __forceinline__ Triple shfl_up(const Triple& v, int d) {
  return {__shfl_up_sync(~0u, v.count, d), __shfl_up_sync(~0u, v.real, d), __shfl_up_sync(~0u, v.padded, d)};
}

// Exclusive scan of one Triple per thread over a block of WARPS warps;
// `total` receives the block sum.  `scratch` holds WARPS entries.
template <int WARPS>
__device__ __forceinline__ Triple block_exclusive(Triple x, Triple* scratch, Triple& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Triple inc = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const Triple o = shfl_up(inc, d);
    if (lane >= d) inc = add(o, inc);
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    Triple w = lane < WARPS ? scratch[lane] : Triple{0, 0, 0};
#pragma unroll
    for (int d = 1; d < WARPS; d <<= 1) {
      const Triple o = shfl_up(w, d);
      if (lane >= d) w = add(o, w);
    }
    if (lane < WARPS) scratch[lane] = w;
  }
  __syncthreads();
  Triple ex = shfl_up(inc, 1);
  if (lane == 0) ex = {0, 0, 0};
  if (warp > 0) ex = add(scratch[warp - 1], ex);
  total = scratch[WARPS - 1];
  return ex;
}

// ----------------------------------------------------------------------------
// row-sized loads and stores, table lookups
// ----------------------------------------------------------------------------
__device__ __forceinline__ int4 load_row(const unsigned char* p, int rb) {
  int4 v = make_int4(0, 0, 0, 0);
  switch (rb) {
    case 16: v = __ldg(reinterpret_cast<const int4*>(p)); break;
    case 8: {
      const uint2 t = __ldg(reinterpret_cast<const uint2*>(p));
      v.x = (int)t.x;
      v.y = (int)t.y;
    } break;
    case 4: v.x = __ldg(reinterpret_cast<const int*>(p)); break;
    case 2: v.x = __ldg(reinterpret_cast<const unsigned short*>(p)); break;
    default: v.x = __ldg(p); break;
  }
  return v;
}

__device__ __forceinline__ void store_row(unsigned char* p, const int4& v, int rb) {
  switch (rb) {
    case 16: *reinterpret_cast<int4*>(p) = v; break;
    case 8: *reinterpret_cast<uint2*>(p) = make_uint2((unsigned)v.x, (unsigned)v.y); break;
    case 4: *reinterpret_cast<int*>(p) = v.x; break;
    case 2: *reinterpret_cast<unsigned short*>(p) = (unsigned short)v.x; break;
    default: *p = (unsigned char)v.x; break;
  }
}

// Largest j in [0, cnt) with cup[j] <= r, given cup[0] <= r < cup[cnt].
// It is never a zero-length sequence: cup[j + 1] > r.
__device__ __forceinline__ int seq_of(const int32_t* cup, int cnt, int64_t r) {
  int lo = 0, hi = cnt;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)cup[mid] <= r) lo = mid;
    else hi = mid;
  }
  return lo;
}

// ----------------------------------------------------------------------------
// bulk asynchronous copies (the TMA engine's non-tensor form) and mbarriers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the asynchronous proxy.
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Arrive once and expect `bytes` more from asynchronous copies.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for phase `parity` of an mbarrier for at most limit_ns; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_ns();
  while (!mbar_try_wait(bar, parity))
    if ((int64_t)(global_ns() - start) >= limit_ns) return false;
  return true;
}

// Global -> shared, `bytes` a multiple of 16, both addresses 16-byte aligned;
// completion is reported to `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(smem_dst)),
               "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// Shared -> global in the current bulk group.
__device__ __forceinline__ void bulk_store(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst), "r"(smem_addr(smem_src)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N bulk groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N bulk groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace pseq
