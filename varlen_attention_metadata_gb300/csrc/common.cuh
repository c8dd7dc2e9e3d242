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

__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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

// Fill `count` elements of elem_bytes at dst with the low elem_bytes of
// `value` (little-endian), with every thread of the block.  dst must start
// on an element boundary.
__device__ __forceinline__ void block_fill(void* dst_, int64_t count, int elem_bytes, int64_t value) {
  unsigned char* dst = static_cast<unsigned char*>(dst_);
  if (count <= 0) return;
  const int tid = threadIdx.x, nt = blockDim.x;
  const uint64_t v = (uint64_t)value;
  const int64_t bytes = count * elem_bytes;
  const uintptr_t d = reinterpret_cast<uintptr_t>(dst);
  int64_t head = (int64_t)((16 - (d & 15)) & 15);
  if (head > bytes) head = bytes;
  // byte j of the region holds byte (j % elem_bytes) of the element
  for (int64_t i = tid; i < head; i += nt) dst[i] = (unsigned char)(v >> (8 * (int)(i % elem_bytes)));
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint32_t byte = (uint32_t)(v >> (8 * (int)((head + k) % elem_bytes))) & 0xffu;
    w[k >> 2] |= byte << (8 * (k & 3));
  }
  const int4 q = make_int4((int)w[0], (int)w[1], (int)w[2], (int)w[3]);
  const int64_t nvec = (bytes - head) >> 4;
  int4* vd = reinterpret_cast<int4*>(dst + head);
  for (int64_t i = tid; i < nvec; i += nt) st_stream(vd + i, q);
  const int64_t done = head + (nvec << 4);
  for (int64_t j = done + tid; j < bytes; j += nt) dst[j] = (unsigned char)(v >> (8 * (int)(j % elem_bytes)));
}

// Fill `count` bytes with `b` using every thread of the block.
__device__ __forceinline__ void block_fill_bytes(uint8_t* dst, int64_t count, uint8_t b) {
  block_fill(dst, count, 1, b);
}

}  // namespace pseq
