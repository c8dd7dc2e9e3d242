// pack_squeeze: the trainer-side squeeze of a padded rectangle into bins.
//
// Follows "Who packs the sequences: the loader, or the trainer?" (NeMo-RL
// #4105 explainer): "Trainer packs" (sources padded to a multiple and laid
// end to end; cu_seqlens from real lengths, cu_seqlens_padded from padded
// lengths) and "Loader packs" (the last padded boundary stretched to the pack
// capacity).
//
// Fused path (up to kFusedMaxMembers members, one launch): a grid of
// (row chunk, bin) CTAs.  Every CTA scans its own bin's members into shared
// memory -- padded lengths, both cumulative sums, the slot where each member
// starts -- and then writes each slot of its chunk once: one thread per slot
// looks its member up in the table and either loads the source token or
// writes pad_value, with the padding mask alongside.  The first chunk of a bin
// writes the bin's cu arrays; CTA (0, 0) also makes one pass over all members
// to fold every bin's checks into the info block.
//
// Two-kernel path (larger inputs): squeeze_meta_kernel gives each bin one
// warp (chunked warp scan); squeeze_copy_kernel (programmatic dependent
// launch) walks the members of its chunk: real tokens are one contiguous
// block copy from the source row, padding slots one block fill.  Every
// output slot is written exactly once.
#include "common.cuh"

namespace pseq {
namespace {

constexpr int kMetaThreads = 256;
constexpr int kMetaWarps = kMetaThreads / 32;
constexpr int kCopyThreads = 512;
constexpr int kFusedThreads = 512;
constexpr int kFusedMaxMembers = 1024;
constexpr int kSlotsPerThread = 4;

struct Workspace {
  int4* bin_stat;    // [num_bins] {status, padded total, largest real, members}
  int32_t* mem_dst;  // [M] slot where the member starts in its bin
  int32_t* mem_real; // [M]
  int32_t* mem_src;  // [M] source row
};

size_t workspace_bytes(int64_t M, int64_t num_bins) {
  return round_up(16 * (size_t)num_bins, 16) + 3 * round_up(4 * (size_t)M, 16);
}

template <typename P>
Workspace carve(P base_, int64_t M, int64_t num_bins) {
  unsigned char* p = (unsigned char*)(base_);
  Workspace w;
  w.bin_stat = reinterpret_cast<int4*>(p);
  p += round_up(16 * (size_t)num_bins, 16);
  w.mem_dst = reinterpret_cast<int32_t*>(p);
  p += round_up(4 * (size_t)M, 16);
  w.mem_real = reinterpret_cast<int32_t*>(p);
  p += round_up(4 * (size_t)M, 16);
  w.mem_src = reinterpret_cast<int32_t*>(p);
  return w;
}

struct MetaArgs {
  const int64_t* real;
  const int32_t* off;
  const int32_t* mem;
  int num_bins, M;
  int64_t N, W, multiple, capacity, width;
  int stretch, check_width;
  int32_t* cu;
  int32_t* cup;
};

__global__ void __launch_bounds__(kMetaThreads) squeeze_meta_kernel(MetaArgs a, Workspace ws) {
  pdl_enter();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x * kMetaWarps + warp;
  if (b >= a.num_bins) return;
  const int lo = __ldg(a.off + b), hi = __ldg(a.off + b + 1);
  const bool bad_offsets = (b == 0 && lo != 0) || (b == a.num_bins - 1 && hi != a.M) || lo < 0 || hi > a.M ||
                           hi <= lo;
  if (bad_offsets) {
    if (lane == 0) ws.bin_stat[b] = make_int4(PSEQ_ERR_VALUE, 0, 0, 0);
    return;
  }
  long long run_real = 0, run_padded = 0;
  int longest = 0;
  bool bad = false;
  for (int base = lo; base < hi; base += 32) {
    const int e = base + lane;
    long long real = 0, padded = 0;
    int src = 0;
    if (e < hi) {
      src = __ldg(a.mem + e);
      if (src < 0 || src >= a.N) {
        bad = true;
      } else {
        real = __ldg(a.real + src);
        if (real < 0 || real > a.W) {
          bad = true;
          real = 0;
        }
      }
      padded = (real + a.multiple - 1) / a.multiple * a.multiple;
      longest = max(longest, (int)real);
    }
    long long ir = real, ip = padded;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const long long r = __shfl_up_sync(~0u, ir, d), q = __shfl_up_sync(~0u, ip, d);
      if (lane >= d) {
        ir += r;
        ip += q;
      }
    }
    if (e < hi) {
      const long long R = run_real + ir - real, Pd = run_padded + ip - padded;
      a.cu[e + b] = (int32_t)R;
      a.cup[e + b] = (int32_t)Pd;
      ws.mem_dst[e] = (int32_t)Pd;
      ws.mem_real[e] = (int32_t)real;
      ws.mem_src[e] = src;
    }
    run_real += __shfl_sync(~0u, ir, 31);
    run_padded += __shfl_sync(~0u, ip, 31);
  }
  bad = __any_sync(~0u, bad);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) longest = max(longest, __shfl_xor_sync(~0u, longest, d));
  if (lane == 0) {
    int status = PSEQ_OK;
    if (bad) status = PSEQ_ERR_VALUE;
    else if (run_padded > a.capacity || (a.check_width && run_padded > a.width)) status = PSEQ_ERR_CAPACITY;
    a.cu[hi + b] = (int32_t)run_real;
    a.cup[hi + b] = a.stretch ? (int32_t)a.capacity : (int32_t)run_padded;
    ws.bin_stat[b] = make_int4(status, (int)min(run_padded, (long long)INT32_MAX), longest, hi - lo);
  }
}

struct CopyArgs {
  const unsigned char* src;
  int64_t W;
  int elem_bytes;
  const int32_t* off;
  int num_bins, M;
  int64_t width, chunk, pad_value;
  unsigned char* out;   // may be NULL (metadata only)
  uint8_t* mask;        // may be NULL
  pseq_info* info;
};

// Largest k in [lo, hi) with dst[k] <= x, given dst[lo] <= x.
__device__ __forceinline__ int warp_find(const int32_t* dst, int lo, int hi, int64_t x) {
  const int lane = threadIdx.x & 31;
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int probe = lo + lane * step;
    const bool ok = probe < hi && (int64_t)__ldcg(dst + probe) <= x;
    const unsigned m = __ballot_sync(~0u, ok);
    lo = lo + (31 - __clz(m)) * step;
    hi = min(lo + step, hi);
  }
  return lo;
}

__global__ void __launch_bounds__(kCopyThreads) squeeze_copy_kernel(CopyArgs c, Workspace ws) {
  __shared__ int s_value, s_capacity, s_longest, s_widest, s_first;
  pdl_enter();
  const int tid = threadIdx.x;
  const int b = blockIdx.y;
  if (blockIdx.x == 0 && b == 0) {
    if (tid == 0) s_value = s_capacity = s_longest = s_widest = 0;
    __syncthreads();
    for (int i = tid; i < c.num_bins; i += kCopyThreads) {
      const int4 st = __ldcg(ws.bin_stat + i);
      if (st.x == PSEQ_ERR_VALUE) s_value = 1;
      if (st.x == PSEQ_ERR_CAPACITY) s_capacity = 1;
      atomicMax(&s_longest, st.z);
      atomicMax(&s_widest, st.y);
    }
    __syncthreads();
    if (tid == 0) {
      const int status = s_value ? PSEQ_ERR_VALUE : (s_capacity ? PSEQ_ERR_CAPACITY : PSEQ_OK);
      *c.info = status == PSEQ_OK ? pseq_info{PSEQ_OK, c.M, s_longest, s_widest} : pseq_info{status, 0, 0, 0};
    }
  }
  if (!c.out || b >= c.num_bins) return;
  const int4 st = __ldcg(ws.bin_stat + b);
  if (st.x != PSEQ_OK) return;
  const int64_t c0 = (int64_t)blockIdx.x * c.chunk;
  const int64_t c1 = min(c0 + c.chunk, c.width);
  if (c0 >= c1) return;
  const int eb = c.elem_bytes;
  const int64_t total = st.y;
  unsigned char* row = c.out + (int64_t)b * c.width * eb;
  uint8_t* mrow = c.mask ? c.mask + (int64_t)b * c.width : nullptr;
  if (c0 < total) {
    const int lo = __ldg(c.off + b), hi = __ldg(c.off + b + 1);
    if (tid < 32) {
      const int k = warp_find(ws.mem_dst, lo, hi, c0);
      if (tid == 0) s_first = k;
    }
    __syncthreads();
    for (int k = s_first; k < hi; ++k) {
      const int64_t s = __ldcg(ws.mem_dst + k);
      if (s >= c1) break;
      const int64_t real_end = s + __ldcg(ws.mem_real + k);
      const int64_t e = (k + 1 < hi) ? (int64_t)__ldcg(ws.mem_dst + k + 1) : total;
      const int64_t a0 = max(s, c0), a1 = min(real_end, c1);
      if (a0 < a1) {
        const int64_t i = __ldcg(ws.mem_src + k);
        block_copy(row + a0 * eb, c.src + (i * c.W + (a0 - s)) * eb, (a1 - a0) * eb);
        if (mrow) block_fill_bytes(mrow + a0, a1 - a0, 0);
      }
      const int64_t p0 = max(real_end, c0), p1 = min(e, c1);
      if (p0 < p1) {
        block_fill(row + p0 * eb, p1 - p0, eb, c.pad_value);
        if (mrow) block_fill_bytes(mrow + p0, p1 - p0, 1);
      }
    }
  }
  const int64_t t0 = max(total, c0);
  if (t0 < c1) {
    block_fill(row + t0 * eb, c1 - t0, eb, c.pad_value);
    if (mrow) block_fill_bytes(mrow + t0, c1 - t0, 1);
  }
}

struct FusedArgs {
  const unsigned char* src;
  const int64_t* real;
  const int32_t* off;
  const int32_t* mem;
  int num_bins, M;
  int64_t N, W, multiple, capacity, width, pad_value;
  int stretch, elem_bytes;
  unsigned char* out;  // may be NULL (metadata only)
  uint8_t* mask;       // may be NULL
  int32_t* cu;
  int32_t* cup;
  pseq_info* info;
};

__device__ __forceinline__ bool offsets_bad(const FusedArgs& a, int b, int lo, int hi) {
  return (b == 0 && lo != 0) || (b == a.num_bins - 1 && hi != a.M) || lo < 0 || hi > a.M || hi <= lo;
}

// CTA (0, 0): one pass over every member to fold all bins' checks into info.
__device__ void squeeze_info_pass(const FusedArgs& a, int32_t* s_off, unsigned long long* s_tot) {
  __shared__ int s_value, s_capacity, s_longest, s_widest;
  const int tid = threadIdx.x;
  if (tid == 0) s_value = s_capacity = s_longest = s_widest = 0;
  for (int i = tid; i <= a.num_bins; i += kFusedThreads) s_off[i] = __ldg(a.off + i);
  for (int i = tid; i < a.num_bins; i += kFusedThreads) s_tot[i] = 0ull;
  __syncthreads();
  for (int b = tid; b < a.num_bins; b += kFusedThreads)
    if (offsets_bad(a, b, s_off[b], s_off[b + 1])) s_value = 1;
  for (int e = tid; e < a.M; e += kFusedThreads) {
    const int b = seq_of(s_off, a.num_bins, e);
    const int i = __ldg(a.mem + e);
    if (i < 0 || i >= a.N) {
      s_value = 1;
      continue;
    }
    const long long real = __ldg(a.real + i);
    if (real < 0 || real > a.W) {
      s_value = 1;
      continue;
    }
    atomicAdd(&s_tot[b], (unsigned long long)((real + a.multiple - 1) / a.multiple * a.multiple));
    atomicMax(&s_longest, (int)real);
  }
  __syncthreads();
  for (int b = tid; b < a.num_bins; b += kFusedThreads) {
    const unsigned long long t = s_tot[b];
    if (t > (unsigned long long)a.capacity || (a.out && t > (unsigned long long)a.width)) s_capacity = 1;
    atomicMax(&s_widest, (int)min(t, (unsigned long long)INT32_MAX));
  }
  __syncthreads();
  if (tid == 0) {
    const int status = s_value ? PSEQ_ERR_VALUE : (s_capacity ? PSEQ_ERR_CAPACITY : PSEQ_OK);
    *a.info = status == PSEQ_OK ? pseq_info{PSEQ_OK, a.M, s_longest, s_widest} : pseq_info{status, 0, 0, 0};
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kFusedThreads) squeeze_fused_kernel(const __grid_constant__ FusedArgs a) {
  __shared__ int32_t s_dst[kFusedMaxMembers + 1];
  __shared__ int32_t s_real[kFusedMaxMembers];
  __shared__ int32_t s_src[kFusedMaxMembers];
  __shared__ int32_t s_off[kFusedMaxMembers + 1];
  __shared__ unsigned long long s_tot[kFusedMaxMembers];
  __shared__ Triple scratch[kFusedThreads / 32];
  __shared__ int s_bad;
  pdl_enter();
  const int tid = threadIdx.x;
  const int b = blockIdx.y;
  if (blockIdx.x == 0 && b == 0) squeeze_info_pass(a, s_off, s_tot);
  const int lo = __ldg(a.off + b), hi = __ldg(a.off + b + 1);
  if (offsets_bad(a, b, lo, hi) || hi - lo > kFusedMaxMembers) return;
  const int n = hi - lo;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  // scan the bin's members: slot where each starts, both cumulative sums
  Triple carry = {0, 0, 0};
  for (int base = 0; base < n; base += kFusedThreads) {
    const int j = base + tid;
    long long real = 0, padded = 0;
    int src = 0;
    if (j < n) {
      src = __ldg(a.mem + lo + j);
      if (src < 0 || src >= a.N) {
        s_bad = 1;
      } else {
        real = __ldg(a.real + src);
        if (real < 0 || real > a.W) {
          s_bad = 1;
          real = 0;
        }
      }
      padded = (real + a.multiple - 1) / a.multiple * a.multiple;
    }
    Triple total;
    const Triple ex = block_exclusive<kFusedThreads / 32>({0, real, padded}, scratch, total);
    if (j < n) {
      const long long R = carry.real + ex.real, Pd = carry.padded + ex.padded;
      s_dst[j] = (int32_t)Pd;
      s_real[j] = (int32_t)real;
      s_src[j] = src;
      if (blockIdx.x == 0) {
        a.cu[lo + b + j] = (int32_t)R;
        a.cup[lo + b + j] = (int32_t)Pd;
      }
    }
    carry = add(carry, total);
  }
  const long long total_pad = carry.padded;
  if (tid == 0) {
    s_dst[n] = (int32_t)min(total_pad, (long long)INT32_MAX);
    if (blockIdx.x == 0) {
      a.cu[hi + b] = (int32_t)carry.real;
      a.cup[hi + b] = a.stretch ? (int32_t)a.capacity : (int32_t)total_pad;
    }
  }
  __syncthreads();
  if (s_bad || total_pad > a.capacity || !a.out || total_pad > a.width) return;
  // every slot of this chunk, once
  const int eb = a.elem_bytes;
  const int64_t chunk = (int64_t)kFusedThreads * kSlotsPerThread;
  const int64_t c0 = (int64_t)blockIdx.x * chunk;
  const int64_t c1 = min(c0 + chunk, a.width);
  unsigned char* row = a.out + (int64_t)b * a.width * eb;
  uint8_t* mrow = a.mask ? a.mask + (int64_t)b * a.width : nullptr;
  int4 v[kSlotsPerThread];
  bool pad[kSlotsPerThread];
  int4 pv = make_int4(0, 0, 0, 0);
  {
    const uint64_t p = (uint64_t)a.pad_value;
    pv.x = (int)(uint32_t)p;
    pv.y = (int)(uint32_t)(p >> 32);
  }
#pragma unroll
  for (int q = 0; q < kSlotsPerThread; ++q) {
    const int64_t t = c0 + tid + (int64_t)q * kFusedThreads;
    pad[q] = true;
    v[q] = pv;
    if (t < c1 && t < total_pad) {
      const int j = seq_of(s_dst, n, t);
      const int64_t off = t - s_dst[j];
      if (off < s_real[j]) {
        pad[q] = false;
        v[q] = load_row(a.src + ((int64_t)s_src[j] * a.W + off) * eb, eb);
      }
    }
  }
#pragma unroll
  for (int q = 0; q < kSlotsPerThread; ++q) {
    const int64_t t = c0 + tid + (int64_t)q * kFusedThreads;
    if (t < c1) {
      store_row(row + t * eb, v[q], eb);
      if (mrow) mrow[t] = pad[q] ? 1 : 0;
    }
  }
}

__global__ void empty_squeeze_kernel(pseq_info* info) {
  pdl_enter();
  *info = {PSEQ_OK, 0, 0, 0};
}

}  // namespace
}  // namespace pseq

using namespace pseq;

extern "C" size_t pack_squeeze_workspace_size(int64_t num_members, int64_t num_bins) {
  if (num_members < 0 || num_bins < 0) return 0;
  return workspace_bytes(num_members, num_bins);
}

extern "C" pseq_status pack_squeeze(const void* src, int64_t N, int64_t W, int32_t elem_bytes,
                                    const int64_t* real_lens, const int32_t* bin_offsets,
                                    const int32_t* bin_members, int64_t num_bins, int64_t num_members,
                                    int64_t multiple, int64_t capacity, int32_t stretch_to_capacity,
                                    int64_t width, int64_t pad_value, void* out, int32_t* cu_seqlens,
                                    int32_t* cu_seqlens_padded, uint8_t* padding_mask, pseq_info* info,
                                    void* workspace, size_t workspace_bytes_, pseq_stream stream) {
  clear_error();
  const char* fn = "pack_squeeze";
  if (N < 0 || W < 0 || num_bins < 0 || num_members < 0 || width < 0 || capacity < 0)
    return fail(PSEQ_ERR_ARG, "%s: negative size", fn);
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
    return fail(PSEQ_ERR_ARG, "%s: elem_bytes must be 1, 2, 4 or 8", fn);
  if (multiple < 1 || multiple > INT32_MAX) return fail(PSEQ_ERR_ARG, "%s: multiple must be in [1, INT32_MAX]", fn);
  if (N > INT32_MAX || W > INT32_MAX || capacity > INT32_MAX || width > INT32_MAX || num_bins > INT32_MAX / 2 ||
      num_members > INT32_MAX / 2)
    return fail(PSEQ_ERR_OVERFLOW, "%s: a size exceeds the int32 range", fn);
  if (num_bins > 65535) return fail(PSEQ_ERR_ARG, "%s: at most 65535 bins per call", fn);
  if ((out == nullptr) != (padding_mask == nullptr) && out == nullptr)
    return fail(PSEQ_ERR_ARG, "%s: padding_mask needs out", fn);
  if (stretch_to_capacity && out && width < capacity)
    return fail(PSEQ_ERR_ARG, "%s: stretching to capacity needs width >= capacity", fn);
  if (!info || !cu_seqlens || !cu_seqlens_padded) return fail(PSEQ_ERR_ARG, "%s: NULL output", fn);
  if (num_bins > 0 && (!bin_offsets || (num_members > 0 && (!bin_members || !real_lens))))
    return fail(PSEQ_ERR_ARG, "%s: NULL bin arrays", fn);
  if (out && num_members > 0 && N * W > 0 && !src) return fail(PSEQ_ERR_ARG, "%s: NULL src", fn);
  if (!aligned(real_lens, 8) || !aligned(bin_offsets, 4) || !aligned(bin_members, 4) || !aligned(cu_seqlens, 4) ||
      !aligned(cu_seqlens_padded, 4) || !aligned(info, 4) || !aligned(src, (uintptr_t)elem_bytes) ||
      !aligned(out, (uintptr_t)elem_bytes))
    return fail(PSEQ_ERR_ARG, "%s: misaligned pointer", fn);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (num_bins == 0) {
    if (num_members != 0) return fail(PSEQ_ERR_ARG, "%s: members without bins", fn);
    const cudaError_t e = launch_pdl(empty_squeeze_kernel, dim3(1), dim3(1), 0, st, info);
    count_launches(1);
    if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    return check_launch(fn);
  }
  const size_t need = workspace_bytes(num_members, num_bins);
  if (!workspace || workspace_bytes_ < need || !aligned(workspace, 16))
    return fail(PSEQ_ERR_ARG, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", fn, need, workspace_bytes_);
  if (num_members <= kFusedMaxMembers && num_bins <= kFusedMaxMembers) {
    FusedArgs a = {};
    a.src = static_cast<const unsigned char*>(src);
    a.real = real_lens;
    a.off = bin_offsets;
    a.mem = bin_members;
    a.num_bins = (int)num_bins;
    a.M = (int)num_members;
    a.N = N;
    a.W = W;
    a.multiple = multiple;
    a.capacity = capacity;
    a.width = width;
    a.pad_value = pad_value;
    a.stretch = stretch_to_capacity ? 1 : 0;
    a.elem_bytes = elem_bytes;
    a.out = static_cast<unsigned char*>(out);
    a.mask = padding_mask;
    a.cu = cu_seqlens;
    a.cup = cu_seqlens_padded;
    a.info = info;
    const int64_t chunk = (int64_t)kFusedThreads * kSlotsPerThread;
    const unsigned gx = out && width > 0 ? (unsigned)((width + chunk - 1) / chunk) : 1u;
    const cudaError_t e = launch_pdl(squeeze_fused_kernel, dim3(gx, (unsigned)num_bins), dim3(kFusedThreads), 0, st, a);
    count_launches(1);
    if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    return check_launch(fn);
  }
  Workspace ws = carve(workspace, num_members, num_bins);

  MetaArgs m = {};
  m.real = real_lens;
  m.off = bin_offsets;
  m.mem = bin_members;
  m.num_bins = (int)num_bins;
  m.M = (int)num_members;
  m.N = N;
  m.W = W;
  m.multiple = multiple;
  m.capacity = capacity;
  m.width = width;
  m.stretch = stretch_to_capacity ? 1 : 0;
  m.check_width = out ? 1 : 0;
  m.cu = cu_seqlens;
  m.cup = cu_seqlens_padded;
  cudaError_t e = launch_pdl(squeeze_meta_kernel, dim3((unsigned)((num_bins + kMetaWarps - 1) / kMetaWarps)),
                             dim3(kMetaThreads), 0, st, m, ws);
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  pseq_status s = check_launch(fn);
  if (s != PSEQ_OK) return s;

  CopyArgs c = {};
  c.src = static_cast<const unsigned char*>(src);
  c.W = W;
  c.elem_bytes = elem_bytes;
  c.off = bin_offsets;
  c.num_bins = (int)num_bins;
  c.M = (int)num_members;
  c.width = width;
  c.pad_value = pad_value;
  c.out = static_cast<unsigned char*>(out);
  c.mask = padding_mask;
  c.info = info;
  dim3 grid(1, 1);
  if (out && width > 0) {
    // chunks of whole 16-byte groups, about four CTAs per SM over the output
    const int64_t slots = num_bins * width;
    const int64_t target = (int64_t)sm_count() * 4;
    int64_t chunk = (slots + target - 1) / target;
    const int64_t per16 = 16 / elem_bytes;
    const int64_t min_chunk = 4096 / elem_bytes;
    if (chunk < min_chunk) chunk = min_chunk;
    chunk = (chunk + per16 - 1) / per16 * per16;
    c.chunk = chunk;
    grid = dim3((unsigned)((width + chunk - 1) / chunk), (unsigned)num_bins);
  } else {
    c.chunk = 1;
  }
  e = launch_pdl(squeeze_copy_kernel, grid, dim3(kCopyThreads), 0, st, c, ws);
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}
