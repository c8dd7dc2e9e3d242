// pack_squeeze: the trainer-side squeeze of a padded rectangle into bins.
//
// Follows "Who packs the sequences: the loader, or the trainer?" (NeMo-RL
// #4105 explainer): "Trainer packs" (sources padded to a multiple and laid
// end to end; cu_seqlens from real lengths, cu_seqlens_padded from padded
// lengths) and "Loader packs" (the last padded boundary stretched to the pack
// capacity).
//
// One launch over (slot window, bin) CTAs.  Every CTA scans its bin's members
// (padded lengths, both cumulative sums) and keeps in shared memory only the
// members whose padded range meets its window of output slots.  Those ranges
// are disjoint and each at least `multiple` slots long, so the table never
// holds more than min(window, window / multiple + 2) entries, whatever the
// number of members; the launch sizes it so, which keeps shared memory from
// limiting the CTAs resident on an SM.  Each thread then owns a fixed number
// of slots of the window (interleaved across the CTA, so that a warp's
// accesses are contiguous): it looks up the member of each slot, issues every
// load before any store, and writes the token or pad_value with its mask
// byte.  Every output slot is written exactly once.
//
// The first window of every bin also writes the bin's cu arrays and adds
// its status and sizes to running totals in the workspace header (atomics
// that return nothing); the last of those CTAs to finish (a wrapping acq_rel
// counter) writes the info block from them and resets them.
#include "common.cuh"

namespace pseq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSlotsNarrow = 4;  // slots per thread when the grid would be small

// Slots per thread on large outputs: 12 (six 16-byte vectors of 8-byte
// elements) lets six CTAs share an SM; 1- and 2-byte elements keep 16 so that
// a thread's slots still make whole 16-byte vectors.
template <int EB>
__host__ __device__ constexpr int slots_wide() {
  return EB >= 4 ? 12 : 16;
}

struct Header {
  unsigned finished;  // bins whose first window is done; wraps back to 0 after each call
  // the call's running totals, reset by the first window that finishes
  // last: a bin with malformed members or offsets (bit 0) or over capacity
  // (bit 1), the longest member, the widest bin
  unsigned flags, longest, widest;
  unsigned pad[28];
};

static_assert(sizeof(Header) == 128, "header is 128 bytes");

size_t workspace_bytes(int64_t) { return sizeof(Header); }

template <int SLOTS>
__host__ __device__ constexpr int window() {
  return kThreads * SLOTS;
}

// A member table entry: output start, real length, source row (int32 each).
constexpr size_t kEntryBytes = 3 * sizeof(int32_t);

// Entries a window of w slots can meet: disjoint ranges, each >= multiple long.
inline int table_entries(int64_t w, int64_t multiple) { return (int)min(w, w / multiple + 2); }

struct Args {
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
  Header* hdr;
};

__device__ __forceinline__ bool offsets_bad(const Args& a, int b, int lo, int hi) {
  return (b == 0 && lo != 0) || (b == a.num_bins - 1 && hi != a.M) || lo < 0 || hi > a.M || hi <= lo;
}

// Exclusive count of set flags over the block; `total` gets the block count.
__device__ __forceinline__ int block_count_exclusive(bool flag, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned m = __ballot_sync(~0u, flag);
  if (lane == 0) s_warp[warp] = __popc(m);
  __syncthreads();
  int before = 0, sum = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int c = s_warp[w];
    before += w < warp ? c : 0;
    sum += c;
  }
  total = sum;
  __syncthreads();
  return before + __popc(m & ((1u << lane) - 1u));
}

template <int EB>
struct Elem;
template <>
struct Elem<1> {
  using T = unsigned char;
};
template <>
struct Elem<2> {
  using T = unsigned short;
};
template <>
struct Elem<4> {
  using T = unsigned int;
};
template <>
struct Elem<8> {
  using T = unsigned long long;
};

// The first window that finishes last: report the call's totals and reset
// them (every other first window has counted itself in).
__device__ __forceinline__ void report(const Args& a) {
  // L2 loads: the counter this CTA acquired ordered every update before it
  const unsigned flags = __ldcg(&a.hdr->flags), longest = __ldcg(&a.hdr->longest), widest = __ldcg(&a.hdr->widest);
  const int status = (flags & 1u) ? PSEQ_ERR_VALUE : ((flags & 2u) ? PSEQ_ERR_CAPACITY : PSEQ_OK);
  *a.info = status == PSEQ_OK ? pseq_info{PSEQ_OK, a.M, (int)longest, (int)widest} : pseq_info{status, 0, 0, 0};
  a.hdr->flags = 0u;
  a.hdr->longest = 0u;
  a.hdr->widest = 0u;
}

// `cap` = table_entries(window, multiple): the table's length in entries.
// Wide windows: five (16 slots) or six (12 slots) CTAs per SM, so that some
// stream while others scan their tables; narrow grids fill less than a wave.
template <int SLOTS, int EB, bool VEC>
__global__ void __launch_bounds__(kThreads, SLOTS >= 16 ? 5 : (SLOTS >= 12 ? 6 : 4))
    squeeze_kernel(const __grid_constant__ Args a, int cap) {
  extern __shared__ __align__(16) int32_t s_table[];
  constexpr int kWindow = window<SLOTS>();
  int32_t* s_dst = s_table;
  int32_t* s_real = s_table + cap;
  int32_t* s_src = s_table + 2 * cap;
  __shared__ Triple scratch[kWarps];
  __shared__ int s_count[kWarps];
  __shared__ int s_bad, s_longest, s_last;
  pdl_enter();
  const int tid = threadIdx.x;
  const int b = blockIdx.y;
  const bool first = blockIdx.x == 0;
  const int lo = __ldg(a.off + b), hi = __ldg(a.off + b + 1);
  const bool bad_offsets = offsets_bad(a, b, lo, hi);
  // the window [c0, c1): width < 2^31 - 2^16 (host check), so int32 holds both
  const int32_t c0 = (int32_t)(blockIdx.x * (unsigned)kWindow);
  const int32_t c1 = (int32_t)min((int64_t)c0 + kWindow, a.width);
  if (tid == 0) {
    s_bad = 0;
    s_longest = 0;
  }
  __syncthreads();
  // the bin's members: both cumulative sums; keep the ones meeting the window
  Triple carry = {0, 0, 0};
  int held = 0;
  if (!bad_offsets) {
    const int n = hi - lo;
    for (int base = 0; base < n; base += kThreads) {
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
        // real <= W and multiple <= INT32_MAX: the rounding fits 32 bits
        const uint32_t m = (uint32_t)a.multiple;
        padded = (long long)(((uint32_t)real + m - 1u) / m) * m;
        atomicMax(&s_longest, (int)real);
      }
      Triple total;
      const Triple ex = block_exclusive<kWarps>({0, real, padded}, scratch, total);
      const long long R = carry.real + ex.real, Pd = carry.padded + ex.padded;
      if (first && j < n) {
        a.cu[lo + b + j] = (int32_t)R;
        a.cup[lo + b + j] = (int32_t)Pd;
      }
      const bool keep = j < n && padded > 0 && Pd < c1 && Pd + padded > c0;
      int kept;
      const int pos = held + block_count_exclusive(keep, s_count, kept);
      if (keep) {
        s_dst[pos] = (int32_t)Pd;
        s_real[pos] = (int32_t)real;
        s_src[pos] = src;
      }
      held += kept;
      carry = add(carry, total);
    }
  }
  __syncthreads();
  const long long total_pad = carry.padded;
  int status = PSEQ_OK;
  if (bad_offsets || s_bad) status = PSEQ_ERR_VALUE;
  else if (total_pad > a.capacity || (a.out && total_pad > a.width)) status = PSEQ_ERR_CAPACITY;
  // First windows add their bin's share and count it in; the counter's
  // old value is looked at only after the window has streamed, so that its
  // round trip overlaps the copy.  The last to arrive reports the totals.
  unsigned ticket = 0;
  if (first && tid == 0) {
    if (!bad_offsets) {
      a.cu[hi + b] = (int32_t)carry.real;
      a.cup[hi + b] = a.stretch ? (int32_t)a.capacity : (int32_t)total_pad;
    }
    // this bin's share of the totals (atomics that return nothing), then the count
    if (status == PSEQ_ERR_VALUE) atomicOr(&a.hdr->flags, 1u);
    else if (status == PSEQ_ERR_CAPACITY) atomicOr(&a.hdr->flags, 2u);
    if (s_longest) atomicMax(&a.hdr->longest, (unsigned)s_longest);
    atomicMax(&a.hdr->widest, (unsigned)min(total_pad, (long long)INT32_MAX));
    ticket = inc_acq_rel(&a.hdr->finished, (unsigned)a.num_bins - 1u);
  }
  auto finish = [&]() {
    if (!first) return;
    if (tid == 0) s_last = ticket == (unsigned)a.num_bins - 1u;
    __syncthreads();
    if (s_last && tid == 0) report(a);
  };
  if (status != PSEQ_OK || !a.out) {
    finish();
    return;
  }
  // every slot of the window, once: loads first, then stores.  A thread's
  // slots ascend, so its member index only moves forward through the table.
  using T = typename Elem<EB>::T;
  const T* src = reinterpret_cast<const T*>(a.src);
  T* row = reinterpret_cast<T*>(a.out) + (int64_t)b * a.width;
  uint8_t* mrow = a.mask ? a.mask + (int64_t)b * a.width : nullptr;
  const T pv = (T)(uint64_t)a.pad_value;
  int j = 0;
  const int32_t lim = (int32_t)min((long long)c1, total_pad);  // slots below are in members
  const int32_t end = c1;
  if constexpr (VEC) {
    // 16-byte vectors of V slots.  The host takes this path only when row
    // pitches, width and multiple keep every member start on a vector
    // boundary, so a vector never spans two members; only the real/padding
    // boundary inside a member can fall inside one.
    constexpr int V = 16 / EB;
    constexpr int NV = SLOTS / V;
    static_assert(NV * V == SLOTS, "window must hold whole vectors");
    T pad_elems[V];
#pragma unroll
    for (int k = 0; k < V; ++k) pad_elems[k] = pv;
    int4 pad4;
    memcpy(&pad4, pad_elems, 16);
    int4 v[NV];
    uint32_t nreal[(NV + 3) / 4];  // real slots of vector q in byte q (fewer registers)
#pragma unroll
    for (int k = 0; k < (NV + 3) / 4; ++k) nreal[k] = 0;
    const int32_t base = c0 + tid * V;
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      const int32_t t = base + q * kThreads * V;
      v[q] = pad4;
      if (t < lim) {
        while (j + 1 < held && s_dst[j + 1] <= t) ++j;
        const int32_t off = t - s_dst[j];
        const int32_t r = s_real[j];
        const T* p = src + (int64_t)s_src[j] * a.W + off;
        if (off + V <= r) {
          v[q] = ld_stream(reinterpret_cast<const int4*>(p));
          nreal[q / 4] |= (uint32_t)V << (8 * (q % 4));
        } else if (off < r) {
          T e[V];
#pragma unroll
          for (int k = 0; k < V; ++k) e[k] = off + k < r ? __ldg(p + k) : pv;
          memcpy(&v[q], e, 16);
          nreal[q / 4] |= (uint32_t)(r - off) << (8 * (q % 4));
        }
      }
    }
#pragma unroll
    for (int q = 0; q < NV; ++q) {
      const int32_t t = base + q * kThreads * V;
      if (t < end) {
        st_stream(reinterpret_cast<int4*>(row + t), v[q]);
        if (mrow) {
          // byte k is 1 for padding: the slots from the vector's real count on
          const int nr = (int)((nreal[q / 4] >> (8 * (q % 4))) & 0xffu);
          uint8_t m[V];
#pragma unroll
          for (int k = 0; k < V; ++k) m[k] = k >= nr ? 1 : 0;
          if constexpr (V == 16) {
            int4 w;
            memcpy(&w, m, 16);
            *reinterpret_cast<int4*>(mrow + t) = w;
          } else if constexpr (V == 8) {
            unsigned long long w;
            memcpy(&w, m, 8);
            *reinterpret_cast<unsigned long long*>(mrow + t) = w;
          } else if constexpr (V == 4) {
            unsigned int w;
            memcpy(&w, m, 4);
            *reinterpret_cast<unsigned int*>(mrow + t) = w;
          } else {
            unsigned short w;
            memcpy(&w, m, 2);
            *reinterpret_cast<unsigned short*>(mrow + t) = w;
          }
        }
      }
    }
  } else {
    T v[SLOTS];
    unsigned padmask = 0;
    const int32_t base = c0 + tid;
#pragma unroll
    for (int q = 0; q < SLOTS; ++q) {
      const int32_t t = base + q * kThreads;
      v[q] = pv;
      bool pad = true;
      if (t < lim) {
        while (j + 1 < held && s_dst[j + 1] <= t) ++j;
        const int32_t off = t - s_dst[j];
        if (off < s_real[j]) {
          pad = false;
          v[q] = __ldg(src + (int64_t)s_src[j] * a.W + off);
        }
      }
      padmask |= (pad ? 1u : 0u) << q;
    }
#pragma unroll
    for (int q = 0; q < SLOTS; ++q) {
      const int32_t t = base + q * kThreads;
      if (t < end) {
        __stcs(row + t, v[q]);
        if (mrow) mrow[t] = (uint8_t)((padmask >> q) & 1u);
      }
    }
  }
  finish();
}

__global__ void empty_squeeze_kernel(pseq_info* info) {
  pdl_enter();
  *info = {PSEQ_OK, 0, 0, 0};
}

template <int SLOTS, int EB, bool VEC>
cudaError_t launch_squeeze(const Args& a, unsigned gy, cudaStream_t st) {
  constexpr int64_t w = window<SLOTS>();
  // the attribute allows the largest table (multiple 1), so that concurrent
  // callers with other multiples never lower it under one another
  const cudaError_t e =
      allow_dynamic_smem(reinterpret_cast<const void*>(squeeze_kernel<SLOTS, EB, VEC>), kEntryBytes * (size_t)w);
  if (e != cudaSuccess) return e;
  const int cap = table_entries(w, a.multiple);
  const unsigned gx = a.out && a.width > 0 ? (unsigned)((a.width + w - 1) / w) : 1u;
  return launch_pdl(squeeze_kernel<SLOTS, EB, VEC>, dim3(gx, gy), dim3(kThreads), kEntryBytes * (size_t)cap, st, a,
                    cap);
}

template <int SLOTS, int EB>
cudaError_t launch_squeeze(const Args& a, bool vec, unsigned gy, cudaStream_t st) {
  if constexpr (SLOTS % (16 / EB) == 0) {
    if (vec) return launch_squeeze<SLOTS, EB, true>(a, gy, st);
  }
  return launch_squeeze<SLOTS, EB, false>(a, gy, st);
}

// Wide windows when they still give every SM two CTAs, else narrow ones.
template <int EB>
cudaError_t launch_squeeze(const Args& a, bool vec, unsigned gy, cudaStream_t st) {
  constexpr int kWide = slots_wide<EB>();
  constexpr int64_t w = window<kWide>();
  const int64_t wide_ctas = (a.out && a.width > 0 ? (a.width + w - 1) / w : 1) * (int64_t)gy;
  return wide_ctas >= 2 * (int64_t)sm_count() ? launch_squeeze<kWide, EB>(a, vec, gy, st)
                                               : launch_squeeze<kSlotsNarrow, EB>(a, vec, gy, st);
}

cudaError_t launch_squeeze(const Args& a, bool vec, unsigned gy, cudaStream_t st) {
  switch (a.elem_bytes) {
    case 8: return launch_squeeze<8>(a, vec, gy, st);
    case 4: return launch_squeeze<4>(a, vec, gy, st);
    case 2: return launch_squeeze<2>(a, vec, gy, st);
    default: return launch_squeeze<1>(a, vec, gy, st);
  }
}

}  // namespace
}  // namespace pseq

using namespace pseq;

extern "C" size_t pack_squeeze_workspace_size(int64_t num_members, int64_t num_bins) {
  if (num_members < 0 || num_bins < 0) return 0;
  return workspace_bytes(num_bins);
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
  if (width > INT32_MAX - 65536) return fail(PSEQ_ERR_OVERFLOW, "%s: width exceeds 2^31 - 2^16", fn);
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
  const size_t need = workspace_bytes(num_bins);
  if (!workspace || workspace_bytes_ < need || !aligned(workspace, 16))
    return fail(PSEQ_ERR_ARG, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", fn, need, workspace_bytes_);
  Args a = {};
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
  a.hdr = static_cast<Header*>(workspace);
  // 16-byte vectors when every member start, row start and window start
  // falls on a 16-byte boundary of both src and out
  const int64_t eb = elem_bytes;
  const bool vec = out && aligned(src, 16) && aligned(out, 16) && aligned(padding_mask, 16) && (W * eb) % 16 == 0 &&
                   (width * eb) % 16 == 0 && (multiple * eb) % 16 == 0;
  const cudaError_t e = launch_squeeze(a, vec, (unsigned)num_bins, st);
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}
