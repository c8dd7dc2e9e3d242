// pack_ffd: first-fit-decreasing bin assignment for the trainer-side squeeze.
//
// In "Who packs the sequences: the loader, or the trainer?", get_packer is the
// step that groups rows into bins under a token budget, and First Fit
// Decreasing is one of the packers the page names.  The textbook algorithm: visit the items largest first (ties:
// smaller index first) and put each into the first open bin with room.
//
// One CTA.  Each item becomes a 64-bit key (inverted size, index) so an
// ascending bitonic sort in shared memory yields the visiting order.  First
// fit is inherently sequential over items, so one warp walks them in order
// with the open bins' remaining room held in registers across its lanes: one
// ballot per item picks the first that fits.  Bins are numbered in the order
// they open, members keep their placement order, and a block scan of the bin
// counts turns the placements into CSR arrays.
#include "common.cuh"

namespace pseq {
namespace {

constexpr int kThreads = 1024;
constexpr int kMaxItems = 8192;

__global__ void __launch_bounds__(kThreads)
    ffd_kernel(const int64_t* __restrict__ lens, int n, int64_t multiple, int64_t capacity, int32_t* bin_offsets,
               int32_t* bin_members, pseq_info* info) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int pow2 = n <= 1 ? 1 : 1 << (32 - __clz(n - 1));
  unsigned long long* key = reinterpret_cast<unsigned long long*>(smem);  // [pow2]
  int32_t* room = reinterpret_cast<int32_t*>(key + pow2);               // [n] per bin
  int32_t* bin_of = room + (n > 0 ? n : 1);                              // [n] per sorted item
  int32_t* slot_of = bin_of + (n > 0 ? n : 1);                           // [n] per sorted item
  int32_t* count = slot_of + (n > 0 ? n : 1);                            // [n] per bin
  __shared__ int s_bad, s_big, s_bins;
  __shared__ long long s_total, s_fullest;
  pdl_enter();
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_bad = s_big = 0;
    s_total = 0;
    s_fullest = 0;
  }
  __syncthreads();
  // keys: (INT32_MAX - size) in the high word sorts sizes descending, the
  // index in the low word breaks ties toward the smaller index
  long long my_total = 0;
  for (int i = tid; i < pow2; i += kThreads) {
    unsigned long long k = ~0ull;  // padding sorts last
    if (i < n) {
      const long long real = lens[i];
      long long size = 0;
      if (real < 0) {
        s_bad = 1;
      } else if (real > capacity) {
        s_big = 1;
      } else {
        size = (real + multiple - 1) / multiple * multiple;
        if (size > capacity) s_big = 1;
        my_total += size;
      }
      if (size > INT32_MAX) size = INT32_MAX;
      k = ((unsigned long long)(INT32_MAX - size) << 32) | (unsigned)i;
    }
    key[i] = k;
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) my_total += __shfl_xor_sync(~0u, my_total, d);
  if ((tid & 31) == 0 && my_total) atomicAdd(reinterpret_cast<unsigned long long*>(&s_total), (unsigned long long)my_total);
  __syncthreads();
  if (n <= 256) {
    // Rank sort: keys are distinct (the index is in the low word), so each
    // key's rank is the number of smaller keys; one pass over the table per
    // thread, reading broadcast from shared memory.
    unsigned long long mine = tid < n ? key[tid] : 0ull;
    int rank = 0;
    if (tid < n) {
#pragma unroll 4
      for (int j = 0; j < n; ++j) rank += key[j] < mine ? 1 : 0;
    }
    __syncthreads();
    if (tid < n) key[rank] = mine;
    __syncthreads();
  } else if (pow2 <= kThreads) {
    // One key per thread, in registers: exchanges within a warp by shuffle,
    // across warps through shared memory.  Whole warps take part (padding
    // keys sort last), so every shuffle has its full warp.
    const int span = pow2 < 32 ? 32 : pow2;
    const bool in = tid < span;
    unsigned long long k = tid < pow2 ? key[tid] : ~0ull;
    for (int width = 2; width <= pow2; width <<= 1) {
      for (int stride = width >> 1; stride > 0; stride >>= 1) {
        unsigned long long other = 0;
        if (stride >= 32) {
          __syncthreads();  // the previous exchange has been read
          if (in) key[tid] = k;
          __syncthreads();
          if (in) other = key[tid ^ stride];
        } else if (in) {
          other = __shfl_xor_sync(~0u, k, stride);
        }
        if (in) {
          // ascending runs where (tid & width) == 0; the lower index of a
          // pair keeps the smaller key of an ascending run
          const bool take_min = ((tid & stride) == 0) == ((tid & width) == 0);
          k = take_min ? (k < other ? k : other) : (k < other ? other : k);
        }
      }
    }
    __syncthreads();
    if (tid < pow2) key[tid] = k;
    __syncthreads();
  } else {
    for (int width = 2; width <= pow2; width <<= 1) {
      for (int stride = width >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < pow2; i += kThreads) {
          const int j = i ^ stride;
          if (j > i) {
            const bool up = (i & width) == 0;
            const unsigned long long a = key[i], b = key[j];
            if ((a > b) == up) {
              key[i] = b;
              key[j] = a;
            }
          }
        }
        __syncthreads();
      }
    }
  }
  if (s_bad || s_big) {
    if (tid == 0) *info = {s_bad ? PSEQ_ERR_VALUE : PSEQ_ERR_CAPACITY, 0, 0, 0};
    return;
  }
  // sizes in visiting order, as int32 (room and count arrays are free yet)
  for (int k = tid; k < n; k += kThreads) bin_of[k] = INT32_MAX - (int)(key[k] >> 32);
  __syncthreads();
  // first fit, one warp, items in visiting order.  While at most 32 bins are
  // open, bin b's remaining room and member count sit in lane b's registers
  // and one ballot per item finds the first bin with room.  Beyond that, lane
  // L holds bins [L*kRegBins, (L+1)*kRegBins): each lane tests its own bins,
  // one ballot picks the first lane with a fit and that lane picks its first
  // register; bins past 32*kRegBins live in shared memory.  The lane that owns
  // the chosen bin records the placement itself, so no value crosses lanes
  // after the ballot; sizes are read two items ahead.
  if (tid < 32) {
    constexpr int kRegBins = 8;
    constexpr int kRegTotal = 32 * kRegBins;
    const int lane = tid;
    int bins = 0;
    int cur = n > 0 ? bin_of[0] : 0;
    int nxt = n > 1 ? bin_of[1] : 0;
    int k = 0;
    int my_room = 0, my_cnt = 0;
    for (; k < n; ++k) {
      const int size = cur;
      const unsigned fits = __ballot_sync(~0u, lane < bins && my_room >= size);
      int chosen = __ffs(fits) - 1;
      if (!fits) {
        if (bins == 32) break;  // a 33rd bin: continue on the general path below
        chosen = bins++;
        if (lane == chosen) {
          my_room = (int)capacity;
          my_cnt = 0;
        }
      }
      cur = nxt;
      if (k + 2 < n) nxt = bin_of[k + 2];  // sizes still staged two items ahead
      if (lane == chosen) {
        my_room -= size;
        slot_of[k] = my_cnt++;
        bin_of[k] = chosen;  // its size was read already
      }
    }
    // general layout: bin b in lane b / kRegBins, register b % kRegBins
    int room_r[kRegBins], count_r[kRegBins];
#pragma unroll
    for (int r = 0; r < kRegBins; ++r) {
      const int b = lane * kRegBins + r;
      const int from_room = __shfl_sync(~0u, my_room, b & 31), from_cnt = __shfl_sync(~0u, my_cnt, b & 31);
      room_r[r] = b < bins ? from_room : 0;
      count_r[r] = b < bins ? from_cnt : 0;
    }
    for (; k < n; ++k) {
      const int size = cur;
      cur = nxt;
      if (k + 2 < n) nxt = bin_of[k + 2];
      bool any = false;
#pragma unroll
      for (int r = 0; r < kRegBins; ++r) any |= lane * kRegBins + r < bins && room_r[r] >= size;
      const unsigned lanes = __ballot_sync(~0u, any);
      if (lanes) {
        const bool owner = lane == __ffs(lanes) - 1;
        int pick = kRegBins;
#pragma unroll
        for (int r = kRegBins - 1; r >= 0; --r)
          if (lane * kRegBins + r < bins && room_r[r] >= size) pick = r;
#pragma unroll
        for (int r = 0; r < kRegBins; ++r)
          if (owner && pick == r) {
            room_r[r] -= size;
            slot_of[k] = count_r[r]++;
            bin_of[k] = lane * kRegBins + r;
          }
        continue;
      }
      int chosen = -1;
      if (bins > kRegTotal) {  // bins that live in shared memory
        for (int base = kRegTotal; chosen < 0 && base < bins; base += 32) {
          const unsigned f = __ballot_sync(~0u, base + lane < bins && room[base + lane] >= size);
          if (f) chosen = base + __ffs(f) - 1;
        }
        if (chosen >= 0) {
          __syncwarp();
          if (lane == 0) {
            room[chosen] -= size;
            slot_of[k] = count[chosen];
            count[chosen] += 1;
            bin_of[k] = chosen;
          }
          __syncwarp();
          continue;
        }
      }
      // open a new bin
      chosen = bins;
      bins += 1;
      if (chosen >= kRegTotal) {
        __syncwarp();
        if (lane == 0) {
          room[chosen] = (int32_t)capacity - size;
          count[chosen] = 1;
          slot_of[k] = 0;
          bin_of[k] = chosen;
        }
        __syncwarp();
      } else {
#pragma unroll
        for (int r = 0; r < kRegBins; ++r)
          if (lane * kRegBins + r == chosen) {
            room_r[r] = (int)capacity - size;
            count_r[r] = 1;
            slot_of[k] = 0;
            bin_of[k] = chosen;
          }
      }
    }
    __syncwarp();
#pragma unroll
    for (int r = 0; r < kRegBins; ++r)
      if (lane * kRegBins + r < bins && lane * kRegBins + r < kRegTotal) {
        room[lane * kRegBins + r] = room_r[r];
        count[lane * kRegBins + r] = count_r[r];
      }
    if (lane == 0) s_bins = bins;
  }
  __syncthreads();
  const int bins = s_bins;
  // bin_offsets = [0] + cumsum(count): a block scan, the bins in chunks
  __shared__ int s_warp[kThreads / 32];
  __shared__ int s_carry;
  if (tid == 0) s_carry = 0;
  __syncthreads();
  for (int base = 0; base < bins; base += kThreads) {
    const int b = base + tid;
    const int c = b < bins ? count[b] : 0;
    int inc = c;
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(~0u, inc, d);
      if (lane >= d) inc += o;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      int w = s_warp[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(~0u, w, d);
        if (lane >= d) w += o;
      }
      s_warp[lane] = w;
    }
    __syncthreads();
    const int excl = s_carry + inc - c + (warp > 0 ? s_warp[warp - 1] : 0);
    if (b < bins) {
      bin_offsets[b] = excl;
      count[b] = excl;  // reuse as the bin's first member position
      const long long load = capacity - room[b];
      atomicMax(reinterpret_cast<unsigned long long*>(&s_fullest), (unsigned long long)load);
    }
    __syncthreads();
    if (tid == 0) s_carry += s_warp[kThreads / 32 - 1];
    __syncthreads();
  }
  for (int k = tid; k < n; k += kThreads) bin_members[count[bin_of[k]] + slot_of[k]] = (int32_t)(key[k] & 0xffffffffu);
  if (tid == 0) {
    bin_offsets[bins] = n;
    *info = {PSEQ_OK, bins, (int32_t)min(s_fullest, (long long)INT32_MAX), (int32_t)min(s_total, (long long)INT32_MAX)};
  }
}

size_t ffd_smem(int n) {
  int pow2 = 1;
  while (pow2 < n) pow2 <<= 1;
  const size_t m = n > 0 ? (size_t)n : 1;
  return round_up(8 * (size_t)pow2 + 4 * m * 4, 16);
}

}  // namespace
}  // namespace pseq

using namespace pseq;

extern "C" pseq_status pack_ffd(const int64_t* lens, int64_t n, int64_t multiple, int64_t capacity,
                                int32_t* bin_offsets, int32_t* bin_members, pseq_info* info, pseq_stream stream) {
  clear_error();
  const char* fn = "pack_ffd";
  if (n < 0 || n > kMaxItems) return fail(PSEQ_ERR_ARG, "%s: n must be in [0, %d]", fn, kMaxItems);
  if (multiple < 1 || multiple > INT32_MAX) return fail(PSEQ_ERR_ARG, "%s: multiple must be in [1, INT32_MAX]", fn);
  if (capacity < 0 || capacity > INT32_MAX) return fail(PSEQ_ERR_ARG, "%s: capacity must be in [0, INT32_MAX]", fn);
  if (!bin_offsets || !info || (n > 0 && (!lens || !bin_members))) return fail(PSEQ_ERR_ARG, "%s: NULL pointer", fn);
  if (!aligned(lens, 8) || !aligned(bin_offsets, 4) || !aligned(bin_members, 4) || !aligned(info, 4))
    return fail(PSEQ_ERR_ARG, "%s: misaligned pointer", fn);
  const size_t smem = ffd_smem((int)n);
  const cudaError_t ea = allow_dynamic_smem(reinterpret_cast<const void*>(ffd_kernel), ffd_smem(kMaxItems));
  if (ea != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(ea));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = launch_pdl(ffd_kernel, dim3(1), dim3(kThreads), smem, st, lens, (int)n, multiple, capacity,
                                   bin_offsets, bin_members, info);
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}
