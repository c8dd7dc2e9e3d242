// thd_mask_from_token_ids: padding by token value, rejecting a pad id that
// also occurs as content.
//
// Follows NeMo AutoModel v0.5 "nemo_automodel.components.distributed.thd_utils",
// thd_padding_mask_from_token_ids: comparing ids with the pad id marks padding
// correctly only if the pad positions form a suffix of the stream, so the
// kernel checks that and reports a pad id that also occurs as content.
//
// One pass.  Each thread compares groups of eight consecutive ids (16-byte
// loads), two groups per round with all loads in flight, and stores each
// group's eight mask bytes at once.  The pad positions form a suffix exactly
// when no pad id is directly followed by another id, so a thread also reads
// the id left of each group and looks for such a step inside and at the left
// edge of the group.  Each CTA adds its pad count, a flag for a step seen
// and one to a finished-CTA count, all packed into one 64-bit word, with a
// single atomic add; the CTA whose add completes the count reads the totals
// from the value the add returns, writes the info block and resets the word.
#include "common.cuh"

namespace pseq {
namespace {

constexpr int kThreads = 512;
constexpr int kGroup = 8;  // ids per thread and step (16 measured slower)
static_assert(kGroup % 8 == 0 && kGroup <= 32, "whole 8-byte mask words, one 32-bit pad mask");

// The call's running totals: pads in bits 0..39, CTAs that saw a pad id
// followed by another id in bits 40..51, finished CTAs in bits 52..63.
constexpr int kBadShift = 40, kDoneShift = 52;
constexpr unsigned long long kField = 0xfffull;
constexpr int kMaxGrid = 4095;  // the finished count's field

struct Header {
  unsigned long long totals;  // zero between calls
  unsigned long long pad[15];
};
static_assert(sizeof(Header) == 128, "header is 128 bytes");

size_t workspace_bytes() { return sizeof(Header); }

template <typename Id, bool kVector>
__global__ void __launch_bounds__(kThreads)
    token_mask_kernel(const Id* __restrict__ ids, int64_t n, Id pad, uint8_t* __restrict__ mask,
                      pseq_info* __restrict__ info, Header* hdr) {
  __shared__ long long s_pads[kThreads / 32];
  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t groups = (n + kGroup - 1) / kGroup;
  long long pads = 0;
  bool step = false;  // a pad id directly followed by another id
  // Two groups per round, every load issued before either group is examined,
  // so a thread with a second group (the grid is one wave) pays one latency.
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  auto load_group = [&](int64_t g, Id* v, Id& left) {
    const int64_t t0 = g * kGroup;
    left = t0 > 0 ? ids[t0 - 1] : pad;
    if (kVector && t0 + kGroup <= n) {
      constexpr int kVec = kGroup * sizeof(Id) / 16;
      const int4* p = reinterpret_cast<const int4*>(ids + t0);
      int4 q[kVec];
#pragma unroll
      for (int k = 0; k < kVec; ++k) q[k] = ld_stream(p + k);
      memcpy(v, q, sizeof(Id) * kGroup);
    } else {
#pragma unroll
      for (int k = 0; k < kGroup; ++k) v[k] = t0 + k < n ? ids[t0 + k] : pad;
    }
  };
  auto do_group = [&](int64_t g, const Id* v, Id left) {
    const int64_t t0 = g * kGroup;
    // one bit per id: which are the pad id
    const int live = t0 + kGroup <= n ? kGroup : (int)(n - t0);
    const unsigned valid = live >= 32 ? ~0u : ((1u << live) - 1u);
    unsigned padbits = 0;
#pragma unroll
    for (int k = 0; k < kGroup; ++k) padbits |= (v[k] == pad ? 1u : 0u) << k;
    padbits &= valid;
    const unsigned content = ~padbits & valid;
    pads += __popc(padbits);
    // bit k of (pad bits, with the left id's as bit -1) next to content bit k
    const unsigned before = (padbits << 1) | (t0 > 0 && left == pad ? 1u : 0u);
    step |= (before & content) != 0;
    if (kVector && live == kGroup) {
#pragma unroll
      for (int w = 0; w < kGroup / 8; ++w) {
        unsigned long long bytes = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) bytes |= (unsigned long long)((padbits >> (8 * w + k)) & 1u) << (8 * k);
        *reinterpret_cast<unsigned long long*>(mask + t0 + 8 * w) = bytes;
      }
    } else {
      for (int k = 0; k < live; ++k) mask[t0 + k] = (uint8_t)((padbits >> k) & 1u);
    }
  };
  for (int64_t g0 = (int64_t)blockIdx.x * kThreads + tid; g0 < groups; g0 += 2 * stride) {
    const int64_t g1 = g0 + stride;
    Id v0[kGroup], v1[kGroup], l0, l1 = pad;
    load_group(g0, v0, l0);
    if (g1 < groups) load_group(g1, v1, l1);
    do_group(g0, v0, l0);
    if (g1 < groups) do_group(g1, v1, l1);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) pads += __shfl_xor_sync(~0u, pads, d);
  if (lane == 0) s_pads[warp] = pads;
  const int cta_step = __syncthreads_or(step ? 1 : 0);  // also publishes s_pads
  if (tid != 0) return;
  long long cta_pads = 0;
  for (int w = 0; w < kThreads / 32; ++w) cta_pads += s_pads[w];
  const unsigned long long add = (unsigned long long)cta_pads | ((unsigned long long)(cta_step ? 1 : 0) << kBadShift) |
                                 (1ull << kDoneShift);
  // the value before this add; the add that completes the count sees every
  // other CTA's share in it
  const unsigned long long old = atomicAdd(&hdr->totals, add);
  if (((old >> kDoneShift) & kField) != gridDim.x - 1) return;
  const unsigned long long all = old + add;
  const long long total = (long long)(all & ((1ull << kBadShift) - 1));
  const bool ok = ((all >> kBadShift) & kField) == 0;
  *info = ok ? pseq_info{PSEQ_OK, (int32_t)total, 0, (int32_t)n} : pseq_info{PSEQ_ERR_VALUE, 0, 0, (int32_t)n};
  hdr->totals = 0;  // for the next call (which starts after this grid completes)
}

// One wave: at most `per_sm` resident CTAs per SM (the workspace is sized for
// the largest any variant can have, 2048 threads' worth).
int grid_for(int64_t n, int per_sm = 2048 / kThreads) {
  const int64_t groups = (n + kGroup - 1) / kGroup;
  const int64_t want = (groups + kThreads - 1) / kThreads;
  int64_t full = (int64_t)sm_count() * per_sm;
  if (full > kMaxGrid) full = kMaxGrid;
  const int64_t g = want < full ? want : full;
  return (int)(g < 1 ? 1 : g);
}

template <typename Id, bool kVector>
int launch_grid(int64_t n) {
  return grid_for(n, occupancy(reinterpret_cast<const void*>(token_mask_kernel<Id, kVector>), kThreads, 0));
}

}  // namespace
}  // namespace pseq

using namespace pseq;

extern "C" size_t thd_mask_from_token_ids_workspace_size(int64_t n) {
  if (n < 0) return 0;
  return workspace_bytes();
}

extern "C" pseq_status thd_mask_from_token_ids(const void* input_ids, int32_t id_bytes, int64_t n,
                                               int64_t padding_token_id, uint8_t* mask, pseq_info* info,
                                               void* workspace, size_t workspace_bytes_, pseq_stream stream) {
  clear_error();
  const char* fn = "thd_mask_from_token_ids";
  if (n < 0) return fail(PSEQ_ERR_ARG, "%s: negative length", fn);
  if (n > INT32_MAX) return fail(PSEQ_ERR_OVERFLOW, "%s: length exceeds INT32_MAX", fn);
  if (id_bytes != 4 && id_bytes != 8) return fail(PSEQ_ERR_ARG, "%s: id_bytes must be 4 or 8", fn);
  if (!info || (n > 0 && (!input_ids || !mask))) return fail(PSEQ_ERR_ARG, "%s: NULL pointer", fn);
  if (!aligned(input_ids, (uintptr_t)id_bytes) || !aligned(info, 4)) return fail(PSEQ_ERR_ARG, "%s: misaligned pointer", fn);
  if (id_bytes == 4 && (padding_token_id < INT32_MIN || padding_token_id > INT32_MAX))
    return fail(PSEQ_ERR_ARG, "%s: padding_token_id does not fit 32-bit ids", fn);
  const size_t need = workspace_bytes();
  if (!workspace || workspace_bytes_ < need || !aligned(workspace, 16))
    return fail(PSEQ_ERR_ARG, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", fn, need, workspace_bytes_);
  Header* hdr = static_cast<Header*>(workspace);
  const bool vec = aligned(input_ids, 16) && aligned(mask, 8);
  const int grid = id_bytes == 4 ? (vec ? launch_grid<int32_t, true>(n) : launch_grid<int32_t, false>(n))
                                 : (vec ? launch_grid<int64_t, true>(n) : launch_grid<int64_t, false>(n));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (id_bytes == 4) {
    const int32_t* p = static_cast<const int32_t*>(input_ids);
    e = vec ? launch_pdl(token_mask_kernel<int32_t, true>, dim3(grid), dim3(kThreads), 0, st, p, n,
                         (int32_t)padding_token_id, mask, info, hdr)
            : launch_pdl(token_mask_kernel<int32_t, false>, dim3(grid), dim3(kThreads), 0, st, p, n,
                         (int32_t)padding_token_id, mask, info, hdr);
  } else {
    const int64_t* p = static_cast<const int64_t*>(input_ids);
    e = vec ? launch_pdl(token_mask_kernel<int64_t, true>, dim3(grid), dim3(kThreads), 0, st, p, n,
                         (int64_t)padding_token_id, mask, info, hdr)
            : launch_pdl(token_mask_kernel<int64_t, false>, dim3(grid), dim3(kThreads), 0, st, p, n,
                         (int64_t)padding_token_id, mask, info, hdr);
  }
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}
