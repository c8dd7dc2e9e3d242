// thd_mask_from_token_ids: padding by token value, rejecting a pad id that
// also occurs as content.
//
// Follows NeMo AutoModel v0.5 "nemo_automodel.components.distributed.thd_utils",
// thd_padding_mask_from_token_ids: comparing ids with the pad id marks padding
// correctly only if the pad positions form a suffix of the stream, so the
// kernel checks that and reports a pad id that also occurs as content.
//
// One pass.  Each thread compares groups of eight consecutive ids (16-byte
// loads), two groups per round with both loads in flight, and stores each
// group's eight mask bytes at once; each CTA reduces the first pad
// position, the last non-pad position and the pad count of its part and
// writes them to its own workspace slot.  The CTA that finishes last (an
// acq_rel counter that wraps back to zero) folds the slots: the input is
// valid exactly when the last content position precedes the first pad.
#include "common.cuh"

namespace pseq {
namespace {

constexpr int kThreads = 512;
constexpr int kGroup = 8;  // ids per thread and step (16 measured slower)
static_assert(kGroup % 8 == 0 && kGroup <= 32, "whole 8-byte mask words, one 32-bit pad mask");

struct Header {
  unsigned int finished;
  unsigned int pad[31];
};

struct Part {
  long long first_pad;     // smallest pad position, or n when none
  long long last_content;  // largest non-pad position, or -1 when none
  long long pads;
  long long unused;
};

size_t workspace_bytes(int64_t ctas) { return sizeof(Header) + sizeof(Part) * (size_t)ctas; }

template <typename Id, bool kVector>
__global__ void __launch_bounds__(kThreads)
    token_mask_kernel(const Id* __restrict__ ids, int64_t n, Id pad, uint8_t* __restrict__ mask,
                      pseq_info* __restrict__ info, Header* hdr, Part* parts) {
  __shared__ long long s_first[kThreads / 32], s_last[kThreads / 32], s_pads[kThreads / 32];
  __shared__ int s_last_cta;
  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t groups = (n + kGroup - 1) / kGroup;
  long long first_pad = n, last_content = -1, pads = 0;
  // Two groups per round, both loads issued before either is examined, so a
  // thread with a second group (the grid is one wave) pays one load latency.
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  auto load_group = [&](int64_t g, Id* v) {
    const int64_t t0 = g * kGroup;
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
  auto do_group = [&](int64_t g, const Id* v) {
    const int64_t t0 = g * kGroup;
    // one bit per id: which are the pad id; the group's statistics from the bits
    const int live = t0 + kGroup <= n ? kGroup : (int)(n - t0);
    const unsigned valid = live >= 32 ? ~0u : ((1u << live) - 1u);
    unsigned padbits = 0;
#pragma unroll
    for (int k = 0; k < kGroup; ++k) padbits |= (v[k] == pad ? 1u : 0u) << k;
    padbits &= valid;
    const unsigned content = ~padbits & valid;
    pads += __popc(padbits);
    if (padbits) first_pad = min(first_pad, (long long)(t0 + __ffs(padbits) - 1));
    if (content) last_content = max(last_content, (long long)(t0 + 31 - __clz(content)));
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
    Id v0[kGroup], v1[kGroup];
    load_group(g0, v0);
    if (g1 < groups) load_group(g1, v1);
    do_group(g0, v0);
    if (g1 < groups) do_group(g1, v1);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    first_pad = min(first_pad, __shfl_xor_sync(~0u, first_pad, d));
    last_content = max(last_content, __shfl_xor_sync(~0u, last_content, d));
    pads += __shfl_xor_sync(~0u, pads, d);
  }
  if (lane == 0) {
    s_first[warp] = first_pad;
    s_last[warp] = last_content;
    s_pads[warp] = pads;
  }
  __syncthreads();
  if (tid == 0) {
    Part p = {(long long)n, -1, 0, 0};
    for (int w = 0; w < kThreads / 32; ++w) {
      p.first_pad = min(p.first_pad, s_first[w]);
      p.last_content = max(p.last_content, s_last[w]);
      p.pads += s_pads[w];
    }
    parts[blockIdx.x] = p;
    s_last_cta = inc_acq_rel(&hdr->finished, gridDim.x - 1) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last_cta) return;
  // fold every CTA's part with the whole block
  long long f = n, l = -1, total = 0;
  for (unsigned c = tid; c < gridDim.x; c += kThreads) {
    // L2 loads: the parts were released by the counter that thread 0 acquired
    f = min(f, __ldcg(&parts[c].first_pad));
    l = max(l, __ldcg(&parts[c].last_content));
    total += __ldcg(&parts[c].pads);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    f = min(f, __shfl_xor_sync(~0u, f, d));
    l = max(l, __shfl_xor_sync(~0u, l, d));
    total += __shfl_xor_sync(~0u, total, d);
  }
  __syncthreads();
  if (lane == 0) {
    s_first[warp] = f;
    s_last[warp] = l;
    s_pads[warp] = total;
  }
  __syncthreads();
  if (tid != 0) return;
  for (int w = 1; w < kThreads / 32; ++w) {
    f = min(f, s_first[w]);
    l = max(l, s_last[w]);
    total += s_pads[w];
  }
  const bool ok = l < f;
  *info = ok ? pseq_info{PSEQ_OK, (int32_t)total, 0, (int32_t)n} : pseq_info{PSEQ_ERR_VALUE, 0, 0, (int32_t)n};
}

// One wave: at most `per_sm` resident CTAs per SM (the workspace is sized for
// the largest any variant can have, 2048 threads' worth).
int grid_for(int64_t n, int per_sm = 2048 / kThreads) {
  const int64_t groups = (n + kGroup - 1) / kGroup;
  const int64_t want = (groups + kThreads - 1) / kThreads;
  const int64_t full = (int64_t)sm_count() * per_sm;
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
  return workspace_bytes(grid_for(n));
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
  const size_t need = workspace_bytes(grid_for(n));
  if (!workspace || workspace_bytes_ < need || !aligned(workspace, 16))
    return fail(PSEQ_ERR_ARG, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", fn, need, workspace_bytes_);
  Header* hdr = static_cast<Header*>(workspace);
  Part* parts = reinterpret_cast<Part*>(static_cast<unsigned char*>(workspace) + sizeof(Header));
  const bool vec = aligned(input_ids, 16) && aligned(mask, 8);
  const int grid = id_bytes == 4 ? (vec ? launch_grid<int32_t, true>(n) : launch_grid<int32_t, false>(n))
                                 : (vec ? launch_grid<int64_t, true>(n) : launch_grid<int64_t, false>(n));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (id_bytes == 4) {
    const int32_t* p = static_cast<const int32_t*>(input_ids);
    e = vec ? launch_pdl(token_mask_kernel<int32_t, true>, dim3(grid), dim3(kThreads), 0, st, p, n,
                         (int32_t)padding_token_id, mask, info, hdr, parts)
            : launch_pdl(token_mask_kernel<int32_t, false>, dim3(grid), dim3(kThreads), 0, st, p, n,
                         (int32_t)padding_token_id, mask, info, hdr, parts);
  } else {
    const int64_t* p = static_cast<const int64_t*>(input_ids);
    e = vec ? launch_pdl(token_mask_kernel<int64_t, true>, dim3(grid), dim3(kThreads), 0, st, p, n,
                         (int64_t)padding_token_id, mask, info, hdr, parts)
            : launch_pdl(token_mask_kernel<int64_t, false>, dim3(grid), dim3(kThreads), 0, st, p, n,
                         (int64_t)padding_token_id, mask, info, hdr, parts);
  }
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}
