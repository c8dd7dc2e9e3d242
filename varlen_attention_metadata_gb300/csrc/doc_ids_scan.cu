// pseq_from_doc_ids: segment boundaries of a neat-packing document map.
//
// Follows NeMo AutoModel "nemo_automodel.components.datasets.packed_seq",
// packed_seq_params_from_doc_ids and PackedSeqParams: a segment is a maximal
// run of one document index within a row, every row start opens a segment,
// padding runs are segments, cu_seqlens ends at B*S, max_seqlen is the
// longest segment.
//
// One pass over doc_ids.  Each CTA takes the next 4096-token tile (dynamic
// tile index, so every tile it waits on is already running), flags the
// boundaries in it, and summarises them as (count, first, last, largest
// inner gap).  The summaries form an associative "followed by" operation,
// so a decoupled look-back over the preceding tiles gives each tile its
// exclusive prefix: the output index of its first boundary and the position
// of the boundary before it, which closes the segment that crosses into the
// tile.  The largest gap over all tiles is max_seqlen, so the segment-length
// maximum rides along with the scan and needs no second pass.  Boundaries
// are compacted through shared memory and written with coalesced stores.
// The last CTA to finish writes cu_seqlens[num_segments] and the info block
// and clears the tile flags, so the workspace is zero again for the next call.
#include <mutex>

#include "common.cuh"

namespace pseq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 16;
constexpr int kTile = kThreads * kItems;  // tokens per tile
constexpr uint32_t kEmpty = 0, kAggregate = 1, kInclusive = 2;

// Boundaries inside a span of tokens: how many, the first and last boundary
// position, and the largest distance between consecutive boundaries.
struct Bounds {
  int count, first, last, gap;
};

__device__ __forceinline__ Bounds none() { return {0, -1, -1, 0}; }

// Summary of span a followed by span b.
__device__ __forceinline__ Bounds join(const Bounds& a, const Bounds& b) {
  Bounds r;
  r.count = a.count + b.count;
  r.first = a.count ? a.first : b.first;
  r.last = b.count ? b.last : a.last;
  r.gap = max(a.gap, b.gap);
  if (a.count && b.count) r.gap = max(r.gap, b.first - a.last);
  return r;
}

__device__ __forceinline__ Bounds shfl_up(const Bounds& v, int d) {
  return {__shfl_up_sync(~0u, v.count, d), __shfl_up_sync(~0u, v.first, d), __shfl_up_sync(~0u, v.last, d),
          __shfl_up_sync(~0u, v.gap, d)};
}

__device__ __forceinline__ Bounds shfl(const Bounds& v, int src) {
  return {__shfl_sync(~0u, v.count, src), __shfl_sync(~0u, v.first, src), __shfl_sync(~0u, v.last, src),
          __shfl_sync(~0u, v.gap, src)};
}

__device__ __forceinline__ int4 pack(const Bounds& b) { return make_int4(b.count, b.first, b.last, b.gap); }
__device__ __forceinline__ Bounds unpack(const int4& v) { return {v.x, v.y, v.z, v.w}; }

struct Header {
  unsigned int next_tile;  // dynamic tile index; wraps back to 0 after each call
  unsigned int finished;   // tiles done; wraps back to 0 after each call
  unsigned int gave_up;    // nonzero when some wait hit its time limit
  unsigned int pad[29];
};
static_assert(sizeof(Header) == 128, "header is 128 bytes");

struct Workspace {
  Header* hdr;
  uint32_t* status;  // [tiles]: kEmpty / kAggregate / kInclusive
  int4* aggregate;   // [tiles]: the tile's own Bounds
  int4* inclusive;   // [tiles]: Bounds of tiles 0..t
};

size_t workspace_bytes(int64_t tiles) {
  return sizeof(Header) + round_up(4 * (size_t)tiles, 16) + 32 * (size_t)tiles;
}

Workspace carve(void* base, int64_t tiles) {
  unsigned char* p = static_cast<unsigned char*>(base);
  Workspace w;
  w.hdr = reinterpret_cast<Header*>(p);
  p += sizeof(Header);
  w.status = reinterpret_cast<uint32_t*>(p);
  p += round_up(4 * (size_t)tiles, 16);
  w.aggregate = reinterpret_cast<int4*>(p);
  p += 16 * (size_t)tiles;
  w.inclusive = reinterpret_cast<int4*>(p);
  return w;
}

template <typename Id>
union Items {
  int4 q[kItems * sizeof(Id) / 16];
  Id v[kItems];
};

template <typename Id, bool kVector>
__global__ void __launch_bounds__(kThreads)
    doc_ids_scan_kernel(const Id* __restrict__ doc, int N, int S, int32_t* __restrict__ cu,
                        pseq_info* __restrict__ info, Workspace ws, int tiles, int64_t wait_ns,
                        int withhold) {
  __shared__ int s_tile;
  __shared__ int s_last_cta;
  __shared__ Bounds s_warp[kWarps];
  __shared__ Bounds s_prefix;
  __shared__ int s_pos[kTile];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    unsigned t = atomicInc(&ws.hdr->next_tile, (unsigned)(tiles - 1));
    if (t >= (unsigned)tiles) {  // the workspace was not zero-filled
      atomicOr(&ws.hdr->gave_up, 2u);
      t %= (unsigned)tiles;
    }
    s_tile = (int)t;
  }
  __syncthreads();
  const int tile = s_tile;
  const int64_t t0 = (int64_t)tile * kTile + (int64_t)tid * kItems;

  // ---- this thread's 16 tokens and the token to their left
  Items<Id> it;
  if (kVector && t0 + kItems <= N) {
    const int4* p = reinterpret_cast<const int4*>(doc + t0);
#pragma unroll
    for (int k = 0; k < (int)(kItems * sizeof(Id) / 16); ++k) it.q[k] = __ldg(p + k);
  } else {
#pragma unroll
    for (int k = 0; k < kItems; ++k) it.v[k] = (t0 + k < N) ? __ldg(doc + t0 + k) : Id(0);
  }
  const Id left = (t0 > 0 && t0 < N) ? __ldg(doc + t0 - 1) : Id(0);

  // ---- boundary flags: row start, or a different index than the left token
  unsigned flags = 0;
  Bounds mine = none();
  int r = (int)(t0 % S);
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int64_t t = t0 + k;
    const Id prev = k ? it.v[k - 1] : left;
    const bool f = (t < N) && (r == 0 || it.v[k] != prev);
    if (f) {
      const int ti = (int)t;
      if (mine.count) mine.gap = max(mine.gap, ti - mine.last);
      else mine.first = ti;
      mine.last = ti;
      mine.count += 1;
      flags |= 1u << k;
    }
    if (++r == S) r = 0;
  }

  // ---- block-wide scan of the summaries (in token order)
  Bounds inc = mine;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const Bounds o = shfl_up(inc, d);
    if (lane >= d) inc = join(o, inc);
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    Bounds w = lane < kWarps ? s_warp[lane] : none();
#pragma unroll
    for (int d = 1; d < kWarps; d <<= 1) {
      const Bounds o = shfl_up(w, d);
      if (lane >= d) w = join(o, w);
    }
    if (lane < kWarps) s_warp[lane] = w;
  }
  __syncthreads();
  Bounds before_me = shfl_up(inc, 1);
  if (lane == 0) before_me = none();
  if (warp > 0) before_me = join(s_warp[warp - 1], before_me);
  const Bounds tile_sum = s_warp[kWarps - 1];

  // ---- publish the tile summary, then look back for the exclusive prefix
  if (warp == 0) {
    Bounds prefix = none();
    if (tile == 0) {
      if (lane == 0 && withhold != 0) {
        __stcg(&ws.inclusive[0], pack(tile_sum));
        st_release(&ws.status[0], kInclusive);
      }
    } else {
      if (lane == 0 && withhold != tile) {
        __stcg(&ws.aggregate[tile], pack(tile_sum));
        st_release(&ws.status[tile], kAggregate);
      }
      Bounds run = none();  // summary of the tiles between the window and this one
      int j = tile - 1;
      bool gave_up = false;
      while (true) {
        const int idx = j - lane;  // lane 0 looks at the nearest predecessor
        uint32_t st = kInclusive;  // lanes before tile 0 stand for an empty prefix
        Bounds b = none();
        if (idx >= 0) {
          st = ld_acquire(&ws.status[idx]);
          if (st == kEmpty) {
            const uint64_t start = global_ns();
            do {
              __nanosleep(32);
              st = ld_acquire(&ws.status[idx]);
            } while (st == kEmpty && (int64_t)(global_ns() - start) < wait_ns);
          }
          if (st == kEmpty) {
            gave_up = true;  // treat as an empty inclusive prefix and finish
            st = kInclusive;
          } else {
            b = unpack(st == kInclusive ? __ldcg(&ws.inclusive[idx]) : __ldcg(&ws.aggregate[idx]));
          }
        }
        const unsigned stop_mask = __ballot_sync(~0u, st == kInclusive);
        const int stop = stop_mask ? __ffs(stop_mask) - 1 : 32;
        Bounds win = none();
        for (int L = (stop < 32 ? stop : 31); L >= 0; --L) win = join(win, shfl(b, L));
        run = join(win, run);
        if (stop < 32) break;
        j -= 32;
      }
      if (__any_sync(~0u, gave_up) && lane == 0) atomicOr(&ws.hdr->gave_up, 1u);
      prefix = run;
      if (lane == 0 && withhold != tile) {
        __stcg(&ws.inclusive[tile], pack(join(prefix, tile_sum)));
        st_release(&ws.status[tile], kInclusive);
      }
    }
    if (lane == 0) s_prefix = prefix;
  }

  // ---- compact this tile's boundary positions and store them
  int li = before_me.count;
#pragma unroll
  for (int k = 0; k < kItems; ++k)
    if (flags & (1u << k)) s_pos[li++] = (int)(t0 + k);
  __syncthreads();
  const int base = s_prefix.count;
  if (base >= 0 && base <= N - tile_sum.count) {
    for (int i = tid; i < tile_sum.count; i += kThreads) cu[base + i] = s_pos[i];
  } else if (tid == 0) {
    atomicOr(&ws.hdr->gave_up, 2u);  // only reachable from a corrupt workspace
  }

  // ---- the last CTA to finish closes the array and resets the workspace
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last_cta = atomicInc(&ws.hdr->finished, (unsigned)(tiles - 1)) == (unsigned)(tiles - 1);
  __syncthreads();
  if (!s_last_cta) return;
  __threadfence();
  if (tid == 0) {
    const Bounds all = unpack(__ldcg(&ws.inclusive[tiles - 1]));
    const unsigned failed = atomicExch(&ws.hdr->gave_up, 0u);
    pseq_info out;
    if (failed || all.count < 1 || all.count > N) {
      out = {(failed & 2u) ? PSEQ_ERR_ARG : PSEQ_ERR_TIMEOUT, 0, 0, N};
    } else {
      cu[all.count] = N;
      out = {PSEQ_OK, all.count, max(all.gap, N - all.last), N};
    }
    *info = out;
  }
  for (int i = tid; i < tiles; i += kThreads) ws.status[i] = kEmpty;
}

__global__ void empty_map_kernel(int32_t* cu, pseq_info* info) {
  cu[0] = 0;
  *info = {PSEQ_OK, 0, 0, 0};
}

template <typename Id>
cudaError_t launch_scan(const void* doc, int N, int S, int32_t* cu, pseq_info* info, Workspace ws,
                        int tiles, cudaStream_t st) {
  const Id* d = static_cast<const Id*>(doc);
  const int64_t wait = wait_limit_ns();
  const int withhold = (int)(withhold_tile() < 0 ? -1 : (withhold_tile() > INT32_MAX ? -1 : withhold_tile()));
  if (aligned(doc, 16))
    doc_ids_scan_kernel<Id, true><<<tiles, kThreads, 0, st>>>(d, N, S, cu, info, ws, tiles, wait, withhold);
  else
    doc_ids_scan_kernel<Id, false><<<tiles, kThreads, 0, st>>>(d, N, S, cu, info, ws, tiles, wait, withhold);
  return cudaSuccess;
}

}  // namespace
}  // namespace pseq

using namespace pseq;

extern "C" size_t pseq_from_doc_ids_workspace_size(int64_t B, int64_t S) {
  if (B < 0 || S < 0) return 0;
  if (B > 0 && S > INT32_MAX / B) return 0;
  const int64_t N = B * S;
  const int64_t tiles = N > 0 ? (N + kTile - 1) / kTile : 1;
  return workspace_bytes(tiles);
}

extern "C" pseq_status pseq_from_doc_ids(const void* doc_ids, int32_t id_bytes, int64_t B, int64_t S,
                                         int32_t* cu_seqlens, pseq_info* info, void* workspace,
                                         size_t ws_bytes, pseq_stream stream) {
  clear_error();
  if (B < 0 || S < 0) return fail(PSEQ_ERR_ARG, "pseq_from_doc_ids: negative shape [%lld, %lld]", (long long)B, (long long)S);
  if (id_bytes != 4 && id_bytes != 8) return fail(PSEQ_ERR_ARG, "pseq_from_doc_ids: id_bytes must be 4 or 8, got %d", id_bytes);
  if (!cu_seqlens || !info) return fail(PSEQ_ERR_ARG, "pseq_from_doc_ids: cu_seqlens and info are required");
  if (B > 0 && S > INT32_MAX / B)
    return fail(PSEQ_ERR_OVERFLOW, "pseq_from_doc_ids: B*S = %lld*%lld exceeds INT32_MAX", (long long)B, (long long)S);
  const int64_t N = B * S;
  if (N > 0 && !doc_ids) return fail(PSEQ_ERR_ARG, "pseq_from_doc_ids: doc_ids is NULL");
  if (!aligned(doc_ids, (uintptr_t)id_bytes) || !aligned(cu_seqlens, 4) || !aligned(info, 4))
    return fail(PSEQ_ERR_ARG, "pseq_from_doc_ids: misaligned pointer");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (N == 0) {
    empty_map_kernel<<<1, 1, 0, st>>>(cu_seqlens, info);
    count_launches(1);
    return check_launch("pseq_from_doc_ids");
  }
  const int64_t tiles = (N + kTile - 1) / kTile;
  const size_t need = workspace_bytes(tiles);
  if (!workspace || ws_bytes < need || !aligned(workspace, 16))
    return fail(PSEQ_ERR_ARG, "pseq_from_doc_ids: workspace needs %zu bytes, 16-byte aligned (got %zu)", need, ws_bytes);
  Workspace ws = carve(workspace, tiles);
  if (id_bytes == 4)
    launch_scan<int32_t>(doc_ids, (int)N, (int)S, cu_seqlens, info, ws, (int)tiles, st);
  else
    launch_scan<int64_t>(doc_ids, (int)N, (int)S, cu_seqlens, info, ws, (int)tiles, st);
  count_launches(1);
  return check_launch("pseq_from_doc_ids");
}

// ----------------------------------------------------------------------------
// pseq_from_doc_ids_static: the same scan with its scratch in a static array.
//
// For callers that cannot allocate device memory at call time -- code running
// under a memory-pool policy that forbids new allocations, inside a plugin or
// callback that has no allocator handle, or in a process that has reserved the
// whole HBM for itself -- this entry point takes only inputs and outputs.  Its
// scratch is a file-scope device array, loaded with the library and held by
// every GPU that loads it until the process exits.
// ----------------------------------------------------------------------------
namespace pseq {
namespace {

constexpr int64_t kStaticMaxTokens = PSEQ_STATIC_MAX_TOKENS;  // B*S limit of the static scratch
constexpr int64_t kStaticMaxTiles = kStaticMaxTokens / kTile;
constexpr size_t kStaticBytes = sizeof(Header) + ((4 * kStaticMaxTiles + 15) / 16) * 16 + 32 * kStaticMaxTiles;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

std::mutex g_static_mu;
void* g_static_ptr[64] = {nullptr};

// Device address of g_static_scratch on the current device, looked up once
// per device.  In host code the array's name is only a stand-in symbol.
pseq_status static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "pseq_from_doc_ids_static: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(PSEQ_ERR_ARG, "pseq_from_doc_ids_static: device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p)
      return fail(PSEQ_ERR_CUDA, "pseq_from_doc_ids_static: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return PSEQ_OK;
}

}  // namespace
}  // namespace pseq

extern "C" pseq_status pseq_from_doc_ids_static(const void* doc_ids, int32_t id_bytes, int64_t B, int64_t S,
                                                int32_t* cu_seqlens, pseq_info* info, pseq_stream stream) {
  clear_error();
  const char* fn = "pseq_from_doc_ids_static";
  if (B < 0 || S < 0) return fail(PSEQ_ERR_ARG, "%s: negative shape [%lld, %lld]", fn, (long long)B, (long long)S);
  if (id_bytes != 4 && id_bytes != 8) return fail(PSEQ_ERR_ARG, "%s: id_bytes must be 4 or 8, got %d", fn, id_bytes);
  if (!cu_seqlens || !info) return fail(PSEQ_ERR_ARG, "%s: cu_seqlens and info are required", fn);
  if (B > 0 && S > kStaticMaxTokens / B)
    return fail(PSEQ_ERR_ARG, "%s: B*S = %lld*%lld exceeds the static scratch limit of %lld tokens", fn, (long long)B,
                (long long)S, (long long)kStaticMaxTokens);
  const int64_t N = B * S;
  if (N > 0 && !doc_ids) return fail(PSEQ_ERR_ARG, "%s: doc_ids is NULL", fn);
  if (!aligned(doc_ids, (uintptr_t)id_bytes) || !aligned(cu_seqlens, 4) || !aligned(info, 4))
    return fail(PSEQ_ERR_ARG, "%s: misaligned pointer", fn);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (N == 0) {
    empty_map_kernel<<<1, 1, 0, st>>>(cu_seqlens, info);
    count_launches(1);
    return check_launch(fn);
  }
  void* scratch = nullptr;
  pseq_status s = static_scratch(&scratch);
  if (s != PSEQ_OK) return s;
  const int64_t tiles = (N + kTile - 1) / kTile;
  // The counters and tile flags must start at zero.  A completed call leaves
  // them zero, but clear them anyway so an interrupted earlier call cannot leak
  // into this one.
  const size_t clear = sizeof(Header) + round_up(4 * (size_t)tiles, 16);
  cudaError_t e = cudaMemsetAsync(scratch, 0, clear, st);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: cudaMemsetAsync: %s", fn, cudaGetErrorString(e));
  Workspace ws = carve(scratch, tiles);
  if (id_bytes == 4)
    launch_scan<int32_t>(doc_ids, (int)N, (int)S, cu_seqlens, info, ws, (int)tiles, st);
  else
    launch_scan<int64_t>(doc_ids, (int)N, (int)S, cu_seqlens, info, ws, (int)tiles, st);
  count_launches(1);
  return check_launch(fn);
}
