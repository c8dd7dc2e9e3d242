// pseq_from_doc_ids: segment boundaries of a neat-packing document map.
//
// Follows NeMo AutoModel "nemo_automodel.components.datasets.packed_seq",
// packed_seq_params_from_doc_ids and PackedSeqParams: a segment is a maximal
// run of one document index within a row, every row start opens a segment,
// padding runs are segments, cu_seqlens ends at B*S, max_seqlen is the
// longest segment.
//
// One pass over doc_ids.  CTA t takes tile t (16384 tokens), flags the
// boundaries in it and summarises them as (count, first, last, largest inner
// gap) -- an associative "followed by" operation -- with a block scan.  A
// decoupled look-back over the preceding tiles then gives the tile its
// exclusive prefix: the output index of its first boundary and the position
// of the boundary before it, which closes the segment crossing into the tile.
// The gap term makes max_seqlen a by-product of the scan.
//
// Every published summary is two 64-bit words, each carrying a valid bit, so
// a single poll returns the summary itself: no flag-then-value round trip and
// no release fence on the publishing side.  A look-back round polls 32
// predecessors at once (one per lane), all loads in flight together, and
// joins them with a shuffle tree.  A map that fits one tile skips all of
// this.  Waits are bounded by a time limit and report PSEQ_ERR_TIMEOUT.
// Boundaries are compacted through shared memory (tile-relative 16-bit
// positions) and stored coalesced.
//
// The last tile, which holds the whole map's summary once its look-back
// ends, writes cu_seqlens[num_segments] and the info block itself.  The tiles
// count themselves done (with any failure they met) in one 64-bit word; the
// CTA whose add completes the count only reports a failure, if any, and
// clears the summary words, so the workspace is zero again for the next call
// and no tile summary is read back at the end.
#include <mutex>

#include "common.cuh"

namespace pseq {
namespace {

#ifndef PSEQ_SCAN_THREADS
#define PSEQ_SCAN_THREADS 1024
#endif
#ifndef PSEQ_SCAN_ITEMS
#define PSEQ_SCAN_ITEMS 16
#endif
constexpr int kThreads = PSEQ_SCAN_THREADS;
constexpr int kItems = PSEQ_SCAN_ITEMS;
constexpr int kPerLane = 1;  // look-back windows of 32 tiles polled together (more unrolled code costs more on a cold instruction cache than extra rounds)
constexpr int kTile = kThreads * kItems;  // tokens per tile
static_assert(kTile <= 65536, "tile-relative positions are 16-bit");

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

// A summary as two self-validating words: {valid, count, last} and
// {valid, gap, first}.  count and gap are below 2^31, positions fit 32 bits
// (-1 for "no boundary" round-trips through the unsigned field).
constexpr unsigned long long kValid = 1ull << 63;

__device__ __forceinline__ unsigned long long word_a(const Bounds& b) {
  return kValid | ((unsigned long long)(unsigned)b.count << 32) | (unsigned)b.last;
}
__device__ __forceinline__ unsigned long long word_b(const Bounds& b) {
  return kValid | ((unsigned long long)(unsigned)b.gap << 32) | (unsigned)b.first;
}
__device__ __forceinline__ Bounds from_words(unsigned long long a, unsigned long long b) {
  return {(int)((a >> 32) & 0x7fffffffu), (int)(unsigned)b, (int)(unsigned)a, (int)((b >> 32) & 0x7fffffffu)};
}

// Header word: tiles done (bits 0..19), tiles whose wait hit its time limit
// (bits 20..39), tiles that found a workspace that was not zero-filled
// (bits 40..59).  A map has at most 2^17 tiles, so no field overflows; the
// tile that completes the count resets the word to zero.
constexpr int kTimeoutShift = 20, kBadShift = 40;
constexpr unsigned long long kCountMask = (1ull << 20) - 1;

struct Header {
  unsigned long long state;
  unsigned long long pad[15];
};
static_assert(sizeof(Header) == 128, "header is 128 bytes");

// Per tile: its own summary and the inclusive one (everything up to it), one
// 128-byte line per tile, so that a tile's publishing and its neighbours'
// polls do not contend for one line (32-byte slots, four to a line, made the
// 2M-token map 4% slower).
struct Slot {
  unsigned long long agg_a, agg_b, inc_a, inc_b;
  unsigned long long pad[12];
};
static_assert(sizeof(Slot) == 128, "slot is 128 bytes");

struct Workspace {
  Header* hdr;
  Slot* slots;  // [tiles]
};

size_t workspace_bytes(int64_t tiles) { return sizeof(Header) + sizeof(Slot) * (size_t)tiles; }

Workspace carve(void* base, int64_t tiles) {
  unsigned char* p = static_cast<unsigned char*>(base);
  (void)tiles;
  return {reinterpret_cast<Header*>(p), reinterpret_cast<Slot*>(p + sizeof(Header))};
}

template <typename Id>
union Items {
  int4 q[kItems * sizeof(Id) / 16];
  Id v[kItems];
};

template <typename Id, bool kVector, int THREADS>
__global__ void __launch_bounds__(THREADS, THREADS <= 512 ? 2 : 1)
    doc_ids_scan_kernel(const Id* __restrict__ doc, int N, int S, int32_t* __restrict__ cu,
                        pseq_info* __restrict__ info, Workspace ws, int tiles, int64_t wait_ns,
                        int withhold) {
  __shared__ Bounds s_warp[(THREADS / 32)];
  __shared__ Bounds s_prefix;
  __shared__ int s_last_cta;
  __shared__ unsigned long long s_state;
  __shared__ unsigned short s_pos[(THREADS * kItems)];

  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x;
  const int64_t tile_base = (int64_t)tile * (THREADS * kItems);
  const int64_t t0 = tile_base + (int64_t)tid * kItems;

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

  // ---- boundary flags, one bit per token: a different index than the left
  // token, or a row start (the first at (S - t0 % S) % S, then every S).
  // Positions fit 32 bits: tiles * kTile < 2^31 + kTile.
  static_assert(kItems <= 32, "one flag bit per token");
  const unsigned pos0 = (unsigned)t0;
  const int live = t0 >= N ? 0 : (int)min((int64_t)kItems, N - t0);
  unsigned flags = 0;
#pragma unroll
  for (int k = 0; k < kItems; ++k) flags |= (unsigned)(it.v[k] != (k ? it.v[k - 1] : left)) << k;
  for (unsigned q = ((unsigned)S - pos0 % (unsigned)S) % (unsigned)S; q < (unsigned)kItems; q += (unsigned)S)
    flags |= 1u << q;
  flags &= live >= 32 ? ~0u : (1u << live) - 1u;
  Bounds mine = none();
  if (flags) {
    mine.count = __popc(flags);
    mine.first = (int)pos0 + __ffs(flags) - 1;
    mine.last = (int)pos0 + 31 - __clz(flags);
    int prev = __ffs(flags) - 1;
    for (unsigned m = flags & (flags - 1); m; m &= m - 1) {
      const int q = __ffs(m) - 1;
      mine.gap = max(mine.gap, q - prev);
      prev = q;
    }
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
    Bounds w = lane < (THREADS / 32) ? s_warp[lane] : none();
#pragma unroll
    for (int d = 1; d < (THREADS / 32); d <<= 1) {
      const Bounds o = shfl_up(w, d);
      if (lane >= d) w = join(o, w);
    }
    if (lane < (THREADS / 32)) s_warp[lane] = w;
  }
  __syncthreads();
  Bounds before_me = shfl_up(inc, 1);
  if (lane == 0) before_me = none();
  if (warp > 0) before_me = join(s_warp[warp - 1], before_me);
  const Bounds tile_sum = s_warp[(THREADS / 32) - 1];

  // ---- one tile: no neighbours, no workspace
  if (tiles == 1) {
    int li = before_me.count;
    for (unsigned m = flags; m; m &= m - 1) s_pos[li++] = (unsigned short)(t0 - tile_base + __ffs(m) - 1);
    __syncthreads();
    for (int i = tid; i < tile_sum.count; i += THREADS) cu[i] = (int32_t)s_pos[i];
    if (tid == 0) {
      cu[tile_sum.count] = N;
      *info = {PSEQ_OK, tile_sum.count, max(tile_sum.gap, N - tile_sum.last), N};
    }
    return;
  }

  // ---- publish the tile summary, then look back for the exclusive prefix
  bool timed_out = withhold == tile;  // (thread 0) a withheld summary is reported as a failed wait
  bool bad_ws = false;                // (thread 0)
  if (warp == 0) {
    Slot* mine_slot = ws.slots + tile;
    Bounds prefix = none();
    if (tile > 0) {
      if (lane == 0 && withhold != tile) {
        st_relaxed_u64(&mine_slot->agg_a, word_a(tile_sum));
        st_relaxed_u64(&mine_slot->agg_b, word_b(tile_sum));
      }
      // Each round polls kPerLane windows of 32 predecessors at once (lane L
      // of window w looks at tile j - 32w - L), waits until every one has
      // published, and joins the tiles after the nearest inclusive summary.
      Bounds run = none();  // summary of the tiles between the polled span and this one
      int j = tile - 1;
      bool gave_up = false;
      while (true) {
        Bounds b[kPerLane];
        bool incl[kPerLane], done[kPerLane];
#pragma unroll
        for (int w = 0; w < kPerLane; ++w) {
          b[w] = none();
          incl[w] = true;  // before tile 0: an empty inclusive prefix
          done[w] = j - 32 * w - lane < 0;
        }
        int polls = 0;
        uint64_t start = 0;
        while (true) {
          // issue every window's loads before looking at any of them, so a
          // round costs one L2 round trip however many windows are open
          unsigned long long ia[kPerLane], ib[kPerLane], aa[kPerLane], ab[kPerLane];
#pragma unroll
          for (int w = 0; w < kPerLane; ++w) {
            ia[w] = ib[w] = aa[w] = ab[w] = 0ull;
            if (!done[w]) {
              const Slot* sl = ws.slots + (j - 32 * w - lane);
              ia[w] = ld_relaxed_u64(&sl->inc_a);
              ib[w] = ld_relaxed_u64(&sl->inc_b);
              aa[w] = ld_relaxed_u64(&sl->agg_a);
              ab[w] = ld_relaxed_u64(&sl->agg_b);
            }
          }
          bool all_done = true;
#pragma unroll
          for (int w = 0; w < kPerLane; ++w) {
            if (done[w]) continue;
            if (ia[w] & ib[w] & kValid) {
              b[w] = from_words(ia[w], ib[w]);
              done[w] = true;
            } else if (aa[w] & ab[w] & kValid) {
              b[w] = from_words(aa[w], ab[w]);
              incl[w] = false;
              done[w] = true;
            } else {
              all_done = false;
            }
          }
          if (all_done) break;
          if (polls++ == 0) {
            start = global_ns();
          } else if ((int64_t)(global_ns() - start) >= wait_ns) {
            gave_up = true;  // treat what is missing as an empty inclusive prefix and finish
#pragma unroll
            for (int w = 0; w < kPerLane; ++w)
              if (!done[w]) {
                b[w] = none();
                incl[w] = true;
                done[w] = true;
              }
            break;
          }
        }
        // nearest inclusive summary: lowest window, then lowest lane
        int stop_w = kPerLane, stop_l = 32;
#pragma unroll
        for (int w = kPerLane - 1; w >= 0; --w) {
          const unsigned m = __ballot_sync(~0u, incl[w]);
          if (m) {
            stop_w = w;
            stop_l = __ffs(m) - 1;
          }
        }
        // Join the counted tiles, farthest first.  Within a window a higher
        // lane holds an earlier tile, so a shuffle-down tree leaves
        // x_31 . x_30 . ... . x_0 in lane 0; tiles past the inclusive one
        // count as empty.
#pragma unroll
        for (int w = 0; w < kPerLane; ++w) {
          if (w > stop_w || (w == stop_w && lane > stop_l)) b[w] = none();
#pragma unroll
          for (int d = 1; d < 32; d <<= 1) {
            const Bounds o = {__shfl_down_sync(~0u, b[w].count, d), __shfl_down_sync(~0u, b[w].first, d),
                              __shfl_down_sync(~0u, b[w].last, d), __shfl_down_sync(~0u, b[w].gap, d)};
            if (lane + d < 32) b[w] = join(o, b[w]);
          }
        }
        Bounds span = none();
#pragma unroll
        for (int w = kPerLane - 1; w >= 0; --w) span = join(span, shfl(b[w], 0));
        run = join(span, run);
        if (stop_w < kPerLane) break;
        j -= 32 * kPerLane;
      }
      if (__any_sync(~0u, gave_up)) timed_out = true;
      prefix = run;
    }
    if (lane == 0) {
      const Bounds all = join(prefix, tile_sum);
      if (withhold != tile) {
        st_relaxed_u64(&mine_slot->inc_a, word_a(all));
        st_relaxed_u64(&mine_slot->inc_b, word_b(all));
      }
      if (tile == tiles - 1 && !timed_out) {
        // the whole map: close the array and report (a failure elsewhere
        // overwrites the report at the end)
        if (all.count >= 1 && all.count <= N) {
          cu[all.count] = N;
          *info = {PSEQ_OK, all.count, max(all.gap, N - all.last), N};
        } else {
          bad_ws = true;
        }
      }
      s_prefix = prefix;
    }
  }

  // ---- compact this tile's boundary positions and store them
  int li = before_me.count;
  for (unsigned m = flags; m; m &= m - 1) s_pos[li++] = (unsigned short)(t0 - tile_base + __ffs(m) - 1);
  __syncthreads();
  const int base = s_prefix.count;
  if (base >= 0 && base <= N - tile_sum.count) {
    for (int i = tid; i < tile_sum.count; i += THREADS) cu[base + i] = (int32_t)(tile_base + s_pos[i]);
  } else if (tid == 0) {
    bad_ws = true;  // only reachable from a workspace that was not zero-filled
  }
  if (tid == 0) {
    const unsigned long long add =
        1ull | ((unsigned long long)timed_out << kTimeoutShift) | ((unsigned long long)bad_ws << kBadShift);
    const unsigned long long old = add_acq_rel_u64(&ws.hdr->state, add);
    s_last_cta = (old & kCountMask) == (unsigned long long)(tiles - 1);
    s_state = old + add;
  }
  __syncthreads();
  if (!s_last_cta) return;

  // ---- last CTA: report a failure, if any, and clear the workspace
  if (tid == 0) {
    const unsigned long long all = s_state;
    const bool timeouts = ((all >> kTimeoutShift) & kCountMask) != 0;
    const bool bad = ((all >> kBadShift) & kCountMask) != 0;
    if (timeouts || bad) *info = {bad ? PSEQ_ERR_ARG : PSEQ_ERR_TIMEOUT, 0, 0, N};
    ws.hdr->state = 0;  // the next call starts after this grid completes
  }
  unsigned long long* words = reinterpret_cast<unsigned long long*>(ws.slots);
  for (int i = tid; i < 4 * tiles; i += THREADS) words[(i >> 2) * 16 + (i & 3)] = 0ull;  // the four words of each slot
}

__global__ void empty_map_kernel(int32_t* cu, pseq_info* info) {
  pdl_enter();
  cu[0] = 0;
  *info = {PSEQ_OK, 0, 0, 0};
}

template <typename Id>
cudaError_t launch_scan(const void* doc, int N, int S, int32_t* cu, pseq_info* info, Workspace ws, int tiles,
                        cudaStream_t st) {
  const Id* d = static_cast<const Id*>(doc);
  const int64_t wait = wait_limit_ns();
  const int withhold = (int)(withhold_tile() < 0 ? -1 : (withhold_tile() > INT32_MAX ? -1 : withhold_tile()));
  // a map that fits half a tile runs as one 512-thread CTA (a 1024-thread
  // CTA would leave half its threads idle)
  constexpr int kSmall = 512;
  const bool small = tiles == 1 && N <= kSmall * kItems;
  if (aligned(doc, 16))
    return small ? launch_pdl(doc_ids_scan_kernel<Id, true, kSmall>, dim3(1), dim3(kSmall), 0, st, d, N, S, cu, info,
                              ws, tiles, wait, withhold)
                 : launch_pdl(doc_ids_scan_kernel<Id, true, kThreads>, dim3(tiles), dim3(kThreads), 0, st, d, N, S, cu,
                              info, ws, tiles, wait, withhold);
  return small ? launch_pdl(doc_ids_scan_kernel<Id, false, kSmall>, dim3(1), dim3(kSmall), 0, st, d, N, S, cu, info,
                            ws, tiles, wait, withhold)
               : launch_pdl(doc_ids_scan_kernel<Id, false, kThreads>, dim3(tiles), dim3(kThreads), 0, st, d, N, S, cu,
                            info, ws, tiles, wait, withhold);
}

cudaError_t launch_empty_map(int32_t* cu, pseq_info* info, cudaStream_t st) {
  return launch_pdl(empty_map_kernel, dim3(1), dim3(1), 0, st, cu, info);
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
    const cudaError_t e = launch_empty_map(cu_seqlens, info, st);
    count_launches(1);
    if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "pseq_from_doc_ids: %s", cudaGetErrorString(e));
    return check_launch("pseq_from_doc_ids");
  }
  const int64_t tiles = (N + kTile - 1) / kTile;
  const size_t need = workspace_bytes(tiles);
  if (!workspace || ws_bytes < need || !aligned(workspace, 16))
    return fail(PSEQ_ERR_ARG, "pseq_from_doc_ids: workspace needs %zu bytes, 16-byte aligned (got %zu)", need, ws_bytes);
  Workspace ws = carve(workspace, tiles);
  const cudaError_t e = id_bytes == 4
                            ? launch_scan<int32_t>(doc_ids, (int)N, (int)S, cu_seqlens, info, ws, (int)tiles, st)
                            : launch_scan<int64_t>(doc_ids, (int)N, (int)S, cu_seqlens, info, ws, (int)tiles, st);
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "pseq_from_doc_ids: %s", cudaGetErrorString(e));
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
constexpr size_t kStaticBytes = sizeof(Header) + sizeof(Slot) * kStaticMaxTiles;

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
    const cudaError_t e = launch_empty_map(cu_seqlens, info, st);
    count_launches(1);
    if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    return check_launch(fn);
  }
  void* scratch = nullptr;
  pseq_status s = static_scratch(&scratch);
  if (s != PSEQ_OK) return s;
  const int64_t tiles = (N + kTile - 1) / kTile;
  // The counters and summary words must start at zero.  A completed call
  // leaves them zero, but clear them anyway so an interrupted earlier call
  // cannot leak into this one.
  const size_t clear = workspace_bytes(tiles);
  cudaError_t e = cudaMemsetAsync(scratch, 0, clear, st);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: cudaMemsetAsync: %s", fn, cudaGetErrorString(e));
  Workspace ws = carve(scratch, tiles);
  e = id_bytes == 4 ? launch_scan<int32_t>(doc_ids, (int)N, (int)S, cu_seqlens, info, ws, (int)tiles, st)
                    : launch_scan<int64_t>(doc_ids, (int)N, (int)S, cu_seqlens, info, ws, (int)tiles, st);
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}
