// pseq_from_doc_ids: segment boundaries of a neat-packing document map.
//
// Follows NeMo AutoModel "nemo_automodel.components.datasets.packed_seq",
// packed_seq_params_from_doc_ids and PackedSeqParams: a segment is a maximal
// run of one document index within a row, every row start opens a segment,
// padding runs are segments, cu_seqlens ends at B*S, max_seqlen is the
// longest segment.
//
// One pass over doc_ids.  CTA t takes tile t (16384 tokens: 1024 threads x
// 16; a 2M-token map is 128 tiles, one per SM), flags the boundaries in it and summarises them as (count, first, last, largest inner
// gap) -- an associative "followed by" operation -- with a block scan.  A
// decoupled look-back over the preceding tiles then gives the tile its
// exclusive prefix: the output index of its first boundary and the position
// of the boundary before it, which closes the segment crossing into the
// tile.  The gap term makes max_seqlen a by-product of the scan.
//
// A tile's summary is one 16-byte slot of two 64-bit words, published first
// as the tile's own aggregate and then overwritten with the inclusive prefix
// (everything up to and including the tile).  Each word carries a published
// bit and an inclusive bit, so one poll returns the summary itself; a poll
// that catches the two words in different states (mid-overwrite) is simply
// repeated.  A look-back round polls 128 predecessors at once (four windows
// of 32, one per lane), all loads in flight together, and joins each window
// with one ballot, two warp reductions and three shuffles; a map of up to
// 129 tiles needs one round.  (Four windows with these joins measured
// faster than one or two on a 2M-token map; 896-thread tiles, which spread
// that map over 147 SMs instead of 128, did not help.)  Waits are bounded by a time limit and report
// PSEQ_ERR_TIMEOUT.
//
// Warp 0 runs the block scan's second level and the look-back; the other
// warps are released by a named barrier as soon as the block prefix is
// known and compact the tile's boundaries into shared memory (tile-relative
// 16-bit positions) while the look-back runs.  After it, the positions are
// stored coalesced with the prefix added.  A map that fits one tile skips
// the look-back and the workspace.
//
// The last tile, which holds the whole map's summary once its look-back
// ends, writes cu_seqlens[num_segments] and the info block itself.  Every
// other tile counts itself done (with any failure it met) in one 64-bit word
// with a release add that returns nothing, so no CTA waits for that round
// trip.  In the last tile, warp 1 waits for the count after its stores,
// then reports a failure, if any, and clears the summary words,
// so the workspace is zero again for the next call and no tile summary is
// read back at the end.
#include <mutex>

#include "common.cuh"

namespace pseq {
namespace {

#ifndef PSEQ_SCAN_THREADS
#define PSEQ_SCAN_THREADS 1024
#endif
#ifndef PSEQ_SCAN_WINDOWS
#define PSEQ_SCAN_WINDOWS 4
#endif
#ifndef PSEQ_SCAN_SLOT_BYTES
#define PSEQ_SCAN_SLOT_BYTES 16
#endif
constexpr int kThreads = PSEQ_SCAN_THREADS;
constexpr int kItems = 16;
constexpr int kWindows = PSEQ_SCAN_WINDOWS;  // windows of 32 predecessors polled per look-back round
constexpr int kSlotWords = PSEQ_SCAN_SLOT_BYTES / 8;
constexpr int kTile = kThreads * kItems;  // tokens per tile
static_assert(kTile <= 65536, "tile-relative positions are 16-bit");
static_assert(kThreads % 32 == 0 && kThreads <= 1024, "whole warps, one CTA");
static_assert(kSlotWords >= 2 && PSEQ_SCAN_SLOT_BYTES % 16 == 0, "a slot holds the two summary words");

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

// A summary as two self-validating words: {published, inclusive, count, last}
// and {published, inclusive, gap, first}.  count and gap are below 2^31 and
// take bits 31..61; positions are below 2^31 - 1 and take bits 0..30, with
// all ones standing for "no boundary".
constexpr unsigned long long kPublished = 1ull << 63;
constexpr unsigned long long kInclusive = 1ull << 62;
constexpr unsigned kNoPos = 0x7fffffffu;

__device__ __forceinline__ unsigned long long pos_bits(int p) { return p < 0 ? kNoPos : (unsigned)p; }
__device__ __forceinline__ int pos_of(unsigned long long w) {
  const unsigned v = (unsigned)(w & kNoPos);
  return v == kNoPos ? -1 : (int)v;
}
__device__ __forceinline__ unsigned long long word_a(const Bounds& b, bool incl) {
  return kPublished | (incl ? kInclusive : 0ull) | ((unsigned long long)(unsigned)b.count << 31) | pos_bits(b.last);
}
__device__ __forceinline__ unsigned long long word_b(const Bounds& b, bool incl) {
  return kPublished | (incl ? kInclusive : 0ull) | ((unsigned long long)(unsigned)b.gap << 31) | pos_bits(b.first);
}
__device__ __forceinline__ Bounds from_words(unsigned long long a, unsigned long long b) {
  return {(int)((a >> 31) & kNoPos), pos_of(b), pos_of(a), (int)((b >> 31) & kNoPos)};
}

// Header word: tiles done (bits 0..19), tiles whose wait hit its time limit
// (bits 20..39), tiles that found a workspace that was not zero-filled
// (bits 40..59).  A map has fewer than 2^18 tiles, so no field overflows;
// the tile that completes the count resets the word to zero.
constexpr int kTimeoutShift = 20, kBadShift = 40;
constexpr unsigned long long kCountMask = (1ull << 20) - 1;
// The last tile's wait for every other tile to count itself done.  Every
// other tile's own waits end within the wait limit (at most 1 s), so this
// bound is only reached after a device fault.
constexpr int64_t kArrivalWaitNs = 2000000000;

struct Header {
  unsigned long long state;
  unsigned long long pad[15];
};
static_assert(sizeof(Header) == 128, "header is 128 bytes");

struct Workspace {
  Header* hdr;
  unsigned long long* slots;  // [tiles][kSlotWords]: word a, word b, padding
};

size_t workspace_bytes(int64_t tiles) { return sizeof(Header) + 8 * (size_t)kSlotWords * (size_t)tiles; }

Workspace carve(void* base) {
  unsigned char* p = static_cast<unsigned char*>(base);
  return {reinterpret_cast<Header*>(p), reinterpret_cast<unsigned long long*>(p + sizeof(Header))};
}

// Named barrier 1: warp 0 arrives once the block prefix is in shared memory,
// the other warps wait for it (barrier 0 stays with __syncthreads).
__device__ __forceinline__ void bar_arrive_1(int threads) { asm volatile("bar.arrive 1, %0;" ::"r"(threads) : "memory"); }
__device__ __forceinline__ void bar_sync_1(int threads) { asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory"); }

template <typename Id>
union Items {
  int4 q[kItems * sizeof(Id) / 16];
  Id v[kItems];
};

// Summary of one look-back window: lane L holds the summary of the L-th tile
// back (higher lanes: earlier tiles); lanes with `use` false count as empty.
// One ballot, two warp reductions and three shuffles, the same in every
// lane.  The gap into a tile with boundaries is closed by the nearest
// earlier tile with boundaries in the window (the one before the window is
// handled when windows are joined).
__device__ __forceinline__ Bounds window_sum(const Bounds& b, bool use) {
  const int lane = threadIdx.x & 31;
  const int cnt = use ? b.count : 0;
  const unsigned nz = __ballot_sync(~0u, cnt > 0);
  Bounds r = none();
  r.count = (int)__reduce_add_sync(~0u, (unsigned)cnt);
  const unsigned earlier = lane == 31 ? 0u : nz & (~0u << (lane + 1));
  const int prev_last = __shfl_sync(~0u, b.last, earlier ? __ffs(earlier) - 1 : lane);
  int g = 0;
  if (cnt > 0) g = earlier ? max(b.gap, b.first - prev_last) : b.gap;
  r.gap = (int)__reduce_max_sync(~0u, (unsigned)g);
  if (nz) {
    r.last = __shfl_sync(~0u, b.last, __ffs(nz) - 1);
    r.first = __shfl_sync(~0u, b.first, 31 - __clz(nz));
  }
  return r;
}

// Joins the summaries of tiles j, j-1, ... going back until one of them is an
// inclusive prefix; returns the summary of everything before tile j + 1.
// Warp-wide; `gave_up` is set in every lane when a wait ran out.
__device__ __forceinline__ Bounds look_back(const unsigned long long* slots, int j, int64_t wait_ns, bool& gave_up) {
  const int lane = threadIdx.x & 31;
  Bounds run = none();  // summary of the tiles between the polled span and tile j + 1
  gave_up = false;
  while (true) {
    // lane L of window w looks at tile j - 32w - L
    Bounds b[kWindows];
    bool incl[kWindows], done[kWindows];
#pragma unroll
    for (int w = 0; w < kWindows; ++w) {
      b[w] = none();
      incl[w] = true;  // before tile 0: an empty inclusive prefix
      done[w] = j - 32 * w - lane < 0;
    }
    int polls = 0;
    uint64_t start = 0;
    bool timed_out = false;
    while (true) {
      // every window's loads are issued before any is looked at, so a round
      // costs one L2 round trip however many windows are open
      unsigned long long wa[kWindows], wb[kWindows];
#pragma unroll
      for (int w = 0; w < kWindows; ++w) {
        wa[w] = wb[w] = 0ull;
        if (!done[w]) {
          const unsigned long long* sl = slots + (size_t)(j - 32 * w - lane) * kSlotWords;
          wa[w] = ld_relaxed_u64(sl);
          wb[w] = ld_relaxed_u64(sl + 1);
        }
      }
      bool all_done = true;
#pragma unroll
      for (int w = 0; w < kWindows; ++w) {
        if (done[w]) continue;
        // both words published and in the same state; otherwise poll again
        if ((wa[w] & wb[w] & kPublished) && !((wa[w] ^ wb[w]) & kInclusive)) {
          b[w] = from_words(wa[w], wb[w]);
          incl[w] = (wa[w] & kInclusive) != 0;
          done[w] = true;
        } else {
          all_done = false;
        }
      }
      if (__all_sync(~0u, all_done)) break;
      if (polls++ == 0) {
        start = global_ns();
      } else if ((int64_t)(global_ns() - start) >= wait_ns) {
        timed_out = true;  // treat what is missing as an empty inclusive prefix and finish
#pragma unroll
        for (int w = 0; w < kWindows; ++w)
          if (!done[w]) {
            b[w] = none();
            incl[w] = true;
            done[w] = true;
          }
        break;
      }
    }
    if (__any_sync(~0u, timed_out)) gave_up = true;
    // nearest inclusive summary: lowest window, then lowest lane
    int stop_w = kWindows, stop_l = 32;
#pragma unroll
    for (int w = kWindows - 1; w >= 0; --w) {
      const unsigned m = __ballot_sync(~0u, incl[w]);
      if (m) {
        stop_w = w;
        stop_l = __ffs(m) - 1;
      }
    }
    // Join the counted tiles, farthest window first; tiles past the inclusive
    // one count as empty.
    Bounds span = none();
#pragma unroll
    for (int w = kWindows - 1; w >= 0; --w)
      span = join(span, window_sum(b[w], w < stop_w || (w == stop_w && lane <= stop_l)));
    run = join(span, run);
    if (stop_w < kWindows) return run;
    j -= 32 * kWindows;
  }
}

template <typename Id, bool kVector, int THREADS>
__global__ void __launch_bounds__(THREADS, 1)
    doc_ids_scan_kernel(const Id* __restrict__ doc, int N, int S, int32_t* __restrict__ cu,
                        pseq_info* __restrict__ info, Workspace ws, int tiles, int64_t wait_ns,
                        int withhold) {
  constexpr int kWarps = THREADS / 32;
  __shared__ Bounds s_warp[kWarps];
  __shared__ Bounds s_prefix;
  __shared__ unsigned long long s_fail;    // this tile's failures, in the header word's layout
  __shared__ unsigned short s_pos[(THREADS * kItems)];

  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x;
  const int64_t tile_base = (int64_t)tile * (THREADS * kItems);
  const int64_t t0 = tile_base + (int64_t)tid * kItems;

  // ---- this thread's 16 tokens and the token to their left (the previous
  // lane's last token; lane 0 loads its own)
  Items<Id> it;
  const Id left0 = (lane == 0 && t0 > 0 && t0 < N) ? __ldg(doc + t0 - 1) : Id(0);
  if (kVector && t0 + kItems <= N) {
    const int4* p = reinterpret_cast<const int4*>(doc + t0);
#pragma unroll
    for (int k = 0; k < (int)(kItems * sizeof(Id) / 16); ++k) it.q[k] = __ldg(p + k);
  } else {
#pragma unroll
    for (int k = 0; k < kItems; ++k) it.v[k] = (t0 + k < N) ? __ldg(doc + t0 + k) : Id(0);
  }
  Id left = __shfl_up_sync(~0u, it.v[kItems - 1], 1);
  if (lane == 0) left = left0;

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

  // ---- warp-level scan of the summaries (in token order)
  Bounds inc = mine;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const Bounds o = shfl_up(inc, d);
    if (lane >= d) inc = join(o, inc);
  }
  if (lane == 31) s_warp[warp] = inc;
  __syncthreads();
  Bounds before_me = shfl_up(inc, 1);
  if (lane == 0) before_me = none();

  // Tile-relative boundary positions, in order, from the thread's index of
  // its first boundary within the tile.
  auto compact = [&](int li) {
    for (unsigned m = flags; m; m &= m - 1) s_pos[li++] = (unsigned short)(t0 - tile_base + __ffs(m) - 1);
  };

  static_assert(THREADS >= 64, "warp 1 counts the tile done");
  bool timed_out = withhold == tile;  // (warp 0) a withheld summary is reported as a failed wait
  bool bad_ws = false;                // (thread 0)
  Bounds tile_sum;
  if (warp == 0) {
    // second level of the block scan: warp totals -> inclusive warp prefixes
    Bounds w = lane < kWarps ? s_warp[lane] : none();
#pragma unroll
    for (int d = 1; d < kWarps; d <<= 1) {
      const Bounds o = shfl_up(w, d);
      if (lane >= d) w = join(o, w);
    }
    if (lane < kWarps) s_warp[lane] = w;
    tile_sum = shfl(w, kWarps - 1);
    bar_arrive_1(THREADS);  // the other warps may compact now
    Bounds prefix = none();
    if (tiles > 1) {
      unsigned long long* mine_slot = ws.slots + (size_t)tile * kSlotWords;
      // publish at once; tile 0's own summary is already its inclusive prefix
      if (lane == 0 && withhold != tile) {
        st_relaxed_u64(mine_slot, word_a(tile_sum, tile == 0));
        st_relaxed_u64(mine_slot + 1, word_b(tile_sum, tile == 0));
      }
      compact(before_me.count);  // warp 0's own boundaries (block prefix: none)
      if (tile > 0) {
        bool gave_up;
        prefix = look_back(ws.slots, tile - 1, wait_ns, gave_up);
        if (gave_up) timed_out = true;
      }
      if (lane == 0) {
        const Bounds all = join(prefix, tile_sum);
        if (tile > 0 && withhold != tile) {
          st_relaxed_u64(mine_slot, word_a(all, true));
          st_relaxed_u64(mine_slot + 1, word_b(all, true));
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
        // a prefix that does not fit only comes from a workspace that was
        // not zero-filled
        if (prefix.count > N - tile_sum.count) bad_ws = true;
        s_fail = ((unsigned long long)timed_out << kTimeoutShift) | ((unsigned long long)bad_ws << kBadShift);
      }
    } else {
      compact(before_me.count);
    }
    if (lane == 0) s_prefix = prefix;
  } else {
    bar_sync_1(THREADS);
    before_me = join(s_warp[warp - 1], before_me);
    tile_sum = s_warp[kWarps - 1];
    compact(before_me.count);
  }
  __syncthreads();

  // ---- store this tile's boundary positions at the prefix
  if (tiles == 1) {
    for (int i = tid; i < tile_sum.count; i += THREADS) cu[i] = (int32_t)s_pos[i];
    if (tid == 0) {
      cu[tile_sum.count] = N;
      *info = {PSEQ_OK, tile_sum.count, max(tile_sum.gap, N - tile_sum.last), N};
    }
    return;
  }
  // Every tile but the last counts itself done (with its failures) with a
  // release add that returns nothing: after the barrier, every read and
  // write of the summaries by this tile has happened, and nobody waits for
  // the round trip.
  const bool last_tile = tile == tiles - 1;
  if (!last_tile && tid == 32) red_release_add_u64(&ws.hdr->state, 1ull | s_fail);
  const int base = s_prefix.count;
  if (base >= 0 && base <= N - tile_sum.count)  // else counted as a bad workspace above
    for (int i = tid; i < tile_sum.count; i += THREADS) cu[base + i] = (int32_t)(tile_base + s_pos[i]);
  if (!last_tile || warp != 1) return;

  // ---- last tile: once every other tile has counted itself done, report a
  // failure, if any, and clear the workspace (warp 1, after its stores)
  unsigned long long others = 0;
  if (lane == 0) {
    others = ld_acquire_u64(&ws.hdr->state);
    const uint64_t start = global_ns();
    while ((others & kCountMask) < (unsigned long long)(tiles - 1) &&
           (int64_t)(global_ns() - start) < kArrivalWaitNs)
      others = ld_acquire_u64(&ws.hdr->state);
  }
  others = __shfl_sync(~0u, others, 0);
  const unsigned long long all = others + s_fail;
  const bool complete = (others & kCountMask) == (unsigned long long)(tiles - 1);
  if (lane == 0) {
    const bool timeouts = !complete || ((all >> kTimeoutShift) & kCountMask) != 0;
    const bool bad = ((all >> kBadShift) & kCountMask) != 0;
    if (timeouts || bad) *info = {bad ? PSEQ_ERR_ARG : PSEQ_ERR_TIMEOUT, 0, 0, N};
    if (complete) ws.hdr->state = 0;  // the next call starts after this grid completes
  }
  // every look-back has ended: no tile reads a summary any more
  if (complete)
    for (int i = lane; i < 2 * tiles; i += 32) ws.slots[(size_t)(i >> 1) * kSlotWords + (i & 1)] = 0ull;
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
  // a map of up to 8192 tokens runs as one 512-thread CTA (a full-size CTA
  // would leave threads idle)
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
  Workspace ws = carve(workspace);
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
constexpr int64_t kStaticMaxTiles = (kStaticMaxTokens + kTile - 1) / kTile;  // a map at the limit fits
constexpr size_t kStaticBytes = sizeof(Header) + 8 * (size_t)kSlotWords * (size_t)kStaticMaxTiles;

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
  Workspace ws = carve(scratch);
  e = id_bytes == 4 ? launch_scan<int32_t>(doc_ids, (int)N, (int)S, cu_seqlens, info, ws, (int)tiles, st)
                    : launch_scan<int64_t>(doc_ids, (int)N, (int)S, cu_seqlens, info, ws, (int)tiles, st);
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}
