// pseq_from_doc_ids: segment boundaries of a neat-packing document map.
//
// Follows NeMo AutoModel "nemo_automodel.components.datasets.packed_seq",
// packed_seq_params_from_doc_ids and PackedSeqParams: a segment is a maximal
// run of one document index within a row, every row start opens a segment,
// padding runs are segments, cu_seqlens ends at B*S, max_seqlen is the
// longest segment.
//
// One pass over doc_ids.  CTA t takes tile t (16384 tokens: 1024 threads x
// 16; a 2M-token map is 128 tiles, one per SM), flags the boundaries in it
// and summarises them as (count, first, last, largest inner gap) -- an
// associative "followed by" operation.  A decoupled look-back over the
// preceding tiles then gives the tile its exclusive prefix: the output index
// of its first boundary and the position of the boundary before it, which
// closes the segment crossing into the tile.  The gap term makes max_seqlen
// a by-product of the scan.
//
// What the look-back waits for comes first: the tile's summary is a
// reduction (per warp one ballot, two warp reductions and three shuffles,
// then the same over the warps in warp 0), published at once.  Row starts
// are found with a multiplication by a precomputed reciprocal of S, not a
// division.  The running count each thread needs to place its boundaries is
// a separate one-field scan, done while warp 0 looks back: every warp
// compacts the tile's boundaries into shared memory as tile-relative 16-bit
// positions, and after the look-back they are stored coalesced with the
// prefix added.  A map that fits one tile skips the look-back and the
// workspace.
//
// A tile's summary is one 32-byte slot of four 64-bit words, published first
// as the tile's own aggregate and then overwritten with the inclusive prefix
// (everything up to and including the tile).  Each word carries the call's
// tag and an inclusive bit, so one poll returns the summary itself; a poll
// that catches the words in different states (mid-overwrite) is simply
// repeated.  A look-back round polls 128 predecessors at once (four windows
// of 32, one per lane), all loads in flight together, and joins each window
// with one ballot, two warp reductions and three shuffles; a map of up to
// 129 tiles needs one round.  Waits are bounded by a time limit and report
// PSEQ_ERR_TIMEOUT.
//
// The tag is one more than the previous call's, read from the workspace
// header, so the slots a call leaves behind are never read as this call's
// and nothing has to be cleared: the kernel ends when the last tile's
// stores do.  The last tile, which holds the whole map's summary once its
// look-back ends, writes cu_seqlens[num_segments] and the counts of the
// info block, and advances the header.  Tile 0, which has no look-back,
// writes the success status early and marks it written (a release off every
// critical path); a tile whose wait ran out waits for that mark and then
// overwrites the status.  The call that takes the last tag zero-fills the
// whole buffer once every tile has counted itself done, and the numbering
// starts again.
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
constexpr int kThreads = PSEQ_SCAN_THREADS;
constexpr int kItems = 16;
constexpr int kWindows = PSEQ_SCAN_WINDOWS;  // windows of 32 predecessors polled per look-back round
constexpr int kSlotWords = 4;                // a tile's summary: count, last, first, gap
constexpr int kTile = kThreads * kItems;     // tokens per tile
static_assert(kTile <= 65536, "tile-relative positions are 16-bit");
static_assert(kThreads % 32 == 0 && kThreads <= 1024, "whole warps, one CTA");

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

// A published summary is four 64-bit words, one per field.  Each carries the
// tag of the call that wrote it (bits 32..63), whether it is an inclusive
// prefix (bit 31) and the field (bits 0..30; a position of all ones stands
// for "no boundary").  Tags run 1, 2, ..., 2^32 - 1 from the workspace
// header; 0 never matches, so a zero-filled slot reads as unpublished.
constexpr unsigned long long kInclusive = 1ull << 31;
constexpr unsigned kNoPos = 0x7fffffffu;
constexpr unsigned kLastTag = 0xffffffffu;

__device__ __forceinline__ unsigned pos_bits(int p) { return p < 0 ? kNoPos : (unsigned)p; }
__device__ __forceinline__ int pos_of(unsigned long long w) {
  const unsigned v = (unsigned)w & kNoPos;
  return v == kNoPos ? -1 : (int)v;
}
__device__ __forceinline__ unsigned long long tagged(unsigned tag, bool incl, unsigned v) {
  return ((unsigned long long)tag << 32) | (incl ? kInclusive : 0ull) | v;
}
__device__ __forceinline__ void publish(unsigned long long* slot, const Bounds& b, bool incl, unsigned tag) {
  st_relaxed_v4_u64(slot, tagged(tag, incl, (unsigned)b.count), tagged(tag, incl, pos_bits(b.last)),
                    tagged(tag, incl, pos_bits(b.first)), tagged(tag, incl, (unsigned)b.gap));
}

// Header.  epoch: the tag of the last call (low 32 bits).  reported: the
// tag of the call whose success status has been written (a tile that failed
// writes its status after that).  state, used only by the call that takes
// the last tag: tiles done (bits 0..19), tiles whose wait hit its time limit
// (bits 20..39), tiles that found a workspace that was not zero-filled (bits
// 40..59); a map has fewer than 2^18 tiles, so no field overflows.
constexpr int kTimeoutShift = 20, kBadShift = 40;
constexpr unsigned long long kCountMask = (1ull << 20) - 1;
// A failed tile's wait for the success status to be written, or the last tile's wait for
// every other tile to count itself done.  Every look-back wait ends within
// the wait limit (at most 1 s), so this bound is only reached after a
// device fault.
constexpr int64_t kArrivalWaitNs = 2000000000;

struct Header {
  unsigned long long epoch;
  unsigned long long reported;
  unsigned long long state;
  unsigned long long pad[13];
};
static_assert(sizeof(Header) == 128, "header is 128 bytes");

struct Workspace {
  Header* hdr;
  unsigned long long* slots;  // [capacity][kSlotWords]
  int64_t capacity;           // slots the caller's buffer holds
};

// The slots start at the first 32-byte boundary after the header (one
// 256-bit access per slot); a 16-byte aligned buffer needs 16 bytes of slack.
constexpr size_t kSlotBytes = 8 * kSlotWords;
constexpr size_t workspace_bytes(int64_t tiles) { return sizeof(Header) + 16 + kSlotBytes * (size_t)tiles; }

Workspace carve(void* base, size_t bytes) {
  const uintptr_t b = reinterpret_cast<uintptr_t>(base);
  const uintptr_t s = (b + sizeof(Header) + kSlotBytes - 1) & ~(uintptr_t)(kSlotBytes - 1);
  return {reinterpret_cast<Header*>(base), reinterpret_cast<unsigned long long*>(s),
          (int64_t)((b + bytes - s) / kSlotBytes)};
}

// Named barrier 1: warp 0 arrives once the tile's output index and its
// boundary positions are in shared memory; the other warps wait for it and
// store (barrier 0 stays with __syncthreads).
__device__ __forceinline__ void bar_arrive_1(int threads) { asm volatile("bar.arrive 1, %0;" ::"r"(threads) : "memory"); }
__device__ __forceinline__ void bar_sync_1(int threads) { asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory"); }

template <typename Id>
union Items {
  int4 q[kItems * sizeof(Id) / 16];
  Id v[kItems];
};

// Summary of the 32 lanes' spans taken in lane order (lane 0 first), in
// every lane: one ballot, two warp reductions (redux add and max) and three
// shuffles.  The gap into a lane with boundaries is closed by the nearest
// lower lane with boundaries.
__device__ __forceinline__ Bounds lanes_sum(const Bounds& b) {
  const int lane = threadIdx.x & 31;
  const unsigned nz = __ballot_sync(~0u, b.count > 0);
  Bounds r = none();
  r.count = (int)__reduce_add_sync(~0u, (unsigned)b.count);
  const unsigned earlier = nz & ((1u << lane) - 1u);
  const int prev_last = __shfl_sync(~0u, b.last, earlier ? 31 - __clz(earlier) : lane);
  int g = 0;
  if (b.count > 0) g = earlier ? max(b.gap, b.first - prev_last) : b.gap;
  r.gap = (int)__reduce_max_sync(~0u, (unsigned)g);
  if (nz) {
    r.first = __shfl_sync(~0u, b.first, __ffs(nz) - 1);
    r.last = __shfl_sync(~0u, b.last, 31 - __clz(nz));
  }
  return r;
}

// Division by an invariant divisor d < 2^31 for dividends n < 2^31: with
// l = ceil(log2 d) and m = ceil(2^(31+l) / d), floor(n / d) =
// floor(n * m / 2^(31+l)) (Granlund and Montgomery, "Division by invariant
// integers using multiplication", 1994, Theorem 4.2 with N = 31), and
// m < 2^32.
struct DivBy {
  unsigned d, m;
  int shift;  // l - 1, or -1 for d == 1
};

DivBy div_by(unsigned d) {
  int l = 0;
  while ((1ull << l) < d) ++l;
  if (l == 0) return {d, 0u, -1};
  return {d, (unsigned)(((1ull << (31 + l)) + d - 1) / d), l - 1};
}

__device__ __forceinline__ unsigned mod_by(unsigned n, DivBy v) {
  const unsigned q = v.shift < 0 ? n : (__umulhi(n, v.m) >> v.shift);
  return n - q * v.d;
}

// Joins the summaries of tiles j, j-1, ... going back until one of them is an
// inclusive prefix of this call (tag); returns the summary of everything
// before tile j + 1.  The boundary count of that span is known before its
// other fields and goes to on_count(count) first (every lane calls it once).
// Warp-wide; `gave_up` is set in every lane when a wait ran out.
template <typename OnCount>
__device__ __forceinline__ Bounds look_back(const unsigned long long* slots, int j, unsigned tag, int64_t wait_ns,
                                            bool& gave_up, OnCount&& on_count) {
  const int lane = threadIdx.x & 31;
  Bounds run = none();  // summary of the tiles between the polled span and tile j + 1
  gave_up = false;
  // the words of an empty inclusive prefix: what lies before tile 0, and what
  // a wait that ran out stands in for
  const unsigned long long e_count = tagged(tag, true, 0u), e_pos = tagged(tag, true, kNoPos);
  while (true) {
    // lane L of window w looks at tile j - 32w - L; the raw words stay live
    // while polling and are decoded once every window is in
    unsigned long long w0[kWindows], w1[kWindows], w2[kWindows], w3[kWindows];
    bool done[kWindows];
#pragma unroll
    for (int w = 0; w < kWindows; ++w) {
      done[w] = j - 32 * w - lane < 0;
      w0[w] = w3[w] = e_count;
      w1[w] = w2[w] = e_pos;
    }
    int polls = 0;
    uint64_t start = 0;
    bool timed_out = false;
    while (true) {
      // every window's loads are issued before any is looked at, so a round
      // costs one L2 round trip however many windows are open
#pragma unroll
      for (int w = 0; w < kWindows; ++w)
        if (!done[w]) {
          const unsigned long long* sl = slots + (size_t)(j - 32 * w - lane) * kSlotWords;
          ld_relaxed_v4_u64(sl, w0[w], w1[w], w2[w], w3[w]);
        }
      bool all_done = true;
#pragma unroll
      for (int w = 0; w < kWindows; ++w) {
        if (done[w]) continue;
        // all four words written by this call and in the same state;
        // otherwise poll again
        const unsigned long long a = w0[w] & w1[w] & w2[w] & w3[w], o = w0[w] | w1[w] | w2[w] | w3[w];
        done[w] = (unsigned)(a >> 32) == tag && (unsigned)(o >> 32) == tag && !((a ^ o) & kInclusive);
        all_done = all_done && done[w];
      }
      if (__all_sync(~0u, all_done)) break;
      if (polls++ == 0) {
        start = global_ns();
      } else if ((int64_t)(global_ns() - start) >= wait_ns) {
        timed_out = true;  // treat what is missing as an empty inclusive prefix and finish
#pragma unroll
        for (int w = 0; w < kWindows; ++w)
          if (!done[w]) {
            w0[w] = w3[w] = e_count;
            w1[w] = w2[w] = e_pos;
          }
        break;
      }
    }
    Bounds b[kWindows];
    bool incl[kWindows];
#pragma unroll
    for (int w = 0; w < kWindows; ++w) {
      b[w] = {(int)((unsigned)w0[w] & kNoPos), pos_of(w2[w]), pos_of(w1[w]), (int)((unsigned)w3[w] & kNoPos)};
      incl[w] = (w0[w] & kInclusive) != 0;
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
    // The span from the inclusive tile (or the farthest polled one) up to tile
    // j, in one pass over all windows: tiles past the inclusive one count as
    // empty.  Each tile with boundaries closes the gap from the nearest
    // earlier tile with boundaries: in its window the next lane up that has
    // some, else the lowest such lane of the nearest earlier window.
    int cnt[kWindows];
    unsigned nz[kWindows];
    int low_last[kWindows];  // last boundary of the window's nearest tile with boundaries
#pragma unroll
    for (int w = 0; w < kWindows; ++w) {
      cnt[w] = (w < stop_w || (w == stop_w && lane <= stop_l)) ? b[w].count : 0;
      nz[w] = __ballot_sync(~0u, cnt[w] > 0);
    }
    int sum = 0;
#pragma unroll
    for (int w = 0; w < kWindows; ++w) {
      sum += cnt[w];
      low_last[w] = __shfl_sync(~0u, b[w].last, nz[w] ? __ffs(nz[w]) - 1 : 0);
    }
    Bounds span = none();
    span.count = (int)__reduce_add_sync(~0u, (unsigned)sum);
    if (stop_w < kWindows) on_count(span.count + run.count);
    int g = 0, carry = -1;  // carry: last boundary before window w, within the span
#pragma unroll
    for (int w = kWindows - 1; w >= 0; --w) {
      const unsigned up = lane == 31 ? 0u : nz[w] & (~0u << (lane + 1));
      const int v = __shfl_sync(~0u, b[w].last, up ? __ffs(up) - 1 : lane);
      const int prev = up ? v : carry;
      if (cnt[w] > 0) g = max(g, prev >= 0 ? max(b[w].gap, b[w].first - prev) : b[w].gap);
      if (nz[w]) carry = low_last[w];
    }
    span.gap = (int)__reduce_max_sync(~0u, (unsigned)g);
    // first: the farthest tile with boundaries; last: the nearest
#pragma unroll
    for (int w = 0; w < kWindows; ++w) {
      const int f = __shfl_sync(~0u, b[w].first, nz[w] ? 31 - __clz(nz[w]) : 0);
      if (nz[w]) span.first = f;
    }
#pragma unroll
    for (int w = kWindows - 1; w >= 0; --w)
      if (nz[w]) span.last = low_last[w];
    run = join(span, run);
    if (stop_w < kWindows) return run;
    j -= 32 * kWindows;
  }
}

template <typename Id, bool kVector, int THREADS>
__global__ void __launch_bounds__(THREADS, 1)
    doc_ids_scan_kernel(const Id* __restrict__ doc, int N, DivBy S, int32_t* __restrict__ cu,
                        pseq_info* __restrict__ info, Workspace ws, int tiles, int64_t wait_ns,
                        int withhold) {
  constexpr int kWarps = THREADS / 32;
  static_assert(kWarps >= 2 && kWarps <= 32, "one lane per warp; warp 1 takes the last tile's tail");
  __shared__ Bounds s_warp[kWarps];
  __shared__ int s_base;  // the tile's first output index
  __shared__ unsigned short s_pos[(THREADS * kItems)];

  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x;
  const int64_t tile_base = (int64_t)tile * (THREADS * kItems);
  const int64_t t0 = tile_base + (int64_t)tid * kItems;
  // the previous call's tag (warp 0, which publishes and polls, and tile 0's
  // warp 1, which writes the success status; the load's latency hides
  // behind the token loads)
  unsigned e0 = 0;
  if ((warp == 0 || (warp == 1 && tile == 0)) && tiles > 1) e0 = (unsigned)ld_relaxed_u64(&ws.hdr->epoch);

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
  {
    const unsigned r = mod_by(pos0, S);  // meaningless past the map (t0 >= N), where every flag is masked off
    for (unsigned q = r ? S.d - r : 0u; q < (unsigned)kItems; q += S.d) flags |= 1u << q;
  }
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

  // ---- the tile's summary first, since the look-back waits for it: each
  // warp's span, then (warp 0) the block's
  {
    const Bounds w = lanes_sum(mine);
    if (lane == 0) s_warp[warp] = w;
  }
  __syncthreads();

  // Tile-relative boundary positions, in token order: this thread's first
  // goes after the boundaries of the warps before it and of the lanes
  // before it.
  auto compact = [&]() {
    int li = (int)__reduce_add_sync(~0u, (unsigned)(lane < warp ? s_warp[lane].count : 0));
    int c = mine.count;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(~0u, c, d);
      if (lane >= d) c += o;
    }
    li += c - mine.count;
    for (unsigned m = flags; m; m &= m - 1) s_pos[li++] = (unsigned short)(t0 - tile_base + __ffs(m) - 1);
  };

  const bool last_tile = tile == tiles - 1;
  if (warp != 0) {
    if (tiles > 1 && tile == 0 && tid == 32) {
      // the success status, before any tile can have failed (a failure
      // takes a wait that ran out, or a look-back; tile 0 has none); a tile
      // that failed sees `reported` and then overwrites it
      const unsigned tag = e0 < kLastTag ? e0 + 1 : 1u;
      info->status = PSEQ_OK;
      st_release_u64(&ws.hdr->reported, tag);
    }
    const int tile_count = (int)__reduce_add_sync(~0u, (unsigned)(lane < kWarps ? s_warp[lane].count : 0));
    compact();
    // ---- once warp 0 has the tile's output index: its boundary positions
    bar_sync_1(THREADS);
    const int base = s_base;
    if (base >= 0 && base <= N - tile_count)  // else reported as a bad workspace
      for (int i = tid - 32; i < tile_count; i += THREADS - 32) cu[base + i] = (int32_t)(tile_base + s_pos[i]);
    return;
  }

  // ---- warp 0: the tile's summary, the look-back and the reports
  const Bounds tile_sum = lanes_sum(lane < kWarps ? s_warp[lane] : none());
  // hands the tile's output index to the other warps, which store
  auto release_stores = [&](int base) {
    if (lane == 0) s_base = base;
    __syncwarp();
    bar_arrive_1(THREADS);
  };
  if (tiles == 1) {
    compact();
    release_stores(0);
    if (lane == 0) {
      cu[tile_sum.count] = N;
      *info = {PSEQ_OK, tile_sum.count, max(tile_sum.gap, N - tile_sum.last), N};
    }
    return;
  }
  const unsigned tag = e0 < kLastTag ? e0 + 1 : 1u;
  unsigned long long* mine_slot = ws.slots + (size_t)tile * kSlotWords;
  // publish at once; tile 0's own summary is already its inclusive prefix
  if (lane == 0 && withhold != tile) publish(mine_slot, tile_sum, tile == 0, tag);
  compact();  // warp 0's own boundaries
  bool timed_out = withhold == tile;  // a withheld summary is reported as a failed wait
  Bounds prefix = none();
  if (tile > 0) {
    bool gave_up;
    prefix = look_back(ws.slots, tile - 1, tag, wait_ns, gave_up, release_stores);
    if (gave_up) timed_out = true;
  } else {
    release_stores(0);
  }
  // a prefix that does not fit only comes from a workspace that was not
  // zero-filled before its first use
  bool bad_ws = prefix.count > N - tile_sum.count;
  if (lane == 0) {
    const Bounds all = join(prefix, tile_sum);
    if (!last_tile) {
      if (tile > 0 && withhold != tile) publish(mine_slot, all, true, tag);
    } else {
      // the whole map: close the array and report (tile 0 writes the
      // status).  Every tile read the header before publishing, and this
      // look-back ended only after every tile had published: the header may
      // take this call's tag.
      if (all.count < 1 || all.count > N) bad_ws = true;
      if (!timed_out && !bad_ws) {
        cu[all.count] = N;
        info->count = all.count;
        info->max_seqlen = max(all.gap, N - all.last);
        info->total = N;
      }
      if (tag != kLastTag) st_relaxed_u64(&ws.hdr->epoch, tag);
    }
  }
  bad_ws = __shfl_sync(~0u, bad_ws, 0);
  const unsigned long long fail =
      ((unsigned long long)timed_out << kTimeoutShift) | ((unsigned long long)bad_ws << kBadShift);

  // A tile that failed writes its status once the success status is out.
  auto report_failure = [&](bool bad) {
    const uint64_t start = global_ns();
    while ((unsigned)ld_acquire_u64(&ws.hdr->reported) != tag && (int64_t)(global_ns() - start) < kArrivalWaitNs) {
    }
    *info = {bad ? PSEQ_ERR_ARG : PSEQ_ERR_TIMEOUT, 0, 0, N};
  };
  if (tag != kLastTag) {
    if (lane == 0 && fail) report_failure(bad_ws);
    return;
  }

  // ---- the call with the last tag (one in 2^32 - 1): every tile counts
  // itself done once it reads no summary any more; the last tile, once all
  // have, reports their failures, zero-fills every slot of the buffer and
  // resets the header, so the next call starts the tags again at 1 and no
  // stale slot can carry them
  if (!last_tile) {
    if (lane == 0) red_release_add_u64(&ws.hdr->state, 1ull | fail);
    return;
  }
  unsigned long long others = 0;
  if (lane == 0) {
    others = ld_acquire_u64(&ws.hdr->state);
    const uint64_t start = global_ns();
    while ((others & kCountMask) < (unsigned long long)(tiles - 1) &&
           (int64_t)(global_ns() - start) < kArrivalWaitNs)
      others = ld_acquire_u64(&ws.hdr->state);
  }
  others = __shfl_sync(~0u, others, 0) + fail;
  const bool complete = (others & kCountMask) == (unsigned long long)(tiles - 1);
  if (lane == 0) {
    const bool timeouts = !complete || ((others >> kTimeoutShift) & kCountMask) != 0;
    const bool bad = ((others >> kBadShift) & kCountMask) != 0;
    if (timeouts || bad) report_failure(bad);
  }
  if (!complete) return;  // the header keeps the previous tag: the next call takes the last tag again
  for (int64_t i = lane; i < ws.capacity * kSlotWords; i += 32) ws.slots[i] = 0ull;
  __syncwarp();
  if (lane == 0) {
    ws.hdr->state = 0;
    ws.hdr->reported = 0;
    ws.hdr->epoch = 0;
  }
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
  const DivBy Sd = div_by((unsigned)S);
  if (aligned(doc, 16))
    return small ? launch_pdl(doc_ids_scan_kernel<Id, true, kSmall>, dim3(1), dim3(kSmall), 0, st, d, N, Sd, cu, info,
                              ws, tiles, wait, withhold)
                 : launch_pdl(doc_ids_scan_kernel<Id, true, kThreads>, dim3(tiles), dim3(kThreads), 0, st, d, N, Sd, cu,
                              info, ws, tiles, wait, withhold);
  return small ? launch_pdl(doc_ids_scan_kernel<Id, false, kSmall>, dim3(1), dim3(kSmall), 0, st, d, N, Sd, cu, info,
                            ws, tiles, wait, withhold)
               : launch_pdl(doc_ids_scan_kernel<Id, false, kThreads>, dim3(tiles), dim3(kThreads), 0, st, d, N, Sd, cu,
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
  Workspace ws = carve(workspace, ws_bytes);
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
constexpr size_t kStaticBytes = workspace_bytes(kStaticMaxTiles);  // a map at the limit, slack included

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
  Workspace ws = carve(scratch, kStaticBytes);
  e = id_bytes == 4 ? launch_scan<int32_t>(doc_ids, (int)N, (int)S, cu_seqlens, info, ws, (int)tiles, st)
                    : launch_scan<int64_t>(doc_ids, (int)N, (int)S, cu_seqlens, info, ws, (int)tiles, st);
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}
