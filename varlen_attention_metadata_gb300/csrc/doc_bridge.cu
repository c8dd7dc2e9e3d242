// pseq_doc_ids_to_lengths: the neat-packing document map of NeMo AutoModel
// "nemo_automodel.components.datasets.packed_seq" (1-based document index per
// token, 0 = padding) turned into the pack-length format that
// "nemo_automodel.components.distributed.thd_utils" process_input_for_thd
// consumes (seq_lens / seq_lens_padded [B, num_packs], filler for unused
// slots), plus per-document position ids.
//
// Readings (the pages connect the two formats but do not spell this out):
// every maximal run of one non-zero index within a row is a sequence whose
// real length is the run length; a padding run that follows a document run
// belongs to that sequence's padded length; a padding run at the start of a
// row is a sequence of real length 0.  Positions count 0, 1, ... inside each
// document run and are 0 on padding.
//
// One pass.  Every row is cut into chunks of 4096 tokens, one CTA each.  A
// chunk summarises its tokens -- how many sequences start in it, its last run
// start, its last sequence start (a commutative join: sum, max, max) -- with
// warp reductions, publishes that summary, and looks back over the chunks
// before it in its row for the row prefix (self-validating words, 32
// predecessors per poll round, stopping at the nearest inclusive prefix,
// bounded waits).  It then walks its tokens: every run end writes its
// sequence's real length, every sequence start closes the padded length of
// the one before it, and the row's last chunk closes the row.  One more CTA
// per row, dispatched after the row's chunks, waits for the row's sequence
// count (the last chunk's inclusive summary) and fills the row's unused
// slots, so no chunk waits for that.  Each chunk adds its share to the
// call's totals in the workspace header (atomics that return nothing); the
// CTA that finishes last (a wrapping acq_rel counter) reads them into the
// info block, resets them and clears the summary words, so the workspace is
// zero again for the next call.
#include "common.cuh"

namespace pseq {
namespace {

constexpr int kThreads = 256;
constexpr int kItems = 16;  // 4096-token chunks; four CTAs per SM, so one wave covers a [64, 32768] map
constexpr int kTile = kThreads * kItems;

struct Header {
  unsigned finished;  // CTAs done with their look-back; wraps back to 0 after each call
  unsigned gave_up;   // a wait hit its time limit
  // the call's running totals, reset by the CTA that finishes last: longest
  // document run, a row that overflowed its slots, most sequences in a row,
  // sequences in all rows
  unsigned longest, overflow, most, total;
  unsigned pad[26];
};

static_assert(sizeof(Header) == 128, "header is 128 bytes");

// Per chunk: its own summary and the inclusive one (the row up to it), each
// as two words carrying a valid bit.
struct Slot {
  unsigned long long agg_a, agg_b, inc_a, inc_b;
};

size_t workspace_bytes(int64_t B, int64_t S) {
  const int64_t chunks = S > 0 ? (S + kTile - 1) / kTile : 1;
  return sizeof(Header) + sizeof(Slot) * (size_t)(B > 0 ? B : 1) * (size_t)chunks;
}

constexpr unsigned long long kValid = 1ull << 63;

// Scan element: sequence starts counted, last run start, last sequence start.
struct Marks {
  int seqs, last_run, last_seq;
};

__device__ __forceinline__ Marks join(const Marks& a, const Marks& b) {
  return {a.seqs + b.seqs, max(a.last_run, b.last_run), max(a.last_seq, b.last_seq)};
}

// The join of every lane's marks, in every lane (three warp reductions).
__device__ __forceinline__ Marks warp_join(const Marks& v) {
  return {(int)__reduce_add_sync(~0u, (unsigned)v.seqs), __reduce_max_sync(~0u, v.last_run),
          __reduce_max_sync(~0u, v.last_seq)};
}

// {valid, seqs, last_run} and {valid, last_seq}; positions -1 ("none") round-
// trip through the unsigned low word.
__device__ __forceinline__ unsigned long long word_a(const Marks& m) {
  return kValid | ((unsigned long long)(unsigned)m.seqs << 32) | (unsigned)m.last_run;
}
__device__ __forceinline__ unsigned long long word_b(const Marks& m) { return kValid | (unsigned)m.last_seq; }
__device__ __forceinline__ Marks from_words(unsigned long long a, unsigned long long b) {
  return {(int)((a >> 32) & 0x7fffffffu), (int)(unsigned)a, (int)(unsigned)b};
}

struct BridgeArgs {
  int B, S, P, chunks;
  int64_t pad_value;
  int64_t* seq_lens;
  int64_t* seq_lens_padded;
  int64_t* positions;  // may be NULL
  pseq_info* info;
  Header* hdr;
  Slot* slots;         // [B * chunks]
  int64_t wait_ns;
  int64_t withhold;    // chunk (row-major) that never publishes: failure tests only
};

// This thread's eight tokens of a row chunk: run starts, sequence starts.
template <typename Id>
__device__ __forceinline__ Marks chunk_flags(const Id* d, int S, int s0, unsigned& runs, unsigned& seqs,
                                             unsigned& nz, unsigned& pnz) {
  Id v[kItems];
  if (s0 + kItems <= S && (reinterpret_cast<uintptr_t>(d + s0) & 15) == 0) {
    // whole group in the row and 16-byte aligned: vector loads
    constexpr int kVec = kItems * (int)sizeof(Id) / 16;
    constexpr int kPer = 16 / (int)sizeof(Id);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int4 q = ld_stream(reinterpret_cast<const int4*>(d + s0) + k);
      if constexpr (kPer == 4) {
        v[4 * k] = (Id)q.x;
        v[4 * k + 1] = (Id)q.y;
        v[4 * k + 2] = (Id)q.z;
        v[4 * k + 3] = (Id)q.w;
      } else {
        v[2 * k] = (Id)(((unsigned long long)(unsigned)q.y << 32) | (unsigned)q.x);
        v[2 * k + 1] = (Id)(((unsigned long long)(unsigned)q.w << 32) | (unsigned)q.z);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < kItems; ++k) v[k] = s0 + k < S ? __ldg(d + s0 + k) : Id(0);
  }
  const Id left = (s0 > 0 && s0 < S) ? __ldg(d + s0 - 1) : Id(0);
  runs = 0;
  seqs = 0;
  nz = 0;
  Marks mine = {0, -1, -1};
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int s = s0 + k;
    if (s >= S) break;
    const Id prev = k ? v[k - 1] : left;
    if (v[k] != 0) nz |= 1u << k;
    if (s == 0 || v[k] != prev) {
      runs |= 1u << k;
      mine.last_run = s;
    }
    if (s == 0 || (v[k] != 0 && v[k] != prev)) {
      seqs |= 1u << k;
      mine.last_seq = s;
      mine.seqs += 1;
    }
  }
  // bit k: the token before token k is a document token
  pnz = (nz << 1) | (left != 0 ? 1u : 0u);
  return mine;
}

// The row prefix of chunk `ch`: join of every earlier chunk of the row,
// looking back in rounds of 32 (lane L polls chunk j - L) and stopping at the
// nearest inclusive summary.  Warp 0 only.
__device__ __forceinline__ Marks row_prefix(const BridgeArgs& a, const Slot* row_slots, int ch, bool& gave_up) {
  const int lane = threadIdx.x & 31;
  Marks run = {0, -1, -1};
  int j = ch - 1;
  while (j >= 0) {
    const int t = j - lane;
    bool done = t < 0, incl = true;
    Marks m = {0, -1, -1};
    // each lane polls its own chunk until it has a summary or its wait runs
    // out; no warp-wide operation inside the loop
    int polls = 0;
    uint64_t start = 0;
    while (!done) {
      const Slot* sl = row_slots + t;
      const unsigned long long ia = ld_relaxed_u64(&sl->inc_a), ib = ld_relaxed_u64(&sl->inc_b);
      const unsigned long long aa = ld_relaxed_u64(&sl->agg_a), ab = ld_relaxed_u64(&sl->agg_b);
      if (ia & ib & kValid) {
        m = from_words(ia, ib);
        done = true;
      } else if (aa & ab & kValid) {
        m = from_words(aa, ab);
        incl = false;
        done = true;
      } else if (polls++ == 0) {
        start = global_ns();
      } else if ((int64_t)(global_ns() - start) >= a.wait_ns) {
        gave_up = true;  // count what is missing as an empty inclusive prefix and finish
        break;
      }
    }
    gave_up = __any_sync(~0u, gave_up);
    // nearest inclusive summary: the lowest lane that has one
    const unsigned inc_lanes = __ballot_sync(~0u, incl && t >= 0);
    const int stop = inc_lanes ? __ffs(inc_lanes) - 1 : 32;
    if (lane > stop || t < 0) m = {0, -1, -1};
    m = warp_join(m);
    run = join(run, m);
    if (inc_lanes || gave_up) break;
    j -= 32;
  }
  return run;
}

// Position ids of this thread's tokens [k_lo, k_hi): the distance to the
// latest run start (lr: the one before the thread's first token), 0 on
// padding.  Two per 16-byte store where the row allows it.
__device__ __forceinline__ void write_positions(int64_t* prow, int S, int s0, unsigned runs, unsigned nz, int lr,
                                                int k_lo, int k_hi) {
  if (s0 + kItems <= S && (reinterpret_cast<uintptr_t>(prow + s0) & 15) == 0) {
#pragma unroll
    for (int k = 0; k < kItems; k += 2) {
      if (runs & (1u << k)) lr = s0 + k;
      const int p0 = (nz >> k) & 1u ? s0 + k - lr : 0;
      if (runs & (2u << k)) lr = s0 + k + 1;
      const int p1 = (nz >> (k + 1)) & 1u ? s0 + k + 1 - lr : 0;
      if (k >= k_lo && k < k_hi) st_stream(reinterpret_cast<int4*>(prow + s0 + k), make_int4(p0, 0, p1, 0));
    }
  } else {
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      if (s0 + k >= S) break;
      if (runs & (1u << k)) lr = s0 + k;
      if (k >= k_lo && k < k_hi) prow[s0 + k] = (nz >> k) & 1u ? s0 + k - lr : 0;
    }
  }
}

// The CTA that finishes last: report the call's totals and reset them (every
// other CTA has counted itself done, so no update is left in flight).
__device__ __forceinline__ void report(const BridgeArgs& a) {
  // L2 loads: the counter this CTA acquired ordered every update before it
  const unsigned failed = __ldcg(&a.hdr->gave_up), longest = __ldcg(&a.hdr->longest),
                 overflow = __ldcg(&a.hdr->overflow), most = __ldcg(&a.hdr->most), total = __ldcg(&a.hdr->total);
  const int status = failed ? PSEQ_ERR_TIMEOUT : (overflow ? PSEQ_ERR_CAPACITY : PSEQ_OK);
  *a.info = pseq_info{status, (int32_t)most, (int32_t)longest, (int32_t)total};
  a.hdr->gave_up = 0u;
  a.hdr->longest = 0u;
  a.hdr->overflow = 0u;
  a.hdr->most = 0u;
  a.hdr->total = 0u;
}

template <typename Id>
__global__ void __launch_bounds__(kThreads, 4) bridge_kernel(const Id* __restrict__ doc, const __grid_constant__ BridgeArgs a) {
  __shared__ Marks s_warp[kThreads / 32];
  __shared__ Marks s_prefix;
  __shared__ int s_longest, s_overflow, s_last, s_used;
  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.y, ch = blockIdx.x;
  const int S = a.S, P = a.P;
  const Id* d = doc + (int64_t)row * S;
  int64_t* real_out = a.seq_lens + (int64_t)row * P;
  int64_t* pad_out = a.seq_lens_padded + (int64_t)row * P;
  if (tid == 0) {
    s_longest = 0;
    s_overflow = 0;
  }
  const unsigned ctas = gridDim.x * gridDim.y;
  // The CTA that finishes last reports the call's totals and leaves the
  // workspace zero.
  auto finish = [&]() {
    __syncthreads();
    if (!s_last) return;
    if (tid == 0) report(a);
    if (a.chunks > 1) {
      unsigned long long* words = reinterpret_cast<unsigned long long*>(a.slots);
      const int64_t n = 4 * (int64_t)a.B * a.chunks;
      for (int64_t i = tid; i < n; i += kThreads) words[i] = 0ull;
    }
  };
  if (a.chunks > 1 && ch == a.chunks) {
    // ---- the row's fill CTA (dispatched right after its chunks): once the
    // row's last chunk has published the row's sequence count, its unused
    // slots [used, P) take pad_value.  The chunks' walks write only slots
    // below `used`, so the fill never meets them.
    if (tid == 0) {
      const Slot* last = a.slots + (int64_t)row * a.chunks + (a.chunks - 1);
      int used = -1, polls = 0;
      uint64_t start = 0;
      while (true) {
        const unsigned long long ia = ld_relaxed_u64(&last->inc_a), ib = ld_relaxed_u64(&last->inc_b);
        if (ia & ib & kValid) {
          used = min(from_words(ia, ib).seqs, P);
          break;
        }
        if (polls++ == 0) {
          start = global_ns();
        } else if ((int64_t)(global_ns() - start) >= a.wait_ns) {
          atomicOr(&a.hdr->gave_up, 1u);  // reported as PSEQ_ERR_TIMEOUT; the slots are left unfilled
          break;
        }
      }
      s_used = used;
    }
    __syncthreads();
    const int used = s_used;
    if (used >= 0) {
      block_fill<8>(real_out + used, P - used, a.pad_value);
      block_fill<8>(pad_out + used, P - used, a.pad_value);
    }
    __syncthreads();
    // this CTA reads no more summary words (release); the last to arrive acquires all
    if (tid == 0) s_last = inc_acq_rel(&a.hdr->finished, ctas - 1u) == ctas - 1u;
    finish();
    return;
  }
  unsigned runs, seqs, nz, pnz;
  const int s0 = ch * kTile + tid * kItems;
  const Marks mine = chunk_flags(d, S, s0, runs, seqs, nz, pnz);
  // The join is commutative (sum, max, max): each warp's marks are three
  // warp reductions, the chunk's are those of the warps' (one barrier).
  {
    const Marks w = warp_join(mine);
    if (lane == 0) s_warp[warp] = w;
  }
  __syncthreads();
  Marks chunk_sum = {0, -1, -1}, wpre = {0, -1, -1};
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const Marks m = s_warp[w];
    chunk_sum = join(chunk_sum, m);
    if (w < warp) wpre = join(wpre, m);
  }
  // marks of the chunk's tokens before this thread's (the row prefix joins
  // later): the sequence starts of the lanes before it, and the last run and
  // sequence starts of the nearest lanes before it that have one
  Marks before;
  {
    int c = mine.seqs;
#pragma unroll
    for (int dd = 1; dd < 32; dd <<= 1) {
      const int o = __shfl_up_sync(~0u, c, dd);
      if (lane >= dd) c += o;
    }
    const unsigned below = (1u << lane) - 1u;
    const unsigned rb = __ballot_sync(~0u, mine.last_run >= 0) & below;
    const unsigned sb = __ballot_sync(~0u, mine.last_seq >= 0) & below;
    const int lr = __shfl_sync(~0u, mine.last_run, rb ? 31 - __clz(rb) : 0);
    const int ls = __shfl_sync(~0u, mine.last_seq, sb ? 31 - __clz(sb) : 0);
    before = join(wpre, Marks{c - mine.seqs, rb ? lr : -1, sb ? ls : -1});
  }
  // Positions after the chunk's first run start do not depend on the row
  // prefix: write them now, while warp 0 looks back.  Only the pairs before
  // this thread's first known run start wait for the prefix.
  // publish this chunk's summary first: the later chunks of the row wait for it
  Slot* row_slots = a.slots + (int64_t)row * a.chunks;
  const bool publish = a.chunks > 1 && (int64_t)row * a.chunks + ch != a.withhold;
  if (ch > 0 && tid == 0 && publish) {
    st_relaxed_u64(&row_slots[ch].agg_a, word_a(chunk_sum));
    st_relaxed_u64(&row_slots[ch].agg_b, word_b(chunk_sum));
  }
  int64_t* prow = a.positions ? a.positions + (int64_t)row * S : nullptr;
  const int known = before.last_run >= 0 ? 0 : (runs ? (__ffs(runs) - 1 + 1) & ~1 : kItems);
  if (prow) write_positions(prow, S, s0, runs, nz, before.last_run, known, kItems);
  // then the row prefix from the chunks before it
  if (warp == 0) {
    Marks prefix = {0, -1, -1};
    if (ch > 0) {
      bool gave_up = false;
      prefix = row_prefix(a, row_slots, ch, gave_up);
      if (gave_up && lane == 0) atomicOr(&a.hdr->gave_up, 1u);
    }
    if (lane == 0) {
      if (publish) {
        const Marks all = join(prefix, chunk_sum);
        st_relaxed_u64(&row_slots[ch].inc_a, word_a(all));
        st_relaxed_u64(&row_slots[ch].inc_b, word_b(all));
      }
      s_prefix = prefix;
    }
  }
  __syncthreads();
  const Marks prefix = s_prefix;
  before = join(prefix, before);
  const Marks row_so_far = join(prefix, chunk_sum);
  // walk this thread's run and sequence starts, in token order
  int last_run = before.last_run, last_seq = before.last_seq, count = before.seqs;
  int longest = 0;
  for (unsigned ev = runs | seqs; ev; ev &= ev - 1) {
    const int k = __ffs(ev) - 1;
    const unsigned bit = 1u << k;
    const int s = s0 + k;
    if (runs & bit) {
      if (s > 0 && (pnz & bit)) {  // the document run [last_run, s) ends here
        const int len = s - last_run;
        if (count - 1 < P) real_out[count - 1] = len;
        longest = max(longest, len);
      }
      last_run = s;
    }
    if (seqs & bit) {
      if (count > 0 && count - 1 < P) pad_out[count - 1] = s - last_seq;
      if (count < P) {
        if (!(nz & bit)) real_out[count] = 0;  // padding before any document
      } else {
        s_overflow = 1;
      }
      last_seq = s;
      count += 1;
    }
  }
  // the positions that waited for the row prefix
  if (prow && known > 0) write_positions(prow, S, s0, runs, nz, before.last_run, 0, known);
  // one shared atomic per warp for the longest document run
#pragma unroll
  for (int dd = 16; dd > 0; dd >>= 1) longest = max(longest, __shfl_xor_sync(~0u, longest, dd));
  if (lane == 0 && longest) atomicMax(&s_longest, longest);
  const bool row_end = ch == a.chunks - 1;
  // the row's last chunk closes the last run and the last sequence
  if (row_end && tid == 0 && S > 0) {
    const int total = row_so_far.seqs;
    if (__ldg(d + S - 1) != 0 && total - 1 < P) {
      real_out[total - 1] = S - row_so_far.last_run;
      atomicMax(&s_longest, S - row_so_far.last_run);
    }
    if (total - 1 < P) pad_out[total - 1] = S - row_so_far.last_seq;
  }
  // With one chunk per row, that chunk fills the row's unused slots [used, P);
  // otherwise the row's fill CTA does.
  if (a.chunks == 1) {
    const int used = min(row_so_far.seqs, P);
    block_fill<8>(real_out + used, P - used, a.pad_value);
    block_fill<8>(pad_out + used, P - used, a.pad_value);
  }
  __syncthreads();
  if (tid == 0) {
    // this chunk's share of the totals (atomics that return nothing)
    if (s_longest) atomicMax(&a.hdr->longest, (unsigned)s_longest);
    if (s_overflow) atomicOr(&a.hdr->overflow, 1u);
    if (row_end) {
      atomicMax(&a.hdr->most, (unsigned)row_so_far.seqs);
      atomicAdd(&a.hdr->total, (unsigned)row_so_far.seqs);
    }
    // this CTA reads no more summary words and has added its share
    // (release); the last one to arrive acquires them all
    s_last = inc_acq_rel(&a.hdr->finished, ctas - 1u) == ctas - 1u;
  }
  finish();
}

// A row of length 0 still has its slots filled; nothing else to do.
__global__ void bridge_empty_rows_kernel(BridgeArgs a) {
  pdl_enter();
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.info = {PSEQ_OK, 0, 0, 0};
  const int64_t cells = (int64_t)a.B * a.P;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < cells; i += (int64_t)gridDim.x * blockDim.x) {
    a.seq_lens[i] = a.pad_value;
    a.seq_lens_padded[i] = a.pad_value;
  }
}

__global__ void empty_bridge_kernel(pseq_info* info) {
  pdl_enter();
  *info = {PSEQ_OK, 0, 0, 0};
}

}  // namespace
}  // namespace pseq

using namespace pseq;

extern "C" size_t pseq_doc_ids_to_lengths_workspace_size(int64_t B, int64_t S) {
  if (B < 0 || S < 0) return 0;
  return workspace_bytes(B, S);
}

extern "C" pseq_status pseq_doc_ids_to_lengths(const void* doc_ids, int32_t id_bytes, int64_t B, int64_t S,
                                               int64_t num_packs, int64_t pad_value, int64_t* seq_lens,
                                               int64_t* seq_lens_padded, int64_t* position_ids, pseq_info* info,
                                               void* workspace, size_t workspace_bytes_, pseq_stream stream) {
  clear_error();
  const char* fn = "pseq_doc_ids_to_lengths";
  if (B < 0 || S < 0 || num_packs < 0) return fail(PSEQ_ERR_ARG, "%s: negative size", fn);
  if (id_bytes != 4 && id_bytes != 8) return fail(PSEQ_ERR_ARG, "%s: id_bytes must be 4 or 8", fn);
  if (B > 0 && S > INT32_MAX / B) return fail(PSEQ_ERR_OVERFLOW, "%s: B*S exceeds INT32_MAX", fn);
  if (S > INT32_MAX - kTile) return fail(PSEQ_ERR_OVERFLOW, "%s: S exceeds 2^31 - 1 - %d", fn, kTile);
  if (B > 0 && num_packs > INT32_MAX / B) return fail(PSEQ_ERR_OVERFLOW, "%s: B*num_packs exceeds INT32_MAX", fn);
  if (B > 65535) return fail(PSEQ_ERR_ARG, "%s: at most 65535 rows per call", fn);
  if (!info || (B * S > 0 && !doc_ids) || (B * num_packs > 0 && (!seq_lens || !seq_lens_padded)))
    return fail(PSEQ_ERR_ARG, "%s: NULL pointer", fn);
  if (!aligned(doc_ids, (uintptr_t)id_bytes) || !aligned(seq_lens, 8) || !aligned(seq_lens_padded, 8) ||
      !aligned(position_ids, 8) || !aligned(info, 4))
    return fail(PSEQ_ERR_ARG, "%s: misaligned pointer", fn);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  BridgeArgs a = {};
  a.B = (int)B;
  a.S = (int)S;
  a.P = (int)num_packs;
  a.chunks = (int)(S > 0 ? (S + kTile - 1) / kTile : 1);
  a.pad_value = pad_value;
  a.seq_lens = seq_lens;
  a.seq_lens_padded = seq_lens_padded;
  a.positions = position_ids;
  a.info = info;
  cudaError_t e;
  int launches = 1;
  if (B == 0) {
    e = launch_pdl(empty_bridge_kernel, dim3(1), dim3(1), 0, st, info);
  } else if (S == 0) {
    e = launch_pdl(bridge_empty_rows_kernel, dim3(64), dim3(256), 0, st, a);
  } else {
    const size_t need = workspace_bytes(B, S);
    if (!workspace || workspace_bytes_ < need || !aligned(workspace, 16))
      return fail(PSEQ_ERR_ARG, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", fn, need,
                  workspace_bytes_);
    a.hdr = static_cast<Header*>(workspace);
    a.slots = reinterpret_cast<Slot*>(static_cast<unsigned char*>(workspace) + sizeof(Header));
    a.wait_ns = wait_limit_ns();
    a.withhold = withhold_tile();
    // each row's chunks, then (with more than one chunk) the row's fill CTA
    const dim3 grid((unsigned)(a.chunks + (a.chunks > 1 ? 1 : 0)), (unsigned)B);
    e = id_bytes == 4 ? launch_pdl(bridge_kernel<int32_t>, grid, dim3(kThreads), 0, st,
                                   static_cast<const int32_t*>(doc_ids), a)
                      : launch_pdl(bridge_kernel<int64_t>, grid, dim3(kThreads), 0, st,
                                   static_cast<const int64_t*>(doc_ids), a);
  }
  count_launches(launches);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}
