// BSHD -> THD conversion: thd_from_batch, thd_meta, thd_gather,
// thd_padding_mask.
//
// Follows NeMo AutoModel v0.5 "nemo_automodel.components.distributed.thd_utils":
// process_input_for_thd (description, Example, Parameters, Returns) and
// _thd_padding_mask.
//
// The length tables are small (B * num_packs entries) and the streams large,
// so the metadata is one block-wide scan and the data movement is a grid-wide
// copy.  Two shapes:
//
//  * fused (tables of up to kFusedMaxEntries entries, the usual case): one
//    launch.  Every CTA scans the whole table into shared memory -- filter,
//    both cumulative sums, in-row source offsets -- so it knows the stream
//    layout without waiting on anyone; CTA 0 also writes cu_seqlens,
//    cu_seqlens_padded, pad_between_seqs and the info block.  Each CTA then
//    moves an equal slice of stream rows.
//  * two kernels (larger tables, and the explicit thd_meta / thd_gather
//    calls): thd_meta_kernel runs the scan in one CTA and leaves the layout in
//    the workspace; thd_gather_kernel (programmatic dependent launch) streams
//    the layout into shared memory in batches and moves its slice.
//
// Moving a slice: sequence pieces are contiguous in the source row and in the
// stream.  Fields whose rows are one aligned access of at most 16 bytes (ids,
// labels, positions) go row by row -- one thread per row, every (field,
// plane) load issued before any store.  Wide rows (embeddings) go piece by
// piece as block copies with 16-byte streaming loads and stores.  The padding
// mask of the slice is written by the same CTA.  Grids are sized from the
// occupancy calculator so they run in a single wave.
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"

namespace pseq {
namespace {

constexpr int kMetaThreads = 1024;
constexpr int kRowThreads = 512;
constexpr int kFusedMaxEntries = 2048;
constexpr int kTableBatch = 1024;
constexpr int kMaxJobs = 16;

struct Header {
  int32_t status;
  int32_t n;      // kept sequences
  int32_t T;      // stream rows that hold sequences (sum of padded lengths)
  int32_t Tmask;  // rows the padding mask covers (T, or total_tokens)
  int32_t pad[28];
};
static_assert(sizeof(Header) == 128, "header is 128 bytes");

struct Workspace {
  Header* hdr;
  int64_t* seq_src;   // [E]   source token (b*S + o) of the sequence's first slot
  int32_t* seq_cup;   // [E+1] stream start of each sequence; [n] = T
  int32_t* seq_real;  // [E]
  int64_t* row_pfx;   // [B]   padded prefix at each row's first entry
};

size_t workspace_bytes(int64_t B, int64_t E) {
  return sizeof(Header) + round_up(8 * (size_t)E, 16) + round_up(4 * (size_t)(E + 1), 16) +
         round_up(4 * (size_t)E, 16) + round_up(8 * (size_t)B, 16);
}

template <typename P>
Workspace carve(P base_, int64_t B, int64_t E) {
  unsigned char* p = (unsigned char*)(base_);
  Workspace w;
  w.hdr = reinterpret_cast<Header*>(p);
  p += sizeof(Header);
  w.seq_src = reinterpret_cast<int64_t*>(p);
  p += round_up(8 * (size_t)E, 16);
  w.seq_cup = reinterpret_cast<int32_t*>(p);
  p += round_up(4 * (size_t)(E + 1), 16);
  w.seq_real = reinterpret_cast<int32_t*>(p);
  p += round_up(4 * (size_t)E, 16);
  w.row_pfx = reinterpret_cast<int64_t*>(p);
  (void)B;
  return w;
}

struct MetaArgs {
  const int64_t* real;
  const int64_t* padded;  // may be NULL
  int B, P;
  int64_t S;
  int64_t pad_value;
  int has_filler;
  int absorb;
  int32_t* cu;           // may be NULL (mask-only use)
  int32_t* cu_padded;    // may be NULL
  uint8_t* pad_between;  // may be NULL
  pseq_info* info;
  int64_t fixed_total;   // >= 0: mask length and info.total (thd_padding_mask)
  int row0;              // source row of this table's first row (chunks)
  int chunks;            // > 1: blockIdx.y selects a chunk of B rows (fused kernel)
  int64_t cu_pad_to;     // > 0: fill cu arrays from n+1 up to this length with pad_value
};

// ----------------------------------------------------------------------------
// the length scan
// ----------------------------------------------------------------------------
struct ScanFlags {
  int bad, mismatch, last_mismatch, max_real;
};

struct ScanResult {
  int n;
  long long real, padded;
};

// Walk the tables in row-major order, dropping filler entries, and call
// put(k, b, o, real, padded, R, Pd) for kept entry k of row b at in-row
// offset o, where R and Pd are the real and padded sums of the kept entries
// before it.  Every thread returns the same totals; the flags are in *fl,
// complete after the caller's next barrier (the last round ends without
// one).  Three barriers per round: the warp sums, their scan in warp 0, and
// the round's end (left to the caller in the last round).  A row's start
// (the padded prefix at its first entry) comes from the warp sums and the
// first entry's in-warp prefix, which that thread leaves in row_pfx before
// the first barrier; in later rounds row_pfx holds the finished value.
template <int THREADS, typename Put>
__device__ ScanResult scan_lengths(const MetaArgs& a, int64_t* row_pfx, Triple* scratch, ScanFlags* fl, Put put) {
  constexpr int kW = THREADS / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) *fl = {0, 0, -1, 0};  // ordered before every update by the round's barriers
  const int E = a.B * a.P;
  Triple carry = {0, 0, 0};
  int done_row = -1;       // the row this thread started in the last round, and its start
  long long done_pfx = 0;
  for (int base = 0; base < E; base += THREADS) {
    if (done_row >= 0) row_pfx[done_row] = done_pfx;  // read after this round's barriers
    done_row = -1;
    const int e = base + tid;
    const bool valid = e < E;
    long long real = 0, padded = 0;
    bool keep = false, bad = false;
    if (valid) {
      real = __ldg(a.real + e);
      padded = a.padded ? __ldg(a.padded + e) : real;
      const bool real_filler = a.has_filler && real == a.pad_value;
      const bool padded_filler = a.has_filler && padded == a.pad_value;
      if (real_filler != padded_filler) {
        bad = true;
      } else if (!real_filler) {
        keep = true;
        if (real < 0 || padded < real) bad = true;
      }
    }
    const Triple x = {keep ? 1 : 0, keep ? real : 0, keep ? padded : 0};
    Triple inc = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const Triple o = shfl_up(inc, d);
      if (lane >= d) inc = add(o, inc);
    }
    const Triple wex = {inc.count - x.count, inc.real - x.real, inc.padded - x.padded};
    const int b = valid ? e / a.P : 0;
    const bool row_first = valid && e % a.P == 0;
    if (lane == 31) scratch[warp] = inc;
    if (row_first) row_pfx[b] = wex.padded;  // this round's part: completed below from the warp sums
    __syncthreads();
    if (warp == 0) {
      Triple w = lane < kW ? scratch[lane] : Triple{0, 0, 0};
#pragma unroll
      for (int d = 1; d < kW; d <<= 1) {
        const Triple o = shfl_up(w, d);
        if (lane >= d) w = add(o, w);
      }
      if (lane < kW) scratch[lane] = w;
    }
    __syncthreads();
    const Triple total = scratch[kW - 1];
    const Triple wpre = warp > 0 ? scratch[warp - 1] : Triple{0, 0, 0};
    const int k = carry.count + wpre.count + wex.count;
    const long long R = carry.real + wpre.real + wex.real;
    const long long Pd = carry.padded + wpre.padded + wex.padded;
    if (row_first) {
      done_row = b;
      done_pfx = Pd;
    }
    if (keep) {
      const int e0 = b * a.P;  // the row's first entry
      long long start;
      if (e0 >= base) {
        const int w0 = (e0 - base) >> 5;
        start = carry.padded + (w0 > 0 ? scratch[w0 - 1].padded : 0) + row_pfx[b];
      } else {
        start = row_pfx[b];
      }
      const long long o = Pd - start;
      if (o + padded > a.S) bad = true;
      put(k, b, o, real, padded, R, Pd);
      if (real != padded) {
        atomicAdd(&fl->mismatch, 1);
        atomicMax(&fl->last_mismatch, k);
      }
      atomicMax(&fl->max_real, (int)min(real, (long long)INT32_MAX));
    }
    if (bad) fl->bad = 1;
    carry = add(carry, total);
    if (base + THREADS < E) __syncthreads();  // the next round reuses scratch and row_pfx
  }
  return {carry.count, carry.real, carry.padded};
}

struct Summary {
  int status, n;
  long long T, cu_last, longest, shown_total;
  int pad_between;
};

// Absorption gate, pad_between_seqs and max_seqlen from the scan totals.
// last_real is the real length of kept sequence n-1 (0 when n == 0).
__device__ __forceinline__ Summary summarize(const MetaArgs& a, const ScanResult& r, const ScanFlags& fl,
                                             long long last_real) {
  Summary s;
  s.n = r.n;
  s.T = r.padded;
  s.status = fl.bad ? PSEQ_ERR_VALUE : PSEQ_OK;
  if (s.status == PSEQ_OK && s.T > INT32_MAX) s.status = PSEQ_ERR_OVERFLOW;
  const bool absorbed = a.absorb && r.n >= 1 && (fl.mismatch == 0 || (fl.mismatch == 1 && fl.last_mismatch == r.n - 1));
  s.cu_last = absorbed ? s.T : r.real;
  s.pad_between = (a.padded && fl.mismatch > 0 && !absorbed) ? 1 : 0;
  long long longest = fl.max_real;
  if (absorbed) longest = max(longest, s.T - (r.real - last_real));
  s.longest = r.n ? longest : 0;
  s.shown_total = a.fixed_total >= 0 ? a.fixed_total : s.T;
  return s;
}

// The cu arrays' filler rows [n+1, cu_pad_to), with every thread of the block.
__device__ __forceinline__ void pad_cu(const MetaArgs& a, const Summary& s) {
  for (int64_t k = s.n + 1 + threadIdx.x; k < a.cu_pad_to; k += blockDim.x) {
    if (a.cu) a.cu[k] = (int32_t)a.pad_value;
    if (a.cu_padded) a.cu_padded[k] = (int32_t)a.pad_value;
  }
}

__device__ __forceinline__ void write_meta(const MetaArgs& a, const Summary& s) {
  if (a.cu) a.cu[s.n] = (int32_t)s.cu_last;
  if (a.cu_padded) a.cu_padded[s.n] = (int32_t)s.T;
  if (a.pad_between) *a.pad_between = (uint8_t)s.pad_between;
  *a.info = s.status == PSEQ_OK ? pseq_info{PSEQ_OK, s.n, (int32_t)s.longest, (int32_t)s.shown_total}
                                : pseq_info{s.status, 0, 0, 0};
}

// ----------------------------------------------------------------------------
// moving stream rows
// ----------------------------------------------------------------------------
struct Fields {
  const unsigned char* src[PSEQ_MAX_FIELDS];
  unsigned char* dst[PSEQ_MAX_FIELDS];
  int64_t row_bytes[PSEQ_MAX_FIELDS];
  int planes[PSEQ_MAX_FIELDS];
  int num;
  int narrow;  // every row of every field is one aligned access of <= 16 bytes
  int bulk;    // every row of every field is >= 256 bytes, a multiple of 16, 16-byte aligned
  int njobs;   // (field, plane) pairs, for the row-by-row path
  int rb_all;  // every field's row is this many bytes (8: int64 ids, labels, positions), else 0
  // per (field, plane) job of the row-by-row path, read at fixed offsets in
  // an unrolled loop: field base pointers, plane, the field's planes, row bytes
  const unsigned char* job_src[kMaxJobs];
  unsigned char* job_dst[kMaxJobs];
  int job_plane[kMaxJobs];
  int job_planes[kMaxJobs];
  int job_rb[kMaxJobs];
};

// The row-by-row path: one thread per stream row, every (field, plane) load
// issued before any store.  A warp finds the sequence of its first row with
// one search that every lane runs alike (broadcast shared-memory reads), and
// each lane walks forward over the few sequence starts among the warp's 32
// rows (a search of its own after 8 steps).  RB = 8 when every row is 8
// bytes (no size switch), else 0.
template <int RB>
__device__ __forceinline__ void narrow_rows(const Fields& f, int64_t plane_in, int64_t T, uint8_t* mask, int64_t lo,
                                            int64_t hi, const int32_t* cup, const int32_t* src_tok,
                                            const int32_t* real, int cnt, int64_t chunk, int64_t chunk_rows) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31;
  for (int64_t rw = lo + (tid - lane); rw < hi; rw += nt) {
    const int64_t r = rw + lane;
    int j = seq_of(cup, cnt, rw);
    if (r < hi) {
      int steps = 0;
      while ((int64_t)cup[j + 1] <= r && steps < 8) {
        ++j;
        ++steps;
      }
      if ((int64_t)cup[j + 1] <= r) j = seq_of(cup, cnt, r);
      const int64_t off = r - cup[j];
      const int64_t tok = (int64_t)src_tok[j] + off;
      for (int g = 0; g < f.njobs; g += 8) {
        int4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (g + q < f.njobs) {
            const int rb = RB ? RB : f.job_rb[g + q];
            const unsigned char* p = f.job_src[g + q] + ((int64_t)f.job_plane[g + q] * plane_in + tok) * rb;
            if (RB == 8) {
              const uint2 t = __ldg(reinterpret_cast<const uint2*>(p));
              v[q] = make_int4((int)t.x, (int)t.y, 0, 0);
            } else {
              v[q] = load_row(p, rb);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (g + q < f.njobs) {
            const int rb = RB ? RB : f.job_rb[g + q];
            unsigned char* p =
                f.job_dst[g + q] + (chunk * f.job_planes[g + q] * chunk_rows + f.job_plane[g + q] * T + r) * rb;
            if (RB == 8)
              *reinterpret_cast<uint2*>(p) = make_uint2((unsigned)v[q].x, (unsigned)v[q].y);
            else
              store_row(p, v[q], rb);
          }
        }
      }
      if (mask) mask[r] = off >= real[j] ? 1 : 0;
    }
  }
}

// Move stream rows [lo, hi) of every field and write their mask bytes.
// Sequences j = 0..cnt-1 of the table start at stream row cup[j] (cup[cnt]
// ends the last one) and at source token src_tok[j]; cup[0] <= lo and
// hi <= cup[cnt].  B is the source's rows per plane; stream `chunk` of a
// chunked result starts chunk * planes * chunk_rows rows into each
// destination (its planes T rows apart), whatever the other chunks' lengths.
__device__ void gather_rows(const Fields& f, int64_t B, int64_t S, int64_t T, uint8_t* mask, int64_t lo,
                            int64_t hi, const int32_t* cup, const int32_t* src_tok, const int32_t* real, int cnt,
                            int64_t chunk, int64_t chunk_rows) {
  if (lo >= hi) return;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int64_t plane_in = B * S;
  if (f.narrow) {
    if (f.rb_all == 8)
      narrow_rows<8>(f, plane_in, T, mask, lo, hi, cup, src_tok, real, cnt, chunk, chunk_rows);
    else
      narrow_rows<0>(f, plane_in, T, mask, lo, hi, cup, src_tok, real, cnt, chunk, chunk_rows);
    return;
  }
  for (int j = seq_of(cup, cnt, lo); j < cnt; ++j) {
    const int64_t cs = cup[j];
    if (cs >= hi) break;
    const int64_t a0 = max(lo, cs), a1 = min(hi, (int64_t)cup[j + 1]);
    if (a0 >= a1) continue;
    const int64_t tok = (int64_t)src_tok[j] + (a0 - cs);
    for (int i = 0; i < f.num; ++i) {
      const int64_t rb = f.row_bytes[i];
      for (int p = 0; p < f.planes[i]; ++p)
        block_copy(f.dst[i] + (chunk * f.planes[i] * chunk_rows + p * T + a0) * rb,
                   f.src[i] + ((int64_t)p * plane_in + tok) * rb, (a1 - a0) * rb);
    }
    if (mask) {
      const int64_t real_end = cs + real[j];
      for (int64_t t = a0 + tid; t < a1; t += nt) mask[t] = t >= real_end ? 1 : 0;
    }
  }
}

// Rows [r0, r1) of a mask of length Tm that CTA blockIdx.x owns.
__device__ __forceinline__ void slice_of(int64_t Tm, int64_t& r0, int64_t& r1) {
  const int64_t G = gridDim.x;
  const int64_t per = (Tm + G - 1) / G;
  r0 = min((int64_t)blockIdx.x * per, Tm);
  r1 = min(r0 + per, Tm);
}

// ----------------------------------------------------------------------------
// kernels
// ----------------------------------------------------------------------------
// Shared-memory tables of one chunk's layout (see fused_scan).
struct Tables {
  int64_t* row;  // [B]
  int32_t* cup;  // [E+1]
  int32_t* src;  // [E]
  int32_t* real; // [E]
};

__device__ __forceinline__ Tables carve_tables(unsigned char* base, int B, int P) {
  const int E = B * P;
  Tables t;
  t.row = reinterpret_cast<int64_t*>(base);
  t.cup = reinterpret_cast<int32_t*>(t.row + (P > 0 ? B : 0));
  t.src = t.cup + E + 1;
  t.real = t.src + E;
  return t;
}

size_t table_bytes(int B, int P) {
  const size_t E = (size_t)B * P;
  return round_up((P > 0 ? 8 * (size_t)B : 0) + 4 * (E + 1) + 8 * E, 16);
}

// The per-chunk view of the arguments: chunk blockIdx.y covers rows
// [c*B, (c+1)*B) of a batch of chunks*B rows.
__device__ __forceinline__ MetaArgs chunk_view(const MetaArgs& a) {
  MetaArgs ac = a;
  if (a.chunks > 1) {
    const int c = blockIdx.y;
    const int64_t e0 = (int64_t)c * a.B * a.P;
    ac.real = a.real + e0;
    ac.padded = a.padded ? a.padded + e0 : nullptr;
    ac.row0 = c * a.B;
    ac.cu = a.cu ? a.cu + c * a.cu_pad_to : nullptr;
    ac.cu_padded = a.cu_padded ? a.cu_padded + c * a.cu_pad_to : nullptr;
    ac.pad_between = a.pad_between ? a.pad_between + c : nullptr;
    ac.info = a.info + c;
  }
  return ac;
}

// Every CTA scans its chunk's whole length table into shared memory; CTA 0
// of the chunk also writes cu_seqlens, cu_seqlens_padded, pad_between_seqs
// and the info block.  Returns the summary (the same in every thread).
__device__ __forceinline__ Summary fused_scan(const MetaArgs& ac, const Tables& t, Triple* scratch, ScanFlags* fl,
                                              int& n) {
  const bool lead = blockIdx.x == 0;
  auto put = [&](int k, int b, long long o, long long real, long long padded, long long R, long long Pd) {
    t.cup[k] = (int32_t)Pd;
    t.src[k] = (int32_t)((ac.row0 + b) * ac.S + o);
    t.real[k] = (int32_t)real;
    if (lead) {
      if (ac.cu) ac.cu[k] = (int32_t)R;
      if (ac.cu_padded) ac.cu_padded[k] = (int32_t)Pd;
    }
  };
  const ScanResult r = scan_lengths<kRowThreads>(ac, t.row, scratch, fl, put);
  if (threadIdx.x == 0) t.cup[r.n] = (int32_t)r.padded;  // the stream's end (= T)
  __syncthreads();  // the tables and the flags are complete
  const Summary s = summarize(ac, r, *fl, r.n ? t.real[r.n - 1] : 0);
  if (lead && threadIdx.x == 0) write_meta(ac, s);
  if (lead) pad_cu(ac, s);
  n = r.n;
  return s;
}

__global__ void __launch_bounds__(kRowThreads, 2)
    thd_fused_kernel(const __grid_constant__ MetaArgs a, const __grid_constant__ Fields f, uint8_t* mask,
                     int64_t mask_cap) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Triple scratch[kRowThreads / 32];
  __shared__ ScanFlags fl;
  pdl_enter();
  const int c = blockIdx.y;
  const MetaArgs ac = chunk_view(a);
  const Tables t = carve_tables(smem, ac.B, ac.P);
  int n;
  const Summary s = fused_scan(ac, t, scratch, &fl, n);
  if (s.status != PSEQ_OK) return;
  const int64_t T = s.T, Tm = s.shown_total;
  if (Tm > mask_cap || T > Tm || T > (int64_t)ac.B * ac.S) return;  // cannot happen for well-formed input
  int64_t r0, r1;
  slice_of(Tm, r0, r1);
  const int64_t chunk_rows = (int64_t)ac.B * ac.S;  // fixed stride of the chunks' streams and masks
  uint8_t* m = mask ? mask + (int64_t)c * chunk_rows : nullptr;
  gather_rows(f, (int64_t)ac.B * a.chunks, ac.S, T, m, r0, min(r1, T), t.cup, t.src, t.real, n, c, chunk_rows);
  if (m) {
    const int64_t tail = max(r0, T);
    if (tail < r1) block_fill_bytes(m + tail, r1 - tail, 1);
  }
}

// Wide rows through the bulk-copy engine: after the table scan, one thread
// streams the CTA's slice global -> shared -> global through a ring of
// kStages buffers of kStage bytes (each load tracked by an mbarrier, each
// store by a bulk group), so the copy needs almost no registers or threads
// while the other threads write the mask.  Every row of every field is a
// multiple of 16 bytes at 16-byte aligned addresses (checked on the host).
#ifndef PSEQ_BULK_STAGES
#define PSEQ_BULK_STAGES 4
#endif
#ifndef PSEQ_BULK_STAGE_KB
#define PSEQ_BULK_STAGE_KB 32
#endif
constexpr int kStages = PSEQ_BULK_STAGES;
constexpr int kStage = PSEQ_BULK_STAGE_KB * 1024;

__global__ void __launch_bounds__(kRowThreads, 1)
    thd_fused_bulk_kernel(const __grid_constant__ MetaArgs a, const __grid_constant__ Fields f, uint8_t* mask,
                          int64_t mask_cap, int64_t wait_ns) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ Triple scratch[kRowThreads / 32];
  __shared__ ScanFlags fl;
  __shared__ __align__(8) uint64_t bar[kStages];
  pdl_enter();
  const int c = blockIdx.y;
  const MetaArgs ac = chunk_view(a);
  unsigned char* ring = smem;
  const Tables t = carve_tables(smem + (size_t)kStages * kStage, ac.B, ac.P);
  int n;
  const Summary s = fused_scan(ac, t, scratch, &fl, n);
  if (s.status != PSEQ_OK) return;
  const int64_t T = s.T, Tm = s.shown_total;
  if (Tm > mask_cap || T > Tm || T > (int64_t)ac.B * ac.S) return;  // cannot happen for well-formed input
  int64_t r0, r1;
  slice_of(Tm, r0, r1);
  const int64_t lo = r0, hi = min(r1, T);
  const int64_t chunk_rows = (int64_t)ac.B * ac.S;  // fixed stride of the chunks' streams and masks
  uint8_t* m = mask ? mask + (int64_t)c * chunk_rows : nullptr;
  if (threadIdx.x == 0 && lo < hi) {
    const int64_t plane_in = (int64_t)ac.B * a.chunks * ac.S;
    // the slice's chunks: sequence pieces x fields x planes, cut at kStage bytes
    int j = seq_of(t.cup, n, lo), i = 0, p = 0;
    int64_t off = 0;
    auto next = [&](const unsigned char*& src, unsigned char*& dst, uint32_t& bytes) -> bool {
      while (j < n) {
        const int64_t cs = t.cup[j];
        if (cs >= hi) return false;
        const int64_t a0 = max(lo, cs), a1 = min(hi, (int64_t)t.cup[j + 1]);
        while (a0 < a1 && i < f.num) {
          const int64_t rb = f.row_bytes[i];
          const int64_t piece = (a1 - a0) * rb;
          if (p < f.planes[i]) {
            if (off < piece) {
              const int64_t tok = (int64_t)t.src[j] + (a0 - cs);
              src = f.src[i] + ((int64_t)p * plane_in + tok) * rb + off;
              dst = f.dst[i] + ((int64_t)c * f.planes[i] * chunk_rows + p * T + a0) * rb + off;
              bytes = (uint32_t)min(piece - off, (int64_t)kStage);
              off += bytes;
              return true;
            }
            off = 0;
            ++p;
            continue;
          }
          p = 0;
          ++i;
        }
        i = 0;
        p = 0;
        off = 0;
        ++j;
      }
      return false;
    };
    for (int k = 0; k < kStages; ++k) mbar_init(&bar[k], 1);
    fence_mbar_init();
    unsigned char* dst_of[kStages];
    uint32_t bytes_of[kStages];
    const unsigned char* src;
    unsigned char* dst;
    uint32_t bytes;
    int loaded = 0;
    for (int k = 0; k < kStages && next(src, dst, bytes); ++k, ++loaded) {
      mbar_expect_tx(&bar[k], bytes);
      bulk_load(ring + (size_t)k * kStage, src, bytes, &bar[k]);
      dst_of[k] = dst;
      bytes_of[k] = bytes;
    }
    bool failed = false;
    for (int q = 0; q < loaded; ++q) {
      const int k = q % kStages;
      if (!mbar_wait(&bar[k], (uint32_t)((q / kStages) & 1), wait_ns)) {
        failed = true;
        break;
      }
      bulk_store(dst_of[k], ring + (size_t)k * kStage, bytes_of[k]);
      bulk_commit();
      // refill the buffer of chunk q - 1 once its store has read it
      if (q >= 1 && next(src, dst, bytes)) {
        const int k1 = (q - 1) % kStages;
        bulk_wait_read<1>();
        mbar_expect_tx(&bar[k1], bytes);
        bulk_load(ring + (size_t)k1 * kStage, src, bytes, &bar[k1]);
        dst_of[k1] = dst;
        bytes_of[k1] = bytes;
        ++loaded;
      }
    }
    if (failed) {
      // a load never arrived: report, then give the loads in flight a bounded
      // chance to land before the shared memory goes away
      atomicMax(&ac.info->status, (int)PSEQ_ERR_TIMEOUT);
      for (int q = 0; q < loaded; ++q) mbar_wait(&bar[q % kStages], (uint32_t)((q / kStages) & 1), wait_ns);
    }
    bulk_wait<0>();
  } else if (m && threadIdx.x > 0) {
    const int nt = blockDim.x - 1, tid = threadIdx.x - 1;
    for (int j = seq_of(t.cup, n, lo); j < n && t.cup[j] < hi; ++j) {
      const int64_t cs = t.cup[j];
      const int64_t a0 = max(lo, cs), a1 = min(hi, (int64_t)t.cup[j + 1]);
      const int64_t real_end = cs + t.real[j];
      for (int64_t x = a0 + tid; x < a1; x += nt) m[x] = x >= real_end ? 1 : 0;
    }
  }
  if (m) {
    __syncthreads();
    const int64_t tail = max(r0, T);
    if (tail < r1) block_fill_bytes(m + tail, r1 - tail, 1);
  }
}

__global__ void __launch_bounds__(kMetaThreads) thd_meta_kernel(const __grid_constant__ MetaArgs a, Workspace ws) {
  __shared__ Triple scratch[kMetaThreads / 32];
  __shared__ ScanFlags fl;
  pdl_enter();
  auto put = [&](int k, int b, long long o, long long real, long long padded, long long R, long long Pd) {
    ws.seq_src[k] = (long long)(a.row0 + b) * a.S + o;
    ws.seq_real[k] = (int32_t)real;
    ws.seq_cup[k] = (int32_t)Pd;
    if (a.cu) a.cu[k] = (int32_t)R;
    if (a.cu_padded) a.cu_padded[k] = (int32_t)Pd;
  };
  const ScanResult r = scan_lengths<kMetaThreads>(a, ws.row_pfx, scratch, &fl, put);
  __syncthreads();  // the flags and the tables are complete
  const Summary s = summarize(a, r, fl, r.n ? ws.seq_real[r.n - 1] : 0);
  pad_cu(a, s);
  if (threadIdx.x != 0) return;
  ws.seq_cup[r.n] = (int32_t)s.T;
  write_meta(a, s);
  Header h = {};
  h.status = s.status;
  h.n = s.n;
  h.T = (int32_t)s.T;
  h.Tmask = (int32_t)s.shown_total;
  *ws.hdr = h;
}

__global__ void __launch_bounds__(kRowThreads, 2)
    thd_gather_kernel(const __grid_constant__ Fields f, int64_t B, int64_t S, uint8_t* __restrict__ mask,
                      Workspace ws, int64_t max_seqs, int64_t max_rows, int64_t plane_rows, int64_t chunk) {
  __shared__ int32_t s_cup[kTableBatch + 1];
  __shared__ int32_t s_src[kTableBatch];
  __shared__ int32_t s_real[kTableBatch];
  __shared__ int s_first;
  pdl_enter();
  const int status = __ldcg(&ws.hdr->status);
  if (status != PSEQ_OK) return;
  const int n = __ldcg(&ws.hdr->n);
  const int64_t T = __ldcg(&ws.hdr->T);
  const int64_t Tm = __ldcg(&ws.hdr->Tmask);
  // a layout that does not fit the buffers did not come from thd_meta: write nothing
  if (n < 0 || n > max_seqs || T < 0 || T > B * S || Tm < T || Tm > max_rows) return;
  int64_t r0, r1;
  slice_of(Tm, r0, r1);
  if (r0 >= r1) return;
  if (mask) mask += chunk * max_rows;  // chunk streams and masks sit max_rows apart
  const int64_t g1 = min(r1, T);
  const int tid = threadIdx.x, lane = tid & 31;
  int64_t lo = r0;
  while (lo < g1) {
    if (tid < 32) {
      // largest k with cup[k] <= lo, 32 probes per round
      int a = 0, b = n;
      while (b - a > 1) {
        const int step = (b - a + 31) / 32;
        const int probe = a + lane * step;
        const bool ok = probe < b && (int64_t)__ldcg(ws.seq_cup + probe) <= lo;
        const unsigned m = __ballot_sync(~0u, ok);
        a = a + (31 - __clz(m)) * step;
        b = min(a + step, b);
      }
      if (tid == 0) s_first = a;
    }
    __syncthreads();
    const int k0 = s_first;
    const int cnt = min(kTableBatch, n - k0);
    for (int i = tid; i <= cnt; i += kRowThreads) s_cup[i] = __ldcg(ws.seq_cup + k0 + i);
    for (int i = tid; i < cnt; i += kRowThreads) {
      s_src[i] = (int32_t)__ldcg(ws.seq_src + k0 + i);
      s_real[i] = __ldcg(ws.seq_real + k0 + i);
    }
    __syncthreads();
    const int64_t hi = min(g1, (int64_t)s_cup[cnt]);
    gather_rows(f, plane_rows, S, T, mask, lo, hi, s_cup, s_src, s_real, cnt, chunk, max_rows);
    lo = hi;
    __syncthreads();
  }
  if (mask) {
    const int64_t tail = max(r0, T);
    if (tail < r1) block_fill_bytes(mask + tail, r1 - tail, 1);
  }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
// One wave of CTAs: about one row per thread on the row-by-row path, every
// resident slot for wide rows.
int row_grid(const void* kernel, size_t smem, int64_t rows, const Fields& f) {
  const int64_t full = (int64_t)sm_count() * occupancy(kernel, kRowThreads, smem);
  int64_t want = f.narrow ? (rows + kRowThreads - 1) / kRowThreads : full;
  if (want > full) want = full;
  return (int)(want < 1 ? 1 : want);
}

pseq_status check_lengths(const char* fn, int64_t B, int64_t S, int64_t P) {
  if (B < 0 || S < 0 || P < 0)
    return fail(PSEQ_ERR_ARG, "%s: negative size (B=%lld S=%lld num_packs=%lld)", fn, (long long)B, (long long)S,
                (long long)P);
  if (B > 0 && S > INT32_MAX / B) return fail(PSEQ_ERR_OVERFLOW, "%s: B*S exceeds INT32_MAX", fn);
  if (B > 0 && P > (INT32_MAX - 1) / B) return fail(PSEQ_ERR_OVERFLOW, "%s: B*num_packs exceeds INT32_MAX", fn);
  return PSEQ_OK;
}

pseq_status check_meta(const char* fn, const MetaArgs& a, const void* workspace, size_t ws_bytes) {
  const int64_t E = (int64_t)a.B * a.P;
  const size_t need = workspace_bytes(a.B, E);
  if (!workspace || ws_bytes < need || !aligned(workspace, 16))
    return fail(PSEQ_ERR_ARG, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", fn, need, ws_bytes);
  if ((E > 0 && !a.real) || !a.info) return fail(PSEQ_ERR_ARG, "%s: NULL lengths or info", fn);
  if (!aligned(a.real, 8) || !aligned(a.padded, 8) || !aligned(a.cu, 4) || !aligned(a.cu_padded, 4) ||
      !aligned(a.info, 4))
    return fail(PSEQ_ERR_ARG, "%s: misaligned pointer", fn);
  return PSEQ_OK;
}

pseq_status build_fields(const char* fn, const pseq_field* fields, int num_fields, int64_t B, int64_t S,
                         Fields& f) {
  if (num_fields < 0 || num_fields > PSEQ_MAX_FIELDS)
    return fail(PSEQ_ERR_ARG, "%s: num_fields must be in [0, %d]", fn, PSEQ_MAX_FIELDS);
  if (num_fields > 0 && !fields) return fail(PSEQ_ERR_ARG, "%s: fields is NULL", fn);
  f = Fields{};
  f.num = num_fields;
  f.narrow = 1;
  int jobs = 0;
  for (int i = 0; i < num_fields; ++i) {
    const pseq_field& x = fields[i];
    if (x.elem_bytes != 1 && x.elem_bytes != 2 && x.elem_bytes != 4 && x.elem_bytes != 8)
      return fail(PSEQ_ERR_ARG, "%s: field %d: elem_bytes must be 1, 2, 4 or 8", fn, i);
    if (x.planes < 1 || x.row_elems < 1)
      return fail(PSEQ_ERR_ARG, "%s: field %d: planes and row_elems must be >= 1", fn, i);
    if (B * S > 0 && (!x.src || !x.dst)) return fail(PSEQ_ERR_ARG, "%s: field %d: NULL src or dst", fn, i);
    if (!aligned(x.src, (uintptr_t)x.elem_bytes) || !aligned(x.dst, (uintptr_t)x.elem_bytes))
      return fail(PSEQ_ERR_ARG, "%s: field %d: misaligned pointer", fn, i);
    const int64_t cells = B * S > 0 ? B * S * (int64_t)x.planes : 1;
    if (x.row_elems > (INT64_MAX / 16) / cells) return fail(PSEQ_ERR_OVERFLOW, "%s: field %d is too large", fn, i);
    const int64_t rb = x.row_elems * x.elem_bytes;
    f.src[i] = static_cast<const unsigned char*>(x.src);
    f.dst[i] = static_cast<unsigned char*>(x.dst);
    f.row_bytes[i] = rb;
    f.planes[i] = x.planes;
    const bool one_access = (rb == 1 || rb == 2 || rb == 4 || rb == 8 || rb == 16) && aligned(x.src, (uintptr_t)rb) &&
                            aligned(x.dst, (uintptr_t)rb);
    if (!one_access) f.narrow = 0;
    for (int p = 0; p < x.planes; ++p) {
      if (jobs < kMaxJobs) {
        f.job_src[jobs] = f.src[i];
        f.job_dst[jobs] = f.dst[i];
        f.job_plane[jobs] = p;
        f.job_planes[jobs] = x.planes;
        f.job_rb[jobs] = (int)rb;
      }
      ++jobs;
    }
  }
  if (jobs > kMaxJobs) f.narrow = 0;
  f.njobs = f.narrow ? jobs : 0;
  f.rb_all = 8;
  for (int i = 0; i < num_fields; ++i)
    if (f.row_bytes[i] != 8) f.rb_all = 0;
  f.bulk = num_fields > 0;
  for (int i = 0; i < num_fields; ++i) {
    const int64_t rb = f.row_bytes[i];
    if (rb < 256 || rb % 16 != 0 || !aligned(f.src[i], 16) || !aligned(f.dst[i], 16)) f.bulk = 0;
  }
  return PSEQ_OK;
}


// Bulk-copy CTAs: one per SM on four fifths of the SMs.  About 120 copy
// engines already saturate HBM (each moves ~55 GB/s here; 88 fall short),
// and the SMs left free let calls that run beside this one -- on another
// stream -- start at once instead of waiting for SMs to drain.
int bulk_ctas() {
  const int n = sm_count() - sm_count() / 5;
  return n > 0 ? n : 1;
}

pseq_status launch_fused(const char* fn, const MetaArgs& a, const Fields& f, uint8_t* mask, int64_t mask_cap,
                         cudaStream_t st) {
  const int64_t rows = a.fixed_total >= 0 ? a.fixed_total : (int64_t)a.B * a.S;
  cudaError_t e;
  if (f.bulk) {
    // one CTA per SM; the ring of bulk-copy buffers sits in front of the tables
    const size_t smem = (size_t)kStages * kStage + table_bytes(a.B, a.P);
    e = allow_dynamic_smem(reinterpret_cast<const void*>(thd_fused_bulk_kernel),
                           (size_t)kStages * kStage + table_bytes(kFusedMaxEntries, 1));
    if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    e = launch_pdl(thd_fused_bulk_kernel, dim3((unsigned)bulk_ctas(), (unsigned)a.chunks), dim3(kRowThreads), smem, st,
                   a, f, mask, mask_cap, wait_limit_ns());
  } else {
    const size_t smem = table_bytes(a.B, a.P);
    const int grid = row_grid(reinterpret_cast<const void*>(thd_fused_kernel), smem, rows, f);
    e = launch_pdl(thd_fused_kernel, dim3(grid, (unsigned)a.chunks), dim3(kRowThreads), smem, st, a, f, mask, mask_cap);
  }
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}

pseq_status launch_meta(const char* fn, const MetaArgs& a, void* workspace, cudaStream_t st) {
  const cudaError_t e =
      launch_pdl(thd_meta_kernel, dim3(1), dim3(kMetaThreads), 0, st, a, carve(workspace, a.B, (int64_t)a.B * a.P));
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}

// plane_rows: source rows per plane (B unless this is one chunk of a larger
// batch); chunk: position of this stream in a chunked result (streams and
// masks B * S rows apart).
pseq_status launch_gather(const char* fn, const Fields& f, int64_t B, int64_t S, int64_t P, uint8_t* mask,
                          const void* workspace, cudaStream_t st, int64_t mask_rows, int64_t plane_rows = -1,
                          int64_t chunk = 0) {
  if (f.num == 0 && !mask) return PSEQ_OK;
  const int64_t E = B * P;
  const int grid = row_grid(reinterpret_cast<const void*>(thd_gather_kernel), 0, mask_rows, f);
  Workspace ws = carve(workspace, B, E);
  cudaError_t e = launch_pdl(thd_gather_kernel, dim3(grid), dim3(kRowThreads), 0, st, f, B, S, mask, ws, E, mask_rows,
                             plane_rows < 0 ? B : plane_rows, chunk);
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}

MetaArgs thd_args(const int64_t* seq_lens, const int64_t* seq_lens_padded, int64_t B, int64_t S, int64_t P,
                  int64_t pad_value, int32_t absorb, int32_t* cu, int32_t* cup, uint8_t* pad_between,
                  pseq_info* info) {
  MetaArgs a = {};
  a.real = seq_lens;
  a.padded = seq_lens_padded;
  a.B = (int)B;
  a.P = (int)P;
  a.S = S;
  a.pad_value = pad_value;
  a.has_filler = 1;
  a.absorb = absorb ? 1 : 0;
  a.cu = cu;
  a.cu_padded = seq_lens_padded ? cup : nullptr;
  a.pad_between = pad_between;
  a.info = info;
  a.fixed_total = -1;
  a.row0 = 0;
  a.chunks = 1;
  a.cu_pad_to = 0;
  return a;
}

}  // namespace
}  // namespace pseq

using namespace pseq;

extern "C" size_t thd_workspace_size(int64_t B, int64_t num_packs) {
  if (B < 0 || num_packs < 0) return 0;
  if (B > 0 && num_packs > (INT32_MAX - 1) / B) return 0;
  return workspace_bytes(B, B * num_packs);
}

extern "C" pseq_status thd_meta(const int64_t* seq_lens, const int64_t* seq_lens_padded, int64_t B, int64_t S,
                                int64_t num_packs, int64_t pad_value, int32_t absorb_trailing_pad,
                                int32_t* cu_seqlens, int32_t* cu_seqlens_padded, uint8_t* pad_between_seqs,
                                pseq_info* info, void* workspace, size_t workspace_bytes_,
                                pseq_stream stream) {
  clear_error();
  const char* fn = "thd_meta";
  pseq_status s = check_lengths(fn, B, S, num_packs);
  if (s != PSEQ_OK) return s;
  if (!cu_seqlens) return fail(PSEQ_ERR_ARG, "%s: cu_seqlens is required", fn);
  const MetaArgs a = thd_args(seq_lens, seq_lens_padded, B, S, num_packs, pad_value, absorb_trailing_pad, cu_seqlens,
                              cu_seqlens_padded, pad_between_seqs, info);
  s = check_meta(fn, a, workspace, workspace_bytes_);
  if (s != PSEQ_OK) return s;
  return launch_meta(fn, a, workspace, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" pseq_status thd_gather(const pseq_field* fields, int32_t num_fields, int64_t B, int64_t S,
                                  int64_t num_packs, uint8_t* padding_mask, const void* workspace,
                                  size_t workspace_bytes_, pseq_stream stream) {
  clear_error();
  const char* fn = "thd_gather";
  pseq_status s = check_lengths(fn, B, S, num_packs);
  if (s != PSEQ_OK) return s;
  const size_t need = workspace_bytes(B, B * num_packs);
  if (!workspace || workspace_bytes_ < need || !aligned(workspace, 16))
    return fail(PSEQ_ERR_ARG, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", fn, need, workspace_bytes_);
  Fields f;
  s = build_fields(fn, fields, num_fields, B, S, f);
  if (s != PSEQ_OK) return s;
  return launch_gather(fn, f, B, S, num_packs, padding_mask, workspace, reinterpret_cast<cudaStream_t>(stream),
                       B * S);
}

extern "C" pseq_status thd_from_batch(const int64_t* seq_lens, const int64_t* seq_lens_padded, int64_t B,
                                      int64_t S, int64_t num_packs, int64_t pad_value,
                                      int32_t absorb_trailing_pad, const pseq_field* fields, int32_t num_fields,
                                      int32_t* cu_seqlens, int32_t* cu_seqlens_padded, uint8_t* padding_mask,
                                      uint8_t* pad_between_seqs, pseq_info* info, void* workspace,
                                      size_t workspace_bytes_, pseq_stream stream) {
  clear_error();
  const char* fn = "thd_from_batch";
  pseq_status s = check_lengths(fn, B, S, num_packs);
  if (s != PSEQ_OK) return s;
  if (!cu_seqlens) return fail(PSEQ_ERR_ARG, "%s: cu_seqlens is required", fn);
  Fields f;
  s = build_fields(fn, fields, num_fields, B, S, f);
  if (s != PSEQ_OK) return s;
  const MetaArgs a = thd_args(seq_lens, seq_lens_padded, B, S, num_packs, pad_value, absorb_trailing_pad, cu_seqlens,
                              cu_seqlens_padded, pad_between_seqs, info);
  s = check_meta(fn, a, workspace, workspace_bytes_);
  if (s != PSEQ_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (B * num_packs <= kFusedMaxEntries) return launch_fused(fn, a, f, padding_mask, B * S, st);
  s = launch_meta(fn, a, workspace, st);
  if (s != PSEQ_OK) return s;
  return launch_gather(fn, f, B, S, num_packs, padding_mask, workspace, st, B * S);
}

extern "C" pseq_status thd_padding_mask(int64_t total_tokens, const int64_t* valid_seq_lens,
                                        const int64_t* valid_seq_lens_padded, int64_t n, uint8_t* mask,
                                        pseq_info* info, void* workspace, size_t workspace_bytes_,
                                        pseq_stream stream) {
  clear_error();
  const char* fn = "thd_padding_mask";
  if (total_tokens < 0 || n < 0) return fail(PSEQ_ERR_ARG, "%s: negative size", fn);
  if (total_tokens > INT32_MAX) return fail(PSEQ_ERR_OVERFLOW, "%s: total_tokens exceeds INT32_MAX", fn);
  if (n > INT32_MAX - 1) return fail(PSEQ_ERR_OVERFLOW, "%s: n exceeds INT32_MAX", fn);
  if (total_tokens > 0 && !mask) return fail(PSEQ_ERR_ARG, "%s: mask is NULL", fn);
  MetaArgs a = thd_args(valid_seq_lens, valid_seq_lens_padded, 1, total_tokens, n, 0, 0, nullptr, nullptr, nullptr,
                        info);
  a.has_filler = 0;
  a.fixed_total = total_tokens;
  pseq_status s = check_meta(fn, a, workspace, workspace_bytes_);
  if (s != PSEQ_OK) return s;
  Fields f;
  build_fields(fn, nullptr, 0, 1, total_tokens, f);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (n <= kFusedMaxEntries) return launch_fused(fn, a, f, mask, total_tokens, st);
  s = launch_meta(fn, a, workspace, st);
  if (s != PSEQ_OK || total_tokens == 0) return s;
  return launch_gather(fn, f, 1, total_tokens, n, mask, workspace, st, total_tokens);
}

extern "C" pseq_status thd_chunks_from_batch(const int64_t* seq_lens, const int64_t* seq_lens_padded, int64_t B,
                                             int64_t S, int64_t num_packs, int64_t num_chunks, int64_t pad_value,
                                             int32_t absorb_trailing_pad, const pseq_field* fields,
                                             int32_t num_fields, int32_t* cu_seqlens, int32_t* cu_seqlens_padded,
                                             uint8_t* padding_mask, uint8_t* pad_between_seqs, pseq_info* infos,
                                             void* workspace, size_t workspace_bytes_, pseq_stream stream) {
  clear_error();
  const char* fn = "thd_chunks_from_batch";
  pseq_status s = check_lengths(fn, B, S, num_packs);
  if (s != PSEQ_OK) return s;
  if (num_chunks < 1 || B % num_chunks != 0)
    return fail(PSEQ_ERR_ARG, "%s: num_chunks must be >= 1 and divide B (B=%lld, num_chunks=%lld)", fn, (long long)B,
                (long long)num_chunks);
  if (num_chunks > 65535) return fail(PSEQ_ERR_ARG, "%s: at most 65535 chunks", fn);
  if (!cu_seqlens || !infos) return fail(PSEQ_ERR_ARG, "%s: cu_seqlens and infos are required", fn);
  const int64_t Bc = B / num_chunks;
  Fields f;
  s = build_fields(fn, fields, num_fields, B, S, f);
  if (s != PSEQ_OK) return s;
  MetaArgs a = thd_args(seq_lens, seq_lens_padded, Bc, S, num_packs, pad_value, absorb_trailing_pad, cu_seqlens,
                        cu_seqlens_padded, pad_between_seqs, infos);
  a.cu_pad_to = Bc * num_packs + 1;
  s = check_meta(fn, a, workspace, workspace_bytes_);
  if (s != PSEQ_OK) return s;
  if (!aligned(seq_lens, 8) || !aligned(seq_lens_padded, 8)) return fail(PSEQ_ERR_ARG, "%s: misaligned pointer", fn);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (Bc * num_packs <= kFusedMaxEntries) {
    a.chunks = (int)num_chunks;
    return launch_fused(fn, a, f, padding_mask, Bc * S, st);
  }
  // large tables: each chunk through the two-kernel path, one after another
  for (int64_t c = 0; c < num_chunks; ++c) {
    MetaArgs ac = a;
    const int64_t e0 = c * Bc * num_packs;
    ac.real = seq_lens + e0;
    ac.padded = seq_lens_padded ? seq_lens_padded + e0 : nullptr;
    ac.row0 = (int)(c * Bc);
    ac.cu = cu_seqlens + c * a.cu_pad_to;
    ac.cu_padded = a.cu_padded ? a.cu_padded + c * a.cu_pad_to : nullptr;
    ac.pad_between = pad_between_seqs ? pad_between_seqs + c : nullptr;
    ac.info = infos + c;
    s = launch_meta(fn, ac, workspace, st);
    if (s != PSEQ_OK) return s;
    s = launch_gather(fn, f, Bc, S, num_packs, padding_mask, workspace, st, Bc * S, B, c);
    if (s != PSEQ_OK) return s;
  }
  return PSEQ_OK;
}
