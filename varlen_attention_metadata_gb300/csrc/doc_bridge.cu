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
// One CTA per row (rows are independent: every row start opens a run).  The
// row is walked in tiles of 4096 tokens; a block scan per tile carries the
// position of the last run start, the last sequence start and the number of
// sequences so far, so every run end writes its sequence's real length and
// every sequence start closes the padded length of the one before it.  The
// CTA that finishes last folds the per-row statistics into the info block.
#include "common.cuh"

namespace pseq {
namespace {

constexpr int kThreads = 512;
constexpr int kItems = 8;
constexpr int kTile = kThreads * kItems;

struct Header {
  unsigned int finished;
  unsigned int pad[31];
};

struct RowStat {
  int overflow, sequences, longest, unused;
};

size_t workspace_bytes(int64_t B) { return sizeof(Header) + sizeof(RowStat) * (size_t)(B > 0 ? B : 1); }

__device__ __forceinline__ unsigned inc_acq_rel(unsigned* p, unsigned limit) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(limit) : "memory");
  return old;
}

// Scan element: sequence starts counted, last run start, last sequence start.
struct Marks {
  int seqs, last_run, last_seq;
};

__device__ __forceinline__ Marks join(const Marks& a, const Marks& b) {
  return {a.seqs + b.seqs, max(a.last_run, b.last_run), max(a.last_seq, b.last_seq)};
}

__device__ __forceinline__ Marks shfl_up(const Marks& v, int d) {
  return {__shfl_up_sync(~0u, v.seqs, d), __shfl_up_sync(~0u, v.last_run, d), __shfl_up_sync(~0u, v.last_seq, d)};
}

struct BridgeArgs {
  int B, S, P;
  int64_t pad_value;
  int64_t* seq_lens;
  int64_t* seq_lens_padded;
  int64_t* positions;  // may be NULL
  pseq_info* info;
  Header* hdr;
  RowStat* stats;
};

template <typename Id>
__global__ void __launch_bounds__(kThreads) doc_bridge_kernel(const Id* __restrict__ doc, BridgeArgs a) {
  __shared__ Marks s_warp[kThreads / 32];
  __shared__ int s_overflow, s_longest, s_last_cta;
  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const int S = a.S, P = a.P;
  const Id* d = doc + (int64_t)row * S;
  int64_t* real_out = a.seq_lens + (int64_t)row * P;
  int64_t* pad_out = a.seq_lens_padded + (int64_t)row * P;
  if (tid == 0) s_overflow = s_longest = 0;
  __syncthreads();
  Marks carry = {0, -1, -1};
  for (int base = 0; base < S; base += kTile) {
    const int s0 = base + tid * kItems;
    Id v[kItems];
#pragma unroll
    for (int k = 0; k < kItems; ++k) v[k] = s0 + k < S ? __ldg(d + s0 + k) : Id(0);
    const Id left = (s0 > 0 && s0 < S) ? __ldg(d + s0 - 1) : Id(0);
    unsigned runs = 0, seqs = 0;
    Marks mine = {0, -1, -1};
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int s = s0 + k;
      if (s >= S) break;
      const Id prev = k ? v[k - 1] : left;
      const bool run_start = s == 0 || v[k] != prev;
      const bool seq_start = s == 0 || (v[k] != 0 && v[k] != prev);
      if (run_start) {
        runs |= 1u << k;
        mine.last_run = s;
      }
      if (seq_start) {
        seqs |= 1u << k;
        mine.last_seq = s;
        mine.seqs += 1;
      }
    }
    // exclusive block scan of the marks, in token order
    Marks inc = mine;
#pragma unroll
    for (int dd = 1; dd < 32; dd <<= 1) {
      const Marks o = shfl_up(inc, dd);
      if (lane >= dd) inc = join(o, inc);
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      Marks w = lane < kThreads / 32 ? s_warp[lane] : Marks{0, -1, -1};
#pragma unroll
      for (int dd = 1; dd < kThreads / 32; dd <<= 1) {
        const Marks o = shfl_up(w, dd);
        if (lane >= dd) w = join(o, w);
      }
      if (lane < kThreads / 32) s_warp[lane] = w;
    }
    __syncthreads();
    Marks before = shfl_up(inc, 1);
    if (lane == 0) before = {0, -1, -1};
    if (warp > 0) before = join(s_warp[warp - 1], before);
    before = join(carry, before);
    const Marks tile_total = s_warp[kThreads / 32 - 1];
    // walk this thread's tokens with the carried marks
    int last_run = before.last_run, last_seq = before.last_seq, count = before.seqs;
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const int s = s0 + k;
      if (s >= S) break;
      const Id prev = k ? v[k - 1] : left;
      if (runs & (1u << k)) {
        if (s > 0 && prev != 0) {  // the document run [last_run, s) ends here
          const int len = s - last_run;
          if (count - 1 < P) real_out[count - 1] = len;
          atomicMax(&s_longest, len);
        }
        last_run = s;
      }
      if (seqs & (1u << k)) {
        if (count > 0 && count - 1 < P) pad_out[count - 1] = s - last_seq;
        if (count < P) {
          if (v[k] == 0) real_out[count] = 0;  // padding before any document
        } else {
          s_overflow = 1;
        }
        last_seq = s;
        count += 1;
      }
      if (a.positions) a.positions[(int64_t)row * S + s] = v[k] != 0 ? s - last_run : 0;
    }
    carry = join(carry, tile_total);
    __syncthreads();
  }
  // the row end closes the last run and the last sequence
  if (tid == 0 && S > 0) {
    const Id tail = __ldg(d + S - 1);
    const int count = carry.seqs;
    if (tail != 0 && count - 1 < P) {
      real_out[count - 1] = S - carry.last_run;
      atomicMax(&s_longest, S - carry.last_run);
    }
    if (count - 1 < P) pad_out[count - 1] = S - carry.last_seq;
  }
  __syncthreads();
  const int used = min(carry.seqs, P);
  for (int k = used + tid; k < P; k += kThreads) {
    real_out[k] = a.pad_value;
    pad_out[k] = a.pad_value;
  }
  if (tid == 0) {
    a.stats[row] = {s_overflow, carry.seqs, s_longest, 0};
    s_last_cta = inc_acq_rel(&a.hdr->finished, gridDim.x - 1) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last_cta || tid != 0) return;
  int overflow = 0, most = 0, longest = 0;
  long long total = 0;
  for (int r = 0; r < (int)gridDim.x; ++r) {
    const RowStat st = a.stats[r];
    overflow |= st.overflow;
    most = max(most, st.sequences);
    longest = max(longest, st.longest);
    total += st.sequences;
  }
  *a.info = overflow ? pseq_info{PSEQ_ERR_CAPACITY, most, 0, 0}
                     : pseq_info{PSEQ_OK, most, longest, (int32_t)min(total, (long long)INT32_MAX)};
}

__global__ void empty_bridge_kernel(pseq_info* info) {
  pdl_enter();
  *info = {PSEQ_OK, 0, 0, 0};
}

}  // namespace
}  // namespace pseq

using namespace pseq;

extern "C" size_t pseq_doc_ids_to_lengths_workspace_size(int64_t B) {
  if (B < 0) return 0;
  return workspace_bytes(B);
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
  if (B > 0 && num_packs > INT32_MAX / B) return fail(PSEQ_ERR_OVERFLOW, "%s: B*num_packs exceeds INT32_MAX", fn);
  if (!info || (B * S > 0 && !doc_ids) || (B * num_packs > 0 && (!seq_lens || !seq_lens_padded)))
    return fail(PSEQ_ERR_ARG, "%s: NULL pointer", fn);
  if (!aligned(doc_ids, (uintptr_t)id_bytes) || !aligned(seq_lens, 8) || !aligned(seq_lens_padded, 8) ||
      !aligned(position_ids, 8) || !aligned(info, 4))
    return fail(PSEQ_ERR_ARG, "%s: misaligned pointer", fn);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (B == 0) {
    e = launch_pdl(empty_bridge_kernel, dim3(1), dim3(1), 0, st, info);
  } else {
    const size_t need = workspace_bytes(B);
    if (!workspace || workspace_bytes_ < need || !aligned(workspace, 16))
      return fail(PSEQ_ERR_ARG, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", fn, need,
                  workspace_bytes_);
    BridgeArgs a = {};
    a.B = (int)B;
    a.S = (int)S;
    a.P = (int)num_packs;
    a.pad_value = pad_value;
    a.seq_lens = seq_lens;
    a.seq_lens_padded = seq_lens_padded;
    a.positions = position_ids;
    a.info = info;
    a.hdr = static_cast<Header*>(workspace);
    a.stats = reinterpret_cast<RowStat*>(static_cast<unsigned char*>(workspace) + sizeof(Header));
    if (id_bytes == 4)
      e = launch_pdl(doc_bridge_kernel<int32_t>, dim3((unsigned)B), dim3(kThreads), 0, st,
                     static_cast<const int32_t*>(doc_ids), a);
    else
      e = launch_pdl(doc_bridge_kernel<int64_t>, dim3((unsigned)B), dim3(kThreads), 0, st,
                     static_cast<const int64_t*>(doc_ids), a);
  }
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}
