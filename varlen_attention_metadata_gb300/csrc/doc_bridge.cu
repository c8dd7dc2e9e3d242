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
// Every row is cut into chunks of 4096 tokens, one CTA each, in two
// launches.  The first summarises every chunk: how many sequences start in
// it, its last run start and its last sequence start (a commutative join:
// sum, max, max).  The second gives each chunk its row prefix by joining the
// summaries of the chunks before it -- no waiting, they are all done -- and
// walks its tokens with a block scan: every run end writes its sequence's
// real length, every sequence start closes the padded length of the one
// before it, and the row's last chunk closes the row and fills unused slots.
// Row statistics reach the info block through atomics (the first launch
// initialises it).
#include "common.cuh"

namespace pseq {
namespace {

constexpr int kThreads = 512;
constexpr int kItems = 8;
constexpr int kTile = kThreads * kItems;

size_t workspace_bytes(int64_t B, int64_t S) {
  const int64_t chunks = S > 0 ? (S + kTile - 1) / kTile : 1;
  return 16 * (size_t)(B > 0 ? B : 1) * (size_t)chunks;
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

__device__ __forceinline__ Marks shfl_xor(const Marks& v, int d) {
  return {__shfl_xor_sync(~0u, v.seqs, d), __shfl_xor_sync(~0u, v.last_run, d), __shfl_xor_sync(~0u, v.last_seq, d)};
}

struct BridgeArgs {
  int B, S, P, chunks;
  int64_t pad_value;
  int64_t* seq_lens;
  int64_t* seq_lens_padded;
  int64_t* positions;  // may be NULL
  pseq_info* info;
  int4* marks;         // [B * chunks]
};

// This thread's eight tokens of a row chunk: run starts, sequence starts.
template <typename Id>
__device__ __forceinline__ Marks chunk_flags(const Id* d, int S, int s0, Id (&v)[kItems], Id& left, unsigned& runs,
                                             unsigned& seqs) {
  if (s0 + kItems <= S && (reinterpret_cast<uintptr_t>(d + s0) & 15) == 0) {
    // whole group in the row and 16-byte aligned: vector loads
    constexpr int kVec = kItems * (int)sizeof(Id) / 16;
    int4 q[kVec];
#pragma unroll
    for (int k = 0; k < kVec; ++k) q[k] = ld_stream(reinterpret_cast<const int4*>(d + s0) + k);
    memcpy(v, q, sizeof(v));
  } else {
#pragma unroll
    for (int k = 0; k < kItems; ++k) v[k] = s0 + k < S ? __ldg(d + s0 + k) : Id(0);
  }
  left = (s0 > 0 && s0 < S) ? __ldg(d + s0 - 1) : Id(0);
  runs = 0;
  seqs = 0;
  Marks mine = {0, -1, -1};
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int s = s0 + k;
    if (s >= S) break;
    const Id prev = k ? v[k - 1] : left;
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
  return mine;
}

template <typename Id>
__global__ void __launch_bounds__(kThreads) bridge_summary_kernel(const Id* __restrict__ doc, BridgeArgs a) {
  __shared__ Marks s_warp[kThreads / 32];
  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.y, ch = blockIdx.x;
  if (row == 0 && ch == 0 && tid == 0) *a.info = {PSEQ_OK, 0, 0, 0};
  Id v[kItems], left;
  unsigned runs, seqs;
  Marks m = chunk_flags(doc + (int64_t)row * a.S, a.S, ch * kTile + tid * kItems, v, left, runs, seqs);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = join(m, shfl_xor(m, d));
  if (lane == 0) s_warp[warp] = m;
  __syncthreads();
  if (tid == 0) {
    Marks t = s_warp[0];
    for (int w = 1; w < kThreads / 32; ++w) t = join(t, s_warp[w]);
    a.marks[(int64_t)row * a.chunks + ch] = make_int4(t.seqs, t.last_run, t.last_seq, 0);
  }
}

template <typename Id>
__global__ void __launch_bounds__(kThreads) bridge_walk_kernel(const Id* __restrict__ doc, BridgeArgs a) {
  __shared__ Marks s_warp[kThreads / 32];
  __shared__ Marks s_prefix;
  __shared__ int s_longest, s_overflow;
  pdl_enter();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.y, ch = blockIdx.x;
  const int S = a.S, P = a.P;
  const Id* d = doc + (int64_t)row * S;
  int64_t* real_out = a.seq_lens + (int64_t)row * P;
  int64_t* pad_out = a.seq_lens_padded + (int64_t)row * P;
  // the row prefix: every earlier chunk's summary (all written by the first launch)
  if (warp == 0) {
    Marks pre = {0, -1, -1};
    for (int c = lane; c < ch; c += 32) {
      const int4 q = __ldcg(a.marks + (int64_t)row * a.chunks + c);
      pre = join(pre, Marks{q.x, q.y, q.z});
    }
#pragma unroll
    for (int dd = 16; dd > 0; dd >>= 1) pre = join(pre, shfl_xor(pre, dd));
    if (lane == 0) {
      s_prefix = pre;
      s_longest = 0;
      s_overflow = 0;
    }
  }
  Id v[kItems], left;
  unsigned runs, seqs;
  const int s0 = ch * kTile + tid * kItems;
  const Marks mine = chunk_flags(d, S, s0, v, left, runs, seqs);
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
  const Marks prefix = s_prefix;
  before = join(prefix, before);
  const Marks row_so_far = join(prefix, s_warp[kThreads / 32 - 1]);
  // walk this thread's tokens
  int last_run = before.last_run, last_seq = before.last_seq, count = before.seqs;
  int longest = 0;
  long long pos[kItems];
#pragma unroll
  for (int k = 0; k < kItems; ++k) {
    const int s = s0 + k;
    pos[k] = 0;
    if (s >= S) break;
    const Id prev = k ? v[k - 1] : left;
    if (runs & (1u << k)) {
      if (s > 0 && prev != 0) {  // the document run [last_run, s) ends here
        const int len = s - last_run;
        if (count - 1 < P) real_out[count - 1] = len;
        longest = max(longest, len);
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
    pos[k] = v[k] != 0 ? s - last_run : 0;
  }
  if (a.positions) {
    int64_t* prow = a.positions + (int64_t)row * S;
    if (s0 + kItems <= S && (reinterpret_cast<uintptr_t>(prow + s0) & 15) == 0) {
#pragma unroll
      for (int k = 0; k < kItems; k += 2)
        st_stream(reinterpret_cast<int4*>(prow + s0 + k),
                  make_int4((int)(uint32_t)pos[k], (int)(pos[k] >> 32), (int)(uint32_t)pos[k + 1],
                            (int)(pos[k + 1] >> 32)));
    } else {
      for (int k = 0; k < kItems && s0 + k < S; ++k) prow[s0 + k] = pos[k];
    }
  }
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
  if (row_end) {
    for (int k = min(row_so_far.seqs, P) + tid; k < P; k += kThreads) {
      real_out[k] = a.pad_value;
      pad_out[k] = a.pad_value;
    }
  }
  __syncthreads();
  if (tid == 0) {
    if (s_longest) atomicMax(&a.info->max_seqlen, s_longest);
    if (s_overflow) atomicMax(&a.info->status, (int)PSEQ_ERR_CAPACITY);
    if (row_end) {
      atomicMax(&a.info->count, row_so_far.seqs);
      atomicAdd(&a.info->total, row_so_far.seqs);
    }
  }
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
    a.marks = static_cast<int4*>(workspace);
    const dim3 grid((unsigned)a.chunks, (unsigned)B);
    if (id_bytes == 4) {
      const int32_t* d = static_cast<const int32_t*>(doc_ids);
      e = launch_pdl(bridge_summary_kernel<int32_t>, grid, dim3(kThreads), 0, st, d, a);
      if (e == cudaSuccess) e = launch_pdl(bridge_walk_kernel<int32_t>, grid, dim3(kThreads), 0, st, d, a);
    } else {
      const int64_t* d = static_cast<const int64_t*>(doc_ids);
      e = launch_pdl(bridge_summary_kernel<int64_t>, grid, dim3(kThreads), 0, st, d, a);
      if (e == cudaSuccess) e = launch_pdl(bridge_walk_kernel<int64_t>, grid, dim3(kThreads), 0, st, d, a);
    }
    launches = 2;
  }
  count_launches(launches);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
}
