// BSHD -> THD conversion: thd_meta, thd_gather, thd_from_batch,
// thd_padding_mask.
//
// Follows NeMo AutoModel v0.5 "nemo_automodel.components.distributed.thd_utils":
// process_input_for_thd (description, Example, Parameters, Returns) and
// _thd_padding_mask.
//
// thd_meta runs in one CTA: the length tables are small (B * num_packs
// entries), so a chunked block scan over them in row-major order drops the
// filler entries, computes both cumulative sums (int64 running totals), the
// in-row source offset of every kept sequence, the absorption gate,
// pad_between_seqs and max_seqlen, and leaves the per-sequence layout
// (source token, stream start, real length) in the workspace.
//
// thd_gather is a persistent grid launched with programmatic dependent
// launch, so its CTAs are resident before thd_meta ends.  Each CTA owns an
// equal slice of stream rows, finds the sequence owning its first row with a
// 32-way warp search, and walks the sequences of its slice.  A sequence's
// rows are contiguous in the source and in the stream, so every piece is one
// contiguous block copy per field and plane (16-byte streaming loads and
// stores when source and destination share their 16-byte alignment).  The
// same CTA writes the padding mask of its slice.
#include "common.cuh"

namespace pseq {
namespace {

constexpr int kMetaThreads = 1024;
constexpr int kMetaWarps = kMetaThreads / 32;
constexpr int kGatherThreads = 512;

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
  int64_t* seq_src;  // [E]  source token (b*S + o) of the sequence's first slot
  int32_t* seq_cup;  // [E+1] stream start of each sequence; [n] = T
  int32_t* seq_real; // [E]
  int64_t* row_pfx;  // [B]  padded prefix at each row's first entry
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
  int32_t* cu;          // may be NULL (mask-only use)
  int32_t* cu_padded;   // may be NULL
  uint8_t* pad_between; // may be NULL
  pseq_info* info;
  int64_t fixed_total;  // >= 0: mask length and info.total (thd_padding_mask)
};

struct Triple {
  int count;
  long long real, padded;
};

__device__ __forceinline__ Triple add(const Triple& a, const Triple& b) {
  return {a.count + b.count, a.real + b.real, a.padded + b.padded};
}

// Exclusive scan of one Triple per thread over the whole block; `total`
// receives the block sum.  Uses `scratch` (kMetaWarps entries).
__device__ __forceinline__ Triple block_exclusive(Triple x, Triple* scratch, Triple& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Triple inc = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    Triple o = {__shfl_up_sync(~0u, inc.count, d), __shfl_up_sync(~0u, inc.real, d),
                __shfl_up_sync(~0u, inc.padded, d)};
    if (lane >= d) inc = add(o, inc);
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    Triple w = scratch[lane];  // kMetaWarps == 32
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      Triple o = {__shfl_up_sync(~0u, w.count, d), __shfl_up_sync(~0u, w.real, d),
                  __shfl_up_sync(~0u, w.padded, d)};
      if (lane >= d) w = add(o, w);
    }
    scratch[lane] = w;
  }
  __syncthreads();
  Triple ex = {__shfl_up_sync(~0u, inc.count, 1), __shfl_up_sync(~0u, inc.real, 1),
               __shfl_up_sync(~0u, inc.padded, 1)};
  if (lane == 0) ex = {0, 0, 0};
  if (warp > 0) ex = add(scratch[warp - 1], ex);
  total = scratch[kMetaWarps - 1];
  return ex;
}

__global__ void __launch_bounds__(kMetaThreads) thd_meta_kernel(MetaArgs a, Workspace ws) {
  static_assert(kMetaWarps == 32, "scan assumes 32 warps");
  __shared__ Triple s_scan[kMetaWarps];
  __shared__ int s_bad, s_mismatch, s_last_mismatch, s_max_real;
  pdl_launch_dependents();  // the gather may start its prologue now

  const int tid = threadIdx.x;
  if (tid == 0) {
    s_bad = 0;
    s_mismatch = 0;
    s_last_mismatch = -1;
    s_max_real = 0;
  }
  __syncthreads();
  const int E = a.B * a.P;
  Triple carry = {0, 0, 0};
  for (int base = 0; base < E; base += kMetaThreads) {
    const int e = base + tid;
    const bool valid = e < E;
    long long real = 0, padded = 0;
    bool keep = false, bad = false;
    if (valid) {
      real = a.real[e];
      padded = a.padded ? a.padded[e] : real;
      const bool real_filler = a.has_filler && real == a.pad_value;
      const bool padded_filler = a.has_filler && padded == a.pad_value;
      if (real_filler != padded_filler) bad = true;
      else if (!real_filler) {
        keep = true;
        if (real < 0 || padded < real) bad = true;
      }
    }
    Triple total;
    const Triple ex = block_exclusive({keep ? 1 : 0, keep ? real : 0, keep ? padded : 0}, s_scan, total);
    const int k = carry.count + ex.count;
    const long long R = carry.real + ex.real;
    const long long Pd = carry.padded + ex.padded;
    const int b = valid ? e / a.P : 0;
    if (valid && e % a.P == 0) ws.row_pfx[b] = Pd;
    __syncthreads();
    if (keep) {
      const long long o = Pd - ws.row_pfx[b];
      if (o + padded > a.S) bad = true;
      ws.seq_src[k] = (long long)b * a.S + o;
      ws.seq_real[k] = (int32_t)real;
      ws.seq_cup[k] = (int32_t)Pd;
      if (a.cu) a.cu[k] = (int32_t)R;
      if (a.cu_padded) a.cu_padded[k] = (int32_t)Pd;
      if (real != padded) {
        atomicAdd(&s_mismatch, 1);
        atomicMax(&s_last_mismatch, k);
      }
      atomicMax(&s_max_real, (int)min(real, (long long)INT32_MAX));
    }
    if (bad) s_bad = 1;
    carry = add(carry, total);
    __syncthreads();
  }
  if (tid != 0) return;
  const int n = carry.count;
  const long long T = carry.padded;
  int status = s_bad ? PSEQ_ERR_VALUE : PSEQ_OK;
  if (status == PSEQ_OK && T > INT32_MAX) status = PSEQ_ERR_OVERFLOW;
  const bool absorbed =
      a.absorb && n >= 1 && (s_mismatch == 0 || (s_mismatch == 1 && s_last_mismatch == n - 1));
  const long long last = absorbed ? T : carry.real;
  if (a.cu) a.cu[n] = (int32_t)last;
  if (a.cu_padded) a.cu_padded[n] = (int32_t)T;
  ws.seq_cup[n] = (int32_t)T;
  if (a.pad_between) *a.pad_between = (a.padded && s_mismatch > 0 && !absorbed) ? 1 : 0;
  long long longest = s_max_real;
  if (absorbed) longest = max(longest, T - (carry.real - ws.seq_real[n - 1]));
  if (n == 0) longest = 0;
  const long long shown_total = a.fixed_total >= 0 ? a.fixed_total : T;
  Header h = {};
  h.status = status;
  h.n = n;
  h.T = (int32_t)T;
  h.Tmask = (int32_t)shown_total;
  *ws.hdr = h;
  pseq_info out = {status, n, (int32_t)longest, (int32_t)shown_total};
  if (status != PSEQ_OK) out = {status, 0, 0, 0};
  *a.info = out;
}

struct Fields {
  const unsigned char* src[PSEQ_MAX_FIELDS];
  unsigned char* dst[PSEQ_MAX_FIELDS];
  int64_t row_bytes[PSEQ_MAX_FIELDS];
  int planes[PSEQ_MAX_FIELDS];
  int num;
};

// Largest k in [0, n) with cup[k] <= x, given cup[0] <= x < cup[n].
// The whole warp searches, 32 probes per round.
__device__ __forceinline__ int warp_find(const int32_t* cup, int n, int64_t x) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) / 32;
    const int probe = lo + lane * step;
    const bool ok = probe < hi && (int64_t)__ldcg(cup + probe) <= x;
    const unsigned m = __ballot_sync(~0u, ok);
    const int L = 31 - __clz(m);
    lo = lo + L * step;
    hi = min(lo + step, hi);
  }
  return lo;
}

__global__ void __launch_bounds__(kGatherThreads)
    thd_gather_kernel(Fields f, int64_t B, int64_t S, uint8_t* __restrict__ mask, Workspace ws,
                      int64_t max_seqs, int64_t max_rows) {
  __shared__ int s_first;
  pdl_wait();
  const int status = __ldcg(&ws.hdr->status);
  if (status != PSEQ_OK) return;
  const int n = __ldcg(&ws.hdr->n);
  const int64_t T = __ldcg(&ws.hdr->T);
  const int64_t Tm = __ldcg(&ws.hdr->Tmask);
  // a layout that does not fit the buffers did not come from thd_meta: write nothing
  if (n < 0 || n > max_seqs || T < 0 || T > B * S || Tm < T || Tm > max_rows) return;
  const int64_t G = gridDim.x;
  const int64_t per = (Tm + G - 1) / G;
  const int64_t r0 = (int64_t)blockIdx.x * per;
  const int64_t r1 = min(r0 + per, Tm);
  if (r0 >= r1) return;
  const int64_t g1 = min(r1, T);
  const int tid = threadIdx.x;
  if (r0 < g1) {
    if (tid < 32) {
      const int k = warp_find(ws.seq_cup, n, r0);
      if (tid == 0) s_first = k;
    }
    __syncthreads();
    for (int k = s_first; k < n; ++k) {
      const int64_t cs = __ldcg(ws.seq_cup + k);
      if (cs >= g1) break;
      const int64_t ce = __ldcg(ws.seq_cup + k + 1);
      const int64_t lo = max(r0, cs), hi = min(g1, ce);
      if (lo >= hi) continue;
      const int64_t src_tok = __ldcg(ws.seq_src + k) + (lo - cs);
      for (int i = 0; i < f.num; ++i) {
        const int64_t rb = f.row_bytes[i];
        for (int p = 0; p < f.planes[i]; ++p)
          block_copy(f.dst[i] + ((int64_t)p * T + lo) * rb, f.src[i] + ((int64_t)p * B * S + src_tok) * rb,
                     (hi - lo) * rb);
      }
      if (mask) {
        const int64_t real_end = cs + __ldcg(ws.seq_real + k);
        for (int64_t t = lo + tid; t < hi; t += kGatherThreads) mask[t] = t >= real_end ? 1 : 0;
      }
    }
  }
  if (mask) {
    const int64_t tail = max(r0, T);
    if (tail < r1) block_fill_bytes(mask + tail, r1 - tail, 1);
  }
}

int gather_grid(int64_t rows, int64_t bytes_per_row) {
  // enough CTAs to keep every SM busy on large streams, fewer on tiny ones
  const int64_t full = (int64_t)sm_count() * (2048 / kGatherThreads);
  const int64_t by_bytes = (rows * (bytes_per_row + 1) + 8191) / 8192;
  int64_t g = by_bytes < full ? by_bytes : full;
  return (int)(g < 1 ? 1 : g);
}

pseq_status check_lengths(const char* fn, int64_t B, int64_t S, int64_t P) {
  if (B < 0 || S < 0 || P < 0)
    return fail(PSEQ_ERR_ARG, "%s: negative size (B=%lld S=%lld num_packs=%lld)", fn, (long long)B, (long long)S,
                (long long)P);
  if (B > 0 && S > INT32_MAX / B) return fail(PSEQ_ERR_OVERFLOW, "%s: B*S exceeds INT32_MAX", fn);
  if (B > 0 && P > (INT32_MAX - 1) / B) return fail(PSEQ_ERR_OVERFLOW, "%s: B*num_packs exceeds INT32_MAX", fn);
  return PSEQ_OK;
}

pseq_status launch_meta(const char* fn, MetaArgs a, void* workspace, size_t ws_bytes, cudaStream_t st) {
  const int64_t E = (int64_t)a.B * a.P;
  const size_t need = workspace_bytes(a.B, E);
  if (!workspace || ws_bytes < need || !aligned(workspace, 16))
    return fail(PSEQ_ERR_ARG, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", fn, need, ws_bytes);
  if ((E > 0 && !a.real) || !a.info) return fail(PSEQ_ERR_ARG, "%s: NULL lengths or info", fn);
  if (!aligned(a.real, 8) || !aligned(a.padded, 8) || !aligned(a.cu, 4) || !aligned(a.cu_padded, 4) ||
      !aligned(a.info, 4))
    return fail(PSEQ_ERR_ARG, "%s: misaligned pointer", fn);
  thd_meta_kernel<<<1, kMetaThreads, 0, st>>>(a, carve(workspace, a.B, E));
  count_launches(1);
  return check_launch(fn);
}

pseq_status launch_gather(const char* fn, const pseq_field* fields, int num_fields, int64_t B, int64_t S,
                          int64_t P, uint8_t* mask, const void* workspace, size_t ws_bytes, cudaStream_t st,
                          int64_t mask_rows) {
  if (num_fields < 0 || num_fields > PSEQ_MAX_FIELDS)
    return fail(PSEQ_ERR_ARG, "%s: num_fields must be in [0, %d]", fn, PSEQ_MAX_FIELDS);
  if (num_fields > 0 && !fields) return fail(PSEQ_ERR_ARG, "%s: fields is NULL", fn);
  const int64_t E = B * P;
  const size_t need = workspace_bytes(B, E);
  if (!workspace || ws_bytes < need || !aligned(workspace, 16))
    return fail(PSEQ_ERR_ARG, "%s: workspace needs %zu bytes, 16-byte aligned (got %zu)", fn, need, ws_bytes);
  Fields f = {};
  f.num = num_fields;
  int64_t bytes_per_row = 0;
  for (int i = 0; i < num_fields; ++i) {
    const pseq_field& x = fields[i];
    if (x.elem_bytes != 1 && x.elem_bytes != 2 && x.elem_bytes != 4 && x.elem_bytes != 8)
      return fail(PSEQ_ERR_ARG, "%s: field %d: elem_bytes must be 1, 2, 4 or 8", fn, i);
    if (x.planes < 1 || x.row_elems < 1) return fail(PSEQ_ERR_ARG, "%s: field %d: planes and row_elems must be >= 1", fn, i);
    if (B * S > 0 && (!x.src || !x.dst)) return fail(PSEQ_ERR_ARG, "%s: field %d: NULL src or dst", fn, i);
    const int64_t rb = x.row_elems * x.elem_bytes;
    if (x.row_elems > (INT64_MAX / 8) / (B * S > 0 ? B * S * x.planes : 1))
      return fail(PSEQ_ERR_OVERFLOW, "%s: field %d is too large", fn, i);
    f.src[i] = static_cast<const unsigned char*>(x.src);
    f.dst[i] = static_cast<unsigned char*>(x.dst);
    f.row_bytes[i] = rb;
    f.planes[i] = x.planes;
    bytes_per_row += rb * x.planes;
  }
  if (num_fields == 0 && !mask) return PSEQ_OK;
  const int grid = gather_grid(mask_rows, bytes_per_row);
  Workspace ws = carve(workspace, B, E);
  cudaError_t e = launch_pdl(thd_gather_kernel, dim3(grid), dim3(kGatherThreads), 0, st, f, B, S, mask, ws, E,
                             mask_rows);
  count_launches(1);
  if (e != cudaSuccess) return fail(PSEQ_ERR_CUDA, "%s: %s", fn, cudaGetErrorString(e));
  return check_launch(fn);
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
  pseq_status s = check_lengths("thd_meta", B, S, num_packs);
  if (s != PSEQ_OK) return s;
  if (!cu_seqlens) return fail(PSEQ_ERR_ARG, "thd_meta: cu_seqlens is required");
  MetaArgs a = {};
  a.real = seq_lens;
  a.padded = seq_lens_padded;
  a.B = (int)B;
  a.P = (int)num_packs;
  a.S = S;
  a.pad_value = pad_value;
  a.has_filler = 1;
  a.absorb = absorb_trailing_pad ? 1 : 0;
  a.cu = cu_seqlens;
  a.cu_padded = seq_lens_padded ? cu_seqlens_padded : nullptr;
  a.pad_between = pad_between_seqs;
  a.info = info;
  a.fixed_total = -1;
  return launch_meta("thd_meta", a, workspace, workspace_bytes_, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" pseq_status thd_gather(const pseq_field* fields, int32_t num_fields, int64_t B, int64_t S,
                                  int64_t num_packs, uint8_t* padding_mask, const void* workspace,
                                  size_t workspace_bytes_, pseq_stream stream) {
  clear_error();
  pseq_status s = check_lengths("thd_gather", B, S, num_packs);
  if (s != PSEQ_OK) return s;
  return launch_gather("thd_gather", fields, num_fields, B, S, num_packs, padding_mask, workspace,
                       workspace_bytes_, reinterpret_cast<cudaStream_t>(stream), B * S);
}

extern "C" pseq_status thd_from_batch(const int64_t* seq_lens, const int64_t* seq_lens_padded, int64_t B,
                                      int64_t S, int64_t num_packs, int64_t pad_value,
                                      int32_t absorb_trailing_pad, const pseq_field* fields, int32_t num_fields,
                                      int32_t* cu_seqlens, int32_t* cu_seqlens_padded, uint8_t* padding_mask,
                                      uint8_t* pad_between_seqs, pseq_info* info, void* workspace,
                                      size_t workspace_bytes_, pseq_stream stream) {
  clear_error();
  pseq_status s = check_lengths("thd_from_batch", B, S, num_packs);
  if (s != PSEQ_OK) return s;
  if (num_fields < 0 || num_fields > PSEQ_MAX_FIELDS || (num_fields > 0 && !fields))
    return fail(PSEQ_ERR_ARG, "thd_from_batch: bad fields / num_fields");
  s = thd_meta(seq_lens, seq_lens_padded, B, S, num_packs, pad_value, absorb_trailing_pad, cu_seqlens,
               cu_seqlens_padded, pad_between_seqs, info, workspace, workspace_bytes_, stream);
  if (s != PSEQ_OK) return s;
  return thd_gather(fields, num_fields, B, S, num_packs, padding_mask, workspace, workspace_bytes_, stream);
}

extern "C" pseq_status thd_padding_mask(int64_t total_tokens, const int64_t* valid_seq_lens,
                                        const int64_t* valid_seq_lens_padded, int64_t n, uint8_t* mask,
                                        pseq_info* info, void* workspace, size_t workspace_bytes_,
                                        pseq_stream stream) {
  clear_error();
  if (total_tokens < 0 || n < 0) return fail(PSEQ_ERR_ARG, "thd_padding_mask: negative size");
  if (total_tokens > INT32_MAX) return fail(PSEQ_ERR_OVERFLOW, "thd_padding_mask: total_tokens exceeds INT32_MAX");
  if (n > INT32_MAX - 1) return fail(PSEQ_ERR_OVERFLOW, "thd_padding_mask: n exceeds INT32_MAX");
  if (total_tokens > 0 && !mask) return fail(PSEQ_ERR_ARG, "thd_padding_mask: mask is NULL");
  MetaArgs a = {};
  a.real = valid_seq_lens;
  a.padded = valid_seq_lens_padded;
  a.B = 1;
  a.P = (int)n;
  a.S = total_tokens;
  a.pad_value = 0;
  a.has_filler = 0;
  a.absorb = 0;
  a.info = info;
  a.fixed_total = total_tokens;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  pseq_status s = launch_meta("thd_padding_mask", a, workspace, workspace_bytes_, st);
  if (s != PSEQ_OK) return s;
  if (total_tokens == 0) return PSEQ_OK;
  return launch_gather("thd_padding_mask", nullptr, 0, 1, total_tokens, n, mask, workspace, workspace_bytes_, st,
                       total_tokens);
}
