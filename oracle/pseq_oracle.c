/*
 * Plain CPU oracle for the packed-sequence metadata path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of the package
 * entry module and the CPU-baseline / reference legs of the benchmark may
 * load this library.  The product path never calls it.  It shares no source,
 * header, table or constant with the CUDA library: every status is reported
 * through this file's own ORC_* codes, mapped by the Python wrapper.
 *
 * Every function is the plain definition written out as loops over rows,
 * tokens and sequences, in the order the pages state the steps.  Nothing is
 * blocked, fused or reordered.  All arithmetic is int64.
 *
 * Pages followed:
 *   [packed_seq]  NeMo AutoModel API reference,
 *                 "nemo_automodel.components.datasets.packed_seq"
 *   [thd_utils]   NeMo AutoModel v0.5 API reference,
 *                 "nemo_automodel.components.distributed.thd_utils"
 *   [who_packs]   "Who packs the sequences: the loader, or the trainer?"
 *                 (NeMo-RL #4105 explainer page)
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_VALUE 3    /* malformed lengths / layout                     */
#define ORC_CAPACITY 4 /* a bin does not fit its capacity or row width   */

/* Read element i of an integer array whose elements are 4 or 8 bytes wide. */
static int64_t read_int(const void* p, int elem_bytes, int64_t i) {
  if (elem_bytes == 4) return (int64_t)((const int32_t*)p)[i];
  return ((const int64_t*)p)[i];
}

/* ------------------------------------------------------------------------
 * O1  packed_seq_params_from_doc_ids
 * [packed_seq] module description and "packed_seq_params_from_doc_ids":
 *   segments are maximal runs of an identical document index within a row,
 *   with a forced boundary at every row start; padding runs (index 0) are
 *   segments of their own; cu_seqlens covers the whole flattened B*S axis and
 *   ends at B*S (PackedSeqParams.cu_seqlens); max_seqlen is the length of the
 *   longest segment (PackedSeqParams.max_seqlen).
 * cu_out must hold B*S+1 entries.  Returns the number of segments.
 * ---------------------------------------------------------------------- */
int64_t oracle_from_doc_ids(const void* doc_ids, int elem_bytes, int64_t B,
                            int64_t S, int32_t* cu_out, int32_t* max_seqlen) {
  int64_t n = 0;
  int64_t total = B * S;
  if (total > 0) cu_out[n++] = 0;
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t s = 0; s < S; ++s) {
      int64_t t = b * S + s;
      if (t == 0) continue;
      int row_start = (s == 0);
      int doc_change = read_int(doc_ids, elem_bytes, t) !=
                       read_int(doc_ids, elem_bytes, t - 1);
      if (row_start || doc_change) cu_out[n++] = (int32_t)t;
    }
  }
  if (total > 0) cu_out[n++] = (int32_t)total;
  else cu_out[n++] = 0;
  int64_t num_segments = n - 1;
  int64_t best = 0;
  for (int64_t k = 0; k < num_segments; ++k) {
    int64_t len = (int64_t)cu_out[k + 1] - (int64_t)cu_out[k];
    if (len > best) best = len;
  }
  *max_seqlen = (int32_t)best;
  return num_segments;
}

/* ------------------------------------------------------------------------
 * O2  process_input_for_thd, metadata part
 * [thd_utils] "process_input_for_thd": description (filter entries equal to
 *   seq_lens_padding_value from seq_lens and seq_lens_padded), Example
 *   (cu_seqlens = [0] + cumsum(real), cu_seqlens_padded = [0] +
 *   cumsum(padded)), Returns 'cu_seqlens' (trailing-pack-pad absorption),
 *   'pad_between_seqs', 'max_seqlen'.
 *
 * Readings where the page is silent:
 *  - the absorption gate (its body is not shown): when absorb is set and
 *    n >= 1 and every kept sequence but the last has real == padded, the
 *    last entry of cu_seqlens is grown to the stream length T;
 *  - T, the stream length, is the sum of the kept padded lengths;
 *  - sequence i of row b is taken from that row at in-row offset o_i, the
 *    sum of the padded lengths of the kept entries before it in that row;
 *  - malformed input (one array has the filler where the other does not, a
 *    negative length, padded < real, a row whose padded lengths exceed S)
 *    is ORC_VALUE;
 *  - seq_lens_padded absent: padded := real, pad_between_seqs = 0.
 * Capacities: cu, cu_padded hold B*P+1; seq_* hold B*P.
 * ---------------------------------------------------------------------- */
int oracle_thd_meta(const int64_t* seq_lens, const int64_t* seq_lens_padded,
                    int64_t B, int64_t S, int64_t P, int64_t pad_value,
                    int absorb, int32_t* cu, int32_t* cu_padded,
                    int64_t* seq_row, int64_t* seq_off, int64_t* seq_real,
                    int64_t* seq_padded, int64_t* n_out, int64_t* T_out,
                    int32_t* max_seqlen, int32_t* pad_between) {
  int have_padded = (seq_lens_padded != 0);
  /* Step 1: filter, row by row, keeping row-major order. */
  int64_t n = 0;
  for (int64_t b = 0; b < B; ++b) {
    int64_t offset_in_row = 0;
    for (int64_t c = 0; c < P; ++c) {
      int64_t real = seq_lens[b * P + c];
      int64_t padded = have_padded ? seq_lens_padded[b * P + c] : real;
      int real_is_filler = (real == pad_value);
      int padded_is_filler = (padded == pad_value);
      if (real_is_filler != padded_is_filler) return ORC_VALUE;
      if (real_is_filler) continue;
      if (real < 0 || padded < real) return ORC_VALUE;
      seq_row[n] = b;
      seq_off[n] = offset_in_row;
      seq_real[n] = real;
      seq_padded[n] = padded;
      offset_in_row += padded;
      if (offset_in_row > S) return ORC_VALUE;
      n += 1;
    }
  }
  /* Step 2: the two cumulative sums. */
  int64_t run_real = 0, run_padded = 0;
  cu[0] = 0;
  cu_padded[0] = 0;
  for (int64_t i = 0; i < n; ++i) {
    run_real += seq_real[i];
    run_padded += seq_padded[i];
    cu[i + 1] = (int32_t)run_real;
    cu_padded[i + 1] = (int32_t)run_padded;
  }
  int64_t T = run_padded;
  /* Step 3: trailing-pack-pad absorption (cp_size == 1). */
  if (absorb && n >= 1) {
    int pad_only_at_end = 1;
    for (int64_t i = 0; i + 1 < n; ++i)
      if (seq_real[i] != seq_padded[i]) pad_only_at_end = 0;
    if (pad_only_at_end) cu[n] = (int32_t)T;
  }
  /* Step 4: pad_between_seqs -- do the complete arrays differ? */
  int differ = 0;
  if (have_padded)
    for (int64_t i = 0; i <= n; ++i)
      if (cu[i] != cu_padded[i]) differ = 1;
  /* Step 5: max_seqlen over the final cu_seqlens. */
  int64_t best = 0;
  for (int64_t i = 0; i < n; ++i) {
    int64_t w = (int64_t)cu[i + 1] - (int64_t)cu[i];
    if (w > best) best = w;
  }
  *n_out = n;
  *T_out = T;
  *max_seqlen = (int32_t)best;
  *pad_between = differ;
  return ORC_OK;
}

/* ------------------------------------------------------------------------
 * O3  process_input_for_thd, gather part
 * [thd_utils] "process_input_for_thd" description and Returns: all
 *   sequences are concatenated along the token axis.  A tensor laid out as
 *   [planes, B, S, row_elems] becomes [planes, T, row_elems]: input_ids and
 *   labels [B,S] (planes 1, row 1), position_ids [B,S] or mRoPE [n_rope,B,S]
 *   (planes n_rope), embeddings [B,S,H] (row H).
 *   out[p, cu_padded[i] + j, :] = in[p, b_i, o_i + j, :] for j < padded_i.
 * Elements are copied as raw bytes: no arithmetic on the payload.
 * ---------------------------------------------------------------------- */
void oracle_thd_gather(const void* src, void* dst, int elem_bytes,
                       int64_t planes, int64_t row_elems, int64_t B, int64_t S,
                       int64_t n, const int64_t* seq_row,
                       const int64_t* seq_off, const int64_t* seq_padded,
                       const int32_t* cu_padded, int64_t T) {
  const unsigned char* in = (const unsigned char*)src;
  unsigned char* out = (unsigned char*)dst;
  int64_t row_bytes = row_elems * elem_bytes;
  for (int64_t p = 0; p < planes; ++p) {
    for (int64_t i = 0; i < n; ++i) {
      for (int64_t j = 0; j < seq_padded[i]; ++j) {
        int64_t src_token = (p * B + seq_row[i]) * S + seq_off[i] + j;
        int64_t dst_token = p * T + (int64_t)cu_padded[i] + j;
        for (int64_t e = 0; e < row_bytes; ++e)
          out[dst_token * row_bytes + e] = in[src_token * row_bytes + e];
      }
    }
  }
}

/* ------------------------------------------------------------------------
 * O4  _thd_padding_mask
 * [thd_utils] "_thd_padding_mask": sequence i occupies
 *   [start_i, start_i + padded_i) and only its first real_i slots hold
 *   tokens; every other slot of the stream of length total_tokens is padding
 *   (True).  start_i is the running sum of the padded lengths (of the real
 *   lengths when no padded lengths are given).
 * Reading: a layout longer than total_tokens, or a negative length or
 *   padded < real, is ORC_VALUE.
 * ---------------------------------------------------------------------- */
int oracle_thd_padding_mask(int64_t total_tokens, const int64_t* valid_seq_lens,
                            const int64_t* valid_seq_lens_padded, int64_t n,
                            uint8_t* mask) {
  for (int64_t t = 0; t < total_tokens; ++t) mask[t] = 1;
  int64_t start = 0;
  for (int64_t i = 0; i < n; ++i) {
    int64_t real = valid_seq_lens[i];
    int64_t padded = valid_seq_lens_padded ? valid_seq_lens_padded[i] : real;
    if (real < 0 || padded < real) return ORC_VALUE;
    if (start + padded > total_tokens) return ORC_VALUE;
    for (int64_t j = 0; j < real; ++j) mask[start + j] = 0;
    start += padded;
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------
 * O5  trainer-side squeeze
 * [who_packs] sections "Trainer packs" and "Loader packs": each source is
 *   padded to a multiple of m; the sources of one bin are concatenated end to
 *   end in the given order; cu_seqlens = [0] + cumsum(real) marks the end of
 *   each source's real tokens, cu_seqlens_padded = [0] + cumsum(padded) the
 *   end of each padded source; with stretch set, the last padded boundary is
 *   set to the pack capacity (36 instead of 20 in the page's example).
 * Readings: only the first real_i tokens of a source row are copied; every
 *   other slot of the [num_bins, width] output holds pad_value and is marked
 *   1 in padding_mask.  A bin whose padded total exceeds capacity or width
 *   is ORC_CAPACITY; an empty bin, a member index outside [0,N), or a real
 *   length outside [0,W] is ORC_VALUE.  Malformed input is reported before
 *   any capacity problem, wherever in the bin list each one sits.
 * Per-bin cu arrays are stored one after the other: bin b starts at
 *   bin_offsets[b] + b and has (members of b) + 1 entries.
 * *max_total receives the largest padded total over bins before stretching.
 * ---------------------------------------------------------------------- */
int oracle_pack_squeeze(const void* src, int64_t N, int64_t W, int elem_bytes,
                        const int64_t* real_lens, const int32_t* bin_offsets,
                        const int32_t* bin_members, int64_t num_bins,
                        int64_t multiple, int64_t capacity, int stretch,
                        int64_t width, int64_t pad_value, void* out,
                        int32_t* cu, int32_t* cu_padded, uint8_t* mask,
                        int64_t* max_total) {
  const unsigned char* in = (const unsigned char*)src;
  unsigned char* o = (unsigned char*)out;
  unsigned char pad_bytes[8];
  memcpy(pad_bytes, &pad_value, 8); /* low-order bytes, little-endian */
  /* Pass 1: the input must be well formed. */
  for (int64_t b = 0; b < num_bins; ++b) {
    int64_t first = bin_offsets[b];
    int64_t count = (int64_t)bin_offsets[b + 1] - first;
    if (count <= 0) return ORC_VALUE;
    for (int64_t k = 0; k < count; ++k) {
      int64_t i = bin_members[first + k];
      if (i < 0 || i >= N) return ORC_VALUE;
      if (real_lens[i] < 0 || real_lens[i] > W) return ORC_VALUE;
    }
  }
  /* Pass 2: lay each bin out. */
  int64_t widest = 0;
  for (int64_t b = 0; b < num_bins; ++b) {
    int64_t first = bin_offsets[b];
    int64_t count = (int64_t)bin_offsets[b + 1] - first;
    int32_t* bcu = cu + first + b;
    int32_t* bcup = cu_padded + first + b;
    /* fill the whole output row with padding first */
    for (int64_t t = 0; t < width; ++t) {
      for (int e = 0; e < elem_bytes; ++e)
        o[(b * width + t) * elem_bytes + e] = pad_bytes[e];
      mask[b * width + t] = 1;
    }
    int64_t run_real = 0, run_padded = 0;
    bcu[0] = 0;
    bcup[0] = 0;
    for (int64_t k = 0; k < count; ++k) {
      int64_t i = bin_members[first + k];
      int64_t real = real_lens[i];
      int64_t padded = ((real + multiple - 1) / multiple) * multiple;
      if (run_padded + padded > capacity) return ORC_CAPACITY;
      if (run_padded + padded > width) return ORC_CAPACITY;
      for (int64_t j = 0; j < real; ++j) {
        int64_t t = run_padded + j;
        for (int e = 0; e < elem_bytes; ++e)
          o[(b * width + t) * elem_bytes + e] = in[(i * W + j) * elem_bytes + e];
        mask[b * width + t] = 0;
      }
      run_real += real;
      run_padded += padded;
      bcu[k + 1] = (int32_t)run_real;
      bcup[k + 1] = (int32_t)run_padded;
    }
    if (run_padded > widest) widest = run_padded;
    if (stretch) bcup[count] = (int32_t)capacity;
  }
  *max_total = widest;
  return ORC_OK;
}

/* ------------------------------------------------------------------------
 * O6  thd_padding_mask_from_token_ids
 * [thd_utils] thd_padding_mask_from_token_ids: padding is marked by
 *   comparing token ids with padding_token_id.  That comparison is sound only
 *   if the pad positions form a suffix of the stream; any other placement is
 *   rejected (the page raises ValueError).
 * Returns ORC_VALUE when a pad token is followed by a non-pad token.
 * ---------------------------------------------------------------------- */
int oracle_mask_from_token_ids(const void* ids, int elem_bytes, int64_t n,
                               int64_t pad_id, uint8_t* mask) {
  for (int64_t t = 0; t < n; ++t)
    mask[t] = (read_int(ids, elem_bytes, t) == pad_id) ? 1 : 0;
  int seen_pad = 0;
  for (int64_t t = 0; t < n; ++t) {
    if (mask[t]) seen_pad = 1;
    else if (seen_pad) return ORC_VALUE; /* content after a pad token */
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------
 * O7  first-fit-decreasing bin assignment
 * [who_packs] get_packer: the packer decides which rows go into one bin under
 *   a token budget; the page names First Fit Decreasing among the packers.  The textbook
 *   algorithm: visit the items largest first (ties: smaller index first) and
 *   put each into the first open bin with room; open a new bin when none has
 *   room.  bin_members lists each bin's items in placement order, bin b
 *   starting at bin_offsets[b].  A negative size is ORC_VALUE, one larger
 *   than capacity ORC_CAPACITY.  *num_bins receives the bin count.
 * ---------------------------------------------------------------------- */
int oracle_ffd(const int64_t* sizes, int64_t n, int64_t capacity,
               int32_t* bin_offsets, int32_t* bin_members, int64_t* num_bins) {
  for (int64_t i = 0; i < n; ++i) {
    if (sizes[i] < 0) return ORC_VALUE;
    if (sizes[i] > capacity) return ORC_CAPACITY;
  }
  int64_t* order = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
  int64_t* room = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
  int64_t* bin_of = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
  /* order: selection sort on (size descending, index ascending) */
  for (int64_t i = 0; i < n; ++i) order[i] = i;
  for (int64_t i = 0; i < n; ++i) {
    int64_t best = i;
    for (int64_t j = i + 1; j < n; ++j) {
      int64_t a = order[j], b = order[best];
      if (sizes[a] > sizes[b] || (sizes[a] == sizes[b] && a < b)) best = j;
    }
    int64_t tmp = order[i];
    order[i] = order[best];
    order[best] = tmp;
  }
  /* first fit */
  int64_t bins = 0;
  for (int64_t k = 0; k < n; ++k) {
    int64_t item = order[k];
    int64_t b = 0;
    while (b < bins && room[b] < sizes[item]) ++b;
    if (b == bins) {
      room[bins] = capacity;
      bins += 1;
    }
    room[b] -= sizes[item];
    bin_of[k] = b;
  }
  /* members of each bin, in placement order */
  int64_t pos = 0;
  for (int64_t b = 0; b < bins; ++b) {
    bin_offsets[b] = (int32_t)pos;
    for (int64_t k = 0; k < n; ++k)
      if (bin_of[k] == b) bin_members[pos++] = (int32_t)order[k];
  }
  bin_offsets[bins] = (int32_t)pos;
  *num_bins = bins;
  free(order);
  free(room);
  free(bin_of);
  return ORC_OK;
}

/* ------------------------------------------------------------------------
 * O8  doc_ids -> seq_lens / seq_lens_padded / position_ids
 * Joins the neat-packing map of [packed_seq] (1-based document index per
 *   token, 0 = padding) to the pack-length format of [thd_utils]
 *   process_input_for_thd (seq_lens and seq_lens_padded [B, num_packs], -1000
 *   for unused slots).  Readings: within a row, every maximal run of one
 *   non-zero index is a sequence whose real length is the run length; a
 *   padding run that follows a document run belongs to that sequence's
 *   padded length; a padding run at the start of a row is a sequence of real
 *   length 0.  position_ids counts 0, 1, ... within each document run and is
 *   0 on padding.  More sequences in a row than num_packs is ORC_CAPACITY.
 * ---------------------------------------------------------------------- */
int oracle_doc_ids_to_lengths(const void* doc_ids, int elem_bytes, int64_t B,
                              int64_t S, int64_t num_packs, int64_t pad_value,
                              int64_t* seq_lens, int64_t* seq_lens_padded,
                              int64_t* position_ids) {
  for (int64_t i = 0; i < B * num_packs; ++i) {
    seq_lens[i] = pad_value;
    seq_lens_padded[i] = pad_value;
  }
  for (int64_t b = 0; b < B; ++b) {
    int64_t slot = -1; /* the sequence being filled in this row */
    for (int64_t s = 0; s < S; ++s) {
      int64_t t = b * S + s;
      int64_t d = read_int(doc_ids, elem_bytes, t);
      int64_t prev = s > 0 ? read_int(doc_ids, elem_bytes, t - 1) : 0;
      int run_start = (s == 0) || (d != prev);
      if (d != 0) {
        if (run_start) { /* a new document run: a new sequence */
          slot += 1;
          if (slot >= num_packs) return ORC_CAPACITY;
          seq_lens[b * num_packs + slot] = 0;
          seq_lens_padded[b * num_packs + slot] = 0;
          position_ids[t] = 0;
        } else {
          position_ids[t] = position_ids[t - 1] + 1;
        }
        seq_lens[b * num_packs + slot] += 1;
        seq_lens_padded[b * num_packs + slot] += 1;
      } else {
        position_ids[t] = 0;
        if (slot < 0) { /* padding before any document: an empty sequence */
          slot = 0;
          if (slot >= num_packs) return ORC_CAPACITY;
          seq_lens[b * num_packs] = 0;
          seq_lens_padded[b * num_packs] = 0;
        }
        seq_lens_padded[b * num_packs + slot] += 1;
      }
    }
  }
  return ORC_OK;
}
