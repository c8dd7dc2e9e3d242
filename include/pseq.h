/*
 * pseq.h -- C ABI of libpseq.so: packed-sequence metadata on the GPU.
 *
 * Every entry point enqueues work on the caller's CUDA stream and returns at
 * once.  It allocates no device memory: the caller owns every buffer (device
 * pointers, unless a comment says otherwise) and passes scratch space as a
 * `workspace` whose size the matching *_workspace_size() call gives.
 *
 * Errors come back on two channels:
 *   - a non-zero pseq_status from the call itself, for anything the host can
 *     see (NULL pointer, negative or too-large size, misaligned pointer,
 *     workspace too small, a CUDA launch error).  Nothing is enqueued then,
 *     and pseq_last_error() describes the problem;
 *   - info->status, written on the device, for anything that depends on the
 *     data (malformed lengths, a bin over capacity, a wait that gave up).
 *     Read the pseq_info block after the stream has reached the call.
 * Outputs are unspecified when either channel reports an error.
 *
 * Pages the operations come from:
 *   [packed_seq]  NeMo AutoModel API reference,
 *                 "nemo_automodel.components.datasets.packed_seq"
 *   [thd_utils]   NeMo AutoModel v0.5 API reference,
 *                 "nemo_automodel.components.distributed.thd_utils"
 *   [who_packs]   "Who packs the sequences: the loader, or the trainer?"
 *                 (NeMo-RL #4105 explainer page)
 */
#ifndef PSEQ_H
#define PSEQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* pseq_stream;

typedef enum pseq_status {
  PSEQ_OK = 0,
  PSEQ_ERR_ARG = 1,      /* bad pointer, size, alignment or workspace       */
  PSEQ_ERR_OVERFLOW = 2, /* a count that does not fit the int32 outputs     */
  PSEQ_ERR_VALUE = 3,    /* malformed lengths or layout (device-detected)   */
  PSEQ_ERR_CAPACITY = 4, /* a bin's padded total exceeds capacity or width  */
  PSEQ_ERR_TIMEOUT = 5,  /* a bounded device-side wait gave up              */
  PSEQ_ERR_CUDA = 6      /* a CUDA runtime call failed                      */
} pseq_status;

/* Result block written on the device by every entry point (16 bytes). */
typedef struct pseq_info {
  int32_t status;     /* pseq_status of the device-side checks          */
  int32_t count;      /* segments / sequences / members produced        */
  int32_t max_seqlen; /* longest segment or sequence                    */
  int32_t total;      /* tokens in the produced stream (see each call)  */
} pseq_info;

/* Library version (major * 10000 + minor * 100 + patch). */
int pseq_version(void);

/* Text of the last host-side error raised on the calling thread ("" if none). */
const char* pseq_last_error(void);

/* Kernel launches this library has issued in this process, all threads. */
int64_t pseq_launch_count(void);

/* Bounded-wait controls, for failure-detection tests.  spin_limit_ns caps
 * every device-side wait of pseq_from_doc_ids, pseq_doc_ids_to_lengths and
 * the bulk-copy path of thd_from_batch; it is clamped to [0, 1e9] ns (the
 * default, 1 s), so no setting makes a wait unbounded.  When withhold_tile
 * >= 0 that scan tile (or bridge chunk, counted row-major over rows and
 * 4096-token chunks) never publishes its partial result, so the ones after
 * it run into the cap and report PSEQ_ERR_TIMEOUT.  Process-wide; pass
 * (-1, -1) to restore the defaults. */
void pseq_debug_set_wait(int64_t spin_limit_ns, int64_t withhold_tile);

/* The wait cap in force, in nanoseconds (after clamping). */
int64_t pseq_debug_wait_limit_ns(void);

/* ------------------------------------------------------------------------
 * pseq_from_doc_ids
 * [packed_seq] "packed_seq_params_from_doc_ids" and PackedSeqParams.
 * doc_ids: [B, S] row-major integers of id_bytes (4 or 8) each; 1-based
 *   document index per token, 0 = padding (any value is accepted; only
 *   equality with the left neighbour matters).  16-byte alignment is faster.
 * A segment is a maximal run of one index within a row; every row start
 *   begins a segment; padding runs are segments too.
 * cu_seqlens: int32, room for B*S+1 entries.  Receives num_segments+1
 *   boundaries: cu_seqlens[0] = 0, cu_seqlens[num_segments] = B*S.
 * info: count = num_segments, max_seqlen = longest segment (padding runs
 *   included; 0 when B*S == 0), total = B*S.
 * workspace: pseq_from_doc_ids_workspace_size(B, S) bytes or more, 16-byte
 *   aligned, ZERO-FILLED before its first use.  Each call stamps what it
 *   writes there with a number one above the previous call's (kept in the
 *   buffer), so nothing a call leaves behind is read by the next: one buffer
 *   serves any number of calls on one stream, of any map size it has room
 *   for, also after a call that failed.  The call that takes the last
 *   number (one call in 2^32 - 1) zero-fills all workspace_bytes and starts
 *   the numbering again.  Calls that may overlap need separate workspaces.
 * Host errors: PSEQ_ERR_ARG (NULL, negative B or S, id_bytes, alignment,
 *   workspace), PSEQ_ERR_OVERFLOW (B*S > INT32_MAX).
 * Device errors: PSEQ_ERR_TIMEOUT (a tile's wait for its predecessor hit the
 *   cap set by pseq_debug_set_wait); PSEQ_ERR_ARG (a workspace that was not
 *   zero-filled before its first use, where that shows).
 * ---------------------------------------------------------------------- */
size_t pseq_from_doc_ids_workspace_size(int64_t B, int64_t S);
pseq_status pseq_from_doc_ids(const void* doc_ids, int32_t id_bytes, int64_t B,
                              int64_t S, int32_t* cu_seqlens, pseq_info* info,
                              void* workspace, size_t workspace_bytes,
                              pseq_stream stream);

/* ------------------------------------------------------------------------
 * pseq_from_doc_ids_static -- pseq_from_doc_ids without a workspace
 * The pages have no counterpart to this entry point; it is an integration
 * variant of the call above.
 * Some callers cannot allocate device memory when they call in: code running
 * under a memory-pool policy that forbids new allocations, a plugin or
 * callback that is handed only input and output pointers, or a process that
 * has reserved all of HBM up front.  This entry point takes the same inputs
 * and outputs as pseq_from_doc_ids and no workspace.  Its scratch is a
 * static device array of about 32 KiB inside libpseq.so (a 128-byte header
 * and 32 bytes per 16384-token tile), which every GPU that loads the library
 * holds until the process exits.
 *  - B*S must not exceed PSEQ_STATIC_MAX_TOKENS; larger maps get
 *    PSEQ_ERR_ARG before anything is enqueued (use pseq_from_doc_ids).
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - Every call clears the part of the array that must start at zero
 *    (cudaMemsetAsync on the caller's stream) and then runs the scan.  All
 *    calls share the one array, so any two calls whose work may overlap on
 *    the GPU race, whatever issued them (other streams, other host threads):
 *    the caller must serialise them.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * Outputs and errors are those of pseq_from_doc_ids.
 * ---------------------------------------------------------------------- */
#define PSEQ_STATIC_MAX_TOKENS (1LL << 24)
pseq_status pseq_from_doc_ids_static(const void* doc_ids, int32_t id_bytes,
                                     int64_t B, int64_t S,
                                     int32_t* cu_seqlens, pseq_info* info,
                                     pseq_stream stream);

/* ------------------------------------------------------------------------
 * BSHD -> THD conversion
 * [thd_utils] "process_input_for_thd" (description, Example, Parameters,
 * Returns) and "_thd_padding_mask".
 *
 * seq_lens, seq_lens_padded: int64 [B, num_packs], 8-byte aligned.  Entries
 *   equal to pad_value (-1000 on the page) are dropped from both; the rest
 *   are the kept sequences in row-major order.  seq_lens_padded may be NULL
 *   (padded := real).
 * Kept sequence i of row b occupies the source slots [o_i, o_i + padded_i)
 *   of that row, o_i being the sum of the padded lengths of the kept entries
 *   before it in the row.  The stream length is T = sum of padded lengths.
 * cu_seqlens: int32 [n+1] = [0] + cumsum(real); when absorb_trailing_pad is
 *   set, n >= 1 and every sequence but the last has real == padded, the
 *   last entry becomes T (the trailing pad is absorbed).  Room: B*num_packs+1.
 * cu_seqlens_padded: int32 [n+1] = [0] + cumsum(padded).  May be NULL.
 * pad_between_seqs: one byte, 1 when the complete cu_seqlens and
 *   cu_seqlens_padded arrays differ after absorption (0 when
 *   seq_lens_padded is NULL).  May be NULL.
 * info: count = n, max_seqlen = max(cu_seqlens[i+1] - cu_seqlens[i]) after
 *   absorption (0 when n == 0), total = T.
 * Device errors: PSEQ_ERR_VALUE when one array holds pad_value where the
 *   other does not, a kept length is negative, padded < real, or a row's
 *   padded lengths exceed S.
 * ---------------------------------------------------------------------- */

/* One tensor to move into the THD stream.
 * src: [planes, B, S, row_elems], dst: [planes, T, row_elems], elements of
 * elem_bytes (1, 2, 4 or 8) copied bit for bit.  input_ids / labels [B,S]:
 * planes 1, row_elems 1; position_ids [B,S] or mRoPE [n_rope,B,S]: planes 1
 * or n_rope; embeddings [B,S,H]: planes 1, row_elems H.  dst needs room for
 * planes * B * S * row_elems elements (T <= B*S); the dst plane stride is T
 * rows, so read T back from info before using a multi-plane dst. */
typedef struct pseq_field {
  const void* src;
  void* dst;
  int32_t elem_bytes;
  int32_t planes;
  int64_t row_elems;
} pseq_field;

#define PSEQ_MAX_FIELDS 8

size_t thd_workspace_size(int64_t B, int64_t num_packs);

/* The whole conversion: the work of thd_meta followed by thd_gather (one
 * launch when B*num_packs <= 2048).  fields may be NULL when num_fields == 0;
 * padding_mask (one byte per stream slot, 1 = padding; room for B*S) may be
 * NULL. */
pseq_status thd_from_batch(const int64_t* seq_lens,
                           const int64_t* seq_lens_padded, int64_t B,
                           int64_t S, int64_t num_packs, int64_t pad_value,
                           int32_t absorb_trailing_pad,
                           const pseq_field* fields, int32_t num_fields,
                           int32_t* cu_seqlens, int32_t* cu_seqlens_padded,
                           uint8_t* padding_mask, uint8_t* pad_between_seqs,
                           pseq_info* info, void* workspace,
                           size_t workspace_bytes, pseq_stream stream);

/* First half: filtering, cumulative sums, absorption and flags.  Leaves the
 * per-sequence layout in the workspace for thd_gather. */
pseq_status thd_meta(const int64_t* seq_lens, const int64_t* seq_lens_padded,
                     int64_t B, int64_t S, int64_t num_packs,
                     int64_t pad_value, int32_t absorb_trailing_pad,
                     int32_t* cu_seqlens, int32_t* cu_seqlens_padded,
                     uint8_t* pad_between_seqs, pseq_info* info,
                     void* workspace, size_t workspace_bytes,
                     pseq_stream stream);

/* Second half: moves every field into the stream and writes the padding
 * mask, from the layout a preceding thd_meta (same B, S, num_packs, same
 * workspace, same stream) left in the workspace.  Does nothing when that
 * thd_meta reported a device error. */
pseq_status thd_gather(const pseq_field* fields, int32_t num_fields,
                       int64_t B, int64_t S, int64_t num_packs,
                       uint8_t* padding_mask, const void* workspace,
                       size_t workspace_bytes, pseq_stream stream);

/* ------------------------------------------------------------------------
 * thd_chunks_from_batch -- split_batch_into_thd_chunks
 * [thd_utils] "split_batch_into_thd_chunks": the batch is split along its
 * rows into num_chunks equal chunks, each chunk is converted as by
 * thd_from_batch, and the results are stacked; cu_seqlens arrays of
 * different lengths are padded with pad_value.
 * num_chunks must divide B; chunk c covers rows [c*B/num_chunks,
 *   (c+1)*B/num_chunks).
 * cu_seqlens, cu_seqlens_padded: int32 [num_chunks, B/num_chunks*num_packs+1];
 *   row c holds the chunk's n_c+1 boundaries followed by pad_value.
 *   cu_seqlens_padded may be NULL.
 * fields: as for thd_from_batch (src rows are rows of the whole batch).  With
 *   Sc = (B / num_chunks) * S, the stream of chunk c starts c * planes * Sc
 *   rows into dst and is [planes, T_c, row_elems] (planes T_c rows apart):
 *   every chunk's stream is defined whatever the other chunks' lengths, and
 *   dst viewed as [num_chunks, planes * Sc, row_elems] holds them at a fixed
 *   stride.  dst room: planes * B * S * row_elems elements.
 * padding_mask: chunk c's T_c bytes start at byte c * Sc (room B*S); may be
 *   NULL.  pad_between_seqs: num_chunks bytes; may be NULL.
 * infos: pseq_info [num_chunks], one per chunk (count n_c, max_seqlen,
 *   total T_c).  Stacking the chunks into one tensor, as the page does, needs
 *   every T_c equal; compare infos[c].total.
 * workspace: thd_workspace_size(B / num_chunks, num_packs) bytes.
 * ---------------------------------------------------------------------- */
pseq_status thd_chunks_from_batch(const int64_t* seq_lens,
                                  const int64_t* seq_lens_padded, int64_t B,
                                  int64_t S, int64_t num_packs,
                                  int64_t num_chunks, int64_t pad_value,
                                  int32_t absorb_trailing_pad,
                                  const pseq_field* fields, int32_t num_fields,
                                  int32_t* cu_seqlens,
                                  int32_t* cu_seqlens_padded,
                                  uint8_t* padding_mask,
                                  uint8_t* pad_between_seqs, pseq_info* infos,
                                  void* workspace, size_t workspace_bytes,
                                  pseq_stream stream);

/* ------------------------------------------------------------------------
 * thd_mask_from_token_ids -- thd_padding_mask_from_token_ids
 * [thd_utils] "thd_padding_mask_from_token_ids": mask[t] = 1 where
 *   input_ids[t] == padding_token_id.  That comparison marks padding
 *   correctly only if the pad positions form a suffix of the stream, so a pad
 *   token followed by any other token is PSEQ_ERR_VALUE (the page raises
 *   ValueError).
 * input_ids: n integers of id_bytes (4 or 8).  mask: n bytes.
 * info: count = number of pad tokens, total = n.
 * workspace: thd_mask_from_token_ids_workspace_size(n) bytes, ZERO-FILLED
 *   before its first use; every completed call leaves its counter at zero.
 *   Do not share it with pseq_from_doc_ids.
 * ---------------------------------------------------------------------- */
size_t thd_mask_from_token_ids_workspace_size(int64_t n);
pseq_status thd_mask_from_token_ids(const void* input_ids, int32_t id_bytes,
                                    int64_t n, int64_t padding_token_id,
                                    uint8_t* mask, pseq_info* info,
                                    void* workspace, size_t workspace_bytes,
                                    pseq_stream stream);

/* ------------------------------------------------------------------------
 * pack_ffd -- first-fit-decreasing bins for pack_squeeze
 * [who_packs] get_packer: the step that groups rows into bins under a token
 *   budget; First Fit Decreasing is one of the packers the page names.  Item i has
 *   size lens[i] rounded up to `multiple`; items are visited largest first
 *   (ties: smaller index first) and each goes into the first open bin with
 *   room; a new bin opens when none has room.
 * lens: int64 [n], n <= 8192.  bin_offsets: int32 [n+1] room (num_bins+1
 *   written); bin_members: int32 [n], each bin's items in placement order --
 *   the CSR input of pack_squeeze.
 * info: count = num_bins, max_seqlen = fullest bin's load, total = sum of
 *   the rounded sizes.
 * Device errors: PSEQ_ERR_VALUE for a negative length, PSEQ_ERR_CAPACITY
 *   for an item larger than capacity.
 * ---------------------------------------------------------------------- */
pseq_status pack_ffd(const int64_t* lens, int64_t n, int64_t multiple,
                     int64_t capacity, int32_t* bin_offsets,
                     int32_t* bin_members, pseq_info* info, pseq_stream stream);

/* ------------------------------------------------------------------------
 * pseq_doc_ids_to_lengths -- from the doc_ids map to pack lengths
 * Joins [packed_seq]'s document map (1-based index per token, 0 = padding)
 * to [thd_utils]' seq_lens / seq_lens_padded [B, num_packs] format (unused
 * slots = pad_value).  Within a row, every maximal run of one non-zero index
 * is a sequence (real length = run length); a padding run after a document
 * run belongs to that sequence's padded length; a padding run at the start
 * of a row is a sequence of real length 0.  position_ids [B, S] (int64, may
 * be NULL) counts 0, 1, ... inside each document run and is 0 on padding.
 * info: count = most sequences in one row, max_seqlen = longest document
 *   run, total = sequences in all rows.
 * Device errors: PSEQ_ERR_CAPACITY when a row holds more than num_packs
 *   sequences (the slots that fit are written).
 * workspace: pseq_doc_ids_to_lengths_workspace_size(B, S) bytes, 16-byte
 *   aligned, ZERO-FILLED before its first use; every call leaves it zero
 *   again (calls sharing one must be ordered).  At most 65535 rows per call.
 * Host errors: PSEQ_ERR_OVERFLOW when B*S or B*num_packs exceeds INT32_MAX
 *   or S exceeds 2^31 - 1 - 4096.
 * Device errors also include PSEQ_ERR_TIMEOUT (a chunk's wait for the chunks
 *   before it in its row, or for the row's last chunk before filling its
 *   share of the unused slots, hit the cap set by pseq_debug_set_wait).
 * ---------------------------------------------------------------------- */
size_t pseq_doc_ids_to_lengths_workspace_size(int64_t B, int64_t S);
pseq_status pseq_doc_ids_to_lengths(const void* doc_ids, int32_t id_bytes,
                                    int64_t B, int64_t S, int64_t num_packs,
                                    int64_t pad_value, int64_t* seq_lens,
                                    int64_t* seq_lens_padded,
                                    int64_t* position_ids, pseq_info* info,
                                    void* workspace, size_t workspace_bytes,
                                    pseq_stream stream);

/* ------------------------------------------------------------------------
 * thd_padding_mask
 * [thd_utils] "_thd_padding_mask": sequence i occupies
 *   [start_i, start_i + padded_i), only its first real_i slots hold tokens;
 *   every other slot of the stream is padding.
 * valid_seq_lens, valid_seq_lens_padded: int64 [n] (already filtered);
 *   valid_seq_lens_padded may be NULL (padded := real).
 * mask: total_tokens bytes, 1 = padding.
 * info: count = n, max_seqlen = largest real length, total = total_tokens.
 * workspace: thd_workspace_size(1, n) bytes, 16-byte aligned.
 * Device errors: PSEQ_ERR_VALUE for a negative length, padded < real, or a
 *   layout longer than total_tokens.
 * ---------------------------------------------------------------------- */
pseq_status thd_padding_mask(int64_t total_tokens,
                             const int64_t* valid_seq_lens,
                             const int64_t* valid_seq_lens_padded, int64_t n,
                             uint8_t* mask, pseq_info* info, void* workspace,
                             size_t workspace_bytes, pseq_stream stream);

/* ------------------------------------------------------------------------
 * pack_squeeze -- the trainer-side squeeze
 * [who_packs] sections "Trainer packs" and "Loader packs", and the note
 * that cu_seqlens_padded ends at the pack capacity.
 *
 * src: [N, W] rectangle of elem_bytes (1, 2, 4 or 8) elements; source i
 *   holds real_lens[i] (int64 [N]) tokens at the start of its row.
 * Bins, in CSR form: bin_offsets int32 [num_bins+1] (bin_offsets[0] = 0,
 *   bin_offsets[num_bins] = num_members), bin_members int32 [num_members];
 *   members keep the given order.
 * Each source is padded to a multiple of `multiple`; a bin's sources are
 *   laid end to end: member k of bin b starts at slot cu_seqlens_padded of
 *   its bin.  Only the real tokens are copied; every other slot of out
 *   [num_bins, width] gets the low elem_bytes of pad_value, and padding_mask
 *   [num_bins, width] (1 = padding) marks it.
 * cu_seqlens / cu_seqlens_padded: int32, num_members + num_bins entries;
 *   bin b's (members + 1) entries start at bin_offsets[b] + b.  cu_seqlens
 *   is [0] + cumsum(real), cu_seqlens_padded is [0] + cumsum(padded); with
 *   stretch_to_capacity its last entry per bin is `capacity` (needs width >=
 *   capacity).
 * out and padding_mask may both be NULL: only the metadata is produced and
 *   width is not checked (size a trainer-style row from info.total).
 * info: count = num_members, max_seqlen = largest real length, total = the
 *   largest padded total over bins before stretching.
 * workspace: pack_squeeze_workspace_size(num_members, num_bins) bytes,
 *   16-byte aligned, zero-filled before the first call; every call leaves it
 *   zero again (a counter of finished bins wraps back to 0).  Calls that
 *   share a workspace must be ordered (one stream).
 * Host errors: PSEQ_ERR_OVERFLOW when a size exceeds the int32 range or
 *   width exceeds 2^31 - 2^16; PSEQ_ERR_ARG for more than 65535 bins.
 * Device errors: PSEQ_ERR_CAPACITY when a bin's padded total exceeds
 *   capacity (or width, when out is given); PSEQ_ERR_VALUE for an empty bin,
 *   non-monotone offsets, a member outside [0, N) or a length outside [0, W].
 * ---------------------------------------------------------------------- */
size_t pack_squeeze_workspace_size(int64_t num_members, int64_t num_bins);
pseq_status pack_squeeze(const void* src, int64_t N, int64_t W,
                         int32_t elem_bytes, const int64_t* real_lens,
                         const int32_t* bin_offsets,
                         const int32_t* bin_members, int64_t num_bins,
                         int64_t num_members, int64_t multiple,
                         int64_t capacity, int32_t stretch_to_capacity,
                         int64_t width, int64_t pad_value, void* out,
                         int32_t* cu_seqlens, int32_t* cu_seqlens_padded,
                         uint8_t* padding_mask, pseq_info* info,
                         void* workspace, size_t workspace_bytes,
                         pseq_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* PSEQ_H */
