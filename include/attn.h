/*
 * attn.h -- C ABI of libattn.so: exact tiled attention with an online softmax
 * on NVIDIA GB300 (sm_103a).
 *
 * The operations (definitions from the pages this library implements):
 *
 *   attention of a query row over the keys it may see --
 *     "Why your local LLM feels dumber than it is" (Part 3.14), section
 *     "What attention is trying to calculate": score_t = scale * dot(q, k_t),
 *     weights exp(score_t) normalised over the visible tokens, output the
 *     weighted sum of the values.
 *
 *   tiled prefill with a running max and running sum --
 *     "Streaming process -- How the SM works inside a transformer", Steps 3-8
 *     and its code snippet.
 *
 *   split-KV decode over a paged cache and the merge of per-group partials --
 *     "GPU Datapath: Where Every Byte Moves in One LLM Inference Step",
 *     section D "Paged decode attention -- the zero-reuse stream", and
 *     "Why your local LLM feels dumber than it is", sections "Why the
 *     calculation is split into groups" and "Backend names expand into four
 *     decode algorithms".
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers (CUDA global memory of the current
 *     device), 16-byte aligned, densely packed in the layout stated, except
 *     the host pointers of attn_prefill_host.  bf16 is
 *     IEEE bfloat16 (2 bytes); LSE values are float32 natural logarithms of
 *     the sum of exp(scaled scores).
 *   - `stream` is a cudaStream_t passed as an opaque pointer (NULL = legacy
 *     default stream).  Kernels are enqueued on it and run asynchronously;
 *     outputs are valid once the stream reaches that point.
 *   - The caller owns all memory.  The library allocates nothing on the
 *     device and keeps no per-call state (attn_prefill_host keeps two copy
 *     streams per device; attn_decode_paged_noalloc uses a fixed array inside
 *     the library).  Argument errors are detected on the host before
 *     anything is enqueued and leave the outputs untouched.
 *   - Grouped-query attention: Hq must be a multiple of Hkv; query head h uses
 *     KV head h / (Hq / Hkv).
 *   - Return value: ATTN_OK, or one of the error codes below.  No exception
 *     crosses the ABI.  Errors detected by a kernel while it runs (a wait that
 *     timed out, a block-table entry out of range) are recorded in a device
 *     status word that attn_device_status() reads.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null pointer, bad shape, misalignment, Hq % Hkv != 0 */
  ATTN_ERR_UNSUPPORTED = 2, /* a head dim or option this build has no kernel for */
  ATTN_ERR_WORKSPACE = 3,   /* decode workspace missing or too small */
  ATTN_ERR_CUDA = 4,        /* a CUDA runtime/driver call or kernel launch failed */
  ATTN_ERR_DEVICE = 5       /* a kernel recorded an error (see attn_device_status) */
} attn_status_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* attn_status_string(attn_status_t status);

/*
 * Prefill forward.
 *   q   [B, S, Hq,  d] bf16      k, v [B, S, Hkv, d] bf16
 *   o   [B, S, Hq,  d] bf16 (output)
 *   lse [B, Hq, S]     f32 (output, may be NULL)
 *   d in {64, 128, 256}; B, S >= 1; Hq, Hkv >= 1 with Hq % Hkv == 0.  d = 256
 *   uses 64-key tiles (the rest 128-key tiles).
 *   scale: multiplier of q.k (for example 1/sqrt(d)); finite and > 0, else
 *   ATTN_ERR_INVALID_ARG (the kernels keep the row maximum in unscaled units
 *   and mask keys with -inf before scaling).  The same holds for every entry
 *   point below that takes a scale.
 *   causal != 0: row i sees keys 0..i (itself included); causal == 0: all S keys.
 * Row i of o is sum_j softmax_j(scale * q_i.k_j) v_j over the visible keys;
 * lse[b, h, i] = ln sum_j exp(scale * q_i.k_j).
 * Arithmetic: bf16 inputs, f32 scores and accumulators, the probabilities
 * rounded to bf16 for P.V while the normaliser sums the unrounded f32 values,
 * output rounded to bf16 (nearest even).
 */
attn_status_t attn_prefill(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                           int Hkv, int S, int d, float scale, int causal, void* stream);

/*
 * Prefill forward over packed sequences of different lengths: the varlen
 * attention call that "GPU Datapath: Where Every Byte Moves in One LLM
 * Inference Step", section "Measuring the Real Kernels, One at a Time", says
 * its attention cells dispatch (cumulative sequence offsets, one packed token
 * dimension).
 *   q, o       [total_tokens, Hq,  d] bf16 (o is output)
 *   k, v       [total_tokens, Hkv, d] bf16
 *   cu_seqlens [num_seqs + 1] int32, DEVICE memory: sequence n holds tokens
 *              cu_seqlens[n] .. cu_seqlens[n+1]-1; cu_seqlens[0] = 0,
 *              non-decreasing, cu_seqlens[num_seqs] <= total_tokens.
 *   max_seqlen upper bound of every sequence length (host value; sizes the
 *              work list).
 *   lse        [Hq, total_tokens] f32 (output, may be NULL).
 * Each sequence is attended on its own, exactly as attn_prefill does for one
 * batch element (causal positions counted from the sequence's first token).
 * Rows of o that belong to no sequence are not written.  A zero-length
 * sequence has no rows.  A cu_seqlens entry that breaks the rules above is
 * recorded as device status 5 and that sequence is skipped.
 * d, Hq, Hkv, scale, causal and the arithmetic are as for attn_prefill.
 */
attn_status_t attn_prefill_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                                  const int32_t* cu_seqlens, int num_seqs, int max_seqlen, int total_tokens, int Hq,
                                  int Hkv, int d, float scale, int causal, void* stream);

/*
 * Chunked prefill against the paged KV cache: the new tokens of each
 * sequence attend to all of its cached tokens (their own K/V already
 * appended to the cache) -- the prefill form of the varlen call with a block
 * table that "GPU Datapath: Where Every Byte Moves in One LLM Inference
 * Step", section "Measuring the Real Kernels, One at a Time", dispatches.
 *   q, o         [total_q, Hq, d] bf16: the new tokens of every sequence,
 *                back to back (o is output)
 *   k_cache,
 *   v_cache      [num_blocks, page_size, Hkv, d] bf16, as for
 *                attn_decode_paged
 *   block_table  [num_seqs, max_blocks_per_seq] int32, DEVICE memory
 *   cu_seqlens_q [num_seqs + 1] int32, DEVICE memory: sequence n's new
 *                tokens are q rows cu_seqlens_q[n] .. cu_seqlens_q[n+1]-1
 *   seq_lens     [num_seqs] int32, DEVICE memory: cached tokens of sequence
 *                n, its new tokens included (they are the last ones)
 *   lse          [Hq, total_q] f32 (output, may be NULL)
 *   max_seqlen_q upper bound of the new tokens per sequence (host value)
 *   d in {64, 128, 256}; page_size == 16.
 * New token i of sequence n sits at position seq_lens[n] - q_len + i; with
 * causal != 0 it sees the keys at positions 0 .. that position, otherwise all
 * seq_lens[n] keys.  Tokens of the last page past seq_len are never used,
 * even if they hold NaN.  A sequence whose offsets break the rules of
 * attn_prefill_varlen or whose seq_len is below its new tokens or beyond its
 * block-table row is recorded as device status 5 and skipped; a block-table
 * entry outside [0, num_blocks) as status 2 (page 0 is read instead).
 * Arithmetic as for attn_prefill.
 */
attn_status_t attn_prefill_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                                 const int32_t* cu_seqlens_q, const int32_t* seq_lens, void* o, float* lse,
                                 int num_seqs, int max_seqlen_q, int total_q, int Hq, int Hkv, int d, int page_size,
                                 int max_blocks_per_seq, int num_blocks, float scale, int causal, void* stream);

/*
 * Causal (or full) prefill of one sequence whose inputs and outputs are in
 * HOST memory, with the transfers inside the call.  The attention is that of
 * attn_prefill with B = 1 ("Why your local LLM feels dumber than it is" (Part
 * 3.14), section "What attention is trying to calculate"); the queries are
 * cut into `chunks` runs of ceil(S / chunks) rows.  Row i only sees keys
 * 0 .. i, so a chunk needs only the keys up to its own last row: each chunk
 * runs as one chunked prefill (attn_prefill_paged, the keys and values seen
 * as a paged cache with an identity block table) as soon as its rows are
 * on the device, while the next chunk is copied in and the previous one
 * copied out.  With causal == 0 every row sees all S keys: all of k and v
 * are copied in before the first chunk, and only the queries and outputs
 * are pipelined.
 *   q_host        [S, Hq, d] bf16, host memory
 *   k_host,
 *   v_host        [S, Hkv, d] bf16, host memory
 *   o_host        [S, Hq, d] bf16, host memory (output)
 *   lse_host      [Hq, S] f32, host memory (output, may be NULL)
 *   chunks        1 .. 64
 *   workspace     DEVICE memory, 256-byte aligned, of at least
 *                 attn_prefill_host_workspace_bytes(S, Hq, Hkv, d, chunks)
 *                 bytes: the device copies of q, k, v, o and LSE, the
 *                 block table and the chunks' offsets.  It must not be in use
 *                 by other work until the call's work on `stream` is done.
 * Host buffers should be page-locked (cudaHostAlloc or cudaHostRegister): the
 * copies then run asynchronously and overlap.  Pageable memory gives the
 * same results, but its copies stop the calling thread and do not overlap.
 * The chunks' prefills run on `stream`; the copies run on two streams the
 * library creates once per device (with four events) and keeps for the life
 * of the process: the only state the library keeps between calls.  The copies
 * start after the work enqueued on `stream` before the call, and work
 * enqueued on `stream` after the call starts after the last copy out, so the
 * host outputs are complete once `stream` reaches that point (for example
 * after cudaStreamSynchronize(stream)).  Enqueueing is serialised across host
 * threads.
 * Errors: argument errors (d, Hq, Hkv, S, chunks, scale, NULL pointers, an
 * unaligned or too small workspace) return before anything is enqueued; a
 * CUDA error while enqueueing returns ATTN_ERR_CUDA with part of the work
 * enqueued and the outputs undefined.
 * Arithmetic as for attn_prefill; every output equals that of attn_prefill on
 * the same sequence.
 */
attn_status_t attn_prefill_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                                float* lse_host, int S, int Hq, int Hkv, int d, float scale, int causal, int chunks,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes attn_prefill_host needs; 0 for invalid arguments. */
size_t attn_prefill_host_workspace_bytes(int S, int Hq, int Hkv, int d, int chunks);

/*
 * Number of partial slots per (sequence, query head) that attn_decode_paged
 * uses for the given split settings (1 means the split kernel writes the
 * output directly and needs no workspace).
 *   split_tokens > 0: groups of split_tokens tokens (must be a multiple of
 *     page_size); slots = ceil(max_blocks_per_seq * page_size / split_tokens).
 *   split_tokens == 0: num_splits (>= 1) groups per sequence.
 * Returns 0 for invalid arguments.
 */
int attn_decode_num_slots(int max_blocks_per_seq, int page_size, int num_splits, int split_tokens);

/*
 * Split-count rule of "Why your local LLM feels dumber than it is" (Part
 * 3.14), section "Why FlashAttention 2 selects 54, 62, or 87 groups": among
 * c = 1 .. min(max_splits, capacity, blocks), a count is a candidate when it
 * changes ceil(blocks / c) compared with c - 1 (c = 1 always is); its
 * estimated efficiency is w / ceil(w) with w = units * c / capacity; the
 * smallest candidate whose efficiency is at least 85% of the best one wins.
 *   units      independent work items per split (sequences x KV heads)
 *   capacity   work items the device runs at once
 *   blocks     key/value blocks of the longest sequence
 * Pure host arithmetic (no CUDA call).  With units = 4, capacity = 2 x SMs and
 * blocks = 431 it gives the page's 54 / 62 / 87 for 132 / 148 / 188 SMs.
 * Returns 0 for invalid arguments.
 */
int attn_split_heuristic(int units, int capacity, int blocks, int max_splits);

/*
 * The same rule restated for this library's split kernel on the current
 * device: units = num_seqs * Hkv, capacity = SMs x resident split-kernel CTAs
 * per SM, blocks = max_blocks_per_seq (16-token pages), at most 128 splits.
 * Pass the result as num_splits to attn_decode_paged (and to
 * attn_decode_num_slots for the workspace size).  Returns 0 for invalid
 * arguments or when no CUDA device can be queried.
 */
int attn_decode_auto_splits(int num_seqs, int Hkv, int d, int max_blocks_per_seq);

/*
 * Length-aware group size for attn_decode_paged (pass the result as
 * split_tokens).  The rule of "Why your local LLM feels dumber than it is"
 * (Part 3.14), section "Why FlashAttention 2 selects 54, 62, or 87 groups",
 * sizes every sequence's groups from the longest one; with mixed lengths that
 * leaves long groups on the long sequences and short ones on the rest.  This
 * rule instead gives every group the same number of pages s, so a sequence's
 * group count is proportional to its length (ceil(pages_n / s)):
 *   items(s) = Hkv * sum_n ceil(pages_n / s) groups, capacity = CTAs the
 *   device runs at once;
 *   one wave: s1 is the smallest page count with items(s1) <= capacity, but
 *   at least 32 pages (512 tokens) or the longest sequence's page count if
 *   that is smaller; it is taken when such a count exists and its groups are
 *   near-equal, i.e. 4 * s1 * capacity <= 5 * (total pages * Hkv), or s1 is
 *   that lower bound;
 *   otherwise (several waves): s is the largest power of two that is at most
 *   max(32, total pages * Hkv / (3 * capacity)), capped by the longest
 *   sequence (about three waves of equal groups).
 *   seq_lens   host array [num_seqs] of the lengths the decode will see
 *              (entries are clamped to [0, max_blocks_per_seq * 16]).
 * Returns s * 16 (a multiple of page_size = 16), or 0 for invalid arguments.
 * attn_split_tokens_rule is the pure host arithmetic with an explicit
 * capacity; attn_decode_auto_split_tokens applies it on the current device
 * (capacity = SMs x resident split-kernel CTAs per SM) and also returns 0 when
 * no CUDA device can be queried.
 */
int attn_split_tokens_rule(const int32_t* seq_lens, int num_seqs, int Hkv, int capacity, int max_blocks_per_seq);
int attn_decode_auto_split_tokens(const int32_t* seq_lens, int num_seqs, int Hkv, int d, int max_blocks_per_seq);

/*
 * Bytes of workspace attn_decode_paged needs: num_seqs * Hq * slots * (d + 2)
 * floats when slots > 1, else 0.
 */
size_t attn_decode_workspace_bytes(int num_seqs, int Hq, int d, int slots);

/*
 * Bytes of workspace attn_decode_paged needs in balanced mode (num_splits == 0
 * and split_tokens == 0) on the current device:
 * (worker warps + Hkv * num_seqs) * (Hq / Hkv) * (d + 2) floats, where the
 * number of worker warps follows the device's SM count.  Returns 0 for
 * invalid arguments or when no CUDA device can be queried.
 */
size_t attn_decode_balanced_workspace_bytes(int num_seqs, int Hq, int Hkv, int d);

/*
 * Single-token decode over a paged KV cache, split over the context.
 *   q            [num_seqs, Hq, d] bf16
 *   k_cache,
 *   v_cache      [num_blocks, page_size, Hkv, d] bf16: physical pages of
 *                page_size consecutive token rows
 *   block_table  [num_seqs, max_blocks_per_seq] int32: physical page of each
 *                logical page (entries past a sequence's last page are ignored)
 *   seq_lens     [num_seqs] int32, 0 <= len <= max_blocks_per_seq * page_size
 *   o            [num_seqs, Hq, d] bf16 (output)
 *   lse          [num_seqs, Hq] f32 (output, may be NULL)
 *   d in {128, 256}; page_size == 16.
 *   Splits: contiguous, page-aligned groups of tokens -- split_tokens per
 *   group if split_tokens > 0, else ceil(pages / num_splits) pages per group.
 *   Each group gives a partial (normalised f32 output, max, sum); when there
 *   is more than one slot the partials go to `workspace` and a second kernel
 *   merges them (same arithmetic as attn_combine).
 *   workspace: device buffer of at least attn_decode_workspace_bytes(...)
 *   bytes (may be NULL when that is 0).
 *   Balanced mode (num_splits == 0 and split_tokens == 0): the pages of all
 *   sequences and KV heads form one list, and every worker warp of a grid
 *   sized to the device takes an equal contiguous share of it, whatever the
 *   mix of lengths; each share yields one partial per (sequence, KV head) it
 *   touches and a second kernel merges them.  Needs
 *   attn_decode_balanced_workspace_bytes(...) bytes of workspace.
 * The query sees all seq_len tokens.  A sequence with seq_len == 0 gets o = 0
 * and lse = -inf.  Tokens of the last page past seq_len are never used, even
 * if they hold NaN.  A block-table entry outside [0, num_blocks) is recorded
 * as ATTN_ERR_DEVICE (page 0 is read instead).
 */
attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                                const int32_t* seq_lens, void* o, float* lse, int num_seqs, int Hq, int Hkv, int d,
                                int page_size, int max_blocks_per_seq, int num_blocks, int num_splits,
                                int split_tokens, float scale, void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * Paged decode that allocates nothing.  The pages have no counterpart to
 * this entry point: it exists for callers that cannot provide a workspace,
 * such as a plugin inside a host framework that owns all device memory and
 * hands out no scratch buffers, or a serving loop that forbids device
 * allocations once it has started.
 *   Arguments, layouts, results and errors are those of attn_decode_paged
 *   (balanced mode included), without workspace / workspace_bytes: the
 *   partials live in a fixed array of ATTN_DECODE_NOALLOC_SCRATCH_BYTES
 *   inside the library's own device memory, present on every device that
 *   loads the library until the process exits.  No cudaMalloc, cudaFree or
 *   other allocating call is made.  The array is passed to attn_decode_paged
 *   as a workspace of that many bytes, so argument errors are reported first,
 *   and a call whose partials need more (attn_decode_workspace_bytes, or
 *   attn_decode_balanced_workspace_bytes in balanced mode) returns
 *   ATTN_ERR_WORKSPACE and enqueues nothing.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current) and keeps it; make that first call
 *   before any stream capture.  The kept address belongs to the device's
 *   primary context: do not reset the device (cudaDeviceReset) while the
 *   library is in use, nor call it from another context on the same device.
 *   All calls share the array: calls whose work overlaps on the GPU (other
 *   streams, other host threads) race on it.  Every partial a call reads was
 *   written earlier in the same call, so leftovers of earlier calls are
 *   harmless.
 */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
attn_status_t attn_decode_paged_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_table, const int32_t* seq_lens, void* o, float* lse,
                                        int num_seqs, int Hq, int Hkv, int d, int page_size, int max_blocks_per_seq,
                                        int num_blocks, int num_splits, int split_tokens, float scale, void* stream);

/*
 * Merge per-group partials ("Why your local LLM feels dumber than it is",
 * section "Backend names expand into four decode algorithms": normalised
 * group outputs merged by their log-sum statistics).
 *   part_o [rows, num_splits, d] f32: normalised output of each group
 *   part_m [rows, num_splits]    f32: max scaled score of the group (-inf if empty)
 *   part_l [rows, num_splits]    f32: sum of exp(score - part_m) (0 if empty)
 *   rows = num_seqs * Hq.
 *   o   [rows, d] bf16 = sum_i w_i part_o_i / sum_i w_i, w_i = part_l_i exp(part_m_i - M),
 *       M = max over non-empty groups; groups with part_l <= 0 carry no weight.
 *   lse [rows] f32 (may be NULL) = M + ln sum_i w_i.  A row with no
 *       non-empty group gets o = 0 and lse = -inf.
 *   d in {64, 128, 256}.
 */
attn_status_t attn_combine(const float* part_o, const float* part_m, const float* part_l, int rows,
                           int num_splits, int d, void* o, float* lse, void* stream);

/*
 * Decode numerics of other backends ("Why your local LLM feels dumber than it
 * is" (Part 3.14), section "Backend names expand into four decode
 * algorithms").  Each backend splits the context into groups in its own way,
 * stores its own per-group value and merges the groups in its own float32
 * order:
 *   ATTN_NUMERICS_TRITON  `partitions` contiguous groups of whole 16-token
 *       tiles (ceil(pages / partitions) pages each; the page's Triton uses
 *       16); stores the float32 weighted-value sum; merge: c_i = exp(m_i - M),
 *       M = max m_i, L = sum l_i c_i, N = sum n_i c_i, out = N / L.
 *   ATTN_NUMERICS_FA2     `partitions` contiguous groups of whole 64-token
 *       blocks (ceil(blocks / partitions) blocks each); stores the float32
 *       normalised output; merge: lse_i = m_i + log l_i, w_i =
 *       exp(lse_i - max lse), out = sum o_i w_i / sum w_i.
 *   ATTN_NUMERICS_XQA     256-token tiles dealt round-robin over
 *       `partitions` groups (group p takes tiles p, p + partitions, ...); the
 *       sum of weights adds the bf16-rounded weights; stores the normalised
 *       output rounded to bf16; merge: w_i = l_i exp(m_i - M),
 *       out = sum o_i w_i / sum w_i.
 *   ATTN_NUMERICS_TRT     one group per 128-token tile (`partitions` is not
 *       used); stores the weighted-value sum rounded to bf16; merge: the
 *       groups one after another, with a running max M' = max(M, m_i),
 *       L = L exp(M - M') + l_i exp(m_i - M'), and likewise for N;
 *       out = N / L.
 * Inside a group the weights are exp(score - group max), and the
 * weighted-value sum multiplies the values by the bf16-rounded weights.  The
 * merges run in group order, with each float32 add, multiply and divide
 * rounded on its own (no fused multiply-add).  exp and log are evaluated in
 * double precision and rounded once to float32.  The group arithmetic itself
 * runs on tensor cores, whose sums have their own order: the emulation holds
 * the geometry, the stored types and the merge order, not the bits of every
 * partial.
 */
typedef enum {
  ATTN_NUMERICS_TRITON = 1,
  ATTN_NUMERICS_FA2 = 2,
  ATTN_NUMERICS_XQA = 3,
  ATTN_NUMERICS_TRT = 4
} attn_numerics_t;

/*
 * Group count that the backend would pick for a batch of num_seqs sequences
 * with Hkv KV heads, the longest max_tokens long, on a GPU of sm_count SMs
 * (pure host arithmetic):
 *   TRITON  16;
 *   FA2     attn_split_heuristic(num_seqs * Hkv, 2 * sm_count,
 *           ceil(max_tokens / 64), 128), which gives the page's 54 / 62 / 87
 *           for 132 / 148 / 188 SMs at 27,525 tokens and 4 KV heads;
 *   XQA     min(max(1, sm_count / (num_seqs * Hkv)), ceil(max_tokens / 256)):
 *           the page's 33 on H200 (132 SMs) and 47 on SM120 (188 SMs);
 *   TRT     ceil(max_tokens / 128), the number of its 128-token groups.
 * Returns 0 for invalid arguments.
 */
int attn_emulated_partitions(int numerics, int num_seqs, int Hkv, int max_tokens, int sm_count);

/*
 * Partial slots per (sequence, query head): `partitions` (1 .. 65535) for
 * TRITON, FA2 and XQA; ceil(max_blocks_per_seq * page_size / 128) for TRT.
 * Returns 0 for invalid arguments (page_size must be 16).
 */
int attn_emulated_num_slots(int numerics, int max_blocks_per_seq, int page_size, int partitions);

/* Workspace bytes of attn_decode_paged_emulated: num_seqs * Hq * slots * (d + 2) floats. */
size_t attn_emulated_workspace_bytes(int num_seqs, int Hq, int d, int slots);

/*
 * Paged decode with the numerics of another backend.  Arguments, layouts and
 * errors are those of attn_decode_paged, with `numerics` and `partitions` (as
 * above) in place of num_splits / split_tokens.  It always writes partials and
 * merges them, even with one group.  The workspace (at least
 * attn_emulated_workspace_bytes(num_seqs, Hq, d, slots) bytes, 16-byte
 * aligned) holds, after the call:
 *   part_o [num_seqs * Hq, slots, d] f32  the stored value of each group
 *   part_m [num_seqs * Hq, slots]    f32  group max of the scaled scores
 *   part_l [num_seqs * Hq, slots]    f32  group sum of weights
 * in that order.  An empty group has m = -inf, l = 0 and part_o = 0.
 * o [num_seqs, Hq, d] bf16 is the merged output rounded to bf16.  lse (may be
 * NULL) is the merge's largest max (FA2: log-sum) plus log of its merged sum.
 */
attn_status_t attn_decode_paged_emulated(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_table, const int32_t* seq_lens, void* o, float* lse,
                                         int num_seqs, int Hq, int Hkv, int d, int page_size, int max_blocks_per_seq,
                                         int num_blocks, int numerics, int partitions, float scale, void* workspace,
                                         size_t workspace_bytes, void* stream);

/*
 * The backend's merge alone, on caller-supplied partials in the layout above:
 *   part_o [rows, num_splits, d] f32, part_m / part_l [rows, num_splits] f32
 *   (a slot with part_l <= 0 is empty and skipped);
 *   o_f32 [rows, d] f32 (may be NULL): the float32 result before the final rounding;
 *   o     [rows, d] bf16 (may be NULL, not both): that result rounded to bf16;
 *   lse   [rows] f32 (may be NULL).
 * A row with no non-empty slot gets 0 and lse = -inf.  1 <= d <= 1024.
 */
attn_status_t attn_merge_emulated(int numerics, const float* part_o, const float* part_m, const float* part_l,
                                  int rows, int num_splits, int d, float* o_f32, void* o, float* lse, void* stream);

/*
 * Device-side status: waits for all work on the current device, then stores
 * the first error code any kernel of this library recorded since the last
 * clear (0 = none; 1 = a pipeline wait timed out; 2 = block-table entry out of
 * range; 3 = a seq_len the block table cannot cover; 4 = shared memory not
 * 1 KB-aligned; 5 = cu_seqlens decreasing, past total_tokens or longer than
 * max_seqlen, or a seq_len that does not fit its chunk or block table) and, if
 * `clear` != 0, resets it.
 */
attn_status_t attn_device_status(uint32_t* code, int clear);

/* Library version as major * 10000 + minor * 100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
