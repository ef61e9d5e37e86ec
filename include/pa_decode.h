/*
 * pa_decode.h -- C ABI of the GB300 (sm_103a) paged-attention decode library.
 *
 * One decode call: every sequence b contributes one query token per query
 * head h, which attends over the first seq_lens[b] tokens of its K/V, stored
 * in a paged pool and found through the block table:
 *
 *     out[b, h, :] = softmax(scale * q[b, h, :] . K_b^T) V_b
 *     token t of sequence b: physical block block_tables[b][t / block_size],
 *                            slot t % block_size
 *     query head h reads kv head  h / (num_heads / num_kv_heads)
 *
 * Method (split-KV, "V2"): the tokens of a sequence are cut into partitions;
 * one CTA per (partition, kv head, sequence) loads each K/V block of its
 * partition once for all query heads of the GQA group and produces the
 * online-softmax partial (max score, exp sum, weighted V); a second kernel
 * merges the partials of each (sequence, head) by a log-sum-exp reduce.
 * Sources: "docs" commit page (GQA-aware grid on kv heads; Phase 1 partition
 * kernel, Phase 2 reduce kernel; the compound partial), the
 * "paged_attention_v2_triton.py" commit page (alpha/beta online-softmax
 * update), the "qwen3_6_scripts/paged_attn.py" commit page (decode dispatch
 * between a single-pass and a partitioned kernel by sequence length;
 * allocate-once buffer reuse).
 *
 * Layouts (all row-major, contiguous):
 *   q, out         fp16 [num_seqs][num_heads][head_dim]
 *   k_cache,
 *   v_cache        fp16 [num_blocks][num_kv_heads][block_size][head_dim]
 *                  (one (block, kv head) is block_size*head_dim contiguous
 *                  halves; the pages do not print a layout, this is the
 *                  library's choice)
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]; entries past
 *                  ceil(seq_lens[b] / block_size) are never read
 *   seq_lens       int32 [num_seqs]
 * Every pointer argument named above is a DEVICE pointer; out, q, k_cache and
 * v_cache must be 16-byte aligned, block_tables and seq_lens 4-byte aligned.
 *
 * Supported: head_dim in {64, 128, 256}; block_size 16; num_heads a multiple
 * of num_kv_heads with a GQA ratio of 1..8.  Other shapes return
 * PA_ERR_UNSUPPORTED.
 *
 * Ownership: the caller owns every buffer it passes and orders it with
 * `stream`; the library never frees caller memory.  Calls are asynchronous on
 * `stream` (a cudaStream_t; NULL is the legacy default stream).
 *
 * Errors: functions return PA_OK (0) or a negative pa_status; nothing is
 * printed and nothing aborts.  Problems only the device can see (a block id
 * outside [0, num_blocks), a sequence length above max_seq_len or above
 * max_blocks_per_seq * block_size, a wait that gave up) set bits of a
 * per-device status word read by pa_get_device_status(); the affected outputs
 * are then unspecified, and no kernel traps.
 */
#ifndef PA_DECODE_H
#define PA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pa_stream_t; /* same type as cudaStream_t */

/* Return codes. */
enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1,  /* null or misaligned pointer, bad size, non-finite scale, ... */
    PA_ERR_UNSUPPORTED = -2,  /* head_dim, block_size, GQA ratio or CTA shape not compiled in */
    PA_ERR_CUDA = -3,         /* a CUDA runtime call or a kernel launch failed */
    PA_ERR_OOM = -4,          /* the library-owned workspace could not be allocated */
    PA_ERR_WORKSPACE = -5     /* caller workspace too small or not 256-byte aligned */
};

/* Bits of the device status word (pa_get_device_status). */
enum {
    PA_DEV_BAD_BLOCK_ID = 1,  /* a block id read from block_tables was outside [0, num_blocks) */
    PA_DEV_BAD_SEQ_LEN = 2,   /* seq_lens[b] < 0, > max_seq_len or > max_blocks_per_seq*block_size */
    PA_DEV_TIMEOUT = 4        /* a shared-memory copy wait gave up (bounded wait, see opts.wait_limit) */
};

/* Execution modes. */
enum {
    PA_MODE_AUTO = 0,   /* library picks SINGLE or SPLIT from the sizes (see pa_decode_plan) */
    PA_MODE_SINGLE = 1, /* one CTA per (kv head, sequence) covers the whole sequence; no reduce */
    PA_MODE_SPLIT = 2,  /* partitions of partition_size tokens + log-sum-exp reduce kernel */
    PA_MODE_FUSED = 3,  /* partitions as SPLIT, one launch: the last CTA of each (sequence, kv head)
                           to finish (an atomic ticket; nobody waits) merges the partials in
                           partition order ("docs" commit page, the cross-partition level of the
                           reduction hierarchy).  When the device holds the whole grid at once
                           (plan.coop) the grid is launched cooperatively: the CTAs of each
                           (sequence, kv head) meet at a bounded group barrier and each merges
                           its own slice of the outputs; otherwise the last CTA to finish merges
                           (an atomic ticket; nobody waits).  For one sequence FUSED takes
                           the one-wave plan (pooled as for SPLIT).  The
                           workspace also holds two 4-byte words per (sequence, kv head) (the
                           ticket or arrivals, and the departures), after the partials and a
                           slot of 8 bytes per (sequence, kv head) for the pooled claim
                           counters, so a pooled SPLIT call of the same shape on the same
                           workspace leaves them alone.  The words must be zero before the first
                           FUSED call on a workspace, and again after the workspace served a
                           call of another shape or a PERSISTENT or FLAT call (whose tables may
                           cover that slot): zero plan.workspace_bytes, e.g. with
                           cudaMemsetAsync.  Every FUSED call leaves them zero, also after a
                           device error */
    PA_MODE_PERSISTENT = 4, /* a fixed grid of (SMs x CTAs per SM) takes the items of a work list
                              that a small kernel builds on the device from a device counter,
                              longest partitions first.  Each sequence gets its own partition size:
                              with partition_size 0 the grid's partitions per kv head are
                              apportioned over the batch with the smallest cap on a partition's
                              blocks that lets them fit (one wave when the sequences are fewer than
                              those partitions), else the fewest partitions of at most
                              partition_size tokens; either way evened out to whole blocks; then the
                              log-sum-exp reduce.  The host never reads the lengths, so the call is
                              graph-safe.  The workspace also holds the work list, the counter,
                              the order and the sizes (rewritten by every call) */
    PA_MODE_FLAT = 5    /* one wave of 256 / head_dim CTAs per SM (one at head_dim 256, so that
                           about 128 KB of copies are in flight per SM), that many times num_SMs /
                           num_kv_heads CTAs per kv head:
                           every CTA reads the lengths on the device and streams an equal share
                           (to within one block) of the batch's concatenated blocks, one partial
                           per sequence its share meets, then the log-sum-exp reduce; no ragged
                           tail of short and long CTAs, whatever the lengths.  At most 256
                           sequences (else PA_ERR_UNSUPPORTED).  The workspace also holds each
                           sequence's partial count (rewritten by every call).  A refinement of
                           the "docs" commit page's partitions: a partition is a CTA's share of
                           one sequence, and the partials and their merge are unchanged */
};

/* Option flags. */
enum {
    PA_FLAG_FORCE_TIMEOUT = 1,   /* test hook: every copy wait gives up before its first poll; the
                                    kernel then drains its copies, sets PA_DEV_TIMEOUT and returns */
    PA_FLAG_PREFIX_WARP_MMA = 2, /* pa_prefix_ex: use the warp-level MMA kernel instead of the
                                    tcgen05 (tensor-memory) one */
    PA_FLAG_POOLED = 4,          /* SPLIT: the partition CTAs of a (sequence, kv head) share its
                                    blocks in chunks of max(2, stages) blocks: each warp takes three
                                    chunks round-robin, then claims the next from a device counter,
                                    so CTAs on faster SMs take more and all finish together.  Same
                                    partials and reduce as SPLIT, but which blocks a partial covers
                                    depends on timing, so results may differ between calls in the
                                    last bits.  Applies when the plan is SPLIT with partition_size
                                    >= warps * 16 * max(2, stages) tokens (plan.pooled).  The
                                    workspace also holds one 8-byte counter per (sequence, kv head)
                                    right after the partials; it needs no initialisation: a counter
                                    whose high word is not the tag the reduce kernel writes there
                                    keeps the round-robin, and the reduce leaves every counter
                                    tagged with a zero count (a call whose reduce launch fails
                                    resets them to zero instead).  Stale bytes left by other calls
                                    are therefore tolerated: this library's partials (bounded by
                                    the fp16 inputs), tickets and work lists never hold the tag.
                                    The planner's one-wave plan for one sequence is pooled without
                                    this flag from 2048-token partitions on.  Source of the split it
                                    refines: "docs" commit page, GQA-aware grid and partition
                                    paragraphs */
    PA_FLAG_DETERMINISTIC = 8,   /* never pool (not even the one-wave plan): each partial covers
                                    fixed blocks, so repeated calls give identical bits */
    PA_FLAG_UNIFORM_LENGTHS = 16, /* AUTO/SPLIT/FUSED without a partition size or CTA shape: the
                                    caller states that the batch's sequences are all about
                                    max_seq_len long.  The planner then gives the batch the
                                    one-wave decomposition it gives a single sequence: 256 /
                                    head_dim 4-warp CTAs per SM (one at head_dim 256), floor(SMs x
                                    that / (kv heads x sequences)) partitions per sequence of
                                    ceil(max_seq_len / that) tokens (rounded up to whole blocks),
                                    when that is at least 2; fixed partitions.
                                    Any lengths stay correct; a batch in which a few sequences are
                                    much longer than the rest runs slower than without the flag
                                    (their partitions get only their share of the SMs) */
    PA_FLAG_PREFIX_GRID = 32     /* pa_prefix_ex / pa_prefix_split, tcgen05 kernel: one CTA per
                                    query tile (and key-split part) instead of the default
                                    persistent form, in which a grid of the CTAs the SMs hold at
                                    once claims the tiles in grid order from a device counter and
                                    each CTA's copy rings run on from one tile to the next.  Both
                                    forms compute every tile alike, so they give the same bits */
};

/* All inputs of one decode call (device pointers; see the layouts above). */
typedef struct {
    void* out;
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* seq_lens;
    int num_seqs;           /* 0..65535 */
    int max_blocks_per_seq; /* row stride of block_tables */
    int max_seq_len;        /* host-side bound, >= every seq_lens[b]; sizes the grid */
    int64_t num_blocks;     /* blocks in the pool; num_blocks*num_kv_heads*block_size < 2^31 */
    int num_heads;
    int num_kv_heads;
    int head_dim;
    int block_size;
    float scale;            /* multiplies q.k before the softmax (finite) */
} pa_decode_args;

/* Tuning and debug options; an all-zero struct means "defaults". */
typedef struct {
    int mode;                    /* PA_MODE_* */
    int partition_size;          /* tokens per partition in SPLIT mode, multiple of block_size; 0 = chosen
                                    by the planner: 512 (256 when that gives fewer CTAs than SMs); for
                                    one sequence over 128 tokens, one wave of 256 / head_dim 4-warp
                                    CTAs per SM (one at head_dim 256), as many partitions per kv head
                                    as that gives (pooled from 2048-token
                                    partitions on, see PA_FLAG_POOLED; fixed below); for a batch whose
                                    longest sequence is over 256 tokens, the same one wave when it gives
                                    at least 4 partitions per sequence of at most 128 tokens (fixed),
                                    or at any length with PA_FLAG_UNIFORM_LENGTHS.  AUTO runs SINGLE
                                    when the longest sequence fits one partition of the plan, e.g.
                                    up to 128 tokens, or up to 512 in larger batches */
    int flags;                   /* PA_FLAG_* */
    unsigned int wait_limit;     /* polls before a copy wait gives up; 0 = library default (2^20) */
    void* event_partition_begin; /* optional cudaEvent_t recorded on `stream` right before ... */
    void* event_partition_end;   /* ... and right after the partition kernel (timing only) */
    int warps;                   /* partition CTA shape: warps per CTA and shared-memory stages per */
    int stages;                  /* warp; 0/0 = library choice; compiled: 2x2, 1x2, 1x3, 4x2
                                    (PERSISTENT: 1x2, 2x2, 4x2; default 4x2, or 1x2 with a
                                    partition_size) */
} pa_decode_opts;

/* What a call will launch (filled by pa_decode_plan; host-only, no CUDA calls). */
typedef struct {
    int mode;              /* PA_MODE_SINGLE, _SPLIT, _FUSED, _PERSISTENT or _FLAT */
    int partition_size;    /* tokens per CTA (SINGLE: max_seq_len rounded up to block_size;
                              PERSISTENT: 0 = apportioned per sequence on the device; FLAT: 0,
                              each CTA's share is fixed on the device) */
    int grid_x, grid_y, grid_z;          /* partition kernel: partitions, kv heads, sequences
                                            (PERSISTENT and FLAT: the fixed grid, 1, 1) */
    int threads;           /* threads per partition CTA */
    int smem_bytes;        /* dynamic shared memory per partition CTA */
    int launch_reduce;     /* 1 if the reduce kernel runs */
    int reduce_grid_x, reduce_grid_y, reduce_grid_z; /* heads, sequences, head_dim / slice
                                                        width (32..256, about 2 CTAs per SM) */
    size_t workspace_bytes; /* caller workspace pa_decode_ex needs (0 when there are no partials) */
    int stages;            /* shared-memory stages per warp of the partition CTA */
    int max_partitions;    /* partials kept per (sequence, head) in the workspace */
    int pooled;            /* 1 if the partition CTAs claim chunks of blocks (PA_FLAG_POOLED) */
    int coop;              /* FUSED: 1 if the grid is launched cooperatively and the CTAs of a
                              (sequence, kv head) merge in parallel after a group barrier */
} pa_decode_plan_t;

/* Decode attention with a library-owned workspace.
 * Sources: "docs" commit page (GQA-aware grid on kv heads, Phase 1 partition
 * and Phase 2 reduce kernels, the compound partial); "paged_attention_v2_triton.py"
 * commit page (the alpha/beta online-softmax update); "qwen3_6_scripts/paged_attn.py"
 * commit page (decode dispatch by sequence length; the buffer-reuse paragraphs).
 * The workspace for the partials is cached per device and grown on demand
 * (allocate once, reuse across calls); growing it synchronises the device, so
 * the first call with a larger size must not be inside a stream capture, and
 * calls on different streams that overlap in time share (and race on) it.
 * num_blocks is the pool size (k_cache.shape[0]); it bounds the block ids the
 * kernel will follow. */
int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
              int max_blocks_per_seq, int max_seq_len, int64_t num_blocks, int num_heads,
              int num_kv_heads, int head_dim, int block_size, float scale, pa_stream_t stream);

/* Decode attention with caller-owned workspace (device memory, 256-byte
 * aligned, at least plan.workspace_bytes; may be NULL when that is 0).
 * Allocates nothing, so it can be captured in a CUDA graph.  opts may be NULL.
 * Same operation and sources as pa_decode; the caller-owned buffer follows the
 * buffer-reuse paragraphs of the "qwen3_6_scripts/paged_attn.py" commit page
 * (allocate once outside the hot loop, pass it in).  The workspace's layout
 * (partials, then the pooled counters, FUSED tickets or PERSISTENT tables) is
 * the library's; its contents between calls are described under the modes and
 * flags above.  Returns PA_ERR_WORKSPACE for a buffer that is too small or
 * misaligned, before launching anything. */
int pa_decode_ex(const pa_decode_args* args, const pa_decode_opts* opts, void* workspace,
                 size_t workspace_bytes, pa_stream_t stream);

/* Validate the arguments and fill *plan with the launches a call would make.
 * num_sms > 0 is the SM count to plan for; 0 asks the current device.  Pure
 * host logic when num_sms > 0.  Returns the same codes a call would.
 * Source: the decode dispatch of the "qwen3_6_scripts/paged_attn.py" commit
 * page (single-CTA kernel vs partitioned kernel by sequence length; the
 * thresholds here are this library's, from GB300 measurements) and the grid
 * arithmetic of the "docs" commit page's GQA-aware grid paragraph
 * ((partitions, kv heads) programs per sequence). */
int pa_decode_plan(const pa_decode_args* args, const pa_decode_opts* opts, int num_sms,
                   pa_decode_plan_t* plan);

/* Workspace bytes of a SPLIT call with these sizes: the compound partials of
 * the "docs" commit page (max score, exp sum, weighted V per partition, fp32),
 * sized once for reuse as the "qwen3_6_scripts/paged_attn.py" commit page's
 * buffer-reuse paragraphs advise.  partition_size 0 gives an upper bound for the
 * automatic partition size, one-wave plans included (PA_FLAG_UNIFORM_LENGTHS
 * too; it asks the device's SM count, and assumes 1024 SMs without a device),
 * and its pooled claim counters.  A pooled SPLIT
 * needs 256-byte-aligned num_seqs * num_kv_heads * 8 bytes more; FUSED that much
 * plus 256-byte-aligned num_seqs * num_kv_heads * 4; PERSISTENT has its own
 * partition count and tables (work list, order, sizes).  pa_decode_plan gives
 * every mode's exact figure.  Returns 0 for non-positive sizes. */
size_t pa_decode_workspace_size(int num_seqs, int max_seq_len, int num_heads, int head_dim,
                                int partition_size);

/* Synchronise `stream`, then read and clear the current device's status word
 * into *status (PA_DEV_* bits).  Returns PA_OK, PA_ERR_INVALID_ARG (status
 * NULL) or PA_ERR_CUDA.  Source: the "qwen3_6_scripts/paged_attn.py" commit
 * page's account of a prefill kernel that hung the GPU for good and of the
 * try/except fallbacks added around it; this library replaces both with
 * bounded waits and this host-read status word (no fallback, no trap). */
int pa_get_device_status(pa_stream_t stream, int* status);

/* Static English text for a return code (never NULL; "unknown status" for a
 * code not listed above).  Part of the same error reporting as
 * pa_get_device_status; the pages print no counterpart. */
const char* pa_status_string(int status);

/* Free the library-owned workspaces of every device (synchronises them, then
 * restores the current device).  The counterpart of the allocate-once cache of
 * the "qwen3_6_scripts/paged_attn.py" commit page's buffer-reuse paragraphs: the
 * next pa_decode allocates again.  Also frees the persistent prefill's counter
 * (the next pa_prefix allocates it again).  Never frees caller memory. */
void pa_release_workspace(void);

/* Chunked-prefill ("prefix") attention over the paged cache.
 * Sequence b has context_lens[b] tokens already in the paged cache (found
 * through block_tables as for decode) and brings a chunk of new tokens: rows
 * query_start_loc[b] .. query_start_loc[b+1]-1 of q, k_new and v_new.  New
 * token i of the chunk attends to every context token and to chunk tokens
 * 0..i (causal inside the chunk):
 *     out[tok, h, :] = softmax(scale * q[tok, h, :] . [K_ctx ; K_new[0..i]]^T) [V_ctx ; V_new[0..i]]
 * Source: "qwen3_6_scripts/paged_attn.py" commit page, prefix path (online
 * softmax over the pre-gathered paged context, then over the current chunk).
 * Layouts: q, out fp16 [num_tokens][num_heads][head_dim]; k_new, v_new fp16
 * [num_tokens][num_kv_heads][head_dim]; query_start_loc int32 [num_seqs + 1]
 * (0 first, num_tokens last, non-decreasing); context_lens int32 [num_seqs];
 * caches and block table as for pa_decode.  max_context_len and max_query_len
 * are host-side bounds that size the grid.  The new tokens' K/V are read from
 * k_new/v_new, not from the cache (the caller appends them afterwards).
 * Same support, alignment, ownership and error rules as pa_decode; a call
 * whose query tiles (of floor(128 / G) tokens) x kv heads x sequences reach
 * 2^31 returns PA_ERR_UNSUPPORTED.  Device-detected bad lengths set
 * PA_DEV_BAD_SEQ_LEN.
 * The tensor-core kernel runs in a persistent form by default: a grid of the
 * CTAs the SMs hold at once claims the query tiles in grid order from a
 * library-owned device counter, and each CTA's copy rings run on from one
 * tile to the next.  There is one counter (256 bytes) per device and stream,
 * allocated and zeroed on the stream by the first such call on it, re-armed
 * by every call and freed by pa_release_workspace; calls on one stream never
 * overlap, so they never share it while running.  A call made while its
 * stream is being captured before that stream's counter exists runs the grid
 * form (one CTA per query tile), which PA_FLAG_PREFIX_GRID also selects; both
 * give the same bits.  A captured call keeps the counter of the stream it was
 * captured on: replays of that graph must not overlap one another or other
 * calls on that stream. */
typedef struct {
    void* out;
    const void* q;
    const void* k_new;
    const void* v_new;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* query_start_loc;
    int num_seqs;
    int num_tokens;
    int max_blocks_per_seq;
    int max_context_len;
    int max_query_len;
    int64_t num_blocks;
    int num_heads;
    int num_kv_heads;
    int head_dim;
    int block_size;
    float scale;
} pa_prefix_args;

int pa_prefix(void* out, const void* q, const void* k_new, const void* v_new, const void* k_cache,
              const void* v_cache, const int32_t* block_tables, const int32_t* context_lens,
              const int32_t* query_start_loc, int num_seqs, int num_tokens, int max_blocks_per_seq,
              int max_context_len, int max_query_len, int64_t num_blocks, int num_heads, int num_kv_heads,
              int head_dim, int block_size, float scale, pa_stream_t stream);

/* The same with an argument struct and options (opts may be NULL; of the
 * options only flags, wait_limit and the two timing events apply). */
int pa_prefix_ex(const pa_prefix_args* args, const pa_decode_opts* opts, pa_stream_t stream);

/* Chunked prefill with the last wave's query tiles split by key range.
 * The tensor-core prefill kernel works on one (query tile, kv head,
 * sequence) at a time per SM, and every tile walks all of its sequence's
 * keys, so the tiles take about the same time and N of them on S SMs run in
 * ceil(N / S) rounds.  When the last round is partly empty, its trailing
 * query tiles (`units`, counted in the grid's order: tile fastest, then kv
 * head, then sequence) each run as `parts` units, part p walking the p-th of
 * `parts` consecutive ranges of the tile's key tiles and leaving, per row,
 * the online-softmax state (m, l, O relative to 2^m) in the workspace; a
 * second kernel then merges a row's parts with the log-sum-exp rule of the
 * decode reduce ("docs" commit page, Phase 2; the alpha/beta fold of the
 * "paged_attention_v2_triton.py" commit page).  The result is the same
 * attention as pa_prefix_ex up to the rounding order of the sums.
 * Split: NULL or parts == 0 takes the library's plan (a model of the rounds
 * on this device, for grids of at most 4 rounds of one CTA per SM; it may
 * split nothing); parts in [1, 64] with units in
 * [0, N] forces that split.  The workspace (caller-owned device memory,
 * 256-byte aligned, contents need no initialisation) must hold
 * pa_prefix_split_workspace_size bytes for the same arguments and split;
 * the call allocates nothing but the persistent form's counter (see
 * pa_prefix), whose parts are units like the whole tiles.  With
 * PA_FLAG_PREFIX_WARP_MMA nothing is split
 * and this is pa_prefix_ex.  Errors as pa_prefix_ex, plus PA_ERR_INVALID_ARG
 * for a workspace that is missing, too small or misaligned, or a split out
 * of range. */
typedef struct {
    int parts; /* key ranges per split query tile; 0 = the library's plan */
    int units; /* trailing query tiles that are split (with parts > 0) */
} pa_prefix_split_opts;

int pa_prefix_split_workspace_size(const pa_prefix_args* args, const pa_prefix_split_opts* split, size_t* bytes);
int pa_prefix_split(const pa_prefix_args* args, const pa_decode_opts* opts, const pa_prefix_split_opts* split,
                    void* workspace, size_t workspace_bytes, pa_stream_t stream);

/* Size of the fixed device scratch that pa_decode_noalloc uses (16 MiB). */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)

/* Decode attention without any device allocation, for callers that cannot
 * call cudaMalloc: a framework that owns every byte of device memory through
 * its own pool, a decode loop that cannot pay the synchronisation of an
 * allocation, code running where allocating CUDA calls are not allowed.  The
 * pages this library follows have no counterpart to this call.
 *
 * Arguments, layouts, modes (AUTO) and results are those of pa_decode.  The
 * split-KV partials go to a file-scope device array of
 * PA_NOALLOC_SCRATCH_BYTES that each GPU loading the library holds until the
 * process exits.
 *  - A call whose partials need more (see pa_decode_plan's workspace_bytes)
 *    returns PA_ERR_WORKSPACE without launching anything.  At the 24-head,
 *    head_dim-256, 512-token-partition shape that is about 64 sequence-
 *    partitions per MiB, e.g. one 100K-token sequence needs 4.95 MB.
 *  - The first call on each device looks up the array's device address with
 *    that device current, so make that first call before any stream capture.
 *  - All calls on a device share the one array: calls that overlap on the
 *    GPU (other streams, other host threads) race and give wrong outputs.
 *    Calls queued on a single stream are safe.
 *  - Nothing in the array has to start at zero: each call writes every partial
 *    it reads, and the pooled split's claim counters tolerate whatever an
 *    earlier call of another shape left there (see PA_FLAG_POOLED). */
int pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                      int max_blocks_per_seq, int max_seq_len, int64_t num_blocks, int num_heads,
                      int num_kv_heads, int head_dim, int block_size, float scale, pa_stream_t stream);

/* Split-KV across devices, step 1 of 2 (no counterpart on the pages beyond
 * their partitions: "docs" commit page, GQA-aware grid and partition
 * paragraphs, and its compound partial).  Sequence b's tokens are cut into
 * partitions of partition_size tokens (partition p holds tokens
 * [p * partition_size, min((p + 1) * partition_size, seq_lens[b])));
 * this call computes partitions partition_begin .. partition_begin +
 * partition_count - 1 of every sequence and writes their partials:
 *   max_logits  fp32 [num_seqs][num_heads][partition_count]: the partition's
 *               largest score in base 2, m = log2(e) * max_t(scale * q . k_t)
 *   exp_sums    fp32 [num_seqs][num_heads][partition_count]:
 *               l = sum_t 2^(log2(e) * scale * q . k_t - m)
 *   tmp_out     fp32 [num_seqs][num_heads][partition_count][head_dim]: the
 *               partition's softmax-weighted V, normalised by l
 * A partition past its sequence's end (or of an empty sequence) gets
 * m = -inf, l = 0 and a zero row.  Each device of a split calls this with its
 * own range over a pool that holds the blocks of that range (the block-table
 * entries outside the range are never read), the devices exchange the arrays
 * (an all-gather of local buffers), and pa_merge_partials finishes.
 * args as for pa_decode_ex except that args->out is not used (may be NULL);
 * partition_size a positive multiple of block_size; partition_begin >= 0,
 * partition_count >= 1.  opts: mode AUTO or SPLIT, warps/stages, wait_limit,
 * PA_FLAG_FORCE_TIMEOUT and the timing events apply; the partitions are fixed
 * (never pooled).  tmp_out 16-byte aligned, the other two 4-byte aligned, all
 * device memory owned by the caller.  Allocates nothing.  Device-detected
 * problems set the status word as for pa_decode; the partials are then
 * unspecified. */
int pa_decode_partials(const pa_decode_args* args, const pa_decode_opts* opts, int partition_size,
                       int partition_begin, int partition_count, float* max_logits, float* exp_sums,
                       float* tmp_out, pa_stream_t stream);

/* Split-KV across devices, step 2 of 2: the log-sum-exp merge of the
 * partials that num_sources calls of pa_decode_partials produced, source r
 * having computed partitions [r * partitions_per_source, (r + 1) *
 * partitions_per_source) with the same partition_size.  The arrays hold the
 * sources one after another, as an all-gather of their buffers along a new
 * leading dimension gives them:
 *   max_logits, exp_sums fp32 [num_sources][num_seqs][num_heads][partitions_per_source]
 *   tmp_out              fp32 [num_sources][num_seqs][num_heads][partitions_per_source][head_dim]
 * out fp16 [num_seqs][num_heads][head_dim] gets, per (sequence, head), the
 * merge of its ceil(seq_lens[b] / partition_size) partials: M = max_p m_p,
 * w_p = l_p 2^(m_p - M), out = sum_p w_p acc_p / sum_p w_p ("docs" commit
 * page, Phase 2 reduce; the alpha/beta fold of the "paged_attention_v2_triton.py"
 * commit page); zero for an empty sequence.  The sources must cover the
 * longest sequence: num_sources * partitions_per_source >= ceil(max_seq_len /
 * partition_size), else PA_ERR_INVALID_ARG.  seq_lens int32 [num_seqs], each in
 * [0, max_seq_len] (a length outside sets PA_DEV_BAD_SEQ_LEN and leaves that
 * output unwritten).  out and tmp_out 16-byte aligned, the rest 4-byte
 * aligned; device memory owned by the caller; allocates nothing; asynchronous
 * on stream.  head_dim in {64, 128, 256}. */
int pa_merge_partials(void* out, const float* max_logits, const float* exp_sums, const float* tmp_out,
                      const int32_t* seq_lens, int num_seqs, int num_heads, int head_dim, int max_seq_len,
                      int partition_size, int num_sources, int partitions_per_source, pa_stream_t stream);

/* Library version, major*10000 + minor*100 + patch.  No counterpart on the pages. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_DECODE_H */
