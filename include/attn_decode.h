/*
 * attn_decode.h -- C ABI of the GB300 (sm_103a) split-KV grouped-query decode
 * attention library, libattn_decode.so.
 *
 * The operation (minfer "10 · R4 -- decode split-attention dim-parallel rewrite",
 * §2.1): for every sequence s and query head h, with one new query row per
 * sequence (decode, nt == 1),
 *
 *     o[s][h] = softmax(q[s][h] · K[s][0:nkv][hk]ᵀ · scale) · V[s][0:nkv][hk]
 *
 * where hk = h / (n_head / n_kv_head) is the KV head shared by the contiguous
 * group of query heads h, and nkv = positions[s] + 1 is read on the device
 * (§2.2), so one launch configuration serves every context length and the call
 * can be captured in a CUDA graph and replayed while positions[] advances.
 *
 * It runs as two kernels (§2.1): a partial kernel with one block per
 * (split, KV head, sequence) that runs the online softmax over its row range
 * [lo, hi) for every query head of the group from a single K/V read and writes
 * the triple (mx, S, oc); and a combine kernel that takes gmx = max mx over the
 * splits, reweights each split by exp(mx - gmx) and writes o = acc / S (0 when
 * every split is empty).
 *
 * Conventions for every entry point below
 *  - Device pointers are caller-owned device memory; the library never frees,
 *    reallocates or synchronises them, and never synchronises the stream except
 *    in attn_read_device_error().
 *  - Layouts are dense row-major:
 *        q, out      float  [n_seq][n_head][head_dim]
 *        k_cache,    f16    [n_seq][cap][n_kv_head][head_dim]   (IEEE binary16, or
 *        v_cache     f16    [n_seq][cap][n_kv_head][head_dim]    bfloat16: ATTN_KV_BF16)
 *        positions   int32  [n_seq]      (device memory; nkv_s = positions[s] + 1)
 *    so row j of sequence s, KV head hk starts at element
 *    ((s * cap + j) * n_kv_head + hk) * head_dim.
 *  - All pointers must be 16-byte aligned.
 *  - Supported shapes: head_dim in {8, 64, 128, 256}; 1 <= n_head / n_kv_head <= 8;
 *    n_head % n_kv_head == 0. Anything else returns ATTN_ERR_UNSUPPORTED; there
 *    is no fallback path.
 *  - Rows [0, nkv_s) are read; rows >= nkv_s are never used. A positions[s]
 *    outside [-1, cap - 1] is clamped (nkv_s to [0, cap]) and sets
 *    ATTN_DEVERR_POSITION_CLAMPED in the device error word.
 *  - Argument errors are returned synchronously, before anything is launched.
 *    Launch failures return ATTN_ERR_CUDA. No entry point aborts the process.
 *  - Thread safety: entry points may be called from several host threads.
 */
#ifndef ATTN_DECODE_H
#define ATTN_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, n_head % n_kv_head != 0 */
    ATTN_ERR_UNSUPPORTED = 2,  /* head_dim or group size outside the compiled set */
    ATTN_ERR_WORKSPACE = 3,    /* workspace too small (or needed growth while capturing) */
    ATTN_ERR_CUDA = 4          /* a CUDA runtime/driver call failed; see attn_last_cuda_error */
} attn_status;

/* Bits of the sticky device error word (attn_read_device_error). */
#define ATTN_DEVERR_POSITION_CLAMPED 0x1u  /* some positions[s] fell outside [-1, cap-1] */
#define ATTN_DEVERR_PIPELINE_TIMEOUT 0x2u  /* a bounded in-kernel wait gave up (block skipped) */

/* Kernel variants for attn_decode_ex. */
#define ATTN_VARIANT_AUTO 0   /* tensor cores where compiled (head_dim % 16 == 0), else CUDA cores;
                                 the tcgen05 kernel for short calls (attn_resolve_variant) */
#define ATTN_VARIANT_SIMT 1   /* CUDA-core f32 partial kernel (every head_dim) */
#define ATTN_VARIANT_TC   2   /* tensor-core partial kernel: 16x8x16 MMA, f32 accumulate, q and
                                 p each carried as a hi + lo pair of the cache's element type (about
                                 22 significant bits for f16, 16 for bf16); head_dim 64, 128, 256
                                 only (ATTN_ERR_UNSUPPORTED otherwise) */
#define ATTN_VARIANT_TCGEN05 3 /* tensor-core partial kernel on tcgen05 (accumulators in tensor
                                 memory): one tile of T rows per block (T = 128; 96 at head_dim
                                 256), q and p as the same hi + lo pairs, a block-wide softmax in
                                 one pass; head_dim 128 or 256 (ATTN_ERR_UNSUPPORTED otherwise);
                                 with attn_decode_multi 16 (query row, head) pairs per block.
                                 Every split must fit one tile: split_len <= T, or by count
                                 n_splits * T >= cap (ATTN_ERR_INVALID_ARG otherwise; the
                                 heuristic picks such a count) */
#define ATTN_VARIANT_TCGEN05_CLUSTER 4 /* the tcgen05 kernel with the combine inside it: the 16
                                 splits of a (sequence, KV head) run as one 16-block thread-block
                                 cluster that merges its blocks' states in distributed shared
                                 memory and writes out directly (no workspace is used, no combine
                                 kernel is launched); each block takes up to 4 tiles of 128 rows.
                                 head_dim 128, one query row, a whole call (not the stage entry
                                 points), splits by count with n_splits 0 or 16, cap <= 8192;
                                 ATTN_ERR_INVALID_ARG otherwise, ATTN_ERR_UNSUPPORTED where the
                                 device cannot hold the cluster. On request only: variant 0
                                 does not take it (measured no faster than the tcgen05 kernel
                                 with its separate combine). */

#define ATTN_VARIANT_TC_TILE 5 /* tensor-core partial kernel for splits of one tile, built for the
                                 shortest chain of dependent steps: 16x8x16 MMAs with operands in
                                 registers (q and p as hi + lo pairs as above), S split by rows
                                 over four warps, one block-wide maximum, O = P·V split by head
                                 dimension over the warps (no merge of warp states). One tile of
                                 T rows per block (T = 128; 96 at head_dim 256) or, one block per
                                 SM, a wide tile of W rows (W = 256 at head_dim 128, 128 at 256)
                                 when a split needs more than T rows (block lengths T+1..W, or
                                 n_splits * T < cap <= n_splits * W);
                                 head_dim 128 or 256 with one query row, head_dim 128 with
                                 several (16 (query row, head) pairs per block, either tile);
                                 ATTN_ERR_UNSUPPORTED otherwise. Every split must fit one tile
                                 (ATTN_ERR_INVALID_ARG otherwise). By count, a chunk
                                 ceil(nkv / n_splits) of more than 3T/4 rows is rounded up to
                                 16 rows, a shorter one to T. By block length, for one query
                                 row, with split_len a multiple of 16 that divides T, one block
                                 serves T / split_len consecutive splits from one tile (cache
                                 rows of that tile past nkv are then read -- all below cap --
                                 but never used). */

/* Cache element type, OR'd into the variant argument: without it K and V are
   IEEE binary16 (f16); with it they are bfloat16 (1 sign, 8 exponent, 7
   fraction bits). k_new / v_new of attn_decode_append use the same type. */
#define ATTN_KV_BF16 0x10

/* Early start, OR'd into the variant argument. Every launch of this library
   is a programmatic dependent launch: its blocks may become resident while the
   kernel before it on the stream still runs, and wait for that kernel to end
   before the first read of anything it could have written. With this flag the
   caller promises that `positions` and the cache rows the call attends (rows
   below positions[s], and row positions[s] itself unless attn_decode_append
   supplies it) are written by nothing that can still be running when the call
   is launched -- in a decode step, true for every attention layer after the
   first once positions has been advanced. The partial kernel then reads
   positions and starts its K/V copies before that wait, so the cache stream
   of this layer overlaps the tail of the previous kernel. q, k_new, v_new
   and the workspace are still touched only after the wait. Breaking the
   promise gives stale rows, not a fault: all reads stay inside the cache. */
#define ATTN_KV_STABLE 0x20

/*
 * attn_decode -- one layer call, single sequence, library-owned workspace.
 *
 * The argument list of the operation itself. n_seq must be 1 (several
 * sequences need their per-sequence row stride: use attn_decode_ex). The cache
 * must hold at least positions[0] + 1 rows; with no capacity argument the
 * library cannot clamp positions[0], so this is the caller's guarantee.
 * The split count comes from attn_split_heuristic(). The workspace is a
 * per-device buffer owned by the library; it grows (cudaMalloc) only outside
 * stream capture, so make one uncaptured call with the largest shape before
 * capturing. Calls that may run concurrently on different streams must use
 * attn_decode_ex with their own workspaces.
 * scale multiplies q·k (1/sqrt(head_dim) for standard attention).
 */
attn_status attn_decode(const float *q, const void *k_cache, const void *v_cache,
                        const int32_t *positions, float *out, int n_seq, int n_head,
                        int n_kv_head, int head_dim, float scale, attn_stream_t stream);

/*
 * attn_decode_ex -- full control.
 *   cap             cache rows per sequence (>= 1); nkv_s is clamped to cap.
 *   n_splits        splits P per (sequence, KV head); 0 = attn_split_heuristic_ex()
 *                   for this call's variant.
 *   split_len       0: split by count, chunk = ceil(nkv / P) rounded up to the
 *                   kernel's row granule: 128 rows (tcgen05: whole tiles; 96 at
 *                   head_dim 256), 64 rows
 *                   (mma.sync, head_dim <= 128, one query row: whole tiles), 16 rows
 *                   (mma.sync otherwise) or 32 rows (CUDA cores) (minfer R4 §2.2);
 *                   the kernel variant 0 runs is reported by attn_resolve_variant;
 *                   > 0: fixed block of split_len
 *                   rows per split (Red Lite dev35 "Change"), which needs
 *                   P * split_len >= cap, else ATTN_ERR_INVALID_ARG; with
 *                   n_splits = 0 the call takes P = ceil(cap / split_len)
 *                   (ATTN_ERR_INVALID_ARG past 4096 splits).
 *   variant         ATTN_VARIANT_*.
 *   workspace       device buffer of at least attn_workspace_size(...) bytes,
 *                   256-byte aligned; NULL selects the library-owned buffer as in
 *                   attn_decode. Its contents on entry do not matter. The
 *                   cluster-fused variant uses none (it may be NULL).
 */
attn_status attn_decode_ex(const float *q, const void *k_cache, const void *v_cache,
                           const int32_t *positions, float *out, int n_seq, int n_head,
                           int n_kv_head, int head_dim, float scale, int64_t cap,
                           int n_splits, int split_len, int variant, void *workspace,
                           size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_decode_append -- append the new token's K/V row to the cache and attend,
 * in the same launches (dotLLM #199 §1: each decode step first writes the new
 * K/V row into the f16 cache, then attends over [0, nkv)).
 *   k_new, v_new    f16 [n_seq][n_kv_head][head_dim], 16-byte aligned: the row
 *                   of the token at position positions[s].
 *   k_cache, v_cache  as in attn_decode_ex, but written: row positions[s] of
 *                   sequence s receives k_new[s] / v_new[s] for every KV head.
 * The result is that of attn_decode_ex on the cache after the write (the new
 * row is attended from the new values, never from the cache's old contents).
 * A positions[s] outside [0, cap - 1] writes nothing for that sequence and is
 * clamped and flagged as in attn_decode_ex. Other arguments as attn_decode_ex.
 */
attn_status attn_decode_append(const float *q, const void *k_new, const void *v_new,
                               void *k_cache, void *v_cache, const int32_t *positions, float *out,
                               int n_seq, int n_head, int n_kv_head, int head_dim, float scale,
                               int64_t cap, int n_splits, int split_len, int variant,
                               void *workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_decode_multi -- several causal query rows per sequence (speculative
 * drafts, short chunks): the variant dotLLM #199 §2 gates out (more than one
 * query row needs a causal mask offset by the query's position).
 *   n_q             query rows per sequence (1 <= n_q <= 1024); n_q == 1 is
 *                   attn_decode_ex.
 *   q, out          float [n_seq][n_q][n_head][head_dim].
 *   positions[s]    position of the sequence's LAST query row; with
 *                   nkv = clamp(positions[s] + 1, 0, cap), query row t sits at
 *                   position nkv - n_q + t and attends cache rows
 *                   [0, nkv - n_q + t] (none when that is negative: o = 0).
 *   workspace       attn_workspace_size(n_seq, n_q * n_head, head_dim, n_splits)
 *                   bytes (the partials of every query row).
 * Needs head_dim % 16 == 0 (tensor-core kernel; ATTN_VARIANT_SIMT and
 * head_dim 8 return ATTN_ERR_UNSUPPORTED). K/V are read once per block of 16
 * (query row, head) pairs of a KV head. Other arguments as attn_decode_ex.
 */
attn_status attn_decode_multi(const float *q, const void *k_cache, const void *v_cache,
                              const int32_t *positions, float *out, int n_seq, int n_q, int n_head,
                              int n_kv_head, int head_dim, float scale, int64_t cap, int n_splits,
                              int split_len, int variant, void *workspace, size_t workspace_bytes,
                              attn_stream_t stream);

/*
 * attn_decode_partial / attn_decode_combine -- the two stages of attn_decode_ex
 * as separate calls (same arguments, same validation), for callers that time
 * the stages apart or merge partials produced elsewhere before combining.
 *
 * attn_decode_partial runs steps a1-a6 ("10 · R4" §2.1 partial kernel) and
 * leaves the partial triples in `workspace`; n_splits must be given (> 0) and
 * workspace must be non-NULL, since both calls have to agree on them.
 * attn_decode_combine runs step a7 (the combine kernel) on a workspace filled
 * by attn_decode_partial with the same n_seq, n_head, head_dim and n_splits,
 * and writes `out`. Workspace layout (all f32, both regions 256-byte aligned):
 *     oc  at byte 0:                      [n_seq][n_head][n_splits][head_dim]
 *     ml  at byte round_up(4 * n_seq * n_head * n_splits * head_dim, 256):
 *                                         [n_seq][n_head][n_splits][2] = (mx, S)
 * where oc is the unnormalised weighted V sum of the split, S its softmax
 * denominator and mx the reference they are scaled to (log2 units): with s a
 * row's score times log2 e, oc = sum 2^(s - mx) v and S = sum 2^(s - mx) over
 * the split's rows. mx is at or near the split's running maximum, or the
 * maximum of the rows a kernel block shares among several splits (a split far
 * below it then holds small or zero S and oc); 2^(s - mx) stays below 2^15. An
 * empty split has mx = -inf, S = 0 and its oc is never read. Splits combine in any order: partials of disjoint row
 * ranges computed elsewhere (another device's shard of the rows, say) can be
 * laid side by side along the split axis and combined with n_splits = the
 * total split count.
 */
attn_status attn_decode_partial(const float *q, const void *k_cache, const void *v_cache,
                                const int32_t *positions, int n_seq, int n_head, int n_kv_head,
                                int head_dim, float scale, int64_t cap, int n_splits,
                                int split_len, int variant, void *workspace,
                                size_t workspace_bytes, attn_stream_t stream);

attn_status attn_decode_combine(const void *workspace, size_t workspace_bytes, float *out,
                                int n_seq, int n_head, int head_dim, int n_splits,
                                attn_stream_t stream);

/*
 * attn_decode_static -- attn_decode_ex for callers that cannot allocate device
 * memory when they call it: an engine step running under CUDA stream capture
 * (no cudaMalloc while capturing), a plugin whose host framework owns all
 * device memory, a process with a fixed device-memory budget. The pages this
 * library follows have no counterpart to this entry point.
 *
 * Same arguments and results as attn_decode_ex without the workspace: the
 * partial triples go to a fixed device array of ATTN_STATIC_SCRATCH_BYTES
 * inside the library, which every GPU that loads the library holds until the
 * process exits. The call allocates nothing (no cudaMalloc/cudaFree, no
 * allocating library routine). The first call on a device, with that device
 * current, looks up the array's device address (cudaGetSymbolAddress); make
 * that first call before any stream capture.
 *   - n_splits == 0 takes the split count attn_decode_ex takes for the same
 *     variant argument (attn_split_heuristic_ex: the kernel variant, the
 *     early-start flag and the cache type all count). A call whose partials
 *     need more than ATTN_STATIC_SCRATCH_BYTES (attn_workspace_size(n_seq,
 *     n_head, head_dim, P)) returns ATTN_ERR_WORKSPACE and launches nothing;
 *     ATTN_VARIANT_TCGEN05_CLUSTER keeps its partials on chip and uses none.
 *   - All calls share the one array and it keeps the last call's contents.
 *     Nothing in it has to start at zero: every split writes its (mx, S) before
 *     the combine reads it, and oc is only read for splits that wrote it in
 *     the same call. Two calls whose kernels can overlap on the GPU (different
 *     streams without ordering, or different host threads) race on the array
 *     and give wrong results; serialise them on one stream.
 */
#define ATTN_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)

attn_status attn_decode_static(const float *q, const void *k_cache, const void *v_cache,
                               const int32_t *positions, float *out, int n_seq, int n_head,
                               int n_kv_head, int head_dim, float scale, int64_t cap,
                               int n_splits, int split_len, int variant, attn_stream_t stream);

/*
 * attn_split_heuristic -- host-only, static split count P for a launch.
 * Chooses P from the shape and the static capacity (never from nkv, which lives
 * on the device). With the capacity known, the chunk is sized so that at full
 * capacity the (sequence, KV head) units fill one wave of resident blocks for a
 * single sequence, eight waves for a batch (whose ragged lengths then balance),
 * rounded up to the kernel's row granule; P = ceil(cap / chunk). cap <= 0
 * means "unknown": one wave. sm_count <= 0 queries the current device (and
 * returns 0 with no device). The same rule serves attn_decode_ex's n_splits = 0.
 */
int attn_split_heuristic(int n_seq, int n_head, int n_kv_head, int head_dim, int64_t cap,
                         int sm_count);

/*
 * attn_split_heuristic_ex -- the same for a call with n_q query rows per
 * sequence (1 for attn_decode_ex / attn_decode_append, n_q for
 * attn_decode_multi, whose blocks each serve 16 (query row, head) pairs) and
 * the call's variant argument (ATTN_VARIANT_*, ATTN_KV_BF16, ATTN_KV_STABLE).
 * With ATTN_KV_STABLE, a single sequence and a short call (at most 4 kernel
 * tiles of rows per block at one block per SM) the wave is one block per SM
 * rather than as many as fit, so that the next flagged call's blocks find room
 * beside this call's and start their copies while it finishes, and a block
 * takes no more rows than its pipeline holds at once (3 tiles of 64 rows at
 * head_dim 128), so that all of its copies start before the previous kernel
 * ends. For the one-tile kernel's wide tiles (256 rows at head_dim 128, 128
 * at 256, one block per SM) the count is the one that gives each SM one block,
 * where that makes splits of more than three quarters of the wide tile at full
 * capacity -- the kernel then rounds such chunks to 16 rows rather than to
 * whole tiles, so the rows spread evenly over the blocks (38 splits of 224 rows
 * for 28 / 4 heads at capacity 8192, 76 of 112 for 16 / 2 heads at 8400, on
 * 152 SMs); otherwise one whole (128- or 96-row) tile per split. Returns 0 for an
 * invalid shape or variant. This is the count-mode plan; a call by block
 * length (split_len > 0) with n_splits = 0 takes P = ceil(cap / split_len)
 * instead.
 */
int attn_split_heuristic_ex(int n_seq, int n_q, int n_head, int n_kv_head, int head_dim,
                            int64_t cap, int sm_count, int variant);

/*
 * attn_resolve_variant -- which partial kernel a call with these arguments and
 * n_splits = 0 runs: ATTN_VARIANT_SIMT, ATTN_VARIANT_TC, ATTN_VARIANT_TCGEN05,
 * ATTN_VARIANT_TCGEN05_CLUSTER or ATTN_VARIANT_TC_TILE (0 for an invalid shape
 * or variant). An explicit variant is returned as is where it supports the
 * shape. ATTN_VARIANT_AUTO picks a one-tile kernel for a short call -- cap > 0
 * and the heuristic's splits, one tile each, in one wave of its blocks: the
 * one-tile mma.sync kernel (ATTN_VARIANT_TC_TILE; 3 blocks per SM at head_dim
 * 128, 2 at 256, or 1 with its wide tiles where one block per SM makes splits
 * longer than the plain tile -- for several query rows with one 16-slot group
 * per KV head) for one query row at head_dim 128 or 256 and for several at 128
 * (ceil(n_q * group / 16) blocks per split and KV head);
 * else tcgen05 for several query rows at head_dim 256 when n_q * group <= 16 (a
 * KV head's (row, head) pairs in one block, 1 block per SM) -- and otherwise the
 * streaming mma.sync tensor-core kernel (head_dim % 16 == 0) or the CUDA-core
 * kernel. With ATTN_KV_STABLE in
 * variant the split count follows the flagged heuristic. With explicit splits
 * that leave a split longer than one tile, or too many blocks for one wave,
 * attn_decode_ex keeps the mma.sync kernel instead. Host only; sm_count <= 0
 * queries the current device.
 */
int attn_resolve_variant(int n_seq, int n_q, int n_head, int n_kv_head, int head_dim, int64_t cap,
                         int sm_count, int variant);

/*
 * attn_plan_call -- the whole plan of one call, host-only: for the arguments
 * of attn_decode_ex (n_q = 1) or attn_decode_multi (n_q rows), including an
 * explicit n_splits or split_len, returns the partial kernel the call runs
 * (*variant_out: ATTN_VARIANT_SIMT, _TC, _TCGEN05 or _TCGEN05_CLUSTER), its
 * split count P (*n_splits_out) and the workspace bytes it needs
 * (*workspace_bytes_out; 0 for the cluster-fused kernel). A call with these
 * arguments and a workspace of that size runs exactly this plan. Any output
 * pointer may be NULL. Uses the current device (its SM count; for
 * ATTN_VARIANT_TCGEN05_CLUSTER, whether it holds the cluster). Returns the
 * status the call itself would return for these arguments (ATTN_ERR_INVALID_ARG
 * also for n_seq == 0, where there is nothing to plan); launches nothing.
 * The planning rules are the ones the ATTN_VARIANT_* descriptions, n_splits
 * and split_len above state (splits by count: minfer "10 · R4" §2.2; by block
 * length: Red Lite dev35 "Change").
 */
attn_status attn_plan_call(int n_seq, int n_q, int n_head, int n_kv_head, int head_dim, int64_t cap,
                           int n_splits, int split_len, int variant, int *variant_out,
                           int *n_splits_out, size_t *workspace_bytes_out);

/*
 * attn_selftest_bounded_wait -- diagnostic: launch one warp that waits on a
 * shared-memory mbarrier nothing ever arrives on, through the same bounded
 * wait the kernels use, with a limit of limit_ns nanoseconds (1 ..
 * 1,000,000,000; the kernels use 1 s). When the limit passes, the warp sets
 * ATTN_DEVERR_PIPELINE_TIMEOUT in the device error word and returns, leaving
 * the context usable; read it with attn_read_device_error. Asynchronous on
 * `stream`; returns the launch status. The pages have no counterpart: it
 * exists to check, without hanging a GPU, that no wait of the library spins
 * forever.
 */
attn_status attn_selftest_bounded_wait(unsigned long long limit_ns, attn_stream_t stream);

/* attn_workspace_size -- bytes of workspace attn_decode_ex needs (host-only). */
size_t attn_workspace_size(int n_seq, int n_head, int head_dim, int n_splits);

/*
 * attn_read_device_error -- synchronises `stream`, returns the sticky device
 * error word (ATTN_DEVERR_* bits) of the current device in *flags and clears it.
 */
attn_status attn_read_device_error(attn_stream_t stream, unsigned int *flags);

/* Human-readable name of a status code (static storage). */
const char *attn_status_string(attn_status status);

/* Last CUDA error seen by the calling thread (cudaError_t value; 0 = none). */
int attn_last_cuda_error(void);

/* Library version, MAJOR*10000 + MINOR*100 + PATCH. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_DECODE_H */
