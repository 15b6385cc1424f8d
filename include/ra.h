/*
 * ra.h - C ABI of the GB300 (sm_103a) ring-ordered blockwise exact attention
 * library (libra.so).
 *
 * The method (web pages on ring and context parallelism):
 *   - "Ring Attention" glossary page (ultralytics.com/tr), section
 *     "Halka Dikkati Nasil Calisir": the sequence is cut into N blocks, one per
 *     ring device; every device keeps its query block while key/value blocks
 *     travel round the ring, so at step s device i meets key/value block
 *     j = (i - s) mod N; partial results are combined with the running softmax
 *     of flash attention (running max, running sum of exponentiated scores,
 *     running score-weighted values, divided at the end); under a causal mask
 *     devices holding early query blocks skip most key blocks, and striped
 *     attention spreads every device's tokens evenly along the sequence to
 *     balance that work.
 *   - "Context Parallelism" glossary page (ultralytics.com/tr), section
 *     "Pratik Kullanim ve Odunlesimler": tensors are [batch, heads, sequence,
 *     dim] with the sequence on dim 2, causal scaled-dot-product attention,
 *     output in the input dtype.
 *   - The same page, section "Baglam Paralelligi Nasil Calisir?": the result
 *     equals full-sequence attention up to ordinary rounding differences.
 *
 * Here the N ring ranks are emulated on one GPU: rank r is an index range of
 * the same HBM buffers, and "receiving block j" is reading it in place.
 *
 * Common conventions for every entry point
 *   - Tensors are dense, row-major, C-contiguous, in NATURAL token order:
 *       q   [B, H,   S, d]        k, v [B, Hkv, S, d]
 *       out [B, H,   S, d]        lse  [B, H,   S]   (fp32, natural log)
 *   - Query head h reads kv head h / (H / Hkv) (grouped-query attention).
 *   - Scores are scaled by 1/sqrt(d).  Causal: key u is visible to query t iff
 *     u <= t in natural positions.  lse = ln sum_u exp(q_t . k_u / sqrt(d)).
 *   - Block length L = S / n_blocks; S must be a multiple of n_blocks.
 *   - layout RA_LAYOUT_CONTIGUOUS: rank r owns tokens [r L, (r + 1) L).
 *     layout RA_LAYOUT_STRIPED: rank r owns tokens t with t mod N == r, in
 *     increasing t (striped attention).
 *   - Pointers are DEVICE pointers owned by the caller, 16-byte aligned, and
 *     stay valid until the enqueued work has finished.  `out` and `lse` must
 *     not overlap any input.
 *   - Every buffer (inputs, outputs, caller workspace) must be device memory
 *     of the CURRENT device: each call checks each one (the allocation its
 *     first byte lies in) with cudaPointerGetAttributes and returns
 *     RA_ERR_INVALID_ARG
 *     (RA_ERR_WORKSPACE for a workspace) for pinned or pageable host memory,
 *     managed memory, or another GPU's memory reached through unified
 *     addressing, before anything is enqueued.  The attention kernels load
 *     tiles with TMA, and the default forward launch multicasts each
 *     key/value tile to both CTAs of a cluster; those copies therefore only
 *     ever read this GPU's own memory.  The library is meant for one process
 *     on one GPU; it holds no multi-GPU code path.
 *   - Every call is asynchronous on `stream` (NULL = legacy default stream):
 *     it validates its arguments, enqueues kernels and returns.  A status
 *     other than RA_OK means nothing was enqueued and nothing was written.
 *     Errors raised later on the device (a bounded wait that ran out) are
 *     reported by ra_check().
 *   - No C++ exception crosses this interface.  The library reads no
 *     environment variables.
 */
#ifndef RA_H_
#define RA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Identical to cudaStream_t; declared here so callers need no CUDA headers. */
typedef struct CUstream_st *ra_stream_t;

typedef enum {
    RA_OK = 0,
    RA_ERR_INVALID_ARG = 1,  /* bad sizes, null/misaligned/overlapping pointers */
    RA_ERR_UNSUPPORTED = 2,  /* valid request outside this build's kernels    */
    RA_ERR_CUDA = 3,         /* a CUDA runtime call failed                     */
    RA_ERR_NO_MEMORY = 4,    /* scratch allocation failed                      */
    RA_ERR_TIMEOUT = 5,      /* a device-side bounded wait ran out             */
    RA_ERR_WORKSPACE = 6,    /* caller workspace too small or misaligned       */
    RA_ERR_SCRATCH_LIMIT = 7 /* problem needs more than the library's fixed
                                scratch array (ra_forward_noalloc only)        */
} ra_status;

typedef enum { RA_LAYOUT_CONTIGUOUS = 0, RA_LAYOUT_STRIPED = 1 } ra_layout;

/* RA_MODE_FUSED: one persistent launch walks, for every query tile, the key
 *   blocks in ring order and keeps the running softmax on chip (problems of
 *   2^19 key/value rows and more: one such launch per (batch, kv head), the
 *   heads being independent; the results are those of a single launch).
 * RA_MODE_PER_STEP: one launch per ring step s writes that step's partial
 *   (out_s, lse_s) for every rank, then ra_merge-style merging folds it into
 *   the running result, as each ring device would after receiving a block.
 * RA_MODE_RING: RA_MODE_PER_STEP with the key/value rotation made explicit:
 *   before step s every rank's block is copied (by the copy engine, on a
 *   second stream of the library's own) from where the previous rank held it
 *   into a double-buffered workspace copy, and step s reads that copy (the
 *   N sends of a step land at the blocks' own offsets, so they are issued as
 *   one copy of k and one of v).  The
 *   copy for step s + 1 overlaps the compute of step s, as the send of the
 *   block to the next device overlaps the block computation on a real ring
 *   ("Ring Attention" page, section "Halka Dikkati Nasil Calisir": each device
 *   passes its key/value block to the next one while it computes).  Same
 *   result as RA_MODE_PER_STEP, bit for bit. */
typedef enum { RA_MODE_FUSED = 0, RA_MODE_PER_STEP = 1, RA_MODE_RING = 2 } ra_mode;

typedef enum { RA_DTYPE_BF16 = 0, RA_DTYPE_F32 = 1 } ra_dtype;

/*
 * ra_forward - ring-ordered blockwise exact attention, bf16 in, bf16 out.
 * Source: "Ring Attention" page, section "Halka Dikkati Nasil Calisir" (ring
 * schedule, running-softmax merge, causal block skipping, striping).
 * q, k, v, out: bf16 (raw 16-bit storage); lse: fp32.  Computes in fp32 with
 * bf16 operands on the tensor cores; out is rounded to bf16 (nearest even).
 * Supported: d in {64, 128}; any block length L >= 1.  Uses RA_MODE_FUSED and
 * allocates its scratch stream-ordered (cudaMallocAsync on `stream`).
 * Small problems, whose work units (pairs of 128-row query tiles) cannot
 * fill half the current device's SMs, have every unit's walk over its key
 * tiles (in ring order) cut into up to SMs / units pieces (at most 16)
 * computed by different CTAs as independent fp32 partials, which a second
 * kernel folds by the running-softmax merge into out and lse (the ring's own
 * decomposition: each block's partial result is merged into the running one,
 * "Ring Attention" page, section "Halka Dikkati Nasil Calisir").
 * Returns RA_ERR_INVALID_ARG for B, H, Hkv, S, n_blocks < 1, H % Hkv != 0,
 * S % n_blocks != 0, layout not in ra_layout, null, misaligned or overlapping
 * pointers; RA_ERR_UNSUPPORTED for other d.
 */
ra_status ra_forward(const void *q, const void *k, const void *v, void *out, float *lse,
                     int B, int H, int Hkv, int S, int d, int n_blocks,
                     int layout, int causal, ra_stream_t stream);

/*
 * ra_forward_f32 - the same computation for fp32 tensors, fp32 arithmetic
 * throughout (no TF32, no reduced-precision operands), for exact checks such
 * as the pages' 4-device, block-8, dim-16 simulation ("Ring Attention" page,
 * section "Halka Dikkati Nasil Calisir", the four-device example).
 * Supported: 1 <= d <= 256, any L >= 1.  Same error rules as ra_forward.
 */
ra_status ra_forward_f32(const float *q, const float *k, const float *v, float *out,
                         float *lse, int B, int H, int Hkv, int S, int d, int n_blocks,
                         int layout, int causal, ra_stream_t stream);

/*
 * ra_workspace_bytes - bytes of scratch ra_forward_ws needs for this problem
 * (striped copies of q, k, v, out and lse; per-step running and partial
 * results; for RA_MODE_RING two rotating copies of k and v; for small bf16
 * fused problems whose walks are split (see ra_forward), the pieces' fp32
 * partials of out and lse).  0 when none is needed (bf16 contiguous fused
 * without a split).  The split depends on the SM count of the CURRENT
 * device, so ask with the device current that ra_forward_ws will run on.
 * dtype is a ra_dtype, mode a ra_mode.  Returns 0 for an invalid request.
 */
size_t ra_workspace_bytes(int B, int H, int Hkv, int S, int d, int n_blocks, int layout,
                          int causal, int mode, int dtype);

/*
 * ra_forward_ws - ra_forward / ra_forward_f32 with an explicit mode and a
 * caller-owned device workspace `ws` of `ws_bytes` bytes (256-byte aligned,
 * at least ra_workspace_bytes(...)); no per-call allocation.  dtype selects the
 * tensor type (RA_DTYPE_BF16: q, k, v, out bf16; RA_DTYPE_F32: all fp32).
 * RA_ERR_WORKSPACE if ws is null, misaligned or too small.  Calls sharing one
 * workspace must be ordered on the GPU (same stream or events).  The ring
 * schedule needs no memory: the kernel enumerates its work units itself.
 */
ra_status ra_forward_ws(const void *q, const void *k, const void *v, void *out, float *lse,
                        int B, int H, int Hkv, int S, int d, int n_blocks, int layout,
                        int causal, int dtype, int mode, void *ws, size_t ws_bytes,
                        ra_stream_t stream);

/*
 * ra_forward_rank_major - ra_forward_ws for tensors already stored in the
 * layout's rank-major order: rank 0's L tokens, then rank 1's, and so on
 * (for RA_LAYOUT_STRIPED, row p = r L + a holds natural token a N + r; for
 * RA_LAYOUT_CONTIGUOUS this is the natural order).  q, k, v, out and lse all
 * use that order and no permutation is launched, as for a model that keeps
 * its activations striped from embedding to output.  Same arguments, types
 * and error rules as ra_forward_ws; the workspace is needed only for
 * RA_MODE_PER_STEP and RA_MODE_RING (ra_workspace_bytes of the contiguous
 * layout).
 * Source: "Ring Attention" page, section "Halka Dikkati Nasil Calisir".
 */
ra_status ra_forward_rank_major(const void *q, const void *k, const void *v, void *out,
                                float *lse, int B, int H, int Hkv, int S, int d, int n_blocks,
                                int layout, int causal, int dtype, int mode, void *ws,
                                size_t ws_bytes, ra_stream_t stream);

/*
 * ra_forward_block - the work of one device of the ring at one ring step:
 * the partial attention of query block `rank` against key/value block
 * j = (rank - step) mod n_blocks, the block that device holds after `step`
 * rotations ("Ring Attention" page, section "Halka Dikkati Nasil Calisir":
 * each device computes attention for its local query block against the key
 * and value block it currently holds, then passes that block on).
 *   q, k, v   device tensors in the layout's rank-major order (as for
 *             ra_forward_rank_major), dtype RA_DTYPE_BF16 or RA_DTYPE_F32;
 *   out_s     fp32 [B,H,S,d], lse_s fp32 [B,H,S] (natural log): only the rows
 *             of block `rank` (rows rank*L .. rank*L + L - 1 of every head)
 *             are written, with the partial normalised by its own sum; rows
 *             that see no key at this step get out 0 and lse -inf (the whole
 *             block when it is masked, e.g. contiguous causal with step > rank).
 * Merging the n_blocks partials of a rank with ra_merge, in any order, gives
 * its rows of ra_forward's result (up to rounding).  Caller-owned buffers,
 * 16-byte aligned; no allocation; asynchronous on `stream`.  Errors:
 * RA_ERR_INVALID_ARG (bad sizes, rank or step outside [0, n_blocks), null,
 * misaligned or overlapping buffers), RA_ERR_UNSUPPORTED (d % 4 != 0, or a
 * bf16 head dimension other than 64 / 128), RA_ERR_CUDA.  Nothing is launched
 * on an error.
 */
ra_status ra_forward_block(const void *q, const void *k, const void *v, float *out_s,
                           float *lse_s, int B, int H, int Hkv, int S, int d, int n_blocks,
                           int layout, int causal, int dtype, int rank, int step,
                           ra_stream_t stream);

/*
 * ra_all_to_all - the all-to-all exchange of DeepSpeed Ulysses, the
 * alternative to the ring named on the "Ring Attention" page (section on
 * ring attention and other kinds of parallelism: every device receives all
 * tokens of a subset of the attention heads), emulated as one relayout of
 * device-major buffers.  With L = S / n_dev and Hg = Hn / n_dev:
 *   sequence-sharded [n_dev][B][Hn][L][d]: device i holds tokens [iL, iL+L)
 *     of every head;
 *   head-sharded     [n_dev][B][Hg][S][d]: device g holds all tokens of
 *     heads [g Hg, g Hg + Hg).
 * inverse = 0 maps sequence-sharded src to head-sharded dst, 1 the reverse.
 * Rows of d elements of elem_bytes bytes (1, 2, 4 or 8) are copied bit-exact.
 * Device pointers, caller-owned, not overlapping; 16-byte aligned when
 * d * elem_bytes % 16 == 0, else 4-byte aligned when it is a multiple of 4.
 * Errors: RA_ERR_INVALID_ARG (sizes, S % n_dev, Hn % n_dev, alignment,
 * overlap), RA_ERR_CUDA.  Asynchronous on `stream`.
 */
ra_status ra_all_to_all(const void *src, void *dst, int B, int Hn, int S, int d,
                        int elem_bytes, int n_dev, int inverse, ra_stream_t stream);

/*
 * ra_ulysses_workspace_bytes - scratch ra_forward_ulysses needs (head-sharded
 * q, k, v and out in the input dtype, lse fp32); 0 for an invalid or
 * unsupported request.
 */
size_t ra_ulysses_workspace_bytes(int B, int H, int Hkv, int S, int d, int n_dev,
                                  int causal, int dtype);

/*
 * ra_forward_ulysses - exact attention over n_dev emulated devices the
 * Ulysses way: all-to-all q, k, v from sequence shards to head shards,
 * attention of every device over the whole sequence for its heads (causal
 * mask on natural positions), all-to-all out and lse back.
 *   q [n_dev][B][H][L][d], k, v [n_dev][B][Hkv][L][d]: sequence shards
 *     (device i holds tokens [iL, iL + L)), dtype RA_DTYPE_BF16 or F32;
 *   out (q's shape and dtype), lse fp32 [n_dev][B][H][L], natural log.
 * The result equals ra_forward's on the same tokens (the shards laid side by
 * side).  Requires H % n_dev == 0 and Hkv % n_dev == 0 (a device holds whole
 * kv heads, so the kv head count bounds the devices): RA_ERR_UNSUPPORTED
 * otherwise; the tensor-core path needs d in {64, 128}.  ws: device scratch
 * of ra_ulysses_workspace_bytes bytes, 256-byte aligned (RA_ERR_WORKSPACE).
 * Other errors as ra_forward.  Asynchronous on `stream`; no allocation.
 */
ra_status ra_forward_ulysses(const void *q, const void *k, const void *v, void *out,
                             float *lse, int B, int H, int Hkv, int S, int d, int n_dev,
                             int causal, int dtype, void *ws, size_t ws_bytes,
                             ra_stream_t stream);

/*
 * ra_backward - gradients of ring attention: dq, dk, dv of the loss
 * sum(dout * out) where (out, lse) = ra_forward(q, k, v, ...).  The pages
 * train through the ring ("Context Parallelism" glossary page, section
 * "Pratik Kullanim ve Odunlesimler": the example calls backward on the
 * attention output); the ring is exact, so these are the gradients of exact
 * attention, computed blockwise in ring order from the saved lse:
 *   P = exp(q k^T / sqrt(d) - lse), dS = P * (dout v^T - rowsum(dout * out)),
 *   dv = P^T dout, dk = dS^T q / sqrt(d), dq = dS k / sqrt(d)
 * (GQA: dk, dv summed over each kv head's query heads).  Key/value block j's
 * gradients accumulate over query blocks i = (j + s) mod N, s = 0..N-1, the
 * order in which they would travel around the ring.
 *   q, out, dout, dq: bf16 [B,H,S,d]; k, v, dk, dv: bf16 [B,Hkv,S,d];
 *   lse: fp32 [B,H,S] as ra_forward wrote it; natural token order; layout,
 *   causal and n_blocks as given to ra_forward.
 * d in {64, 128} (RA_ERR_UNSUPPORTED otherwise); any L >= 1.  Device
 * pointers, 16-byte aligned, caller-owned; dq, dk, dv must not overlap any
 * other argument (RA_ERR_INVALID_ARG).  Scratch is allocated stream-ordered
 * (RA_ERR_NO_MEMORY); asynchronous on `stream`; a device-side timeout is
 * reported by ra_check.
 */
ra_status ra_backward(const void *q, const void *k, const void *v, const void *out,
                      const float *lse, const void *dout, void *dq, void *dk, void *dv,
                      int B, int H, int Hkv, int S, int d, int n_blocks, int layout,
                      int causal, ra_stream_t stream);

/* ra_backward_f32 - ra_backward with every tensor in fp32 (exact SIMT path,
 * no tensor cores, no bf16 rounding; any 1 <= d <= 256), for checks at fp32
 * precision.  Same arguments and error rules as ra_backward. */
ra_status ra_backward_f32(const float *q, const float *k, const float *v, const float *out,
                          const float *lse, const float *dout, float *dq, float *dk, float *dv,
                          int B, int H, int Hkv, int S, int d, int n_blocks, int layout,
                          int causal, ra_stream_t stream);

/* ra_backward_workspace_bytes - scratch ra_backward_ws needs (delta per row;
 * for the striped layout, rank-major copies of the inputs and gradients);
 * 0 for an invalid request. */
size_t ra_backward_workspace_bytes(int B, int H, int Hkv, int S, int d, int n_blocks,
                                   int layout, int causal);

/* ra_backward_ws - ra_backward with a caller-owned workspace (256-byte
 * aligned, at least ra_backward_workspace_bytes; RA_ERR_WORKSPACE). */
ra_status ra_backward_ws(const void *q, const void *k, const void *v, const void *out,
                         const float *lse, const void *dout, void *dq, void *dk, void *dv,
                         int B, int H, int Hkv, int S, int d, int n_blocks, int layout,
                         int causal, void *ws, size_t ws_bytes, ra_stream_t stream);

/*
 * ra_forward_noalloc - ra_forward for callers that cannot allocate device
 * memory.  No counterpart on the pages: this is a deployment variant of the
 * same computation, with the same arguments, result and error rules as
 * ra_forward (bf16, fused ring, natural token order).  It enqueues the same
 * kernels as ra_forward, including the forward kernel variant chosen with
 * ra_set_kernel_variant, so its out and lse equal ra_forward's bit for bit.
 *
 * Who needs it: code that runs under a memory manager that owns every byte
 * of device memory (a framework's caching allocator or an inference server
 * that reserves its whole budget at start-up and forbids allocation after
 * that), and latency-critical loops that must not meet an allocation-time
 * synchronisation or an out-of-memory failure half way through.  ra_forward
 * gets its striped scratch with cudaMallocAsync; this entry point does not.
 *
 * Its scratch is exactly the workspace ra_forward would allocate
 * (ra_workspace_bytes with RA_MODE_FUSED: for RA_LAYOUT_STRIPED the striped
 * copies of q, k, v, out and lse, 2 (B H + 2 B Hkv) S d + 4 B H S bytes; for
 * small problems whose walks are split, the pieces' fp32 partials; large
 * contiguous problems need none).  It
 * lives in one fixed array of RA_NOALLOC_SCRATCH_BYTES (64 MiB) that is part
 * of the library's device image: every GPU that loads the library holds it
 * until the process exits.  A problem whose scratch would not fit returns
 * RA_ERR_SCRATCH_LIMIT and enqueues nothing.  Nothing in the array has to
 * start at zero: every byte a call reads was written earlier by the same call.
 *
 * All calls on a device share the one array and it keeps the last call's
 * contents, so calls that can overlap on the GPU (different streams without
 * ordering between them) race: order them on one stream or with events.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Calls no cudaMalloc, cudaMallocAsync, cudaFree
 * or other allocating routine.
 */
#define RA_NOALLOC_SCRATCH_BYTES (64ull << 20)
ra_status ra_forward_noalloc(const void *q, const void *k, const void *v, void *out, float *lse,
                             int B, int H, int Hkv, int S, int d, int n_blocks, int layout,
                             int causal, ra_stream_t stream);

/*
 * ra_permute - move the sequence axis between natural and striped order.
 * Source: "Ring Attention" page, section "Halka Dikkati Nasil Calisir"
 * (striped attention).  With L = S / n_blocks, striped row p = r L + a holds
 * natural token t = a n_blocks + r.  src and dst are [B * Hn, S, row] with
 * row = d * elem_bytes bytes; inverse = 0 gathers natural -> striped
 * (dst[p] = src[t(p)]), inverse = 1 scatters back (dst[t(p)] = src[p]).
 * Bit-exact copy; elem_bytes in {1, 2, 4, 8}; src and dst must not overlap.
 */
ra_status ra_permute(const void *src, void *dst, int B, int Hn, int S, int d, int elem_bytes,
                     int n_blocks, int inverse, ra_stream_t stream);

/*
 * ra_merge - fold one ring step's partial result into the running one.
 * Source: "Ring Attention" page, section "Halka Dikkati Nasil Calisir"
 * (partial results combined with the running softmax of flash attention).
 * Per row: lse = ln(e^lse_run + e^lse_s);
 *          out_run = e^(lse_run - lse) out_run + e^(lse_s - lse) out_s;
 *          lse_run = lse.
 * A side with lse = -inf (no visible key) contributes nothing; if both are
 * -inf the row stays out 0, lse -inf.  out_run, out_s: fp32 [rows, d];
 * lse_run, lse_s: fp32 [rows].  1 <= d <= 256, d % 4 == 0 (16-byte vectors).
 */
ra_status ra_merge(float *out_run, float *lse_run, const float *out_s, const float *lse_s,
                   long long rows, int d, ra_stream_t stream);

/*
 * ra_check - synchronise `stream`, then read and clear the device error word
 * that bounded waits set.  RA_OK, RA_ERR_TIMEOUT, or RA_ERR_CUDA when the
 * stream reported a CUDA error.
 */
ra_status ra_check(ra_stream_t stream);

/* Human-readable name of a ra_status value; never NULL. */
const char *ra_status_string(int status);

/*
 * ra_set_kernel_variant - choose the bf16 tensor-core kernel for the calls
 * that follow (process-wide): 0 = automatic (the library's default choice,
 * currently variant 3), 1 = one CTA per SM computing two 128-row query
 * tiles, 3 = variant 1 launched as clusters of two CTAs whose units walk the
 * same key/value tiles and share each tile load by TMA multicast (when every
 * kv head serves a multiple of four query heads; otherwise variant 1).  Both
 * compute the same result bit for bit (same ring order, same running
 * softmax); they differ in how work maps onto SMs.  2 (a CTA-pair kernel in
 * earlier versions) is no longer a valid value.  Returns the previous
 * setting, or -1 for an invalid value (nothing changes).
 * Source: "Ring Attention" page, section "Halka Dikkati Nasil Calisir" (the
 * per-device blockwise kernel the ring runs).
 */
int ra_set_kernel_variant(int variant);

/*
 * ra_set_wait_timeout_ns - bound, in nanoseconds of the GPU's global timer,
 * on every mbarrier wait inside the tensor-core kernel launched after this
 * call (0 restores the default of 4 s).  A wait that runs out records
 * RA_ERR_TIMEOUT in the device error word, the kernel drains its in-flight
 * copies and MMAs, frees tensor memory and returns; ra_check() reports it.
 * Source: the "Context Parallelism" page of freenetmedia.pl, section "Typowe
 * bledy i pulapki": synchronisation mistakes give wrong results or hangs; here
 * a broken handshake turns into an error status instead of a hang.
 */
void ra_set_wait_timeout_ns(unsigned long long timeout_ns);

/*
 * ra_wait_probe - launch a one-thread kernel that waits, with the same
 * bounded wait the tensor-core kernel uses, on an mbarrier that nothing ever
 * arrives at, for at most timeout_ns (1 ms .. 10 s).  The wait runs out, the
 * kernel records RA_ERR_TIMEOUT in the device error word and returns, and the
 * next ra_check() reports RA_ERR_TIMEOUT; the context stays usable.  Exists to
 * test the failure path without faulting or hanging a GPU.
 * RA_ERR_INVALID_ARG for a timeout outside the range.  Same source as above.
 */
ra_status ra_wait_probe(unsigned long long timeout_ns, ra_stream_t stream);

/* Number of CUDA kernels this library has launched in the process so far
 * (all entry points, all devices).  Lets a caller count the launches inside
 * a timed region. */
unsigned long long ra_launch_count(void);

/* Library version string, e.g. "ra 0.1.0 sm_103a". */
const char *ra_version(void);

/*
 * ra_schedule_stats - host-only view of the ring-step scheduler, no GPU
 * needed.  For layout, causal, n_blocks and block length L, writes for every
 * (rank i, step s) the number of visible (query, key) pairs that rank i
 * computes at step s into pairs[i * n_blocks + s], and the number of
 * 128 x 128 tiles it launches into tiles[i * n_blocks + s] (either array may
 * be NULL).  Returns the total number of visible pairs, or -1 on bad input.
 */
long long ra_schedule_stats(int layout, int causal, int n_blocks, int L,
                            long long *pairs, long long *tiles);

/*
 * ra_schedule_units - host-only view of the tensor-core kernel's work units
 * for ring steps [s_begin, s_end) (all steps, or a single step), in the order
 * the kernel deals them to CTAs (heaviest first).  Unit u is written to
 * units[8u .. 8u + 7] as {bh0, ta0, bh1, ta1, rank, cost, tile1_valid, 0}: two
 * 128-row query tiles (batch*H + head, tile index within the rank's block) of
 * rank `rank` that share a kv head, and the number of 128-key tiles they visit.
 * Writes at most `capacity` units (units may be NULL); returns the total
 * count, or -1 on bad input.  Source: as for ra_schedule_stats.
 */
long long ra_schedule_units(int B, int H, int Hkv, int S, int n_blocks, int layout, int causal,
                            int s_begin, int s_end, int *units, long long capacity);

/*
 * ra_schedule_block_units - host-only view of the units ra_forward_block
 * launches for (rank, step): the same enumeration and record format as
 * ra_schedule_units, restricted to query block `rank` at ring step `step`.
 * Returns the count (0 when the block is fully masked), or -1 on bad input.
 * Source: as for ra_schedule_stats.
 */
long long ra_schedule_block_units(int B, int H, int Hkv, int S, int n_blocks, int layout, int causal,
                                  int rank, int step, int *units, long long capacity);

/*
 * ra_backward_tile_pairs - host-only view of the backward pass's work: the
 * (query tile, key tile) pairs each kernel visits, unit by unit, in order.
 * which = 0: the dK/dV kernel (one unit per 128-key tile; query blocks in the
 * order the key block travels the ring, i = (j + s) mod N); which = 1: the dQ
 * kernel (one unit per 128-row query tile; key blocks j = (i - s) mod N).
 * Pair n is written to pairs[8n .. 8n + 7] as {unit, batch*H + query head,
 * query block i, query tile ta, key block j, key tile tb, position within the
 * unit, 0}.  Writes at most `capacity` pairs (pairs may be NULL); returns the
 * total, or -1 on bad input.  Source: as for ra_backward.
 */
long long ra_backward_tile_pairs(int B, int H, int Hkv, int S, int n_blocks, int layout,
                                 int causal, int which, int *pairs, long long capacity);

#ifdef __cplusplus
}
#endif

#endif /* RA_H_ */
