/*
 * ra.h - C ABI of the GB300 (sm_103a) exact ring-attention library.
 *
 * What is computed.  Ring attention as the tutorial "06 - Sequence / Context
 * Parallelism" (section 4, "Ring Attention - the core algorithm") gives it:
 * every rank i keeps its queries Q_i; the K/V blocks circulate round a ring;
 * at each step rank i attends Q_i to the block it currently holds and folds
 * the partial result into an online-softmax state (out_i, m_i, l_i), which
 * is rescaled whenever a block raises the running maximum (the quiz
 * "Sequence Parallelism and Ring Attention", questions 3 and 7); after the
 * last step out_i / l_i is the exact softmax attention.  The sequence is
 * split over c ranks contiguously (tutorial section 1) or zig-zag (plate
 * "Splitting the Sequence": 2c chunks, rank k owns chunks k and 2c-1-k), and
 * the causal mask compares global token positions (plate, and quiz
 * questions 6 and 8).  In this library all c ranks are virtual and run on
 * one GPU: the ring pass is a change of which block a rank reads, so no
 * bytes move and no collective is called.
 *
 * Conventions shared by every entry point.
 *  - Tensors are row-major and contiguous:  q [B, Sq, Hq, D];  k, v
 *    [B, Sk, Hkv, D]; out [B, S, Hq, D]; lse [B, Hq, S].  Query head h reads
 *    key/value head h / (Hq / Hkv).
 *  - The online-softmax state of a query row is (o, m, l): o [B, S, Hq, D]
 *    float32 is the unnormalised accumulator; m, l [B, Hq, S] float32.  m is
 *    the running maximum of  scale * log2(e) * q.k  over the keys seen so far
 *    (base-2 units), and l = sum over those keys of 2^(scale*log2(e)*q.k - m).
 *    A row that has seen no key has o = 0, m = -inf, l = 0.  The natural log
 *    sum exp is  lse = ln(2) * (m + log2(l)).
 *  - The causal mask is inclusive: query position p sees key position p'
 *    when p' <= p.
 *  - The caller owns every buffer.  The library never allocates device or
 *    pinned memory (it only registers one page of its own host memory, the
 *    error mirror below); where it needs scratch the caller passes a workspace
 *    of the size the matching *_workspace_size function returns.
 *  - Device pointers must be 16-byte aligned.  Positions are int32.
 *  - Calls are asynchronous and stream-ordered on the given stream (NULL is
 *    the legacy default stream), except where noted.  Arguments are checked
 *    on the host before anything is launched; on a bad argument the call
 *    returns RA_ERR_INVALID or RA_ERR_UNSUPPORTED and launches nothing.
 *  - Every device-side wait in the kernels is bounded.  A wait that runs out
 *    sets a device error word and the kernel returns early; ra_device_error()
 *    reports it as RA_ERR_TIMEOUT and clears it.  Until it is cleared, kernels
 *    launched on that device return without computing anything, so every
 *    entry point that launches work first reads a host-mapped mirror of the
 *    word (no synchronisation) and, if an error is pending, returns
 *    RA_ERR_TIMEOUT without launching.  Work already enqueued when a wait runs
 *    out is not recalled: it finishes as a no-op, and only ra_device_error()
 *    (or a call with a report) tells.  The mirror is one page of the
 *    library's own host memory, registered with the CUDA driver on the first
 *    call in a process; each device's first call also publishes its address
 *    to the device with a synchronous copy, so make that first call before
 *    any stream capture.
 *  - Nothing here is thread-safe across concurrent calls that share a
 *    workspace.
 */
#ifndef RA_H_
#define RA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL selects the default stream. */
typedef struct CUstream_st* ra_stream_t;

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID = -1,      /* an argument is out of range, null or misaligned */
  RA_ERR_UNSUPPORTED = -2,  /* valid request the library does not implement  */
  RA_ERR_CUDA = -3,         /* a CUDA runtime/driver call failed              */
  RA_ERR_TIMEOUT = -4,      /* a bounded device-side wait ran out             */
  RA_ERR_WORKSPACE = -5     /* workspace missing or smaller than required     */
} ra_status;

typedef enum { RA_BF16 = 0, RA_F32 = 1 } ra_dtype;

/* Shard layouts.  Contiguous: rank k owns tokens [k*S/c, (k+1)*S/c)
 * (tutorial, section 1).  Zig-zag: the sequence is cut into 2c chunks and
 * rank k (counted from 0) owns chunks k and 2c-1-k, in increasing position
 * (plate "Splitting the Sequence").  Striped: round robin, rank k owns the
 * tokens whose position is k mod c, in increasing position (tutorial
 * section 5, "striped / zigzag attention"). */
typedef enum { RA_CONTIGUOUS = 0, RA_ZIGZAG = 1, RA_STRIPED = 2 } ra_layout;

/* How ra_ring_forward executes the ring.
 * RA_MODE_FUSED: one launch; each (rank, query tile, head) block walks the
 *   ring steps t = 0..c-1 in order, keeping its state on chip, and writes
 *   the normalised output at the end.
 * RA_MODE_PER_STEP: one launch per ring step t over all ranks; the state
 *   lives in the workspace between steps; a final normalisation pass.
 * Both visit the same tiles in the same order with the same arithmetic and
 * give bitwise identical results.
 * RA_MODE_ALLGATHER: the all-gather form of context parallelism the plate
 *   "Splitting the Sequence" reports for Llama 3: every rank gathers all c
 *   shards and attends its queries to them in one step (no ring; work counts
 *   are reported at step 0).  Same result up to rounding. */
typedef enum { RA_MODE_FUSED = 0, RA_MODE_PER_STEP = 1, RA_MODE_ALLGATHER = 2 } ra_mode;

typedef struct {
  int32_t B;       /* batch                                   */
  int32_t Sq;      /* query rows (ring: S)                    */
  int32_t Sk;      /* key/value rows (ring: S, must equal Sq) */
  int32_t Hq;      /* query heads                             */
  int32_t Hkv;     /* key/value heads, Hq % Hkv == 0          */
  int32_t D;       /* head dim: 64 or 128                     */
  int32_t dtype;   /* ra_dtype of q, k, v (and of out)        */
  float scale;     /* softmax scale applied to q.k (finite)   */
} ra_shape;

/* Work of one (rank, ring step), summed over batch and query heads.  Tiles
 * are 128 query rows x 128 keys of the two shards' local order (the last
 * tile of a shard may be short).  A tile pair is skipped when the causal
 * mask hides all of it, full when it hides none of it, partial otherwise;
 * pairs counts the visible (query, key) pairs.  (Tutorial section 10
 * exercise B asks for per-rank compute instrumentation.) */
typedef struct {
  uint64_t pairs;
  uint64_t tiles_full;
  uint64_t tiles_partial;
  uint64_t tiles_skipped;
} ra_work;

/* Host-side report of one ring_forward call (all pointers host memory). */
typedef struct {
  int32_t c;
  ra_work* per_rank_step;      /* [c*c], index rank*c + step, or NULL; counted on the GPU */
  int32_t* schedule;           /* [c*c], index step*c + rank = source rank, or NULL */
  double imbalance_pairs;      /* max over ranks / mean of the per-rank pairs */
  double imbalance_tiles;      /* same with executed (full + partial) tiles  */
  uint64_t ring_kv_bytes;      /* tutorial section 4: S*Hkv*D*2*bytes*B per layer and device */
  uint64_t ring_kv_bytes_sent; /* plate form: (c-1)/c of that (own block not sent) */
  uint64_t algorithmic_flop;   /* 4*B*Hq*D*(visible pairs)                     */
} ra_report;

/* ---------------------------------------------------------------------- */

/* Human-readable name of a status code.  Never NULL. */
const char* ra_status_string(int status);

/* Library version string, e.g. "ra-gb300 0.1 sm_103a". */
const char* ra_version(void);

/* Text of the last CUDA failure or device timeout seen by a call on this
 * host thread ("" if none): the failing step, the CUDA error name and its
 * description.  Owned by the library; valid until the next call. */
const char* ra_last_error(void);

/* Initialise an online-softmax state for Sq rows: o = 0, m = -inf, l = 0
 * (tutorial section 4, "out_i, m_i, l_i = initialize()").  o: device
 * [B, Sq, Hq, D] float32; m, l: device [B, Hq, Sq] float32. */
ra_status ra_state_init(ra_shape shp, float* o, float* m, float* l, ra_stream_t stream);

/* One ring step of one rank (tutorial section 4, "compute partial
 * attention: Q_i against the K,V currently held" and "update out_i, m_i,
 * l_i with online softmax rescaling"): attends q to (k, v) and folds the
 * result into the state (o, m, l) in place.
 *   q      device [B, Sq, Hq, D] in shp.dtype
 *   k, v   device [B, Sk, Hkv, D] in shp.dtype
 *   q_pos  device int32 [Sq], global token positions of the query rows
 *   k_pos  device int32 [Sk], global token positions of the key rows
 *   causal nonzero: key position p' is visible to query position p iff p' <= p
 *   o,m,l  device state as described above, read and written
 *   work   device ra_work[1] to which this call's counts are ADDED, or NULL
 * bf16 runs on the tensor cores (fp32 accumulation, P rounded to bf16 before
 * the P.V product); f32 runs in exact fp32 on the CUDA cores.  Sq or Sk = 0
 * (or B = 0) is a no-op. */
ra_status ra_block_attn(const void* q, const void* k, const void* v,
                        const int32_t* q_pos, const int32_t* k_pos, int causal,
                        ra_shape shp, float* o, float* m, float* l,
                        ra_work* work, ra_stream_t stream);

/* Merge P partial states over disjoint key sets and normalise (tutorial
 * section 4's final out_i / l_i; section 7's gather of partial results for
 * decode):  M = max_p m_p, L = sum_p l_p 2^(m_p - M),
 * out = (sum_p o_p 2^(m_p - M)) / L,  lse = ln(2) * (M + log2 L).
 *   outs, ms, ls  HOST arrays of P device pointers, each state laid out as
 *                 above for shp.Sq rows; 1 <= P <= RA_MERGE_MAX_PARTIALS
 *   out           device [B, Sq, Hq, D] in shp.dtype (bf16 or f32)
 *   lse           device [B, Hq, Sq] float32, or NULL
 * Rows with L = 0 get out = 0 and lse = -inf. */
#define RA_MERGE_MAX_PARTIALS 64
ra_status ra_lse_merge(int P, const float* const* outs, const float* const* ms,
                       const float* const* ls, ra_shape shp, void* out, float* lse,
                       ra_stream_t stream);

/* Bytes of device workspace ra_ring_forward / ra_ring_prepare /
 * ra_ring_attend need for this problem (shp.Sq = shp.Sk = S).  Returns 0 for
 * an invalid request. */
size_t ra_ring_forward_workspace_size(ra_shape shp, int c, int layout, int mode);

/* Full ring attention over c virtual ranks on this GPU:
 * ra_ring_prepare followed by ra_ring_attend.
 *   q, k, v    device, natural token order, [B, S, Hq|Hkv, D] in shp.dtype
 *   c          ranks, 1 <= c; S % c == 0 (contiguous, striped) or S % (2c) == 0
 *              (zig-zag)
 *   out_dtype  element type of out: shp.dtype, or RA_F32 to receive the
 *              float32 result before its rounding to bf16 (the bf16 output is
 *              exactly that result rounded to nearest even)
 *   out        device [B, S, Hq, D] in out_dtype, natural order
 *   lse        device [B, Hq, S] float32 natural log, or NULL
 *   workspace  device, >= ra_ring_forward_workspace_size(...) bytes
 *   report     host, or NULL.  When non-NULL the call synchronises the
 *              stream, fills the report (work counted on the GPU, schedule
 *              and derived quantities from the host scheduler) and returns
 *              RA_ERR_TIMEOUT if a device wait ran out. */
ra_status ra_ring_forward(const void* q, const void* k, const void* v, ra_shape shp,
                          int c, int layout, int causal, int mode, int out_dtype,
                          void* out, float* lse, void* workspace, size_t ws_bytes,
                          ra_report* report, ra_stream_t stream);

/* First half of ra_ring_forward: copies q, k, v into rank-major shard order
 * in the workspace (each rank's shard contiguous, as on a real ring), writes
 * the global position of every shard row, and orders the query blocks
 * heaviest-first for causal calls (largest position first).  Bandwidth-bound. */
ra_status ra_ring_prepare(const void* q, const void* k, const void* v, ra_shape shp,
                          int c, int layout, void* workspace, size_t ws_bytes,
                          ra_stream_t stream);

/* Second half of ra_ring_forward: the ring steps and the normalisation,
 * reading the shards ra_ring_prepare left in the same workspace.
 * count_work nonzero zeroes and fills the per-(rank, step) counters kept in
 * the workspace (read them with ra_ring_read_work). */
ra_status ra_ring_attend(ra_shape shp, int c, int layout, int causal, int mode, int out_dtype,
                         void* out, float* lse, void* workspace, size_t ws_bytes,
                         int count_work, ra_stream_t stream);

/* Copy the c*c per-(rank, step) counters of the last ra_ring_attend with
 * count_work set into host memory (synchronises the stream). */
ra_status ra_ring_read_work(ra_shape shp, int c, int layout, int mode, const void* workspace,
                            size_t ws_bytes, ra_work* host_per_rank_step, ra_stream_t stream);

/* ra_ring_forward with HOST inputs and outputs: copies q, k, v from host
 * memory (pinned for overlap), runs the ring, copies out and lse back, all
 * on `stream`; returns after the stream has finished.  The device buffers
 * for q, k, v, out and lse are carved from the workspace, whose size is
 * ra_ring_forward_hostio_workspace_size().  When out_host (or lse_host) is
 * pinned memory mapped into the device's address space, the kernels write it
 * directly over the CPU-GPU link while they run; otherwise the result is
 * copied back after the attention.  The fused bf16 ring with pinned q and a
 * mapped out in the contiguous or zig-zag layout is pipelined: K, V and the
 * positions are packed first, each rank's query rows are copied on an
 * internal copy stream, and each rank's query blocks run as a launch of their
 * own once those rows have landed, alternating between `stream` and an
 * internal stream; the output goes to device memory and each rank's rows are
 * copied to out_host on another internal stream once its launch is done (all
 * joined back into `stream`; the internal streams and events are created on
 * first use per device and kept). */
size_t ra_ring_forward_hostio_workspace_size(ra_shape shp, int c, int layout, int mode,
                                             int out_dtype);
ra_status ra_ring_forward_hostio(const void* q_host, const void* k_host, const void* v_host,
                                 ra_shape shp, int c, int layout, int causal, int mode,
                                 int out_dtype, void* out_host, float* lse_host, void* workspace,
                                 size_t ws_bytes, ra_stream_t stream);

/* ra_ring_forward for callers that cannot allocate device memory.  The
 * pages have no counterpart: this is a deployment convenience of this
 * library.  Some callers cannot call cudaMalloc where they run attention
 * (cudaMalloc may synchronise the device and may fail part-way through a
 * job; some host frameworks own all device memory).  This entry point takes
 * no workspace: its scratch is a fixed array of RA_NOALLOC_SCRATCH_BYTES
 * (64 MiB) that the library reserves on every GPU where it is used, until the
 * process exits.  It allocates nothing itself (no cudaMalloc, cudaFree or
 * allocating library call).
 *   Arguments and results as ra_ring_forward (no report).
 *   Problems whose workspace (ra_ring_forward_workspace_size) exceeds the
 *   scratch are rejected with RA_ERR_WORKSPACE before anything is launched.
 *   The first call on a device looks up the scratch's device address; make
 *   that first call before any stream capture.
 *   All calls share the one scratch array: calls that overlap on the GPU
 *   (other streams, other host threads on the same device) race. */
#define RA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
ra_status ra_ring_forward_noalloc(const void* q, const void* k, const void* v, ra_shape shp,
                                  int c, int layout, int causal, int mode, int out_dtype,
                                  void* out, float* lse, ra_stream_t stream);

/* The ring with its K/V pass made real (tutorial section 4: "SEND K,V to
 * GPU (i+1) mod N, RECV K,V from GPU (i-1) mod N", and the point that the
 * SEND can be overlapped with the compute of the current block; section 10
 * exercise C measures it with and without overlap).  Each rank's held block
 * lives in its own slot of a double buffer; after step t every holder's slot
 * receives the block of holder i-1 (device-to-device copies), and step t+1
 * attends to what arrived.  With overlap != 0 the copies run on copy_stream
 * while step t computes (ordered by events); with overlap == 0 they run on
 * `stream` between the steps.  The attention arithmetic is that of
 * RA_MODE_PER_STEP, so the results are bitwise identical to it.
 *   copy_stream  a stream other than `stream` (used only when overlap != 0) */
size_t ra_ring_rotate_workspace_size(ra_shape shp, int c, int layout);
ra_status ra_ring_forward_rotate(const void* q, const void* k, const void* v, ra_shape shp,
                                 int c, int layout, int causal, int overlap, int out_dtype,
                                 void* out, float* lse, void* workspace, size_t ws_bytes,
                                 ra_stream_t stream, ra_stream_t copy_stream);

/* Decode over keys and values spread across c shards (tutorial section 7:
 * decode has one query per step, and attention over the distributed keys needs
 * a gather of partial results, like a FlashDecoding split-K): every shard's
 * keys are cut into 128-key tiles (each contiguous stretch of a shard on its
 * own), a block of the tensor-core kernel computes one partial state (o, m, l)
 * over a fixed set of tiles, and the partials are merged in a fixed order into
 * the normalised output.  D = 64 or 128; every layout.
 *   shp        B, Sq = R new tokens, Sk = S keys, Hq, Hkv, D, dtype (bf16), scale
 *   q          device [B, R, Hq, D] bf16;  q_pos device int32 [R] global positions
 *   k, v       device [B, S, Hkv, D] bf16, natural order; the shards are those of
 *              `layout` over c ranks (S divisible as for ra_ring_forward)
 *   out        device [B, R, Hq, D] in out_dtype (bf16 or RA_F32); lse [B, Hq, R] or NULL
 *   workspace  device, >= ra_decode_workspace_size() bytes (the partials) */
size_t ra_decode_workspace_size(ra_shape shp, int c, int layout);
ra_status ra_decode_forward(const void* q, const int32_t* q_pos, const void* k, const void* v,
                            ra_shape shp, int c, int layout, int causal, int out_dtype, void* out,
                            float* lse, void* workspace, size_t ws_bytes, ra_stream_t stream);

/* ---- host-side scheduler (no GPU needed) ------------------------------ */

/* Ring schedule: table[step*c + rank] = the rank whose K/V block `rank`
 * holds at `step`, i.e. (rank - step) mod c (each rank sends to rank+1 and
 * receives from rank-1 after every step; tutorial section 4). */
ra_status ra_schedule(int c, int32_t* table);

/* Global positions of the S tokens in rank-major shard order:
 * pos[rank*(S/c) + i] = position of the i-th token of `rank`. */
ra_status ra_shard_positions(int S, int c, int layout, int32_t* pos);

/* Expected per-(rank, step) work of ONE batch and ONE query head, computed
 * on the host from the layout: out[rank*c + step]. */
ra_status ra_work_expected(int S, int c, int layout, int causal, ra_work* out);

/* Wait for `stream`, then read and clear the device error word.  Returns
 * RA_OK, RA_ERR_TIMEOUT or RA_ERR_CUDA. */
ra_status ra_device_error(ra_stream_t stream);

/* Self-test of the device-timeout path (the pages have no counterpart: they
 * assume the ring completes).  Clears any pending device error, then runs one
 * block that waits, through the same bounded wait as the attention kernels, on
 * a barrier that nothing ever arrives on.  The wait gives up after about
 * limit_us microseconds (1 .. 1000000; the check runs every 256 polls, so the
 * real time can be longer), sets its bit in the device error word and the
 * kernel returns.  Returns RA_ERR_TIMEOUT when the path works as designed,
 * RA_ERR_INVALID for a bad limit, RA_ERR_CUDA if a CUDA call fails.  With
 * leave_pending == 0 the error word is cleared again before the return; with
 * leave_pending != 0 it stays set, as after a real timeout, so that a caller
 * can check that later calls are refused until ra_device_error() clears it.
 * The device stays usable afterwards. */
ra_status ra_selftest_wait_timeout(uint32_t limit_us, int leave_pending, ra_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* RA_H_ */
