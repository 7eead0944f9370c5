/*
 * cpa.h -- chunked prefill attention with past, fused RoPE, KV-cache append and
 * padded-append rollback for NVIDIA GB300 (sm_103a).
 *
 * Sources (page title, section):
 *   [P1] "functiongemma: chunk prefill-with-past graph gemma_prefill_with_past"
 *        (SKaiNET-transformers PR 417): Why; Change (additive); Validation.
 *   [P2] "[quanization] Enable prefill-decode modeling" (Samsung TICO issue 586):
 *        Runtime behavior; Mask/cache layout used in the runtime.
 *   [P4] "Pad the chunked-prefill tail for sliding-window models" (cactus PR 716):
 *        Problem; Fix; review sweep; Declined with rationale.
 *
 * Conventions shared by every entry point
 *   - All tensors are caller-owned device memory; the library allocates nothing
 *     and keeps no pointer after a call returns ([P2, Runtime behavior]: the KV
 *     cache is managed by the runtime, not inside the graph).
 *   - Every call is asynchronous and stream-ordered on `stream` (a cudaStream_t;
 *     NULL means the legacy default stream).  A call returns after host-side
 *     validation and kernel launch; it never synchronises.
 *   - bf16 means IEEE bfloat16 bit patterns (uint16).  "Contiguous" means
 *     row-major with the last index fastest.
 *   - Host-side argument errors return a cpa_status and launch nothing.
 *     Errors that depend on device data (lengths) are reported by OR-ing
 *     CPA_EBIT_* bits into the caller's device int32 word `err`, which the
 *     library never clears; the caller reads it after synchronising.
 *   - Supported head dims D: 64, 128, 256.  Hq must be a multiple of Hkv
 *     (GQA: q head h reads kv head h / (Hq / Hkv)).
 *   - Pointers to bf16 / fp32 tensors must be 16-byte aligned; cache strides
 *     must be multiples of 8 elements.
 */
#ifndef CPA_H_
#define CPA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cpa_stream; /* same type as cudaStream_t */

typedef enum {
  CPA_OK = 0,
  CPA_ERR_NULL = 1,              /* a required pointer is NULL */
  CPA_ERR_SHAPE = 2,             /* a size is out of range or inconsistent */
  CPA_ERR_ALIGN = 3,             /* pointer or stride misaligned */
  CPA_ERR_UNSUPPORTED = 4,       /* valid but not implemented (e.g. D = 96) */
  CPA_ERR_WINDOW_TOO_SMALL = 5,  /* sliding window W <= C + S ([P4, review]) */
  CPA_ERR_WORKSPACE = 6,         /* workspace / scratch smaller than required */
  CPA_ERR_CUDA = 7               /* a CUDA launch error */
} cpa_status;

/* Bits OR-ed into the device error word. */
#define CPA_EBIT_CAPACITY 1       /* global append: len + n > cap; that sequence untouched */
#define CPA_EBIT_PAST_GT_SPAN 2   /* attention: past_len outside [0, P]; clamped */
#define CPA_EBIT_NREAL_GT_C 4     /* n_real / n_rows outside [0, C]; clamped */
#define CPA_EBIT_SLIDING_N 8      /* sliding append: n > W - S or len > W; sequence untouched */
#define CPA_EBIT_SNAPSHOT 16      /* rollback: cache length does not match the snapshot */
#define CPA_EBIT_TIMEOUT 32       /* a bounded in-kernel pipeline wait ran out */
#define CPA_EBIT_BOUNDS 64        /* checked builds only: a computed index fell outside
                                     its buffer; the access was skipped */

enum { CPA_CACHE_GLOBAL = 0, CPA_CACHE_SLIDING = 1 };
/* Element format of a cache's K and V ([P4, Declined with rationale] names a
 * runtime option that keeps the KV cache in fp16). */
enum { CPA_KV_BF16 = 0, CPA_KV_F16 = 1 };

/*
 * A KV cache for one layer.  Element (b, h, s, d) of K (and of V) lives at
 * k[b*stride_b + h*stride_h + s*stride_s + d] (strides in elements, d fastest).
 *   GLOBAL  ([P2, Mask/cache layout]): rows are packed first; `len[b]` rows
 *           hold data; appends go to slots [len, len + n); capacity `cap`.
 *   SLIDING ([P4, Fix]): at most `window` rows (window <= cap): `sink` pinned
 *           rows, then the newest rows in chronological order; an append that
 *           overflows evicts the oldest non-sink rows and compacts.
 * Rows at or beyond len[b] are dead: the library never promises their bytes
 * ([P4, Declined with rationale]: nothing reads past the length).  With the
 * implicit mask their bytes never reach an output, whatever they hold (NaN
 * and infinity patterns included); the same holds for the chunk's pad rows.
 * dtype CPA_KV_F16: K and V hold IEEE half values.  Appends round the fp32
 * rotation of each key (the same arithmetic as for bf16) to half, nearest
 * even, and convert value rows bf16 -> half (exact inside the half range;
 * larger values become infinite).  The attention then runs its products in
 * fp16: Q and the chunk keys are rotated to half, the chunk values and P are
 * half, accumulation is fp32 and the output stays bf16.
 */
typedef struct {
  void* k;
  void* v;
  int64_t stride_b, stride_h, stride_s;
  int32_t* len;     /* device int32 [B] */
  int32_t cap;
  int32_t kind;     /* CPA_CACHE_GLOBAL or CPA_CACHE_SLIDING */
  int32_t window;   /* SLIDING: W rows (<= cap); GLOBAL: ignored */
  int32_t sink;     /* SLIDING: S pinned rows; GLOBAL: ignored */
  int32_t dtype;    /* CPA_KV_BF16 or CPA_KV_F16 */
} cpa_cache;

/*
 * Arguments of one chunk-prefill attention step ([P1, Change]).
 *
 * Shapes: B sequences, Hq query heads, Hkv kv heads, head dim D, C chunk rows
 * (pads included), P past slots visible to the step.
 *   q      bf16 [B, Hq, C, D]  contiguous  query rows, before RoPE
 *   k_new  bf16 [B, Hkv, C, D] contiguous  chunk keys, before RoPE
 *   v_new  bf16 [B, Hkv, C, D] contiguous  chunk values
 *   cos, sin  fp32 [B, C, D] contiguous    per-row RoPE tables; row i of
 *          sequence b carries the angles of that row's absolute position.
 *          Rotation (rotate-half pairing d, d + D/2, fp32 products and sums
 *          without fused multiply-add, rounded to bf16 nearest-even):
 *            y[d]     = x[d]*cos[d] - x[d+D/2]*sin[d]
 *            y[d+D/2] = x[d+D/2]*cos[d+D/2] + x[d]*sin[d+D/2]
 *   cache  slots [0, P) of cache->k / cache->v are the past keys/values
 *          (already rotated when they were appended).  The step reads the
 *          cache as it is before this chunk is appended.
 *   Key columns are the P past slots followed by the C chunk rows.
 *   mask   NULL: implicit mask from (past_len, n_real, window, causal):
 *            query row i sits at position past_len[b] + i; past slot j is
 *            visible iff j < past_len[b] and (window == 0 or
 *            past_len[b] + i - j < window); chunk row t is visible iff
 *            t < n_real[b], (causal == 0 or t <= i) and (window == 0 or
 *            |i - t| < window).  ([P1, Change]: causal band, zero padding,
 *            512-position window; [P2, Mask/cache layout]: packed past,
 *            unfilled slots masked.)  A SLIDING cache with sink S > 0 also
 *            keeps its pinned slots [0, min(S, past_len[b])) visible to
 *            every row whatever the window; its other slots hold the newest
 *            tokens in order, so the window rule above applies to them
 *            ([P4, Fix]: pinned sink rows, chronological compaction).
 *          non-NULL: explicit additive fp32 mask [B, Hq, C, P + C],
 *            contiguous, 0 = attend, -1e30 = masked ([P1, Change]); entries
 *            <= -1e29 (or not a number) count as masked; other entries are
 *            added to the scaled scores.  Every cache slot in [0, P) and every
 *            chunk row must then hold finite values.  The explicit and the
 *            implicit form of one mask give identical output bits.
 *   past_len, n_real  device int32 [B]; required for the implicit mask;
 *          n_real also gives the default selected row.  Out-of-range values
 *          are clamped and flagged (CPA_EBIT_PAST_GT_SPAN / _NREAL_GT_C).
 *   scale  softmax scale; <= 0 selects 1/sqrt(D).
 *   sel_row  device int32 [B] or NULL (NULL: n_real[b] - 1) -- the row whose
 *          fp32 output is copied to out_sel ([P1, Change]: one-hot select;
 *          [P1, Validation]: row 51 of a 52-token chunk).
 *   out    bf16 [B, Hq, C, D]: softmax-weighted values of every row (pad rows
 *          included); a row with no visible key is all zeros.
 *   out_sel  fp32 [B, Hq*D] or NULL: row sel_row[b] of every head, before
 *          bf16 rounding.
 *   workspace  device memory of at least cpa_attn_workspace_size(...) bytes
 *          (the work plan the call builds on the device, split-KV partial
 *          results, rotated copies of the chunk's queries and keys; with an
 *          explicit mask, the classes of its key tiles and, given
 *          cpa_attn_workspace_size_mask(...) bytes, its bit copy); may be
 *          NULL when that size is 0.  Its contents need no initialisation
 *          and are meaningless after the call.
 *   err    device int32 error word (required).
 *   sm_budget  0, or the number of SMs the call may occupy: a value below
 *          the device's SM count sizes the persistent grid for that many
 *          SMs and keeps the call's follow-up kernels from taking SMs before
 *          its attention grid ends, so that work issued on another stream
 *          (for example a decode batch beside a prefill chunk, the mixed
 *          batch of chunked prefill serving) runs on the rest.  The result
 *          does not depend on it beyond rounding order.  Negative ->
 *          CPA_ERR_SHAPE.
 */
typedef struct {
  int B, Hq, Hkv, D, C, P;
  float scale;
  const void* q;
  const void* k_new;
  const void* v_new;
  const float* cos;
  const float* sin;
  const cpa_cache* cache;
  const float* mask;
  const int32_t* past_len;
  const int32_t* n_real;
  int window;
  int causal;
  const int32_t* sel_row;
  void* out;
  float* out_sel;
  void* workspace;
  size_t workspace_bytes;
  int32_t* err;
  int sm_budget;
} cpa_attn_args;

/* One chunk of C rows against the cache ([P1, Change]; cost scales with C,
 * [P1, Validation]).  C == 1 is allowed.  Returns CPA_OK after launch. */
cpa_status cpa_chunk_prefill_attn(const cpa_attn_args* args, cpa_stream stream);

/* One-token decode step: the C == 1 case ([P2, Runtime behavior]: a single-token
 * step against the static past; [P2, Mask/cache layout]: the valid past slots and
 * the current token are unmasked, no causal mask).  Requires C == 1; the mask
 * is implicit unless args->mask is given.  Append the token afterwards with
 * cpa_kv_append (n_rows = 1). */
cpa_status cpa_decode_step(const cpa_attn_args* args, cpa_stream stream);

/* Bytes of workspace cpa_chunk_prefill_attn / cpa_decode_step need for these
 * sizes: the plan, split-KV partials and rotated copies described under
 * `workspace` above (0 only for a one-token step that needs no partials). */
size_t cpa_attn_workspace_size(int B, int Hq, int Hkv, int D, int C, int P);

/* Bytes of workspace for a call with an explicit mask at these sizes: at
 * least cpa_attn_workspace_size(...).  On the two-tile path (D = 64 or 128
 * with more than 128 packed query rows per kv head) a pre-pass reads the
 * fp32 mask once and classifies every key tile; with this much workspace it
 * also keeps a one-bit copy of each row's entries that are exactly 0 (1/32
 * of the mask's bytes), so that tiles holding only 0 and masked entries
 * ([P1, Change]: 0 = attend, -1e30 = masked) are never read in fp32 again.
 * With only cpa_attn_workspace_size(...) bytes the attention re-reads the
 * fp32 values of the tiles it visits.  The results are the same bits either
 * way. */
size_t cpa_attn_workspace_size_mask(int B, int Hq, int Hkv, int D, int C, int P);

/*
 * cpa_chunk_prefill_attn for callers that cannot allocate device memory.  The
 * pages have no counterpart: this exists for callers with no way to obtain a
 * workspace -- code running while a CUDA graph is captured, runtimes whose
 * device memory is planned once from static shapes, and plugins inside a host
 * framework that owns the allocator.  Arguments and results are those of
 * cpa_chunk_prefill_attn; args->workspace and args->workspace_bytes are
 * ignored.  The call's workspace (what cpa_attn_workspace_size counts) is one
 * 16 MiB array compiled into the library (held on every GPU that loads the
 * library until the process exits); the call itself allocates nothing.
 *   - Returns CPA_ERR_WORKSPACE, launching nothing, when the sizes need more
 *     than 16 MiB (cpa_attn_workspace_size(...) > 16 MiB).
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call shares the array, and no byte of it needs to start at zero
 *     (each call writes every partial it reads).  Calls whose kernels overlap
 *     on the GPU (different streams without ordering) race on the array.
 */
cpa_status cpa_chunk_prefill_attn_noalloc(const cpa_attn_args* args, cpa_stream stream);

/*
 * Append rows [0, n_rows[b]) of the chunk to the cache ([P2, Runtime
 * behavior]: the runtime writes the step's K/V into the external cache;
 * [P1, Change]: K/V extended by the chunk).  K rows are rotated with cos/sin
 * exactly as cpa_chunk_prefill_attn rotates them (same bytes); V rows are
 * copied.  k_new/v_new bf16 [B, Hkv, C, D], cos/sin fp32 [B, C, D],
 * n_rows device int32 [B] (each in [0, C]).
 *   GLOBAL: rows go to slots [len, len + n); len += n.  If len + n > cap the
 *     sequence is left unchanged and CPA_EBIT_CAPACITY is set.
 *   SLIDING ([P4, Fix]): e = max(0, len + n - W) oldest non-sink rows are
 *     evicted, the rest move down, the n rows are written at the end and
 *     len = min(len + n, W).  n must be <= W - S (else CPA_EBIT_SLIDING_N).
 *     Needs `scratch` of cpa_cache_scratch_size(...) bytes.
 * scratch may be NULL for a GLOBAL cache.
 */
cpa_status cpa_kv_append(const cpa_cache* cache, const void* k_new, const void* v_new,
                         const float* cos, const float* sin, const int32_t* n_rows,
                         int B, int Hkv, int D, int C,
                         void* scratch, size_t scratch_bytes, int32_t* err, cpa_stream stream);

/*
 * Attention and global append in one call ([P1, Change]: "K/V extended by
 * the chunk"; [P2, Runtime behavior]: the runtime writes the new K/V into its
 * buffers after the step).  Same results as cpa_chunk_prefill_attn(args)
 * followed by cpa_kv_append(args->cache, args->k_new, args->v_new, args->cos,
 * args->sin, n_rows, ...): identical outputs, identical cache bytes in rows
 * [0, len) and len, identical error bits.  The RoPE pre-pass that rotates
 * the chunk keys for the attention also writes them (and the values) to the
 * cache slots [len_b, len_b + n_b), and len advances once the attention has
 * read it, so the keys are rotated once and the append costs no extra pass.
 *   n_rows   device int32 [B], 16-byte aligned: rows to append (as
 *            cpa_kv_append's n_rows).
 * The cache must be GLOBAL (CPA_ERR_UNSUPPORTED otherwise: a sliding append
 * evicts rows the attention reads; use the separate calls).  The new rows are
 * written before the attention reads the cache, into slots the attention
 * does not see when past_len <= len (always with the implicit mask; an
 * explicit mask must keep slots >= len masked, as it must for dead rows).
 * One-token chunks run the attention and then the separate append kernels.
 * Errors as cpa_chunk_prefill_attn and cpa_kv_append.
 */
cpa_status cpa_chunk_prefill_attn_append(const cpa_attn_args* args, const int32_t* n_rows, cpa_stream stream);

/* Scratch bytes a SLIDING cache needs for cpa_kv_append and the padded-append
 * snapshot / rollback with chunk size C (0 for a GLOBAL cache). */
size_t cpa_cache_scratch_size(const cpa_cache* cache, int B, int Hkv, int D, int C);

/*
 * Before a padded append of C rows of which n_real[b] are real, save the rows
 * that the padded append would evict beyond an exact append ([P4, Fix]:
 * snapshot_cache_padded_append).  With e_pad = max(0, len + C - W) and
 * e_ex = max(0, len + n - W) the rows [S + e_ex, S + e_pad) are saved, with
 * the lengths, into `scratch`.  SLIDING caches only.  Returns
 * CPA_ERR_WINDOW_TOO_SMALL when W <= C + S ([P4, review]: sink-aware guard).
 * Sequence: snapshot -> cpa_chunk_prefill_attn (reads the cache before the
 * append) -> cpa_kv_append(n_rows = C) -> rollback.
 */
cpa_status cpa_kv_snapshot_padded_append(const cpa_cache* cache, const int32_t* n_real,
                                         int B, int Hkv, int D, int C,
                                         void* scratch, size_t scratch_bytes,
                                         int32_t* err, cpa_stream stream);

/*
 * After the padded append, drop the C - n pad rows and reinsert the saved rows
 * at slot S ([P4, Fix]: rollback_cache_padded_append), leaving rows [0, len)
 * and len byte-identical to cpa_kv_append with n_rows = n_real.  Bytes past
 * the final length are unspecified ([P4, Declined with rationale]).  If the
 * cache length is not the one the snapshot predicts, nothing changes and
 * CPA_EBIT_SNAPSHOT is set.
 */
cpa_status cpa_kv_rollback_padded_append(const cpa_cache* cache, int B, int Hkv, int D, int C,
                                         void* scratch, size_t scratch_bytes,
                                         int32_t* err, cpa_stream stream);

/*
 * Tail policy ([P4, Fix] and the review's padded-versus-scalar sweep; its
 * follow-up list proposes a small tail-chunk variant).  A runtime whose chunk
 * calls have fixed shapes feeds the last t real tokens of a prompt either as
 *   CPA_TAIL_SCALAR: t one-token steps (cpa_decode_step + cpa_kv_append of one
 *                    row each), or
 *   CPA_TAIL_PADDED: one chunk of c_pad rows, the t real rows first and zero
 *                    pad rows after; on a SLIDING cache wrapped in snapshot ->
 *                    attention -> cpa_kv_append(n_rows = c_pad) -> rollback, on
 *                    a GLOBAL cache followed by cpa_kv_append(n_rows = t).
 * Both leave the same cache bytes.  Arguments:
 *   t          real tail tokens, 1 <= t <= C;
 *   C          the full chunk rows (c_pad never exceeds it);
 *   window     W of a SLIDING cache, 0 for a GLOBAL cache;  sink: S (0 if none);
 *   buckets    the chunk sizes the caller can run, ascending, each in [1, C];
 *              NULL (n_buckets = 0) means {C} alone;
 *   crossover  the smallest t for which the padded chunk is faster;
 *              <= 0 means CPA_TAIL_CROSSOVER_DEFAULT;
 *   force      CPA_TAIL_AUTO, CPA_TAIL_FORCE_SCALAR (the kill switch) or
 *              CPA_TAIL_FORCE_PADDED.
 * Results: *mode and *c_pad (the smallest bucket >= t that a SLIDING cache
 * can snapshot, i.e. with W > c_pad + S; t for CPA_TAIL_SCALAR).  With no such
 * bucket the tail runs scalar (AUTO) or the call returns
 * CPA_ERR_WINDOW_TOO_SMALL (FORCE_PADDED), following [P4, review]'s
 * sink-aware guard.  Host only: no device memory, no stream.
 * Returns CPA_ERR_NULL for NULL mode / c_pad, CPA_ERR_SHAPE for t outside
 * [1, C], an unsorted or out-of-range bucket list, or W < 0, S < 0.
 */
#define CPA_TAIL_SCALAR 0
#define CPA_TAIL_PADDED 1
#define CPA_TAIL_AUTO 0
#define CPA_TAIL_FORCE_SCALAR 1
#define CPA_TAIL_FORCE_PADDED 2
/* Measured on GB300: D = 256, 8 q / 1 kv heads, a full 512-row window cache,
 * buckets {16, 32, 64, 128}, every sequence replayed as one CUDA graph. */
#define CPA_TAIL_CROSSOVER_DEFAULT 2
cpa_status cpa_tail_plan(int t, int C, int window, int sink, const int32_t* buckets, int n_buckets,
                         int crossover, int force, int32_t* mode, int32_t* c_pad);

/* Text for a status code (static storage). */
const char* cpa_status_str(cpa_status status);

/* Library version string (static storage). */
const char* cpa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CPA_H_ */
