/*
 * dustin.h -- C ABI of the GB300 (sm_103a) sparse-verification hot path.
 *
 * The calls follow the method described in "Technical Summary: Dustin"
 * (gist.science/paper/2606.24957):
 *   dustin_score       section 1 "Hybrid Attention Aggregation" + section 2
 *                      "Efficient Estimation via Semantic Retrieval Heads":
 *                      draft-look-ahead and target-historical attention on a few
 *                      SRH heads, summed into a global per-token importance map.
 *   dustin_select      section 1: fixed-size verification set I_verify -- a
 *                      protected sink prefix and recent window, then the top-m
 *                      tokens by the draft signal, then the rest of the budget by
 *                      the target signal.
 *   dustin_verify_attn section 3 "Verification Workflow", steps 3-4: the target
 *                      verifies the gamma+1 draft/bonus queries against the
 *                      selected rows only.
 *   dense_verify_attn  "Problem Statement": standard verification that loads
 *                      the full KV cache (the comparator).
 *   dustin_kv_append   section 3, step 5: accepted tokens are appended.
 *   dustin_verify_step score -> select -> verify in one call on one stream.
 *
 * Conventions (all calls):
 *  - The caller owns every buffer.  Pointers named "device" are CUDA device
 *    pointers; "host" arrays are read during the call only.  No call allocates
 *    device memory: scratch lives in a caller-provided workspace of
 *    dustin_workspace_bytes() bytes (256-byte aligned), initialised once with
 *    dustin_workspace_init().
 *  - Arguments are validated on the host before anything is launched; on any
 *    error the call returns a negative dustin_status and launches nothing.
 *  - Work is enqueued asynchronously on the given stream.  Kernels never trap:
 *    device-side anomalies (an index outside the context, a NaN importance
 *    value, an append past the capacity, a bounded wait that gave up) set bits
 *    of a sticky error word in the workspace, read by dustin_check().
 *  - bf16 tensors are raw bf16 bit patterns; fp32 outputs are IEEE floats.
 *  - Context length per sequence is the device array seq_len[B]; positions at
 *    or beyond seq_len[b] are never read.
 *  - No call is thread-safe with respect to a shared workspace.
 */
#ifndef DUSTIN_H
#define DUSTIN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DUSTIN_OK = 0,
  DUSTIN_EINVAL = -1,     /* bad argument: null pointer, size, stride, alignment */
  DUSTIN_ERANGE = -2,     /* a size beyond the library's limits (see DUSTIN_MAX_*) */
  DUSTIN_ECUDA = -3,      /* a CUDA runtime/driver call failed */
  DUSTIN_EDEVICE = -4,    /* dustin_check: a kernel flagged an anomaly */
  DUSTIN_EWORKSPACE = -5  /* workspace null, misaligned or smaller than required */
} dustin_status;

/* Bits of the device error word (dustin_check). */
#define DUSTIN_DEV_INDEX   1   /* an I_verify entry outside [-1, seq_len[b]) (skipped) */
#define DUSTIN_DEV_NAN     2   /* a NaN or negative importance value (ranked as 0) */
#define DUSTIN_DEV_APPEND  4   /* n_accept outside [0, gamma+1] or append past Lcap (skipped) */
#define DUSTIN_DEV_TIMEOUT 8   /* a bounded wait on an on-chip barrier gave up */
#define DUSTIN_DEV_SEQLEN 16   /* seq_len[b] outside [0, Lcap] (sequence skipped) */

/* Limits. */
#define DUSTIN_MAX_SRH 32           /* SRH entries per call */
#define DUSTIN_MAX_PAIRS 32         /* (SRH head x query row) pairs sharing one KV head */
#define DUSTIN_MAX_LAYERS 16        /* layers per verify / append call */
#define DUSTIN_MAX_QROWS 128        /* (gamma+1) * (Hq/Hkv) verify query rows per KV head */
#define DUSTIN_MAX_BLOCK 64         /* gamma+1 draft-block rows per verify call */
#define DUSTIN_MAX_LCAP (1 << 20)   /* positions per cache */

/* A bf16 KV-cache view, element (b, g, pos, j) at
 *   ptr + b*sb + g*sh + pos*sl + j          (strides in elements).
 * d must be 64 or 128; rows (j = 0..d-1) are contiguous.  ptr must be 16-byte
 * aligned and sb, sh, sl multiples of 8.  The cache holds Lcap positions. */
typedef struct {
  void* ptr;
  int32_t hkv;
  int32_t d;
  int64_t sb, sh, sl;
} dustin_kv;

/* Budget and shape parameters shared by all calls. */
typedef struct {
  int32_t B;       /* sequences in the batch, >= 1 */
  int32_t Lcap;    /* capacity (positions) of every cache, 1..DUSTIN_MAX_LCAP */
  int32_t gamma;   /* draft block length (>= 0); verification uses gamma+1 queries */
  int32_t sinks;   /* protected prefix length */
  int32_t window;  /* protected recent-window length; sinks + window <= k */
  int32_t m;       /* draft-tier size (clipped to what the budget leaves) */
  int32_t k;       /* budget |I_verify|, >= 1 */
} dustin_params;

/* One attention signal used for scoring (section 1 of the pages): the draft
 * model's look-ahead queries (channel 0, nq = gamma rows) or the target
 * model's previous-step queries (channel 1, nq = gamma+1 rows). */
typedef struct {
  int32_t n_layers;        /* entries of q[] and k[] */
  int32_t hq;              /* query heads of that model; k[l].hkv must divide it */
  int32_t nq;              /* query rows per sequence */
  const void* const* q;    /* host array [n_layers] of device pointers,
                              bf16 [B][nq][hq][d] contiguous (entries of layers
                              that hold no SRH may be NULL) */
  const dustin_kv* k;      /* host array [n_layers] of key-cache views */
} dustin_signal;

/* One Semantic Retrieval Head: channel 0 = draft look-ahead, 1 = target
 * historical; layer indexes that channel's dustin_signal; q_head < hq. */
typedef struct {
  int32_t channel;
  int32_t layer;
  int32_t q_head;
} dustin_srh;

/* One target layer for verification. */
typedef struct {
  const void* q;    /* device, bf16 [B][gamma+1][hq][d]: verify queries */
  dustin_kv k, v;   /* that layer's full caches (same hkv, d, strides) */
  const void* kb;   /* device, bf16 [B][hkv][gamma+1][d]: the draft block's keys */
  const void* vb;   /* device, bf16 [B][hkv][gamma+1][d]: the draft block's values */
  float* o;         /* device, fp32 [B][gamma+1][hq][d]: output */
} dustin_verify_layer;

/* Arguments of dustin_verify_step. */
typedef struct {
  dustin_params p;
  const dustin_signal* draft;          /* channel 0 */
  const dustin_signal* target;         /* channel 1 */
  const dustin_srh* srh;
  int32_t n_srh;
  int32_t hq;                          /* target query heads for verification */
  int32_t n_layers;                    /* verified layers, all sharing one I_verify */
  const dustin_verify_layer* layers;   /* host array [n_layers] */
  const int32_t* seq_len;              /* device [B] */
  float* importance;                   /* device fp32 [B][2][Lcap] (output) */
  int32_t* i_verify;                   /* device int32 [B][k] (output) */
  cudaEvent_t* stage_events;           /* NULL, or host array of 5 events recorded on
                                          the stream: before score, after the stream
                                          kernel of the first scoring group (before its
                                          normalise kernel), after all score kernels,
                                          after select, after verify */
} dustin_step;

/* Library version string (static storage). */
const char* dustin_version(void);

/* Bytes of workspace needed by every call made with these arguments: score
 * sizes its per-KV-head partial maps from the SRH list, verification its
 * per-unit partials from (hq, hkv, d, n_layers).  Pass n_srh = 0 (and NULL
 * pointers) when nothing is scored and n_layers = 0 when nothing is verified.
 * Returns 0 if the arguments are invalid.  Every workspace holds at least
 * 256 + 65536 bytes (the error word and a reserved area). */
size_t dustin_workspace_bytes(const dustin_params* p, const dustin_signal* draft,
                              const dustin_signal* target, const dustin_srh* srh,
                              int32_t n_srh, int32_t hq, int32_t hkv, int32_t d,
                              int32_t n_layers);

/* Clears the error word and the reserved area of a workspace
 * (asynchronously, on stream).  Call it once before first use, and again
 * after dustin_check has reported DUSTIN_DEV_TIMEOUT. */
int dustin_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream);

/* Synchronises the stream, returns the error word in *flags (if non-NULL),
 * clears it, and returns DUSTIN_EDEVICE if it was non-zero. */
int dustin_check(void* ws, cudaStream_t stream, int32_t* flags);

/* Hybrid SRH importance scoring (section 1 + 2 of the pages).
 * importance: device fp32 [B][2][Lcap]; channel 0 = draft look-ahead, 1 =
 *   target historical.  importance[b][c][i] = sum over the SRHs of channel c
 *   and their query rows t of softmax_i(q_t . k_i / sqrt(d)) over the
 *   seq_len[b] context positions; entries at or beyond seq_len[b] are 0.
 * seq_len: device int32 [B]. */
int dustin_score(const dustin_params* p, const dustin_signal* draft,
                 const dustin_signal* target, const dustin_srh* srh, int32_t n_srh,
                 const int32_t* seq_len, float* importance, void* ws, size_t ws_bytes,
                 cudaStream_t stream);

/* Budgeted tiered selection (section 1 of the pages).
 * i_verify: device int32 [B][k] = [sinks | window | draft tier | target tier],
 *   each segment ascending; the draft tier holds the top-m' unprotected
 *   positions by importance[b][0] (m' = min(m, k - |protected|)), the target
 *   tier the top remaining ones by importance[b][1]; equal values go to the
 *   lower position.  If k >= seq_len[b] the row is 0..seq_len[b]-1 followed by
 *   -1 padding. */
int dustin_select(const dustin_params* p, const float* importance, const int32_t* seq_len,
                  int32_t* i_verify, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Sparse verification attention (section 3, steps 3-4 of the pages).
 * For sequence b, verify query t (0..gamma) of head h (KV head
 * g = h / (hq/hkv)) attends to the cache rows i_verify[b][*] (entries -1
 * skipped) plus the draft-block rows u <= t, with softmax(q.k/sqrt(d)) weights
 * over values; o = fp32 [B][gamma+1][hq][d].  q, kb, vb as in
 * dustin_verify_layer. */
int dustin_verify_attn(const dustin_params* p, int32_t hq, const void* q, dustin_kv k,
                       dustin_kv v, const void* kb, const void* vb, const int32_t* i_verify,
                       const int32_t* seq_len, float* o, void* ws, size_t ws_bytes,
                       cudaStream_t stream);

/* Dense (full-cache) verification: dustin_verify_attn with every context
 * row 0..seq_len[b]-1 (the pages' "Problem Statement" comparator). */
int dense_verify_attn(const dustin_params* p, int32_t hq, const void* q, dustin_kv k,
                      dustin_kv v, const void* kb, const void* vb, const int32_t* seq_len,
                      float* o, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Append accepted draft rows (section 3, step 5 of the pages).
 * For every layer l and sequence b: rows 0..n_accept[b]-1 of kb[l]/vb[l]
 * (device bf16 [B][hkv][gamma+1][d]) are copied to positions
 * seq_len[b].. of k[l]/v[l]; then seq_len[b] += n_accept[b].  A sequence whose
 * n_accept is outside [0, gamma+1] or whose append would pass Lcap is left
 * untouched and flagged (DUSTIN_DEV_APPEND). */
int dustin_kv_append(const dustin_params* p, int32_t n_layers, const dustin_kv* k,
                     const dustin_kv* v, const void* const* kb, const void* const* vb,
                     const int32_t* n_accept, int32_t* seq_len, void* ws, size_t ws_bytes,
                     cudaStream_t stream);

/* The literal "compressed target KV cache" of section 3, step 3 of the pages,
 * for callers that verify several passes against one selection.  For every
 * layer l, sequence b, KV head g and j < k: row j of kc[l]/vc[l] (bf16
 * [B][hkv][>= k][d], same hkv and d as k[l]/v[l]) becomes row i_verify[b][j]
 * of k[l]/v[l]; entries -1 give zero rows, other indices outside
 * [0, seq_len[b]) give zero rows and set DUSTIN_DEV_INDEX.  seq_len_c[b]
 * (device, out) = the number of entries of i_verify[b] before its first -1
 * (the -1 entries must form a suffix, as dustin_select writes them).
 * dense_verify_attn over (kc, vc, seq_len_c) with Lcap = k then gives the same
 * result as dustin_verify_attn over (k, v, i_verify).  That equality holds
 * only for calls that do not set DUSTIN_DEV_INDEX: sparse verification skips
 * an invalid entry, while dense verification over the compact cache attends
 * to its zero row.  seq_len_c must not be seq_len (other CTAs still read
 * seq_len while it is written): DUSTIN_EINVAL.  dustin_verify_attn itself
 * gathers the rows in-kernel and never writes such a copy. */
int dustin_compact_kv(const dustin_params* p, int32_t n_layers, const dustin_kv* k,
                      const dustin_kv* v, const int32_t* i_verify, const int32_t* seq_len,
                      const dustin_kv* kc, const dustin_kv* vc, int32_t* seq_len_c, void* ws,
                      size_t ws_bytes, cudaStream_t stream);

/* score -> select -> sparse verify of every layer, on one stream. */
int dustin_verify_step(const dustin_step* s, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Host-only query (no device work): how many kernels one dustin_verify_step
 * call with these arguments launches, and how many sequences each scoring
 * group holds.  Scoring runs over groups of *group_size sequences so that a
 * group's logits stay resident in L2; each group takes two kernels (stream,
 * normalise), select takes one, and verification two (the stream-K kernel and
 * the merge of the units it split).  Returns DUSTIN_EINVAL / DUSTIN_ERANGE for arguments
 * dustin_verify_step would reject while planning the scoring. */
int dustin_step_launches(const dustin_step* s, int32_t* n_launches, int32_t* group_size);

/* Host-only query (no device work): the stream-K split that
 * dustin_verify_attn (dense = 0), dense_verify_attn (dense = 1) and the
 * verification of dustin_verify_step use on the current device for this
 * shape.  Units are (layer, sequence, KV head) triples, unit
 * u = (l * B + b) * hkv + g, each of *tiles_per_unit tiles of 64 keys (the
 * context tiles, then one draft-block tile); the T = units * tiles_per_unit
 * tiles are cut among *grid CTAs, CTA c taking tiles [c*T/grid,
 * (c+1)*T/grid).  The grid is two CTAs per SM when (gamma+1)*hq/hkv <= 64
 * and two CTAs' shared-memory layouts fit an SM, else one (at most T).  A
 * unit whose tiles fall to several CTAs is merged by the second verification
 * kernel.  DUSTIN_EINVAL / DUSTIN_ERANGE as the
 * verification calls would return for the shape. */
int dustin_verify_split(const dustin_params* p, int32_t hq, int32_t hkv, int32_t d,
                        int32_t n_layers, int32_t dense, int32_t* grid, int32_t* tiles_per_unit);

/* Self-test of the bounded waits (no counterpart in the pages).  Every
 * on-chip wait of the kernels above gives up after 2 s, sets
 * DUSTIN_DEV_TIMEOUT in the error word and raises a CTA-wide abort flag that
 * makes the CTA's other waits give up at once.  This call runs that wait in
 * one CTA on an mbarrier that nothing ever arrives on, with no copy or MMA in
 * flight: one thread waits limit_ns nanoseconds (1000 .. 1e9) and gives up,
 * a second waits with the kernels' own 2 s limit and stops when the first
 * raises the abort flag.  waited_ns: device int64 [2], 8-byte aligned (out):
 * how long each waited (-1 if its wait had succeeded).  Afterwards
 * dustin_check(ws) reports DUSTIN_DEV_TIMEOUT and the context stays usable.
 * ws needs only its 256-byte header. */
int dustin_wait_selftest(int64_t limit_ns, int64_t* waited_ns, void* ws, size_t ws_bytes,
                         cudaStream_t stream);

/* Bytes of the library-owned scratch array used by dustin_score_noalloc. */
#define DUSTIN_NOALLOC_SCRATCH_BYTES (16u << 20)

/* dustin_score without a caller workspace.  The pages have no counterpart to
 * this call: it exists for callers that cannot call cudaMalloc (or any other
 * allocator) at the point where they score -- for example code running inside
 * an allocator-free runtime, a host callback, or a component that must not
 * touch the process's memory pools.  Results are the same as dustin_score's.
 *
 * Scratch lives in one file-scope device array of DUSTIN_NOALLOC_SCRATCH_BYTES
 * (16 MiB) inside the library; every GPU that loads the library holds it
 * until the process exits.  The call allocates nothing: no cudaMalloc,
 * cudaFree or allocating library routine.  The first call on each device
 * looks up the array's device address (cudaGetSymbolAddress, with that device
 * current); make that first call before any stream capture.
 *
 * Limits: the scratch of at least one sequence -- its logits (SRH pairs x
 * Lcap x 4 bytes) and their statistics, plus a 256-byte header -- must fit in
 * the array; larger batches are scored in groups of sequences that fit.
 * Otherwise DUSTIN_ERANGE is returned and nothing is launched.
 *
 * The device error word (DUSTIN_DEV_* bits) lives in the array's first bytes.
 * It is sticky across calls, like a workspace's: dustin_score_noalloc_check
 * reads and clears it.
 *
 * All calls share the one array and it keeps the last call's contents: calls
 * that overlap on the GPU (different streams, or different host threads
 * without ordering) race on it and must be serialised by the caller. */
int dustin_score_noalloc(const dustin_params* p, const dustin_signal* draft,
                         const dustin_signal* target, const dustin_srh* srh, int32_t n_srh,
                         const int32_t* seq_len, float* importance, cudaStream_t stream);

/* dustin_check for the static array of dustin_score_noalloc on the current
 * device: synchronises the stream, returns the error word of every
 * dustin_score_noalloc call since the last check in *flags (if non-NULL),
 * clears it, and returns DUSTIN_EDEVICE if it was non-zero.  Allocates
 * nothing; DUSTIN_ECUDA if a CUDA call fails. */
int dustin_score_noalloc_check(cudaStream_t stream, int32_t* flags);

#ifdef __cplusplus
}
#endif

#endif /* DUSTIN_H */
