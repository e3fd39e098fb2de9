/*
 * vsamp.h -- C ABI of libvsamp.so, the GB300 (sm_103a) per-row vocabulary sampling stage.
 *
 * For each row of a [B, V] logits batch the stage computes an online max / log-sum-exp, an exact
 * top-k select with index-ordered ties, a top-p nucleus cut (probability-space predicate, row maximum
 * always kept), a min-p filter, a Philox4x32-10 Gumbel-max draw and the selected token's
 * log-probability.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers: every array argument is a DEVICE pointer unless its comment says otherwise. The caller
 *   allocates and owns every buffer; the library keeps no pointer after a call returns and allocates
 *   no device memory.
 * Layout: logits / scores are row-major [B, ld] with ld >= V (elements, not bytes); row r starts at
 *   element r * ld. Only the first V (or lengths[r]) elements of a row are read.
 * Streams: `stream` is a cudaStream_t (NULL = the legacy default stream). Every call only enqueues
 *   work on `stream` and returns without synchronising; outputs are valid once the stream reaches
 *   that point.
 * Errors: the return value reports problems the host can see before launch (NULL pointers, sizes,
 *   dtype, a device that cannot hold the row) and launch failures (VSAMP_ERR_CUDA). Nothing is
 *   enqueued when the return value is not VSAMP_OK. Data-dependent problems are reported per row in
 *   `row_status[r]` (when the caller passes it) with the row's outputs set to sentinels (token -1,
 *   logprob NaN, indices -1); the device never traps or asserts.
 * Keys: `pivot_key` values are the order-preserving 32-bit key of the fp32 value (bf16 values are
 *   widened exactly): positive floats get the sign bit set, negative floats are bit-inverted, and
 *   -0.0 is read as +0.0 ("[Kernel] Make persistent_topk deterministic", Changes: signed zeros are
 *   one key).
 *
 * Per-row parameters (arrays of length B; NULL selects the default in brackets):
 *   temperature [1.0]  T > 0 scales scores as (x - max) / T; T <= 0 is greedy (the lowest-index
 *                      maximum, all filters keep one token) and log-probabilities then use T = 1.
 *   top_k [off]        0 < k < V keeps the k largest by (value desc, index asc); k <= 0 or k >= V: off.
 *   top_p [off]        0 < p < 1 keeps the shortest prefix of that order whose mass reaches p * S_k,
 *                      S_k the mass kept by top-k; p >= 1: off; p <= 0 or NaN: row error.
 *   min_p [off]        0 < q <= 1 keeps tokens with exp((x - max)/T) >= q; q <= 0: off; q > 1 or NaN:
 *                      row error.
 *   seed, step [0]     Philox4x32-10 key = (seed mod 2^32, seed >> 32); token v of a row uses output
 *                      word v & 3 of the counter (v >> 2, row_id, step mod 2^32, step >> 32).
 *   row_id [r]         32-bit counter word identifying the row (use the global row index when a batch
 *                      is split across devices, or a per-request id for batch-invariant draws).
 * Transform order: temperature -> top-k -> top-p -> min-p ("[WS2][Logprob] Deterministic SM90
 * linear_logp ...", Integration). The kept set is always a prefix of the order (value desc, index
 * asc) and holds at least the row maximum ("Split top-p numerical reference and conservative gate",
 * Source basis).
 */
#ifndef VSAMP_H_
#define VSAMP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum vsamp_status {
  VSAMP_OK = 0,
  VSAMP_ERR_INVALID_ARG = 1,   /* bad pointer / size / parameter */
  VSAMP_ERR_UNSUPPORTED = 2,   /* this device cannot hold the row (shared memory, cluster size) */
  VSAMP_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch, attribute) */
  VSAMP_ERR_NONFINITE = 4,     /* per row: NaN or +-inf in the row */
  VSAMP_ERR_TIMEOUT = 5,       /* per row: a bounded device-side wait gave up */
  VSAMP_ERR_SCRATCH_LIMIT = 6  /* vsamp_sample_static: the batch needs more than its fixed scratch array */
} vsamp_status;

typedef enum vsamp_dtype {
  VSAMP_F32 = 0,
  VSAMP_BF16 = 1
} vsamp_dtype;

/* Cut descriptor of one row: token v is kept iff key(x_v) > pivot_key, or key(x_v) == pivot_key and
 * v <= idx_cut. (pivot_key, idx_cut) are the key and index of the last kept token in the order
 * (value desc, index asc); kept is the number of kept tokens. */
typedef struct vsamp_cut {
  uint32_t pivot_key;
  int32_t idx_cut;
  int32_t kept;
  int32_t status;      /* vsamp_status of the row */
} vsamp_cut;

/* Device limits the library works with (filled by vsamp_device_info). */
typedef struct vsamp_limits {
  int32_t sm_count;
  int32_t smem_optin_bytes;       /* cudaDevAttrMaxSharedMemoryPerBlockOptin */
  int32_t max_cluster;            /* largest cluster size the row kernels may use on this device */
  int64_t max_row_f32;            /* longest fp32 row a cluster can hold in shared memory */
  int64_t max_row_bf16;           /* longest bf16 row */
} vsamp_limits;

/* Online max / log-sum-exp ("[WS2][Logprob] Deterministic SM90 linear_logp ...", Design: the numeric
 * contract: m = max_v x_v, S = sum_v exp(x_v - m), lse = m + log S; temperature applied to the
 * statistics, stored logits left unscaled).
 *   row_max[r]    = max_v x[r, v] (fp32)
 *   row_logsum[r] = log sum_v exp((x[r, v] - row_max[r]) / T_r), T_r <= 0 read as 1.
 * The sum is accumulated in 64-bit fixed point (2^-40 units), so it does not depend on scheduling,
 * batch size or neighbouring rows. Either output may be NULL. */
vsamp_status vsamp_softmax_lse(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                               const float* temperature, float* row_max, float* row_logsum,
                               int32_t* row_status, void* stream);

/* Deterministic exact top-k select ("[Kernel] Make persistent_topk deterministic", Changes: a radix
 * select whose pivot is exact, then an index-ordered emission of everything above the pivot and the
 * lowest-index elements equal to it; output in ascending index order, identical across calls).
 *   scores   [B, ld] fp32 or bf16; row r has lengths[r] valid elements (NULL: max_len for all rows).
 *            +-inf are ordinary keys; NaN inside the length is a row error.
 *   k        [B] per-row k (NULL: k_max for every row); k <= 0 selects nothing; k > k_max is a row
 *            error.
 *   out_idx  [B, k_max] int32: the first min(k, len) slots hold the selected indices in ascending
 *            order, the remaining slots -1 (also on error). */
vsamp_status vsamp_topk_select(const void* scores, vsamp_dtype dt, int64_t B, int64_t max_len,
                               int64_t ld, const int32_t* lengths, const int32_t* k, int32_t k_max,
                               int32_t* out_idx, int32_t* row_status, void* stream);

/* Top-p / min-p cut after top-k ("Split top-p numerical reference and conservative gate", Source
 * basis: mask with the probability-space predicate and always keep the row maximum; Independent
 * binary64 numerical reference: the smallest prefix of (value desc, index asc) whose mass reaches
 * p * normaliser; "Sorting-free top-k/top-p/min-p sampling ... #901", Background: min-p pivot =
 * max * p). No logit-space threshold is ever rebuilt.
 *   cut   [B] descriptor of the kept prefix (required).
 *   mask  [B, V] uint8, 1 = kept (NULL: not written).
 *   stats [B, 4] int32 or NULL: {full passes over the row, radix rounds, kept, path flags}. */
vsamp_status vsamp_topp_minp_mask(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                                  const float* temperature, const int32_t* top_k, const float* top_p,
                                  const float* min_p, vsamp_cut* cut, uint8_t* mask, int32_t* stats,
                                  void* stream);

/* The fused stage: LSE, top-k, top-p, min-p, then a Gumbel-max draw over the kept tokens and the
 * drawn token's log-probability ("[vLLM PR #45996] use log1p(-u) to improve FP32 Gumbel sampling
 * precision": noise -log(-log1p(-u)), masked arg-max over logits + noise with the lowest index among
 * equal maxima; temperature 0 returns the arg-max).
 *   u = (b + 0.5) * 2^-32 for the token's 32-bit Philox word b; score = (x - max)/T + noise.
 *   token   [B] int32 (required): the drawn token, -1 on a row error.
 *   logprob [B] fp32 or NULL: min((x_t - max)/T - log S, 0) over the full row ("[WS2][Logprob]
 *           ...", Design: logp = min(z_t - lse, 0)).
 *   stats   [B, 4] int32 or NULL: as for vsamp_topp_minp_mask. */
vsamp_status vsamp_sample(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                          const float* temperature, const int32_t* top_k, const float* top_p,
                          const float* min_p, const uint64_t* seed, const uint64_t* step,
                          const uint32_t* row_id, int32_t* token, float* logprob,
                          int32_t* row_status, int32_t* stats, void* stream);

/* vsamp_sample with a workspace: the same draw by two streaming launches over fixed 4 KB pieces of every row
 * (2048 bf16 or 1024 fp32 logits) instead of one thread-block cluster per row. In the first, each warp reads
 * pieces from HBM once and writes their statistics (maximum, count of maxima, mass relative to the maximum)
 * and, for rows without top-k and with T > 0, a 4-bit code per 16-byte vector from the smallest Philox word of
 * its tokens (the words do not depend on the logits). In the second, one CTA per row combines the row's pieces
 * in a fixed order, plans the cut (radix rounds re-read the row, mostly from L2, only when the cut leaves the
 * maximum's tie group) and draws: only vectors whose code passes the prune bound are scored again.
 * Results are deterministic and do not depend on the batch; they agree with vsamp_sample except for the last
 * bits of the row mass (piece masses are rescaled to the row maximum in binary64), which moves a top-p cut
 * only inside the 1e-6 tolerance band. Rows with top-k are drawn by scanning their kept tokens instead; for
 * rows whose kept set is small relative to V, vsamp_sample is usually faster.
 *   workspace        device buffer of at least vsamp_sample_workspace_size(dt, B, V) bytes, 16-byte aligned.
 *                    It needs no initialisation: every call writes what it reads. Calls sharing a workspace
 *                    must not run at the same time (use one workspace per stream).
 *   workspace_bytes  its size in bytes; too small, unaligned or NULL is VSAMP_ERR_INVALID_ARG.
 * Every other argument is as for vsamp_sample. Two launches on `stream`. */
vsamp_status vsamp_sample_ws(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                             const float* temperature, const int32_t* top_k, const float* top_p,
                             const float* min_p, const uint64_t* seed, const uint64_t* step,
                             const uint32_t* row_id, int32_t* token, float* logprob,
                             int32_t* row_status, int32_t* stats, void* workspace, size_t workspace_bytes,
                             void* stream);

/* Workspace bytes vsamp_sample_ws needs for B rows of V logits of type dt (0 for invalid arguments):
 * 256 + 160 B * ceil(V / piece) with pieces of 2048 bf16 or 1024 fp32 logits. */
size_t vsamp_sample_workspace_size(vsamp_dtype dt, int64_t B, int64_t V);

/* Bytes of the fixed device array that vsamp_sample_static uses as its workspace. */
#define VSAMP_STATIC_SCRATCH_BYTES 4194304

/* vsamp_sample_ws on a fixed scratch array of VSAMP_STATIC_SCRATCH_BYTES bytes that the library holds in
 * device memory (a file-scope __device__ array of its module), so the call allocates nothing: no device
 * allocation by the library or by the caller. The sampling method has no counterpart of this call; it
 * exists for callers that must not allocate (for instance while a memory pool is frozen).
 *   Size limit: vsamp_sample_workspace_size(dt, B, V) must not exceed VSAMP_STATIC_SCRATCH_BYTES, else
 *     the call returns VSAMP_ERR_SCRATCH_LIMIT and enqueues nothing.
 *   Set-up: the first call on each device (with that device current) looks up the array's address once.
 *   Contents: the array keeps what the last call left in it. As for vsamp_sample_ws nothing needs clearing
 *     (every call writes what it reads), so each call enqueues only the two kernels.
 *   Largest batch (from vsamp_sample_workspace_size): V = 151,936: 175 rows fp32, 349 rows bf16;
 *     V = 262,144: 102 rows fp32, 204 rows bf16.
 *   Races: one array per device is shared by every caller of this function, so calls whose kernels
 *     overlap on one device (from two streams or two host threads) race on it and give wrong results;
 *     serialise them, or use vsamp_sample_ws with a workspace per stream.
 * Every other argument, the results and the errors are as for vsamp_sample_ws. */
vsamp_status vsamp_sample_static(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                                 const float* temperature, const int32_t* top_k, const float* top_p,
                                 const float* min_p, const uint64_t* seed, const uint64_t* step,
                                 const uint32_t* row_id, int32_t* token, float* logprob,
                                 int32_t* row_status, int32_t* stats, void* stream);

/* Selected-token log-probability ("[WS2][Logprob] ...", Design: logp = min(z_t - lse, 0), temperature
 * applied to the statistics):
 *   out[r] = min((x[r, t] - row_max[r]) / T_r - row_logsum[r], 0), t = token[r], T_r <= 0 read as 1.
 * row_max and row_logsum must both be given (from vsamp_softmax_lse at the same temperature) or both
 * be NULL, in which case they are recomputed from the row. token[r] outside [0, V) is a row error. */
vsamp_status vsamp_logprob(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                           const float* temperature, const int32_t* token, const float* row_max,
                           const float* row_logsum, float* out, int32_t* row_status, void* stream);

/* Processed log-probability of given tokens: the softmax renormalised over the kept set of the cut that
 * vsamp_topp_minp_mask computes (temperature, then top-k, top-p, min-p; greedy rows keep the first maximum)
 * ("[WS2][Logprob] ...", Background: the rollout's processed_logprobs, derived from its logits after the
 * sampling transforms; the clamp of the Design's logp = min(z_t - lse, 0)):
 *   out[r] = min((x[r, t] - m) / T_r - log S_kept, 0) if token t = token[r] is kept, -inf if it is not;
 *   m = row maximum, S_kept = sum over the kept tokens of exp((x - m) / T_r) (T_r <= 0 read as 1).
 * Parameters and errors as for vsamp_topp_minp_mask; token[r] outside [0, V) is a row error; error rows
 * give NaN. One launch on `stream`, one read of each row. */
vsamp_status vsamp_kept_logprob(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                                const float* temperature, const int32_t* top_k, const float* top_p,
                                const float* min_p, const int32_t* token, float* out, int32_t* row_status,
                                void* stream);

/* Top-N log-probability lists ("[Kernel] Make persistent_topk deterministic", details of the probe: per
 * generated token the list of the 20 most probable (token, logprob) pairs, hashed to compare runs; the
 * log-probabilities follow "[WS2][Logprob] ...", Design: logp = min(z_v - lse, 0)).
 *   N            list length, 1 <= N <= VSAMP_TOPN_MAX (else VSAMP_ERR_INVALID_ARG, nothing enqueued).
 *   row_max, row_logsum  [B] fp32, required: written as by vsamp_softmax_lse at the row's temperature.
 *   out_idx      [B, N] int32: slot j holds the (j+1)-th token of the row in the order (logit descending,
 *                index ascending); equal logits keep ascending index order, -0 equals +0.
 *   out_lp       [B, N] fp32: min((x[r, v] - row_max[r]) / T_r - row_logsum[r], 0) for the token in slot j,
 *                T_r <= 0 read as 1.
 *   Slots past min(N, V), and every slot of an error row (a non-finite logit, a NaN or infinite
 *   temperature; row_status as vsamp_softmax_lse reports it), hold -1 and NaN.
 * Two launches on `stream`: one pass over each row (row statistics and the top-k cut with k = N, the N
 * indices emitted in ascending order), then one CTA per row that orders the N
 * tokens (O(N^2 / 256) comparisons per thread) and writes their log-probabilities. The list is a function
 * of the row alone: it does not depend on B, the launch geometry or neighbouring rows. */
#define VSAMP_TOPN_MAX 4096
vsamp_status vsamp_topn_logprobs(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                                 const float* temperature, int32_t N, float* row_max, float* row_logsum,
                                 int32_t* out_idx, float* out_lp, int32_t* row_status, void* stream);

/* The dual-pivot rejection sampler ("Sorting-free top-k/top-p/min-p sampling with dual-pivot rejection
 * kernels #901", Background and Task): a draw from the same filtered law as vsamp_sample (temperature, then
 * top-k, top-p on the top-k mass, min-p; the kept set is a prefix of the order value desc / index asc) without
 * sorting the row or forming the cut. Each round draws a candidate from the fixed-point CDF of a prefix of
 * that order (pivot_0 = its logit), counts the tokens and mass above pivot_0 and above pivot_1 = (pivot_0 +
 * high) / 2, accepts the candidate if it lies in the kept prefix, and otherwise shrinks the prefix. Rounds
 * are capped at 32; a row that reaches the cap takes the exact cut and one draw inside it.
 *   Random numbers: round r uses word 0 of Philox4x32-10 at counter (2^32 - 1 - r, row_id, step mod 2^32,
 *   step >> 32) with the row's key (the cap's draw uses r = 32). Tokens therefore differ from vsamp_sample's
 *   (which draws a Gumbel word per token); the law is the same.
 *   stats [B, 4] int32 or NULL: {passes over the row, rounds, 0, path flags; 64 = the cap was reached}.
 * Every other argument, the log-probability and the errors are as for vsamp_sample. One launch, one CTA per
 * row; the row is read from global memory at every pass. */
vsamp_status vsamp_sample_rejection(const void* logits, vsamp_dtype dt, int64_t B, int64_t V, int64_t ld,
                                    const float* temperature, const int32_t* top_k, const float* top_p,
                                    const float* min_p, const uint64_t* seed, const uint64_t* step,
                                    const uint32_t* row_id, int32_t* token, float* logprob, int32_t* row_status,
                                    int32_t* stats, void* stream);

/* ---------------------------------------------------------------------------------------------------
 * Vocabulary-sharded sampling ("[WS2][Logprob] Deterministic SM90 linear_logp ...", Tensor parallelism:
 * rank order + owned merge: each rank computes rank-local tile summaries over its vocabulary shard, the
 * partials are exchanged without reduction in transit (an all-gather) and placed in rank order, and one
 * fixed merge owned by the library folds them).
 *
 * A row's vocabulary [0, V) is split over R shards in rank order; shard r holds the logits [v0_r, v0_r + V_r)
 * of every row. Protocol:
 *   1. every shard calls vsamp_shard_partial on its logits: it writes NP piece records per row (the tile
 *      summaries: one per 4 KB piece of the shard) and one winner record per row;
 *   2. the records of all shards are gathered in rank order into recs [R, B, NP] and wins [R, B] (for
 *      example with an all-gather; on one device the shards simply write their slices of these arrays);
 *   3. vsamp_shard_merge folds them: the row maximum, log S (piece masses rescaled to the maximum and summed
 *      as integers), the drawn token and its log-probability, and the log-probability of a target token
 *      taken from the one shard that owns it.
 * The draw is a Philox4x32-10 Gumbel-max over the full temperature-scaled distribution (no top-k, top-p or
 * min-p: those cuts depend on the whole row). Max and arg-max decompose over shards, so the token equals the
 * unsharded vsamp_sample / vsamp_sample_ws token with top_k, top_p and min_p off. When every shard boundary
 * v0_r is a multiple of the piece length (2048 bf16 or 1024 fp32 logits), the records are exactly those of an
 * unsharded row, and every output is bit-identical to vsamp_sample_ws for any R; otherwise the fold differs
 * only in the last bits of S.
 * --------------------------------------------------------------------------------------------------- */
typedef struct vsamp_piece_rec {   /* 32 bytes: a piece's summary */
  float m;                         /* maximum (NaN: a non-finite value in the piece) */
  uint32_t cnt;                    /* elements equal to m */
  uint64_t s;                      /* sum of exp((x - m) / T) over the piece, 2^-40 fixed point */
  float mn;                        /* minimum */
  uint32_t reserved[3];
} vsamp_piece_rec;

typedef struct vsamp_shard_win {   /* 16 bytes: a shard's winner for one row */
  int32_t idx;                     /* global index of the shard's Gumbel-max winner (-1 on a row error) */
  float x;                         /* its logit */
  float xt;                        /* the target token's logit when this shard owns it */
  int32_t flags;                   /* bit 0: owns the target; bits 8..15: the shard's row status */
} vsamp_shard_win;

/* Piece records per row that a shard of V_shard logits of type dt writes (ceil(V_shard / piece)); the NP of
 * vsamp_shard_partial / vsamp_shard_merge is the largest of these over the shards (0 for invalid arguments). */
int64_t vsamp_shard_pieces(vsamp_dtype dt, int64_t V_shard);

/* Workspace bytes of vsamp_shard_partial for B rows of a shard of V_shard logits (0 for invalid arguments). */
size_t vsamp_shard_workspace_size(vsamp_dtype dt, int64_t B, int64_t V_shard);

/* Rank-local summaries of one vocabulary shard.
 *   logits     [B, ld] the shard's logits; element j of row r is the logit of token v0 + j.
 *   v0         the shard's first token (a multiple of 8 for bf16, 4 for fp32, so that the Philox groups of four
 *              tokens start inside the shard).
 *   NP         record slots per row in recs (>= vsamp_shard_pieces(dt, V_shard)); slots past the shard's pieces
 *              get empty records (maximum -inf, no mass).
 *   temperature, seed, step, row_id: as for vsamp_sample (the same arrays on every shard).
 *   target     [B] global token ids whose log-probability the merge reports, or NULL.
 *   recs       [B, NP] vsamp_piece_rec (device): this shard's slice of the gathered records.
 *   win        [B] vsamp_shard_win (device).
 *   workspace  device buffer of vsamp_shard_workspace_size bytes, 16-byte aligned (no initialisation needed).
 * Two launches on `stream`. */
vsamp_status vsamp_shard_partial(const void* logits, vsamp_dtype dt, int64_t B, int64_t V_shard, int64_t ld,
                                 int64_t v0, int64_t NP, const float* temperature, const uint64_t* seed,
                                 const uint64_t* step, const uint32_t* row_id, const int32_t* target,
                                 vsamp_piece_rec* recs, vsamp_shard_win* win, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* The owned merge of R shards' records, rank order: recs [R, B, NP], wins [R, B] (device).
 *   V          the full vocabulary size.
 *   outputs    [B] each, any may be NULL: row_max (fp32), row_logsum = log S at temperature T (T <= 0 read
 *              as 1), token (-1 on error), logprob = min((x_t - max) / T - log S, 0) of the drawn token,
 *              target_logprob of the target given to vsamp_shard_partial, row_status.
 *   Row errors: a non-finite logit or a NaN / infinite temperature; a requested target that no shard owns.
 * One launch on `stream`; it reads only the records, never the logits. */
vsamp_status vsamp_shard_merge(const vsamp_piece_rec* recs, const vsamp_shard_win* wins, int32_t R, int64_t B,
                               int64_t NP, int64_t V, const float* temperature, const uint64_t* seed,
                               const uint64_t* step, const uint32_t* row_id, float* row_max, float* row_logsum,
                               int32_t* token, float* logprob, float* target_logprob, int32_t* row_status,
                               void* stream);

/* Static description of a status code. */
const char* vsamp_status_string(vsamp_status s);

/* Limits on `device` (queried once per device and cached; thread-safe). Host pointer `out`. */
vsamp_status vsamp_device_info(int device, vsamp_limits* out);

/* ABI version: (major << 16) | minor. */
int32_t vsamp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VSAMP_H_ */
