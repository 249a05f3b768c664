/*
 * spec_verify_shard.h -- the verify step over a vocabulary split across ranks.
 *
 * Where this comes from.  The DFlash/Spec V2 page serves its large target
 * with tensor parallelism 8 on one 8-GPU node and fuses the all-reduce into
 * its kernels (section "A4 实验环境与运行配置": hardware TP=8, launch flag
 * --enable-flashinfer-allreduce-fusion).  A tensor-parallel LM head leaves
 * each rank the logits of one vocabulary range only: rank q holds columns
 * [v_q, v_q + V_q) of every target and every draft row, the ranges tiling
 * [0, V) in rank order.  The verify step (spec_verify.h: accept test
 * u * p_d(x) < p_t(x), the first rejection, the replacement or bonus draw
 * over ascending ids, the label c* = sum_v min(p_t, p_d), greedy argmax)
 * needs statistics over the whole vocabulary, so the ranks exchange three
 * small per-row buffers.  The results are those of spec_verify on the whole
 * rows: the same rules, only the fp32 summation order differs.
 *
 * Protocol (every rank runs every step on its own stream; the library does
 * no communication -- between steps the caller all-gathers the named buffer
 * of every rank, in rank order, into one [world, ...] array, by NCCL, gloo,
 * or a plain copy when all shards live on one device):
 *
 *   1. spec_verify_shard_stats  -> rec   [N_t][SV_SHARD_REC_WORDS]   (all-gather)
 *      spec_verify_shard_merge  <- recs  [world][N_t][...]
 *         row statistics over the whole vocabulary, the accept decisions,
 *         the first rejection a_r and accepted tokens of every request;
 *         greedy: also the final token.
 *   2. spec_verify_shard_masses -> mass  [N_t][SV_SHARD_MASS_WORDS]  (all-gather)
 *         per row this rank's share of sum min(p_t, p_d), of the residual
 *         sum max(0, p_t - p_d) and of sum p_t.  Needed for labels or for
 *         sampling.
 *   3. spec_verify_shard_draw   <- masses [world][N_t][...]
 *         labels (shares summed in rank order); sampling: the rank whose
 *         range holds the draw walks its range, every other rank reports
 *         -1  -> cand [B]                                        (all-gather)
 *      spec_verify_shard_finish <- cands [world][B]: the final token.
 *
 * Every rank computes the same merged statistics, decisions and labels
 * bit for bit (the same kernels over the same gathered bytes, summed in
 * rank order), so no rank has to broadcast them.  Only unfiltered calls are
 * taken (top_k and top_p over a split vocabulary would need a distributed
 * select); at most SV_SHARD_MAX_WORLD ranks.
 *
 * Layout, ownership, streams, errors: as in spec_verify.h.  Row r's target
 * rows, draft rows and uniforms are placed as there; N_t = row_offsets[B],
 * N_d = N_t - B.  Shard logits are row-major [N_t, V_q] and [N_d, V_q] with
 * row stride V_q elements and need only element alignment (2 bytes for
 * bf16, 4 for fp32); every other device pointer is 4-byte aligned.  Drafted
 * tokens are ids of the whole vocabulary [0, V).  Every call only enqueues
 * work on `stream` and returns without synchronising; host-visible argument
 * errors (SV_ERR_*) are returned before anything is enqueued; data problems
 * are OR-ed into *dev_error (SV_DEVERR_*).  The buffers of one rank's steps
 * are ordered by its stream; the gathered arrays must be complete before the
 * step that reads them is enqueued.
 */
#ifndef SPEC_VERIFY_SHARD_H
#define SPEC_VERIFY_SHARD_H

#include "spec_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

#define SV_SHARD_MAX_WORLD 32 /* ranks of one split */

/* Step 1 record of one target row (int32 words; floats stored bit for bit):
 * this rank's partial statistics of the target row and of its draft partner
 * as sum_v 2^(x_v sc) = s 2^h with sc = log2(e) / T, the raw maximum and
 * the lowest id holding it (ids of the whole vocabulary), the two logits at
 * the drafted token when this rank holds it, and error bits. */
#define SV_SHARD_REC_WORDS 12
enum {
  SV_SREC_HT = 0, SV_SREC_ST, SV_SREC_MT, SV_SREC_IT,
  SV_SREC_HD, SV_SREC_SD, SV_SREC_MD, SV_SREC_ID,
  SV_SREC_XT, SV_SREC_XD, SV_SREC_HASX, SV_SREC_FLAGS
};

/* Merged row of step 1 (written by spec_verify_shard_merge, read by the
 * later steps): reference h and normaliser z of the target row (p_t(v) =
 * 2^(x_v sc - h_t) / z_t) and of the draft partner, the target argmax, the
 * accept decision of the row's drafted token, its error bits, and a pad
 * word. */
#define SV_SHARD_ROW_WORDS 8
enum {
  SV_SROW_HT = 0, SV_SROW_ZT, SV_SROW_HD, SV_SROW_ZD,
  SV_SROW_ARGT, SV_SROW_ACC, SV_SROW_FLAGS, SV_SROW_PAD
};

/* Step 2 shares of one target row, float32: sum over this rank's range of
 * min(p_t, p_d) (drafted rows), of max(0, p_t - p_d) (drafted rows), and of
 * p_t (every row). */
#define SV_SHARD_MASS_WORDS 4
enum { SV_SMASS_C = 0, SV_SMASS_R, SV_SMASS_P, SV_SMASS_PAD };

/*
 * Step 1, this rank: partial statistics of its columns of every target row
 * and draft partner.
 *  target_shard  [N_t, V_shard] device, dtype.
 *  draft_shard   [N_d, V_shard] device, dtype; may be NULL when N_d == 0.
 *  V_shard       columns held here (>= 1); v_begin their first id;
 *                v_begin + V_shard <= V.
 *  draft_tokens  [N_d] int32 ids in [0, V) (others raise SV_DEVERR_TOKEN in
 *                the merge).
 *  verify_lens, row_offsets, B, n_target_rows, max_len: as spec_verify.
 *  temperature   > 0 and finite.
 *  out_rec       [N_t][SV_SHARD_REC_WORDS] int32 device.
 * Data errors (NaN or +inf in a row) are recorded in the row's
 * SV_SREC_FLAGS word and raised by the merge.
 */
int spec_verify_shard_stats(const void* target_shard, const void* draft_shard, int32_t V_shard,
                            int32_t v_begin, int32_t V, const int32_t* draft_tokens,
                            const int32_t* verify_lens, const int32_t* row_offsets, int32_t B,
                            int32_t n_target_rows, int32_t max_len, int32_t dtype,
                            float temperature, int32_t* out_rec, void* stream);

/*
 * Step 1, every rank: merge the gathered records.
 *  recs           [world][N_t][SV_SHARD_REC_WORDS] int32 device, rank order.
 *  world          1 .. SV_SHARD_MAX_WORLD.
 *  uniforms       [N_t] float32 device, as spec_verify.
 *  mode           SV_GREEDY or SV_SAMPLE.
 *  out_merged     [N_t][SV_SHARD_ROW_WORDS] int32 device.
 *  out_tokens     [N_t] int32: the accepted drafts, -1 after the final
 *                 token; greedy also writes the final token (the argmax of
 *                 row a_r), sampling leaves it to spec_verify_shard_finish.
 *  out_accept_len [B] int32: a_r.
 *  out_row_stats  [N_t + N_d][3] float32 or NULL: m = max z, Z = sum
 *                 exp(z - m), argmax (int32 bits), as spec_verify.
 */
int spec_verify_shard_merge(const int32_t* recs, int32_t world, const int32_t* draft_tokens,
                            const float* uniforms, const int32_t* verify_lens,
                            const int32_t* row_offsets, int32_t B, int32_t V,
                            int32_t n_target_rows, int32_t max_len, float temperature,
                            int32_t mode, int32_t* out_merged, int32_t* out_tokens,
                            int32_t* out_accept_len, float* out_row_stats, int32_t* dev_error,
                            void* stream);

/*
 * Step 2, this rank: its shares of the masses, given the merged statistics.
 *  all_rows   1: every target row (labels wanted); 0: only the stopping row
 *             off_r + a_r of each request (sampling without labels).
 *  accept_len [B] int32 device: a_r from the merge.
 *  out_mass   [N_t][SV_SHARD_MASS_WORDS] float32 device; rows not visited
 *             are left as they are.
 */
int spec_verify_shard_masses(const void* target_shard, const void* draft_shard, int32_t V_shard,
                             const int32_t* merged, const int32_t* verify_lens,
                             const int32_t* row_offsets, const int32_t* accept_len, int32_t B,
                             int32_t n_target_rows, int32_t max_len, int32_t dtype,
                             float temperature, int32_t all_rows, float* out_mass, void* stream);

/*
 * Step 3, every rank: labels and, sampling, the draw on the rank that owns
 * it.  The draw follows spec_verify: the residual masses R_q of the ranks
 * are summed in rank order; a residual at or below 2^-21 falls back to p_t
 * (the masses P_q); the target u * total (u of the request's last row)
 * picks the first rank whose running sum passes it, and that rank walks
 * its columns in ascending id with the mass left over (strict ">").
 *  masses    [world][N_t][SV_SHARD_MASS_WORDS] float32 device, rank order.
 *  rank      this rank (0 .. world - 1); target_shard, draft_shard,
 *            V_shard, v_begin: its columns, as in step 1.
 *  out_conf  [N_d] float32 or NULL: c* of every drafted row.
 *  out_cand  [B] int32 (sampling; may be NULL for greedy): the drawn token
 *            where this rank owns the draw, else -1.
 */
int spec_verify_shard_draw(const float* masses, int32_t world, int32_t rank,
                           const void* target_shard, const void* draft_shard, int32_t V_shard,
                           int32_t v_begin, const int32_t* merged, const float* uniforms,
                           const int32_t* verify_lens, const int32_t* row_offsets,
                           const int32_t* accept_len, int32_t B, int32_t n_target_rows,
                           int32_t max_len, int32_t dtype, float temperature, int32_t mode,
                           float* out_conf, int32_t* out_cand, int32_t* dev_error, void* stream);

/*
 * Step 3, every rank: the final token of each request from the gathered
 * candidates (exactly one rank owns each draw).  A request with no owner
 * (no mass anywhere: non-finite statistics) raises SV_DEVERR_NAN and takes
 * the target argmax of its stopping row.
 *  cands  [world][B] int32 device, rank order.
 */
int spec_verify_shard_finish(const int32_t* cands, int32_t world, const int32_t* merged,
                             const int32_t* verify_lens, const int32_t* row_offsets,
                             const int32_t* accept_len, int32_t B, int32_t n_target_rows,
                             int32_t* out_tokens, int32_t* dev_error, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_SHARD_H */
