/* Batched modified-ALSD RNN-T beam search with an end-of-utterance class
 * (C ABI): many independent streams, beam width K <= 8, over projected encoder
 * frames that arrive chunk by chunk.
 *
 * Follows "Fast Accuracy-Preserving RNNT Beam Search on Apple Silicon":
 *   §2.2 — one alignment iteration: every running hypothesis takes the joint at
 *   its own frame, an fp32 log-softmax and its top K labels, adds its score;
 *   blank is forced where the per-frame symbol limit fired; the global top K
 *   of the K*K candidates survive (pruning first), identical survivors are then
 *   merged by log-sum-exp into the best-scoring one without refilling; the
 *   predictor advances on the selected labels and keeps the parent's state on
 *   blank; acoustic time advances only on blank.
 *   §2.3 — survivors are identical when transcript, last label and non-blank
 *   length match (compared here on the token sequences themselves).
 *   §2.4 — max_symbols forces blank; score normalisation orders the finals.
 *   §4.1 — fixed storage per stream: per-hypothesis score, time, last label,
 *   length, symbols at the current frame, predictor state and transcript.
 * The predictor and joint are those of cac_decode.h (fp32 single-layer LSTM on
 * the last non-blank class, its projection, joint = W_out ReLU(z + p) + b_out;
 * a stream starts from h = c = 0 and one predictor step on blank).
 *
 * Readings where the pages are silent: the beam starts as one hypothesis
 * (score 0, empty, last label blank) and K - 1 empty slots; a hypothesis at
 * the utterance's last frame is final and stays as one candidate with its
 * score; every top-K breaks ties to the lower index (class, then candidate
 * position parent * K + j); a hypothesis at the symbol limit offers only
 * blank; a merged hypothesis keeps all but the score from its best member.
 * Streaming: iterations keep every hypothesis at one alignment length, so the
 * search of a stream pauses when a running hypothesis needs a frame that has
 * not arrived and resumes on the next step; only a final step ends the
 * utterance.  The chunked search therefore equals the one-shot search.
 *
 * Class ids: tokens 0 .. vocab-1, blank = vocab, EOU = vocab + 1.
 * Errors: every call returns CAC_OK (0) or a negative CAC_E_* code of cac.h.
 * Device-side failures (a grid barrier that gave up, a transcript longer than
 * max_tokens) are latched and reported by cac_beam_check.
 */
#ifndef CAC_BEAM_H
#define CAC_BEAM_H

#include <stddef.h>

#include "cac_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct cac_beam cac_beam;

/* Weights: the host fp32 blob of cac_decoder_create (same layout and config).
 * beam: K, 1 .. 8.  max_streams: stream ids 0 .. max_streams-1, all starting
 * fresh.  max_tokens: transcript capacity per hypothesis; a label that would
 * exceed it is dropped from the search and CAC_E_LIMIT is latched. */
int cac_beam_create(const cac_dec_config* cfg, const float* weights, size_t n_floats, int beam, int max_streams,
                    int max_tokens, cac_beam** out);
void cac_beam_destroy(cac_beam* bd);

/* Start the listed streams again (host [n] ids); the device state is
 * re-initialised by their next step. */
int cac_beam_reset(cac_beam* bd, int n, const int* ids);

/* Advance n streams over T new projected encoder frames each.
 *   ids      host [n] distinct ids of streams not finished since their reset
 *   z        device fp32, slot b's new frame t at z + b * z_bstride + t * joint_dim
 *            (may be NULL when T == 0); frames continue the stream's earlier ones
 *   is_final 1: these are the utterance's last frames — the search runs to the
 *            end and the streams are finished until their reset; the call then
 *            waits for the device (it relaunches until every stream is done)
 *   0 < T <= 1024 unless is_final (T = 0 allowed).  Asynchronous on `stream`
 *   (a cudaStream_t, 0 = legacy default) when is_final == 0. */
int cac_beam_step(cac_beam* bd, int n, const int* ids, const float* z, long long z_bstride, int T, int is_final,
                  void* stream);

/* Reads the device status word (synchronises); returns and clears the first
 * latched error (CAC_E_TIMEOUT, CAC_E_LIMIT) or CAC_OK. */
int cac_beam_check(cac_beam* bd);

/* The beam of one stream (synchronises the device): scores [K] (-inf for an
 * empty slot), lengths [K], tokens [K][max_tokens] (the first lengths[k] of
 * row k), and in *best the slot that wins by score / (length + 1) when
 * score_norm, else by score (ties to the lower slot).  Output pointers are
 * host memory; tokens may be NULL. */
int cac_beam_get(cac_beam* bd, int id, int score_norm, float* scores, int* lengths, int* tokens, int* best);

#ifdef __cplusplus
}
#endif

#endif /* CAC_BEAM_H */
