/* Batched greedy RNN-T decoding with an end-of-utterance class (C ABI).
 *
 * Follows "Parakeet-EOU-120M — Streaming ASR Model", §Architecture (an fp32
 * single-step LSTM predictor on the previous non-blank token; a joint over one
 * projected encoder frame and the predictor output giving logits for
 * vocabulary + blank + EOU; greedy decoding per encoder frame that advances the
 * predictor only on non-blank emissions) and "True streaming encode —
 * implementation spec", §Decoder state carry (per-stream h/c kept across calls;
 * a reset starts a stream from the blank token).  Projections are hoisted as
 * in "Fast Accuracy-Preserving RNNT Beam Search on Apple Silicon", §3: the
 * encoder frames arrive already projected (the encoder's joint projection), the
 * predictor output is projected once per emitted prefix.
 *
 * Class ids: tokens 0 .. vocab-1, blank = vocab, EOU = vocab + 1.  An argmax
 * tie goes to the lowest id.  After max_symbols emissions on one frame the
 * decoder moves to the next frame.  EOU is a non-blank emission: it is output
 * and the predictor advances on it.  All arithmetic is fp32.
 *
 * Errors: every call returns CAC_OK (0) or a negative CAC_E_* code of cac.h;
 * device-side failures (a grid barrier that gave up) are latched and reported
 * by cac_decoder_check.
 */
#ifndef CAC_DECODE_H
#define CAC_DECODE_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct cac_dec_config {
    int vocab;        /* tokens; classes = vocab + 2 (blank, EOU) */
    int pred_dim;     /* LSTM width (embedding and hidden), multiple of 64 */
    int joint_dim;    /* width of both joint projections, multiple of 64 */
    int max_symbols;  /* emissions per encoder frame before a forced blank, >= 1 */
} cac_dec_config;

typedef struct cac_decoder cac_decoder;

/* Weights: host fp32 blob, concatenated in this order (linears [out][in]):
 *   emb [C][P], lstm.w_ih [4P][P], lstm.w_hh [4P][P], lstm.b_ih [4P],
 *   lstm.b_hh [4P], pred.w [J][P], pred.b [J], out.w [C][J], out.b [C]
 * with C = vocab + 2, P = pred_dim, J = joint_dim; LSTM gate rows in the order
 * input, forget, cell, output.  The library copies what it needs to the current
 * device; the caller keeps the blob.  max_streams: stream ids 0 .. max_streams-1
 * each own one predictor state (h, c and its projection), all starting reset.
 * Every CTA of the step kernel keeps a copy of the per-slot decoding state in
 * shared memory beside its weight slices, which bounds max_streams (about
 * 1,600 for the 1024-token, 640-wide decoder on a 152-SM GPU); beyond that,
 * or for pred_dim / joint_dim above 1024, the call returns CAC_E_UNSUPPORTED. */
int cac_decoder_create(const cac_dec_config* cfg, const float* weights, size_t n_floats, int max_streams,
                       cac_decoder** out);
void cac_decoder_destroy(cac_decoder* d);

/* Mark streams as starting: their next step begins from h = c = 0 with one
 * predictor step on the blank token.  ids: host array of n stream ids.
 * Asynchronous on `stream` (a cudaStream_t, 0 = legacy default). */
int cac_decoder_reset(cac_decoder* d, int n, const int* ids, void* stream);

/* One decoding step of n streams over T projected encoder frames each.
 *   ids     host [n] distinct stream ids
 *   z       device fp32, slot b's frame t at z + b * z_bstride + t * joint_dim
 *   tokens  device int32 [n][T * max_symbols]: emitted class ids in order
 *   frames  device int32 [n][T * max_symbols]: frame (0 .. T-1) of each emission
 *   counts  device int32 [n]: emissions of the slot
 * T = 0 decodes nothing (z, tokens, frames may be NULL) but still sets counts to 0 and primes
 * reset streams.  T <= 1024.
 * Entries of tokens/frames past counts[b] are left unchanged.  Pointers must be
 * 4-byte aligned, z 16-byte aligned with z_bstride a multiple of 4.
 * Asynchronous on `stream`; the per-stream state is updated on the device.
 * Calls on one decoder (step and reset) share its device scratch and pinned
 * id slots: issue them on one CUDA stream, or order them across streams. */
int cac_decoder_step(cac_decoder* d, int n, const int* ids, const float* z, long long z_bstride, int T,
                     int* tokens, int* frames, int* counts, void* stream);

/* Synchronizes and returns CAC_OK or the latched device error (and clears it). */
int cac_decoder_check(cac_decoder* d);

/* Copy one stream's predictor state to the host: h [P], c [P], p [J]
 * (p = the predictor projection of h) and primed (0 after a reset until the
 * next step).  Synchronous. */
int cac_decoder_get_state(cac_decoder* d, int id, float* h, float* c, float* p, int* primed);

#ifdef __cplusplus
}
#endif

#endif
