/* Streaming log-mel front end on the GPU (C ABI): 16 kHz audio in, 128-bin
 * log-mel frames out, for many independent streams per call.
 *
 * What it computes (the same frames as a one-shot transform of the whole
 * signal, however the audio is split into pushes):
 *   - "Parakeet-EOU-120M — Streaming ASR Model", §Config: 16 kHz audio, a
 *     160-sample (10 ms) hop, 128 mel bins;
 *   - "Fast Accuracy-Preserving RNNT Beam Search on Apple Silicon", §1.3: a
 *     window of 240,000 samples gives 1,501 frames, i.e. frames centred on every
 *     hop with half a transform of zero padding on both sides;
 *   - "True streaming encode — implementation spec", §Status: padding only at
 *     the top of a stream and at the bottom on flush; streamed output equals
 *     the one-shot output.
 * Where those pages are silent this follows the usual filterbank front end:
 * pre-emphasis y[n] = x[n] - 0.97 x[n-1] (x[-1] = 0), a 512-point transform of
 * 400-sample frames weighted by a symmetric Hann window centred in the 512
 * points, frame t centred on sample 160 t of the pre-emphasised signal (zeros
 * before sample 0 and, on flush, after the last sample), power spectrum of the
 * 257 non-negative frequencies, 128 triangular filters from 0 to 8 kHz on the
 * Slaney mel scale each scaled by 2 / (bandwidth in Hz), natural log of
 * (energy + 2^-24).  No dither, no normalisation.  Arithmetic is fp32.
 *
 * Frame schedule: a push emits every frame whose 512-sample window lies
 * inside the samples received so far (frame t needs samples up to
 * 160 t + 255); a flush treats the rest as zeros and emits the frames a
 * one-shot transform of all N samples has, 1 + N / 160 in total.
 *
 * Ownership: the caller owns the audio and mel device buffers; the library
 * owns per-stream state (a 512-sample raw tail per stream on the device, sample
 * and frame counters on the host).  Calls are asynchronous on the given
 * cudaStream_t (0 = legacy default stream); calls for one front end must be
 * ordered (one CUDA stream, or the caller's own ordering).
 *
 * Errors: every call returns CAC_OK (0) or a negative CAC_E_* code of cac.h
 * and changes no state when it fails.  The kernels have no waits, so there is
 * no latched device status.
 */
#ifndef CAC_FRONTEND_H
#define CAC_FRONTEND_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct cac_frontend cac_frontend;

/* Stream ids 0 .. max_streams-1 (max_streams <= 65535) each own one front-end
 * state, all starting fresh.  Allocates on the current device. */
int cac_frontend_create(int max_streams, cac_frontend** out);
void cac_frontend_destroy(cac_frontend* fe);

/* Start the listed streams again (no samples, next frame 0, not flushed).
 * ids: host [n] stream ids.  Host-side only; the next push of a reset stream
 * reads no old device state. */
int cac_frontend_reset(cac_frontend* fe, int n, const int* ids);

/* Append n_samples new samples to each of n streams and emit their newly
 * complete frames.
 *   ids            host [n] distinct ids of streams not flushed since their reset
 *   audio          device fp32, slot b's samples at audio + b * audio_bstride
 *                  (may be NULL when n_samples == 0); audio_bstride >= n_samples
 *   mel            device fp32, slot b's frames at mel + b * mel_bstride,
 *                  frame f's 128 bins contiguous at + f * 128;
 *                  mel_bstride >= 128 * max_frames
 *   max_frames     capacity per slot; a push that would emit more returns
 *                  CAC_E_LIMIT and does nothing
 *   n_frames_out   host [n]: frames emitted per slot (known when the call
 *                  returns; the mel values are ready when the stream reaches
 *                  the call's work) */
int cac_frontend_push(cac_frontend* fe, int n, const int* ids, const float* audio, long long audio_bstride,
                      int n_samples, float* mel, long long mel_bstride, int max_frames, int* n_frames_out,
                      void* stream);

/* Last samples of each of n streams (n_samples_each: host [n], each >= 0, may
 * differ), then every remaining frame with zeros past the end; the streams are
 * finished until their reset.  Arguments otherwise as cac_frontend_push;
 * audio_bstride >= the largest n_samples_each. */
int cac_frontend_flush(cac_frontend* fe, int n, const int* ids, const float* audio, long long audio_bstride,
                       const int* n_samples_each, float* mel, long long mel_bstride, int max_frames,
                       int* n_frames_out, void* stream);

/* Host counters of one stream: samples received, frames emitted, flushed. */
int cac_frontend_get_state(const cac_frontend* fe, int id, long long* samples, long long* frames, int* finished);

/* The constant tables the kernel uses (host arithmetic only; needs no
 * device): window [512] (zero outside the centred 400 points), twiddles [256]
 * as (cos, -sin)(2 pi k / 512) pairs, and the mel filters as 16-bin rows:
 * mel_start [128] (first bin of row m) and mel_w [128][16] (weights of bins
 * mel_start[m] .. mel_start[m] + 15; every nonzero weight of filter m lies in
 * that span).  Each value is computed in fp64 and rounded once to fp32.
 * Returns CAC_OK, CAC_E_INVAL for a NULL pointer. */
int cac_frontend_tables(float* window, float* twiddles, int* mel_start, float* mel_w);

/* Frames a push (flush = 0) or a flush (flush = 1) of n_samples emits for a
 * stream that has received samples_before samples and emitted frames_before
 * frames (host arithmetic only; needs no device).  Returns the count, or
 * CAC_E_INVAL for negative arguments. */
long long cac_frontend_schedule(long long samples_before, long long frames_before, long long n_samples, int flush);

#ifdef __cplusplus
}
#endif

#endif /* CAC_FRONTEND_H */
