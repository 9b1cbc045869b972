/*
 * cac.h — C ABI of the GB300 cache-aware Conformer streaming encoder.
 *
 * The operation is the cache-aware Conformer encoder chunk step of the
 * streaming Parakeet-EOU RNN-T recognizer, batched over many independent
 * streams ("True streaming encode — implementation spec", §Per-chunk flow):
 *   1. mel staging over [melTail | new mel] (14-frame tail, §State),
 *   2. causal 8x subsampling, causal padding only at stream start,
 *   3. per layer: FF1, LN -> Q/K/V, rectangular rel-pos attention over
 *      [kCache | K_new] with the chunked-causal mask on absolute positions,
 *      softmax, probs@V, pw1 + GLU, causal depthwise conv over
 *      [convCache | glu_new], pw2, FF2, ln_out, K/V and conv cache update,
 *   4. the encoder-side joint projection of every new frame (640 wide,
 *      "Fast Accuracy-Preserving RNNT Beam Search", §1.3).
 * Stream life cycle and API shape follow the same page's §Goal / §Status
 * (push / reset / finish, createEncodeStream / encodeStreamPush /
 * encodeStreamFlush) and the explicit state tensors of "Parakeet-EOU-120M —
 * Streaming ASR Model", §Architecture.  The offline encode is the full-sequence
 * pass with the same mask, which already emulates streaming ("True streaming
 * encode", §Why this is provably correct).
 *
 * Conventions
 *   - Every call returns CAC_OK (0) or a negative CAC_E_* code; no call throws.
 *   - "device" pointers are CUDA global memory on the model's device, owned by
 *     the caller, and must stay valid until the work queued on `stream`
 *     completes.  "host" pointers are read or written before the call returns
 *     unless stated otherwise.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls that take it are asynchronous on it.  All calls on one
 *     pool must be ordered: issue them on one stream (or synchronize between).
 *   - Layouts are row-major, float32 unless stated.  mel frames are
 *     [frames][mel_bins]; encoder frames [frames][d_model]; joint frames
 *     [frames][joint_dim].
 *   - The library owns weights, per-stream state pools and scratch.
 *   - Errors detected on the device (a non-finite input, a bounded wait that
 *     gave up) are latched in a device status word and reported by
 *     cac_pool_check() / cac_model_check().
 */
#ifndef CAC_H_
#define CAC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define CAC_OK          0
#define CAC_E_INVAL    -1   /* bad argument (null pointer, id out of range, duplicate id, bad config) */
#define CAC_E_ALIGN    -2   /* push not a multiple of att_chunk * 8 mel frames (160 ms for chunk 2) */
#define CAC_E_STATE    -3   /* wrong stream state (push after flush without reset, dead id) */
#define CAC_E_NOMEM    -4   /* device or pinned-host allocation failed, or pool full */
#define CAC_E_CUDA     -5   /* a CUDA runtime/driver call failed */
#define CAC_E_DEVICE   -6   /* an error latched on the device (see cac_pool_check) */
#define CAC_E_NONFINITE -7  /* non-finite value found in an input mel chunk */
#define CAC_E_TIMEOUT  -8   /* a bounded device-side wait gave up */
#define CAC_E_UNSUPPORTED -9 /* configuration outside what the kernels implement */
#define CAC_E_LIMIT    -10  /* request larger than the fixed scratch of cac_encode_offline_noalloc */
#define CAC_E_BOUNDS   -11  /* an index outside its buffer: caught (and the access skipped) by the checked
                               build, or a pool guard zone found overwritten (cac_pool_check_guards) */

#define CAC_DTYPE_F32  0    /* everything fp32 (SIMT GEMMs) */
#define CAC_DTYPE_BF16 1    /* bf16 weights, GEMM operands and caches; fp32 accumulation,
                               residual stream, LayerNorm, softmax and conv arithmetic */

/* Model shape.  Parakeet-EOU-120M: 17 layers, d_model 512, 8 heads, ff 2048,
 * dw_kernel 9, att_left 70, att_chunk 2, 128 mel bins, joint 640
 * ("Parakeet-EOU-120M", §Config; "True streaming encode", §State). */
typedef struct cac_config {
    int32_t n_layers;
    int32_t d_model;
    int32_t n_heads;
    int32_t ff_dim;
    int32_t dw_kernel;       /* must be 9 (conv cache of 8 columns) */
    int32_t att_left;        /* left attention context in subsampled frames (70) */
    int32_t att_chunk;       /* chunk of the chunked-causal mask (2 = 160 ms) */
    int32_t mel_bins;        /* must be 128 */
    int32_t joint_dim;       /* encoder-side joint projection width (640) */
    int32_t dtype;           /* CAC_DTYPE_* */
    int32_t right_context;   /* 0: chunked-causal (exact streaming).  >0: window mask
                                [p - att_left, p + right_context] with a provisional tail */
    int32_t emit_frames;     /* provisional tail: frames emitted per pass (C*k) */
    int32_t lookahead_frames;/* provisional tail: extra frames computed per pass (B) */
    int32_t gemm_simt;       /* debugging aid: 1 runs bf16 GEMMs on the SIMT kernel
                                instead of tcgen05 (same arithmetic, slower) */
} cac_config;

typedef struct cac_model cac_model;
typedef struct cac_pool cac_pool;

/* Number of floats in the weight blob for `cfg`.  The blob is the
 * concatenation, in this order, of (all linears [out][in], subsampling convs
 * [out][tap][in], depthwise [channel][tap]):
 *   sub.w1[D][3][mel] sub.b1[D] sub.w2[D][3][D] sub.b2[D] sub.w3[D][3][D] sub.b3[D]
 *   sub.wo[D][D] sub.bo[D]
 *   per layer l:
 *     ff1.ln_g[D] ff1.ln_b[D] ff1.w1[F][D] ff1.b1[F] ff1.w2[D][F] ff1.b2[D]
 *     att.ln_g[D] att.ln_b[D] att.wq[D][D] att.bq[D] att.wk[D][D] att.bk[D]
 *     att.wv[D][D] att.bv[D] att.wo[D][D] att.bo[D] att.wpos[D][D]
 *     att.pbu[H][D/H] att.pbv[H][D/H]
 *     conv.ln_g[D] conv.ln_b[D] conv.w_pw1[2D][D] conv.b_pw1[2D] conv.w_dw[D][9]
 *     conv.b_dw[D] conv.bn_g[D] conv.bn_b[D] conv.w_pw2[D][D] conv.b_pw2[D]
 *     ff2.(same six as ff1) out.ln_g[D] out.ln_b[D]
 *   joint.w[J][D] joint.b[J]
 * Returns 0 for an invalid config. */
size_t cac_weights_size(const cac_config* cfg);

/* Create a model on the current CUDA device from a host fp32 blob of
 * `n_floats` values (layout above).  In bf16 mode the values are rounded to
 * bf16 on upload.  The caller keeps ownership of `weights`. */
int  cac_model_create(const cac_config* cfg, const float* weights, size_t n_floats, cac_model** out);

/* The same model with its weight matrices stored as 6-bit palettes ("Fast
 * Accuracy-Preserving RNNT Beam Search on Apple Silicon", §1.3: the encoder
 * keeps every matrix as a 64-entry lookup table and 6-bit indices; vectors
 * and the depthwise taps stay dense).  bf16 mode on the tcgen05 path only
 * (else CAC_E_UNSUPPORTED).
 *   weights  the dense blob of cac_model_create, every palettised matrix
 *            holding its decoded values (table entries);
 *   tables   host fp32 [n_tables / 64][64], one table per matrix in this order:
 *            sub.w1, sub.w2, sub.w3, sub.wo, joint.w, then for each layer
 *            ff1.w1, ff1.w2, att.wq, att.wk, att.wv, att.wo, att.wpos,
 *            conv.w_pw1, conv.w_pw2, ff2.w1, ff2.w2 (n_tables = 64 (5 + 11 L));
 *            every entry a bf16 value.
 * The library finds each weight's index in its matrix's table (exact match,
 * the lowest index among equal entries), packs the indices 6 bits per weight
 * (0.75 bytes instead of 2) and the projections' GEMMs decode them into bf16
 * tiles on the device; att.wpos only enters the position table computed at
 * load.  A weight absent from its table, or a table entry that is not a bf16
 * value, returns CAC_E_INVAL.  The caller keeps ownership of both arrays. */
int  cac_model_create_palette(const cac_config* cfg, const float* weights, size_t n_floats, const float* tables,
                              size_t n_tables, cac_model** out);
void cac_model_destroy(cac_model* m);

/* Per-stream state pool for up to `max_streams` concurrent streams and at
 * most `max_frames_per_step` subsampled frames per internal step (1..8;
 * larger pushes are split into several steps).  Allocates the GPU-resident
 * caches: K/V rings [streams][layers][heads][R][head_dim], conv tail
 * [streams][layers][8][d_model], melTail [streams][14][128] (fp32), subT. */
int  cac_pool_create(cac_model* m, int max_streams, int max_frames_per_step, cac_pool** out);
void cac_pool_destroy(cac_pool* p);

/* Stream ids are small integers in [0, max_streams). */
int  cac_stream_create(cac_pool* p, int* id);
int  cac_stream_destroy(cac_pool* p, int id);

/* reset(): zero subT, the caches and melTail of the listed host `ids` (the
 * caches are invalidated by position, so no memory is cleared); queued on
 * `stream`, ordered before later pushes on the same stream. */
int  cac_stream_reset(cac_pool* p, int n, const int* ids, void* stream);

/* push(): encode `n_mel` new mel frames for each of `n` streams.
 *   ids   host [n] distinct live, unfinished stream ids
 *   mel   device [n][n_mel][mel_bins]
 *   enc   device [n][n_mel/8][d_model]   (may be NULL)
 *   joint device [n][n_mel/8][joint_dim] (may be NULL)
 *   n_out host [n], receives the frames emitted per stream; stream b's frames
 *         are rows 0 .. n_out[b]-1 of its enc/joint slab
 * Chunked-causal mode: n_mel must be a positive multiple of 8*att_chunk
 * (CAC_E_ALIGN otherwise); exactly n_mel/8 frames are emitted per stream.
 * Provisional-tail mode: n_mel must be a positive multiple of 8*emit_frames;
 * a stream emits frames only once lookahead_frames of lookahead exist, so
 * n_out[b] may be 0 (a fresh stream filling its lookahead). */
int  cac_stream_push(cac_pool* p, int n, const int* ids, const float* mel, int n_mel,
                     float* enc, float* joint, int* n_out, void* stream);

/* Same as cac_stream_push with HOST buffers: copies mel in and enc/joint out
 * on `stream` and synchronizes `stream` before returning (enc/joint are valid
 * on return).  Page-locked caller buffers (cudaHostAlloc / cudaHostRegister)
 * are copied directly; pageable ones go through pinned staging owned by the
 * pool (one extra host copy each way). */
int  cac_stream_push_host(cac_pool* p, int n, const int* ids, const float* mel, int n_mel,
                          float* enc, float* joint, int* n_out, void* stream);

/* Asynchronous form of cac_stream_push_host: queues the copy of mel in, the
 * push and the copies of enc/joint out on `stream`, and returns without
 * waiting for them.  mel, enc and joint (enc/joint may be NULL) must be
 * page-locked host memory (cudaHostAlloc / cudaHostRegister); a pageable
 * buffer returns CAC_E_INVAL before anything is queued.  Until `stream` has
 * passed this call's work (cudaStreamSynchronize, or an event recorded on
 * `stream` after the call), the caller must not modify mel nor read or reuse
 * enc/joint.  n_out is written before the call returns.  A caller can thus
 * queue push k+1 while push k runs and read push k's frames meanwhile, so the
 * GPU does not idle while the host prepares the next chunk.  The first call
 * (and one needing larger buffers than any before it) grows the pool's
 * device staging and synchronizes `stream` to do so. */
int  cac_stream_push_host_async(cac_pool* p, int n, const int* ids, const float* mel, int n_mel,
                                float* enc, float* joint, int* n_out, void* stream);

/* flush(): final partial chunk of each listed stream; afterwards the stream
 * needs cac_stream_reset before it can push again.
 *   mel        device [n][mel_stride][mel_bins]; stream b uses its first
 *              n_mel_each[b] (>= 0) frames
 *   enc/joint  device [n][out_stride][d_model / joint_dim] (may be NULL)
 *   n_out_each host [n] receives ceil(n_mel_each[b] / 8) in chunked mode, and
 *              every frame still held back in provisional-tail mode
 * out_stride must be >= the largest n_out_each (see cac_stream_flush_frames). */
int  cac_stream_flush(cac_pool* p, int n, const int* ids, const float* mel, int mel_stride,
                      const int* n_mel_each, float* enc, float* joint, int out_stride,
                      int* n_out_each, void* stream);
/* Frames the flush of stream `id` with `n_mel` remaining mel frames emits. */
int  cac_stream_flush_frames(cac_pool* p, int id, int n_mel, int* frames);

/* Offline chunked-causal encode of B independent windows (no streaming state).
 *   mel     device [B][t_mel_max][mel_bins]; window b uses mel_len[b] frames
 *   mel_len host [B], 1 <= mel_len[b] <= t_mel_max
 *   enc     device [B][T][d_model], T = ceil(ceil(ceil(t_mel_max/2)/2)/2)
 *   joint   device [B][T][joint_dim] (may be NULL)
 *   out_len host [B] receives ceil(ceil(ceil(mel_len[b]/2)/2)/2)
 * Frames past out_len[b] are unspecified.  Scratch is owned by the model and
 * grows on demand (the growth synchronizes `stream`). */
int  cac_encode_offline(cac_model* m, int B, const float* mel, const int* mel_len, int t_mel_max,
                        float* enc, float* joint, int* out_len, void* stream);

/* cac_encode_offline without allocation.  No counterpart on the pages: this
 * entry point exists for callers that may not allocate device memory once
 * they are running.  cudaMalloc can block the calling thread and synchronize
 * the device, which a real-time audio callback cannot afford, and some hosts
 * hand the library a fixed device-memory budget up front (a sandbox, a
 * serving process that reserves memory per model at start).
 * cac_encode_offline grows a model-owned workspace with cudaMalloc when a
 * larger batch arrives; this variant runs the same kernels on a fixed array of
 * CAC_NOALLOC_SCRATCH_BYTES (32 MiB) that the library declares in device
 * memory: every GPU that loads the library holds it until the process exits.
 *   - Arguments, layouts and results are those of cac_encode_offline.
 *   - Requests whose scratch exceeds the array (roughly B x t_mel_max beyond
 *     ~11,000 mel frames for the 17-layer d_model-512 model, less for wider
 *     models) return CAC_E_LIMIT and do nothing.
 *   - It calls no cudaMalloc / cudaFree and no allocating library routine.
 *     It copies the B lengths from mel_len to the device and waits for that
 *     copy on `stream` before it returns (mel_len may be pageable memory).
 *   - The model's device must be the current device (CAC_E_INVAL otherwise):
 *     the array used is the current device's.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - All calls on a device share the one array and leave their contents in
 *     it; calls whose GPU work overlaps (different streams, or different
 *     models, without ordering between them) race on it and must be
 *     serialized by the caller. */
#define CAC_NOALLOC_SCRATCH_BYTES (32u << 20)
int  cac_encode_offline_noalloc(cac_model* m, int B, const float* mel, const int* mel_len, int t_mel_max,
                                float* enc, float* joint, int* out_len, void* stream);

/* Logical state of one stream, for snapshots and migration ("Parakeet-EOU-120M",
 * §Architecture: state tensors passed in and returned each step).  All
 * buffers are host memory sized by the caller (NULL skips that part):
 *   mel_tail   [14][mel_bins]                rows oldest first (zeros before start)
 *   k_cache    [n_layers][att_left][d_model] rows oldest first; first Lc rows valid
 *   v_cache    [n_layers][att_left][d_model]
 *   conv_cache [n_layers][8][d_model]        GLU outputs, oldest first
 * get_state synchronizes the device; set_state is visible to the next push. */
typedef struct cac_stream_state {
    int32_t subT;      /* subsampled frames consumed (emitted, in chunked mode) */
    int32_t Lc;        /* valid attention-cache rows = min(subT, att_left) */
    int32_t finished;  /* 1 after flush */
    int32_t x0_rows;   /* provisional tail: subsampled frames waiting to be emitted */
    float* mel_tail;
    float* k_cache;
    float* v_cache;
    float* conv_cache;
    float* x0;         /* provisional tail only: [emit_frames + lookahead_frames][d_model] */
} cac_stream_state;

int  cac_stream_get_state(cac_pool* p, int id, cac_stream_state* st);
int  cac_stream_set_state(cac_pool* p, int id, const cac_stream_state* st);

/* Synchronize the device and return the latched device status (CAC_OK,
 * CAC_E_NONFINITE, CAC_E_TIMEOUT ...), clearing it. */
int  cac_pool_check(cac_pool* p);
int  cac_model_check(cac_model* m);

/* Capture each (batch, frames, buffers) step shape into a CUDA graph on its
 * second use and replay it afterwards (1), or launch kernels directly (0,
 * default). */
int  cac_pool_set_graphs(cac_pool* p, int enable);

/* Kernels this library launched on the pool since creation (a host-side
 * counter; a graph replay counts its kernel nodes). */
long long cac_pool_launch_count(cac_pool* p);

/* The number of concurrent sub-batches a push of n_streams streams with
 * n_frames frames each runs as (1 when the step is not split; a profiled push
 * keeps the split).  Host-only; CAC_E_INVAL for bad arguments. */
int  cac_pool_sub_batches(cac_pool* p, int n_streams, int n_frames);

/* Chained steps (1): on the tensor-core path a chunked step runs the
 * projections and LayerNorms between two attention launches as one
 * persistent kernel whose 128-row blocks advance phase by phase on
 * completion counters ("True streaming encode", §Per-chunk flow steps 2-4,
 * as one submission per stretch of the layer stack), all streams as one
 * batch.  0 (default): one launch per projection, the step split into
 * concurrent sub-batches of 64 streams, each replayed from its own CUDA
 * graph — measured faster on a GB300 (1.43 against 3.2 ms for 256 streams),
 * because a chained phase's latency (main loop, epilogue, completion signal)
 * is exposed while the sub-batches overlap one another's.  Both compute the
 * same step; split-K sums differ in order only.  Synchronizes the device.
 * CAC_CHAIN=1 in the environment turns chains on for every pool. */
int  cac_pool_set_chains(cac_pool* p, int enable);

/* Per-layer intermediate taps of the most recent push, for kernel-level
 * parity checks.  enable=1 makes every later push copy, per layer, the fp32
 * rows of: 0 x after FF1, 1 attention output before the out-projection,
 * 2 x after attention, 3 GLU output, 4 conv-module activation before pw2,
 * 5 x after the conv module, 6 x after ln_out; tap 7 = subsampled input x0
 * (layer ignored).  Rows are the last internal step's [n][frames]. */
int  cac_pool_set_trace(cac_pool* p, int enable);
int  cac_pool_read_trace(cac_pool* p, int layer, int tap, float* host, size_t n_floats);

/* Per-kernel-class timing with CUDA events recorded on the launching stream
 * around every kernel of later pushes and resets (launches run eagerly while
 * enabled).  cac_pool_read_profile synchronizes the device and fills, for each
 * class 0 .. cac_profile_classes()-1, the summed kernel time in ms and the
 * launch count since the previous read, then clears them.  Class names:
 * cac_profile_class_name ("gemm_ff_up", "attention", "dwconv", ...). */
int  cac_pool_set_profile(cac_pool* p, int enable);
int  cac_pool_read_profile(cac_pool* p, int n_classes, double* total_ms, long long* launches);
int  cac_profile_classes(void);
const char* cac_profile_class_name(int cls);

/* Guard zones: every per-stream device pool (K/V rings, conv ring, provisional
 * x0 ring) sits between two 4 KiB zones filled with NaN bit patterns at pool
 * creation.  Synchronizes the device and returns CAC_OK when all zones are
 * intact, CAC_E_BOUNDS when a kernel wrote into one. */
int  cac_pool_check_guards(cac_pool* p);

/* 1 when this library was built with CAC_CHECKED: every kernel of the
 * streaming step checks stream ids, positions and ring slots before it uses
 * them, latches CAC_E_BOUNDS in the status word and skips the access when one
 * is out of range (a stand-in for a memory checker; no trap, no wait).  0 in
 * the default build. */
int  cac_build_checked(void);

const char* cac_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* CAC_H_ */
