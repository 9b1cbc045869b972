// Streaming log-mel front end: 16 kHz audio -> 128-bin log-mel frames for many
// streams per launch.  What the frames are is stated in include/cac_frontend.h
// ("Parakeet-EOU-120M — Streaming ASR Model", §Config; "Fast
// Accuracy-Preserving RNNT Beam Search on Apple Silicon", §1.3; "True streaming
// encode — implementation spec", §Status).
//
// One launch per push: grid (frame blocks + 1, slots), 4 warps per block, one
// warp per frame.  A warp gathers its frame's 512 samples from the stream's
// raw-sample tail and the new audio (pre-emphasis recomputed from raw samples,
// so a push boundary can fall anywhere), weights them with the window, runs a
// radix-2 decimation-in-time FFT of 512 complex points in shared memory (bit-
// reversed load, nine butterfly stages, twiddles from an fp64-built table),
// squares the 257 bins and applies the mel filters as a sparse table (each
// filter's support fits 16 consecutive bins).  The extra block of each slot
// copies the newest 512 raw samples into the other half of the stream's
// ping-pong tail, so nothing in the launch reads what it writes.
//
// Work per frame: ~23 K flops of FFT + 4 K of filters; per 160 ms push of 256
// streams ~2.6 MB of audio in and ~2.1 MB of mel out — a short, latency- and
// HBM-bound kernel (no tensor-core contraction here).
#include <cmath>
#include <cstring>
#include <vector>

#include <cuda_runtime.h>

#include "cac.h"
#include "cac_frontend.h"
#include "status.cuh"

namespace {

constexpr int HOP = 160;             // samples per frame step
constexpr int NFFT = 512;            // transform points
constexpr int WIN = 400;             // window length, centred in the transform
constexpr int NBIN = NFFT / 2 + 1;   // non-negative frequencies
constexpr int NMEL = 128;
constexpr int TAIL = 512;            // raw samples kept per stream
constexpr int MW = 16;               // filter support width in bins (sparse table)
constexpr int FE_WARPS = 4;          // frames per block
constexpr int RING = 4;              // staging slots for per-call slot tables
constexpr double PI = 3.14159265358979323846;

struct FeSlot {                      // one batch slot of a call (32 bytes)
    long long nprev;                 // samples of the stream before this call
    long long t0;                    // first frame to emit
    int id;                          // stream id
    int par;                         // tail half holding samples nprev-TAIL .. nprev-1
    int nf;                          // frames to emit
    int ns;                          // new samples in this call
};

struct FeArgs {
    const float* audio;
    long long lda;
    float* mel;
    long long ldm;
    const FeSlot* slots;
    float* tails;                    // [S][2][TAIL]
    const float* win;                // [NFFT], zero outside the centred window
    const float2* tw;                // [NFFT/2]: (cos, -sin)(2 pi k / NFFT)
    const int* mstart;               // [NMEL] first bin of each filter's table row
    const float* mw;                 // [NMEL][MW]
    int fblocks;                     // frame blocks per slot (grid.x - 1)
};

// Raw sample j of the stream of slot `sl`: zero before the stream start; the
// tail for the samples of earlier calls (the frame schedule never reaches
// further back than TAIL samples; anything older reads as zero rather than
// out of bounds); the new audio; zero past the end (flush padding).
__device__ __forceinline__ float fe_raw(const FeSlot& sl, const float* tail, const float* au, long long j) {
    if (j < 0) return 0.f;
    if (j < sl.nprev) {
        const long long k = j - (sl.nprev - TAIL);
        return k >= 0 ? tail[k] : 0.f;
    }
    const long long k = j - sl.nprev;
    return k < sl.ns ? au[k] : 0.f;
}

__global__ void __launch_bounds__(FE_WARPS * 32) fe_kernel(FeArgs a) {
    __shared__ float2 buf[FE_WARPS][NFFT];
    __shared__ float pw[FE_WARPS][NBIN + 7];
    __shared__ float2 tw[NFFT / 2];

    const FeSlot sl = a.slots[blockIdx.y];
    const float* tail = a.tails + ((long long)sl.id * 2 + sl.par) * TAIL;
    const float* au = a.audio ? a.audio + (long long)blockIdx.y * a.lda : nullptr;

    if ((int)blockIdx.x == a.fblocks) {  // tail block: newest TAIL raw samples into the other half
        float* out = a.tails + ((long long)sl.id * 2 + (sl.par ^ 1)) * TAIL;
        const long long n1 = sl.nprev + sl.ns;
        for (int i = threadIdx.x; i < TAIL; i += blockDim.x) out[i] = fe_raw(sl, tail, au, n1 - TAIL + i);
        return;
    }

    for (int k = threadIdx.x; k < NFFT / 2; k += blockDim.x) tw[k] = a.tw[k];
    __syncthreads();

    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int f = blockIdx.x * FE_WARPS + w;
    if (f >= sl.nf) return;  // no block-wide barrier follows
    const long long t = sl.t0 + f;
    const long long j0 = t * HOP - NFFT / 2;  // signal index of the frame's first point
    const long long end = sl.nprev + sl.ns;   // samples of the stream after this call
    float2* B = buf[w];

    // windowed, pre-emphasised samples into bit-reversed positions
#pragma unroll 4
    for (int r = 0; r < NFFT / 32; ++r) {
        const int i = lane + 32 * r;
        const float wv = a.win[i];
        float v = 0.f;
        const long long j = j0 + i;
        if (wv != 0.f && j >= 0 && j < end)
            v = (fe_raw(sl, tail, au, j) - 0.97f * fe_raw(sl, tail, au, j - 1)) * wv;
        B[__brev((unsigned)i) >> 23] = make_float2(v, 0.f);
    }
    __syncwarp();

    // nine radix-2 stages; stage s joins pairs `half` apart, 256 disjoint butterflies per stage
#pragma unroll
    for (int s = 0; s < 9; ++s) {
        const int half = 1 << s;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int b = lane + 32 * q;
            const int pos = b & (half - 1);
            const int i = ((b >> s) << (s + 1)) + pos, j = i + half;
            const float2 c = tw[pos << (8 - s)];
            const float2 u = B[i], x = B[j];
            const float vr = x.x * c.x - x.y * c.y, vi = x.x * c.y + x.y * c.x;
            B[i] = make_float2(u.x + vr, u.y + vi);
            B[j] = make_float2(u.x - vr, u.y - vi);
        }
        __syncwarp();
    }

    float* P = pw[w];
    for (int k = lane; k < NBIN; k += 32) {
        const float2 c = B[k];
        P[k] = c.x * c.x + c.y * c.y;
    }
    __syncwarp();

    float* out = a.mel + (long long)blockIdx.y * a.ldm + (long long)f * NMEL;
#pragma unroll
    for (int r = 0; r < NMEL / 32; ++r) {
        const int m = lane + 32 * r;
        const int st = a.mstart[m];
        const float* wm = a.mw + m * MW;
        float e = 0.f;
#pragma unroll
        for (int q = 0; q < MW; ++q) e = fmaf(wm[q], P[st + q], e);
        out[m] = logf(e + 5.9604644775390625e-8f);  // + 2^-24
    }
}

// ---------------------------------------------------------------------------
// host tables, built in fp64 and rounded once
// ---------------------------------------------------------------------------
double hz_to_mel(double f) {  // Slaney: linear below 1 kHz (200/3 Hz per mel), log above (x6.4 per 27 mels)
    return f >= 1000.0 ? 15.0 + std::log(f / 1000.0) * 27.0 / std::log(6.4) : f * 3.0 / 200.0;
}
double mel_to_hz(double m) {
    return m >= 15.0 ? 1000.0 * std::exp((m - 15.0) * std::log(6.4) / 27.0) : m * 200.0 / 3.0;
}

struct Tables {
    std::vector<float> win;
    std::vector<float2> tw;
    std::vector<int> mstart;
    std::vector<float> mw;
};

// false if a filter's support does not fit MW bins (never for these constants)
bool build_tables(Tables& T) {
    T.win.assign(NFFT, 0.f);
    const int off = (NFFT - WIN) / 2;
    for (int k = 0; k < WIN; ++k) T.win[off + k] = (float)(0.5 - 0.5 * std::cos(2.0 * PI * k / (WIN - 1)));
    T.tw.resize(NFFT / 2);
    for (int k = 0; k < NFFT / 2; ++k)
        T.tw[k] = make_float2((float)std::cos(2.0 * PI * k / NFFT), (float)-std::sin(2.0 * PI * k / NFFT));
    double edge[NMEL + 2];
    const double top = hz_to_mel(8000.0);
    for (int i = 0; i < NMEL + 2; ++i) edge[i] = mel_to_hz(top * i / (NMEL + 1));
    T.mstart.assign(NMEL, 0);
    T.mw.assign((size_t)NMEL * MW, 0.f);
    std::vector<double> row(NBIN);
    for (int m = 0; m < NMEL; ++m) {
        int first = -1, last = -1;
        for (int k = 0; k < NBIN; ++k) {
            const double fq = 8000.0 * k / (NBIN - 1);
            const double rise = (fq - edge[m]) / (edge[m + 1] - edge[m]);
            const double fall = (edge[m + 2] - fq) / (edge[m + 2] - edge[m + 1]);
            row[k] = std::fmax(0.0, std::fmin(rise, fall)) * 2.0 / (edge[m + 2] - edge[m]);
            if (row[k] != 0.0) {
                if (first < 0) first = k;
                last = k;
            }
        }
        if (first < 0) first = last = 0;
        const int st = first < NBIN - MW ? first : NBIN - MW;
        if (last - st + 1 > MW) return false;
        T.mstart[m] = st;
        for (int q = 0; q < MW; ++q) T.mw[(size_t)m * MW + q] = (float)row[st + q];
    }
    return true;
}

long long complete_frames(long long n) { return n >= NFFT / 2 ? (n - NFFT / 2) / HOP + 1 : 0; }

}  // namespace

struct cac_frontend {
    int S = 0;
    std::vector<long long> n, t;  // samples received, frames emitted
    std::vector<int> par;         // tail half holding the newest samples
    std::vector<unsigned char> finished;
    float* tails = nullptr;
    float* win = nullptr;
    float2* tw = nullptr;
    int* mstart = nullptr;
    float* mw = nullptr;
    FeSlot* d_slots = nullptr;    // [RING][S]
    FeSlot* h_slots = nullptr;    // pinned [RING][S]
    cudaEvent_t ev[RING] = {};
    int ring = 0;
    std::vector<FeSlot> plan;     // this call's slots, before staging
};

extern "C" long long cac_frontend_schedule(long long samples_before, long long frames_before, long long n_samples,
                                           int flush) {
    if (samples_before < 0 || frames_before < 0 || n_samples < 0) return CAC_E_INVAL;
    const long long n1 = samples_before + n_samples;
    const long long last = flush ? 1 + n1 / HOP : complete_frames(n1);
    return last > frames_before ? last - frames_before : 0;
}

extern "C" int cac_frontend_tables(float* window, float* twiddles, int* mel_start, float* mel_w) {
    if (!window || !twiddles || !mel_start || !mel_w) return CAC_E_INVAL;
    Tables T;
    if (!build_tables(T)) return CAC_E_UNSUPPORTED;
    std::memcpy(window, T.win.data(), sizeof(float) * NFFT);
    std::memcpy(twiddles, T.tw.data(), sizeof(float2) * NFFT / 2);
    std::memcpy(mel_start, T.mstart.data(), sizeof(int) * NMEL);
    std::memcpy(mel_w, T.mw.data(), sizeof(float) * NMEL * MW);
    return CAC_OK;
}

extern "C" void cac_frontend_destroy(cac_frontend* fe) {
    if (!fe) return;
    for (cudaEvent_t e : fe->ev)
        if (e) cudaEventDestroy(e);
    for (void* p : {(void*)fe->tails, (void*)fe->win, (void*)fe->tw, (void*)fe->mstart, (void*)fe->mw,
                    (void*)fe->d_slots})
        if (p) cudaFree(p);
    if (fe->h_slots) cudaFreeHost(fe->h_slots);
    delete fe;
}

extern "C" int cac_frontend_create(int max_streams, cac_frontend** out) {
    if (!out || max_streams < 1 || max_streams > 65535) return CAC_E_INVAL;
    *out = nullptr;
    Tables T;
    if (!build_tables(T)) return CAC_E_UNSUPPORTED;
    auto* fe = new cac_frontend();
    fe->S = max_streams;
    fe->n.assign(max_streams, 0);
    fe->t.assign(max_streams, 0);
    fe->par.assign(max_streams, 0);
    fe->finished.assign(max_streams, 0);
    const size_t S = (size_t)max_streams;
    bool ok = cudaMalloc(&fe->tails, sizeof(float) * 2 * TAIL * S) == cudaSuccess &&
              cudaMemset(fe->tails, 0, sizeof(float) * 2 * TAIL * S) == cudaSuccess &&
              cudaMalloc(&fe->win, sizeof(float) * NFFT) == cudaSuccess &&
              cudaMalloc(&fe->tw, sizeof(float2) * NFFT / 2) == cudaSuccess &&
              cudaMalloc(&fe->mstart, sizeof(int) * NMEL) == cudaSuccess &&
              cudaMalloc(&fe->mw, sizeof(float) * NMEL * MW) == cudaSuccess &&
              cudaMalloc(&fe->d_slots, sizeof(FeSlot) * RING * S) == cudaSuccess &&
              cudaHostAlloc(reinterpret_cast<void**>(&fe->h_slots), sizeof(FeSlot) * RING * S,
                            cudaHostAllocDefault) == cudaSuccess;
    if (!ok) {
        cac_frontend_destroy(fe);
        return cac::nomem();
    }
    ok = cudaMemcpy(fe->win, T.win.data(), sizeof(float) * NFFT, cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(fe->tw, T.tw.data(), sizeof(float2) * NFFT / 2, cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(fe->mstart, T.mstart.data(), sizeof(int) * NMEL, cudaMemcpyHostToDevice) == cudaSuccess &&
         cudaMemcpy(fe->mw, T.mw.data(), sizeof(float) * NMEL * MW, cudaMemcpyHostToDevice) == cudaSuccess;
    for (int k = 0; ok && k < RING; ++k) ok = cudaEventCreateWithFlags(&fe->ev[k], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cac_frontend_destroy(fe);
        return CAC_E_CUDA;
    }
    *out = fe;
    return CAC_OK;
}

extern "C" int cac_frontend_reset(cac_frontend* fe, int n, const int* ids) {
    if (!fe || n < 0 || (n > 0 && !ids)) return CAC_E_INVAL;
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= fe->S) return CAC_E_INVAL;
    for (int i = 0; i < n; ++i) {
        const int id = ids[i];
        fe->n[id] = fe->t[id] = 0;
        fe->par[id] = 0;
        fe->finished[id] = 0;
    }
    return CAC_OK;
}

extern "C" int cac_frontend_get_state(const cac_frontend* fe, int id, long long* samples, long long* frames,
                                      int* finished) {
    if (!fe || id < 0 || id >= fe->S) return CAC_E_INVAL;
    if (samples) *samples = fe->n[id];
    if (frames) *frames = fe->t[id];
    if (finished) *finished = fe->finished[id];
    return CAC_OK;
}

namespace {

// Shared body of push (ns_each == nullptr: every slot gets ns) and flush.
int fe_call(cac_frontend* fe, int n, const int* ids, const float* audio, long long lda, int ns,
            const int* ns_each, bool flush, float* mel, long long ldm, int max_frames, int* nf_out,
            cudaStream_t st) {
    if (!fe || n < 1 || n > fe->S || !ids || !nf_out || lda < 0 || max_frames < 0) return CAC_E_INVAL;
    if (ldm < (long long)NMEL * max_frames) return CAC_E_INVAL;
    std::vector<unsigned char> seen(fe->S, 0);
    int ns_max = 0;
    for (int b = 0; b < n; ++b) {
        const int id = ids[b];
        if (id < 0 || id >= fe->S || seen[id]) return CAC_E_INVAL;
        seen[id] = 1;
        if (fe->finished[id]) return CAC_E_STATE;
        const int nsb = ns_each ? ns_each[b] : ns;
        if (nsb < 0) return CAC_E_INVAL;
        ns_max = nsb > ns_max ? nsb : ns_max;
    }
    if (ns_max > 0 && (!audio || lda < ns_max)) return CAC_E_INVAL;
    fe->plan.resize(n);
    int fmax = 0;
    for (int b = 0; b < n; ++b) {
        const int id = ids[b];
        FeSlot& s = fe->plan[b];
        s.nprev = fe->n[id];
        s.t0 = fe->t[id];
        s.id = id;
        s.par = fe->par[id];
        s.ns = ns_each ? ns_each[b] : ns;
        const long long nf = cac_frontend_schedule(s.nprev, s.t0, s.ns, flush ? 1 : 0);
        if (nf > max_frames) return CAC_E_LIMIT;
        s.nf = (int)nf;
        fmax = s.nf > fmax ? s.nf : fmax;
    }
    if (fmax > 0 && !mel) return CAC_E_INVAL;

    const int k = fe->ring;
    if (cudaEventSynchronize(fe->ev[k]) != cudaSuccess) return CAC_E_CUDA;
    FeSlot* h = fe->h_slots + (size_t)k * fe->S;
    FeSlot* d = fe->d_slots + (size_t)k * fe->S;
    std::memcpy(h, fe->plan.data(), sizeof(FeSlot) * n);
    if (cudaMemcpyAsync(d, h, sizeof(FeSlot) * n, cudaMemcpyHostToDevice, st) != cudaSuccess) return CAC_E_CUDA;
    FeArgs a;
    a.audio = ns_max > 0 ? audio : nullptr;
    a.lda = lda;
    a.mel = mel;
    a.ldm = ldm;
    a.slots = d;
    a.tails = fe->tails;
    a.win = fe->win;
    a.tw = fe->tw;
    a.mstart = fe->mstart;
    a.mw = fe->mw;
    a.fblocks = (fmax + FE_WARPS - 1) / FE_WARPS;
    fe_kernel<<<dim3(a.fblocks + 1, n), FE_WARPS * 32, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess) return CAC_E_CUDA;
    if (cudaEventRecord(fe->ev[k], st) != cudaSuccess) return CAC_E_CUDA;
    fe->ring = (k + 1) % RING;

    for (int b = 0; b < n; ++b) {
        const FeSlot& s = fe->plan[b];
        fe->n[s.id] += s.ns;
        fe->t[s.id] += s.nf;
        fe->par[s.id] ^= 1;
        if (flush) fe->finished[s.id] = 1;
        nf_out[b] = s.nf;
    }
    return CAC_OK;
}

}  // namespace

extern "C" int cac_frontend_push(cac_frontend* fe, int n, const int* ids, const float* audio, long long audio_bstride,
                                 int n_samples, float* mel, long long mel_bstride, int max_frames,
                                 int* n_frames_out, void* stream) {
    if (n_samples < 0) return CAC_E_INVAL;
    return fe_call(fe, n, ids, audio, audio_bstride, n_samples, nullptr, false, mel, mel_bstride, max_frames,
                   n_frames_out, static_cast<cudaStream_t>(stream));
}

extern "C" int cac_frontend_flush(cac_frontend* fe, int n, const int* ids, const float* audio, long long audio_bstride,
                                  const int* n_samples_each, float* mel, long long mel_bstride, int max_frames,
                                  int* n_frames_out, void* stream) {
    if (!n_samples_each) return CAC_E_INVAL;
    return fe_call(fe, n, ids, audio, audio_bstride, 0, n_samples_each, true, mel, mel_bstride, max_frames,
                   n_frames_out, static_cast<cudaStream_t>(stream));
}
