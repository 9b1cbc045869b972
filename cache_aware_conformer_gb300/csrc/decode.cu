// Batched greedy RNN-T decoding with an end-of-utterance class ("Parakeet-EOU-
// 120M — Streaming ASR Model", §Architecture: fp32 LSTM predictor on the last
// non-blank token, joint over one projected encoder frame and the predictor
// output -> vocabulary + blank + EOU, greedy loop per frame advancing the
// predictor only on non-blank emissions; "True streaming encode —
// implementation spec", §Decoder state carry: h/c persist per stream).
//
// One step decodes n streams over T frames in ONE cooperative launch of a
// persistent kernel (one 256-thread CTA per SM).  The streams advance in
// lockstep iterations; each iteration is
//   A  joint + argmax: logits of every still-active slot at its current frame,
//      tiled (32 slots x 64 classes) over the CTAs, K = joint_dim, written as
//      per-tile partial maxima;
//   B  decisions: per active slot the first maximum over the partials; blank
//      (or max_symbols reached) moves the slot to its next frame, anything else
//      is emitted and queued for the predictor;
//   C  LSTM step of the queued slots, tiled (32 slots x 16 hidden units = 64
//      gate rows): gates = tab[token] + W_hh h, with tab = emb W_ih^T + b_ih +
//      b_hh computed once at load (the input half of the gates depends on the
//      token only), then the cell update in the tile;
//   D  predictor projection p = W_pred h' + b_pred of the queued slots.
// Grid-wide barriers separate the phases: an arrival counter and a generation
// word in global memory, every spin bounded (about a second) after which the
// kernel latches CAC_E_TIMEOUT, raises an abort word that releases every
// other waiter, and returns.  Everything is fp32 on the CUDA cores (the pages
// fix fp32 for the decoder, so every argmax is decided in fp32).
#include <cfloat>
#include <cstring>
#include <mutex>
#include <vector>

#include "cac.h"
#include "cac_decode.h"
#include "common.cuh"

namespace cac {
namespace {

constexpr int DT = 256;        // threads per CTA
constexpr int TS = 32;         // slots per tile
constexpr int TN = 64;         // output columns per tile
constexpr int KC = 64;         // K chunk staged in shared memory
constexpr int WLD = KC + 4;    // row stride of the staged weight chunk
constexpr int OLD = TN + 1;    // row stride of the output tile

struct DecParams {
    int n, T, C, P, J, max_sym, blank, nct, maxit;
    const int* ids;
    const float* z;
    long long zb;
    int *tokens, *frames, *counts;
    const float *tab, *whh, *wpp, *bpp, *wout, *bout;
    float *h, *c, *p;
    int* primed;
    int *frame, *sym, *act, *em, *emk, *cnt;
    float* pval;
    int* pidx;
    float* hnext;
    unsigned* bar;  // [0] arrivals, [1] generation
    int* abort_flag;
    int* status;
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier of a cooperative launch; false when it gave up (timeout or
// another CTA's abort), in which case the caller returns.
__device__ bool grid_sync(const DecParams& d) {
    __shared__ int ok_s;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const unsigned gen = ld_acquire(&d.bar[1]);
        __threadfence();
        if (atomicAdd(&d.bar[0], 1u) == gridDim.x - 1) {
            atomicExch(&d.bar[0], 0u);
            __threadfence();
            atomicAdd(&d.bar[1], 1u);
        } else {
            const long long t0 = clock64();
            for (unsigned it = 0;; ++it) {
                if (ld_acquire(&d.bar[1]) != gen) break;
                if (*(volatile int*)d.abort_flag) { ok = 0; break; }
                if ((it & 63u) == 63u && clock64() - t0 > (1ll << 31)) {
                    latch_error(d.status, CAC_E_TIMEOUT);
                    atomicExch(d.abort_flag, 1);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
        ok_s = ok;
    }
    __syncthreads();
    return ok_s != 0;
}

__device__ __forceinline__ float sigm(float x) { return 1.f / (1.f + expf(-x)); }

// acc[s][j] += sum_k As[slot row][k] * W[row j][k] for the thread's 2 slots (sx,
// sx + 16) and 4 columns (cx + 16 j); W rows come from wrow(r) (nullptr: zero),
// K a multiple of KC.  As: [TS][K + 4] in shared memory, filled by the caller.
template <class WRow>
__device__ __forceinline__ void mac_tile(int K, const float* As, float* Ws, WRow wrow, float (&acc)[2][4]) {
    const int tid = threadIdx.x, sx = tid & 15, cx = tid >> 4;
    const int lda = K + 4;
    for (int k0 = 0; k0 < K; k0 += KC) {
        for (int e = tid; e < TN * KC / 4; e += DT) {
            const int r = e >> 4, q = e & 15;
            const float* src = wrow(r);
            const float4 w = src ? __ldg(reinterpret_cast<const float4*>(src + k0) + q) : make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(Ws + r * WLD + 4 * q) = w;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < KC; kk += 4) {
            const float4 a0 = *reinterpret_cast<const float4*>(As + sx * lda + k0 + kk);
            const float4 a1 = *reinterpret_cast<const float4*>(As + (sx + 16) * lda + k0 + kk);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 w = *reinterpret_cast<const float4*>(Ws + (cx + 16 * j) * WLD + kk);
                acc[0][j] = fmaf(a0.x, w.x, acc[0][j]);
                acc[0][j] = fmaf(a0.y, w.y, acc[0][j]);
                acc[0][j] = fmaf(a0.z, w.z, acc[0][j]);
                acc[0][j] = fmaf(a0.w, w.w, acc[0][j]);
                acc[1][j] = fmaf(a1.x, w.x, acc[1][j]);
                acc[1][j] = fmaf(a1.y, w.y, acc[1][j]);
                acc[1][j] = fmaf(a1.z, w.z, acc[1][j]);
                acc[1][j] = fmaf(a1.w, w.w, acc[1][j]);
            }
        }
        __syncthreads();
    }
}

// thread's accumulators into the output tile Os [TS][OLD]
__device__ __forceinline__ void store_tile(float* Os, const float (&acc)[2][4]) {
    const int tid = threadIdx.x, sx = tid & 15, cx = tid >> 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        Os[sx * OLD + cx + 16 * j] = acc[0][j];
        Os[(sx + 16) * OLD + cx + 16 * j] = acc[1][j];
    }
}

// Phase C: LSTM step of the queued slots em[0 .. ne) with tokens emk[.]:
// tile (32 slots, 16 hidden units = the 4 x 16 gate rows of those units).
__device__ void phase_lstm(const DecParams& d, const int* em, const int* emk, int ne, float* As, float* Ws,
                           float* Os) {
    const int P = d.P, lda = P + 4, tid = threadIdx.x;
    const int ut = P / 16, tiles = ((ne + TS - 1) / TS) * ut;
    int loaded = -1;  // slot tile whose h rows sit in As
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int st = t / ut, j0 = (t % ut) * 16;
        if (st != loaded) {
            __syncthreads();
            for (int e = tid; e < TS * P / 4; e += DT) {
                const int r = e / (P / 4), q = e % (P / 4), i = st * TS + r;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < ne) {
                    const int id = d.ids[__ldcg(em + i)];
                    v = __ldcg(reinterpret_cast<const float4*>(d.h + (long long)id * P) + q);
                }
                *reinterpret_cast<float4*>(As + r * lda + 4 * q) = v;
            }
            __syncthreads();
            loaded = st;
        }
        float acc[2][4] = {};
        mac_tile(P, As, Ws, [&](int r) { return d.whh + (long long)((r >> 4) * P + j0 + (r & 15)) * P; }, acc);
        store_tile(Os, acc);
        __syncthreads();
        // cell update of (slot r, unit jj): two per thread
        for (int e = tid; e < TS * 16; e += DT) {
            const int r = e >> 4, jj = e & 15, i = st * TS + r;
            if (i >= ne) continue;
            const int b = __ldcg(em + i), k = __ldcg(emk + i), id = d.ids[b], j = j0 + jj;
            const float* tb = d.tab + (long long)k * 4 * P;
            const float gi = Os[r * OLD + jj] + __ldg(tb + j);
            const float gf = Os[r * OLD + 16 + jj] + __ldg(tb + P + j);
            const float gg = Os[r * OLD + 32 + jj] + __ldg(tb + 2 * P + j);
            const float go = Os[r * OLD + 48 + jj] + __ldg(tb + 3 * P + j);
            float* cp = d.c + (long long)id * P + j;
            const float c2 = sigm(gf) * __ldcg(cp) + sigm(gi) * tanhf(gg);
            *cp = c2;
            d.hnext[(long long)b * P + j] = sigm(go) * tanhf(c2);
        }
        __syncthreads();
    }
}

// Phase D: p = W_pred h' + b_pred for the queued slots, and h <- h'.
__device__ void phase_proj(const DecParams& d, const int* em, int ne, float* As, float* Ws) {
    const int P = d.P, J = d.J, lda = P + 4, tid = threadIdx.x;
    const int jt = J / TN, tiles = ((ne + TS - 1) / TS) * jt;
    int loaded = -1;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int st = t / jt, c0 = (t % jt) * TN;
        if (st != loaded) {
            __syncthreads();
            for (int e = tid; e < TS * P / 4; e += DT) {
                const int r = e / (P / 4), q = e % (P / 4), i = st * TS + r;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < ne) {
                    const int b = __ldcg(em + i);
                    v = __ldcg(reinterpret_cast<const float4*>(d.hnext + (long long)b * P) + q);
                }
                *reinterpret_cast<float4*>(As + r * lda + 4 * q) = v;
            }
            __syncthreads();
            loaded = st;
        }
        if (c0 == 0) {  // the first column tile of each slot tile commits h <- h'
            for (int e = tid; e < TS * P / 4; e += DT) {
                const int r = e / (P / 4), q = e % (P / 4), i = st * TS + r;
                if (i < ne)
                    reinterpret_cast<float4*>(d.h + (long long)d.ids[__ldcg(em + i)] * P)[q] =
                        *reinterpret_cast<const float4*>(As + r * lda + 4 * q);
            }
        }
        float acc[2][4] = {};
        mac_tile(P, As, Ws, [&](int r) { return d.wpp + (long long)(c0 + r) * P; }, acc);
        const int sx = tid & 15, cx = tid >> 4;
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
            const int i = st * TS + sx + 16 * s2;
            if (i >= ne) continue;
            const int id = d.ids[__ldcg(em + i)];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = c0 + cx + 16 * j;
                d.p[(long long)id * J + col] = acc[s2][j] + __ldg(d.bpp + col);
            }
        }
    }
}

// Phase A: logits of the active slots act[0 .. na) at their current frame,
// partial first-maximum per 64-class tile into pval / pidx [slot][nct].
__device__ void phase_joint(const DecParams& d, const int* act, int na, float* As, float* Ws, float* Os) {
    const int J = d.J, C = d.C, lda = J + 4, tid = threadIdx.x;
    const int tiles = ((na + TS - 1) / TS) * d.nct;
    int loaded = -1;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int st = t / d.nct, ct = t % d.nct, c0 = ct * TN;
        if (st != loaded) {
            __syncthreads();
            for (int e = tid; e < TS * J / 4; e += DT) {
                const int r = e / (J / 4), q = e % (J / 4), i = st * TS + r;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < na) {
                    const int b = __ldcg(act + i), id = d.ids[b], f = __ldcg(d.frame + b);
                    const float4 zz = __ldg(reinterpret_cast<const float4*>(d.z + b * d.zb + (long long)f * J) + q);
                    const float4 pp = __ldcg(reinterpret_cast<const float4*>(d.p + (long long)id * J) + q);
                    v = make_float4(fmaxf(zz.x + pp.x, 0.f), fmaxf(zz.y + pp.y, 0.f), fmaxf(zz.z + pp.z, 0.f),
                                    fmaxf(zz.w + pp.w, 0.f));
                }
                *reinterpret_cast<float4*>(As + r * lda + 4 * q) = v;
            }
            __syncthreads();
            loaded = st;
        }
        float acc[2][4] = {};
        mac_tile(J, As, Ws, [&](int r) { return c0 + r < C ? d.wout + (long long)(c0 + r) * J : nullptr; }, acc);
        store_tile(Os, acc);
        __syncthreads();
        if (tid < TS) {
            const int i = st * TS + tid;
            if (i < na) {
                float best = -FLT_MAX;
                int bi = c0;
                for (int q = 0; q < TN && c0 + q < C; ++q) {
                    const float v = Os[tid * OLD + q] + __ldg(d.bout + c0 + q);
                    if (v > best) { best = v; bi = c0 + q; }
                }
                const int b = __ldcg(act + i);
                d.pval[(long long)b * d.nct + ct] = best;
                d.pidx[(long long)b * d.nct + ct] = bi;
            }
        }
        __syncthreads();
    }
}

// The whole step (see the top of the file).  Iteration it reads the active
// list act[it & 1] (length cnt[2 it]) and writes the next one act[(it + 1) & 1]
// (length cnt[2 it + 2]) and its emissions em/emk[it & 1] (length cnt[2 it +
// 1]); iteration 0 only builds the first active list and primes reset streams.
__global__ void __launch_bounds__(DT, 1) dec_step_kernel(DecParams d) {
    extern __shared__ float smem[];
    const int K = d.P > d.J ? d.P : d.J;
    float* As = smem;
    float* Ws = As + TS * (K + 4);
    float* Os = Ws + TN * WLD;
    const int gtid = blockIdx.x * DT + threadIdx.x, gstride = gridDim.x * DT;
    const long long tsym = (long long)d.T * d.max_sym;

    for (int b = gtid; b < d.n; b += gstride) {
        const int id = d.ids[b];
        d.frame[b] = 0;
        d.sym[b] = 0;
        d.counts[b] = 0;
        if (d.T > 0) d.act[d.n + atomicAdd(&d.cnt[2], 1)] = b;
        if (__ldcg(d.primed + id) == 0) {  // stream start: zero state, one predictor step on blank
            for (int j = 0; j < d.P; ++j) {
                d.h[(long long)id * d.P + j] = 0.f;
                d.c[(long long)id * d.P + j] = 0.f;
            }
            d.primed[id] = 1;
            const int q = atomicAdd(&d.cnt[1], 1);
            d.em[q] = b;
            d.emk[q] = d.blank;
        }
    }
    if (!grid_sync(d)) return;
    int ne = __ldcg(d.cnt + 1);
    if (ne > 0) {
        phase_lstm(d, d.em, d.emk, ne, As, Ws, Os);
        if (!grid_sync(d)) return;
        phase_proj(d, d.em, ne, As, Ws);
        if (!grid_sync(d)) return;
    }
    for (int it = 1; it <= d.maxit; ++it) {
        const int na = __ldcg(d.cnt + 2 * it);
        if (na == 0) break;
        const int* act = d.act + (it & 1) * d.n;
        phase_joint(d, act, na, As, Ws, Os);
        if (!grid_sync(d)) return;
        int* nact = d.act + ((it + 1) & 1) * d.n;
        int* em = d.em + (it & 1) * d.n;
        int* emk = d.emk + (it & 1) * d.n;
        for (int i = gtid; i < na; i += gstride) {
            const int b = __ldcg(act + i);
            const long long pb = (long long)b * d.nct;
            float best = __ldcg(d.pval + pb);
            int k = __ldcg(d.pidx + pb);
            for (int q = 1; q < d.nct; ++q) {  // tiles in class order: strict > keeps the lowest index
                const float v = __ldcg(d.pval + pb + q);
                if (v > best) {
                    best = v;
                    k = __ldcg(d.pidx + pb + q);
                }
            }
            int f = __ldcg(d.frame + b), sy = __ldcg(d.sym + b);
            bool next = k == d.blank;
            if (!next) {
                const int cn = __ldcg(d.counts + b);
                d.tokens[b * tsym + cn] = k;
                d.frames[b * tsym + cn] = f;
                d.counts[b] = cn + 1;
                const int q = atomicAdd(&d.cnt[2 * it + 1], 1);
                em[q] = b;
                emk[q] = k;
                next = ++sy == d.max_sym;
            }
            if (next) {
                ++f;
                sy = 0;
            }
            d.frame[b] = f;
            d.sym[b] = sy;
            if (f < d.T) nact[atomicAdd(&d.cnt[2 * it + 2], 1)] = b;
        }
        if (!grid_sync(d)) return;
        ne = __ldcg(d.cnt + 2 * it + 1);
        if (ne > 0) {
            phase_lstm(d, em, emk, ne, As, Ws, Os);
            if (!grid_sync(d)) return;
            phase_proj(d, em, ne, As, Ws);
            if (!grid_sync(d)) return;
        }
    }
}

// tab[k][r] = sum_m W_ih[r][m] emb[k][m] + b_ih[r] + b_hh[r], fp64 sums rounded to fp32
__global__ void dec_tab_kernel(const float* emb, const float* wih, const float* bih, const float* bhh, float* tab,
                               int C, int P) {
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= (long long)C * 4 * P) return;
    const int k = (int)(e / (4 * P)), r = (int)(e % (4 * P));
    double s = (double)bih[r] + (double)bhh[r];
    for (int m = 0; m < P; ++m) s += (double)wih[(long long)r * P + m] * (double)emb[(long long)k * P + m];
    tab[e] = (float)s;
}

__global__ void dec_reset_kernel(const int* ids, int n, int* primed) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) primed[ids[i]] = 0;
}

constexpr int ID_SLOTS = 4;
constexpr int MAX_T = 1024;

}  // namespace
}  // namespace cac

using namespace cac;

struct cac_decoder {
    cac_dec_config cfg{};
    int C = 0, S = 0, nct = 0, grid = 0;
    size_t smem = 0;
    std::vector<void*> allocs;
    float *tab = nullptr, *whh = nullptr, *wpp = nullptr, *bpp = nullptr, *wout = nullptr, *bout = nullptr;
    float *h = nullptr, *c = nullptr, *p = nullptr;
    int* primed = nullptr;
    // step scratch for up to S slots
    int *ids = nullptr, *frame = nullptr, *sym = nullptr, *act = nullptr, *em = nullptr, *emk = nullptr;
    int* cnt = nullptr;  // [2 (maxit + 2)] iteration counters, then arrivals / generation / abort
    int cnt_ints = 0;
    float* pval = nullptr;
    int* pidx = nullptr;
    float* hnext = nullptr;
    int* status = nullptr;
    int* pinned = nullptr;  // ID_SLOTS x S host ids
    cudaEvent_t slot_ev[ID_SLOTS] = {};
    int slot = 0;
};

namespace {

int dalloc(cac_decoder* d, size_t bytes, void** out) {
    if (cudaMalloc(out, bytes) != cudaSuccess) return CAC_E_NOMEM;
    d->allocs.push_back(*out);
    return CAC_OK;
}

template <class T>
int dalloc_t(cac_decoder* d, size_t count, T** out) {
    void* v = nullptr;
    const int r = dalloc(d, count * sizeof(T), &v);
    *out = static_cast<T*>(v);
    return r;
}

int maxit_for(const cac_dec_config& c, int T) { return T * (c.max_symbols + 1) + 1; }

}  // namespace

extern "C" void cac_decoder_destroy(cac_decoder* d) {
    if (!d) return;
    cudaDeviceSynchronize();
    for (void* a : d->allocs) cudaFree(a);
    if (d->pinned) cudaFreeHost(d->pinned);
    for (auto& e : d->slot_ev)
        if (e) cudaEventDestroy(e);
    delete d;
}

extern "C" int cac_decoder_create(const cac_dec_config* cfg, const float* weights, size_t n_floats, int max_streams,
                                  cac_decoder** out) {
    if (!cfg || !weights || !out || max_streams < 1 || cfg->vocab < 1 || cfg->max_symbols < 1 ||
        cfg->pred_dim < 64 || cfg->joint_dim < 64)
        return CAC_E_INVAL;
    if (cfg->pred_dim % 64 || cfg->joint_dim % 64) return CAC_E_UNSUPPORTED;
    const size_t C = (size_t)cfg->vocab + 2, P = cfg->pred_dim, J = cfg->joint_dim;
    const size_t need = C * P + 2 * 4 * P * P + 2 * 4 * P + J * P + J + C * J + C;
    if (n_floats != need) return CAC_E_INVAL;
    *out = nullptr;
    cac_decoder* d = new cac_decoder();
    d->cfg = *cfg;
    d->C = (int)C;
    d->S = max_streams;
    d->nct = (int)((C + TN - 1) / TN);
    auto fail = [&](int code) {
        cac_decoder_destroy(d);
        return code;
    };
    const float* w = weights;
    const float *emb = w, *wih = emb + C * P, *whh = wih + 4 * P * P, *bih = whh + 4 * P * P, *bhh = bih + 4 * P,
                *wpp = bhh + 4 * P, *bpp = wpp + J * P, *wout = bpp + J, *bout = wout + C * J;
    auto upload = [&](const float* src, size_t nf, float** dst) {
        int r = dalloc_t(d, nf, dst);
        if (r == CAC_OK && cudaMemcpy(*dst, src, nf * 4, cudaMemcpyHostToDevice) != cudaSuccess) r = CAC_E_CUDA;
        return r;
    };
    int r;
    float *emb_d = nullptr, *wih_d = nullptr, *bih_d = nullptr, *bhh_d = nullptr;
    if ((r = upload(emb, C * P, &emb_d)) || (r = upload(wih, 4 * P * P, &wih_d)) || (r = upload(bih, 4 * P, &bih_d)) ||
        (r = upload(bhh, 4 * P, &bhh_d)) || (r = upload(whh, 4 * P * P, &d->whh)) || (r = upload(wpp, J * P, &d->wpp)) ||
        (r = upload(bpp, J, &d->bpp)) || (r = upload(wout, C * J, &d->wout)) || (r = upload(bout, C, &d->bout)))
        return fail(r);
    if ((r = dalloc_t(d, C * 4 * P, &d->tab))) return fail(r);
    {
        const long long nt = (long long)C * 4 * P;
        dec_tab_kernel<<<(unsigned)((nt + 255) / 256), 256>>>(emb_d, wih_d, bih_d, bhh_d, d->tab, (int)C, (int)P);
        if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return fail(CAC_E_CUDA);
    }
    const size_t S = max_streams;
    if ((r = dalloc_t(d, S * P, &d->h)) || (r = dalloc_t(d, S * P, &d->c)) || (r = dalloc_t(d, S * J, &d->p)) ||
        (r = dalloc_t(d, S, &d->primed)) || (r = dalloc_t(d, S, &d->ids)) || (r = dalloc_t(d, S, &d->frame)) ||
        (r = dalloc_t(d, S, &d->sym)) || (r = dalloc_t(d, 2 * S, &d->act)) || (r = dalloc_t(d, 2 * S, &d->em)) ||
        (r = dalloc_t(d, 2 * S, &d->emk)) || (r = dalloc_t(d, S * d->nct, &d->pval)) ||
        (r = dalloc_t(d, S * d->nct, &d->pidx)) || (r = dalloc_t(d, S * P, &d->hnext)) ||
        (r = dalloc_t(d, 1, &d->status)))
        return fail(r);
    d->cnt_ints = 2 * (maxit_for(*cfg, MAX_T) + 2) + 4;
    if ((r = dalloc_t(d, d->cnt_ints, &d->cnt))) return fail(r);
    if (cudaMemset(d->primed, 0, S * 4) != cudaSuccess || cudaMemset(d->status, 0, 4) != cudaSuccess ||
        cudaMemset(d->h, 0, S * P * 4) != cudaSuccess || cudaMemset(d->c, 0, S * P * 4) != cudaSuccess ||
        cudaMemset(d->p, 0, S * J * 4) != cudaSuccess)
        return fail(CAC_E_CUDA);
    if (cudaMallocHost(reinterpret_cast<void**>(&d->pinned), sizeof(int) * S * ID_SLOTS) != cudaSuccess)
        return fail(CAC_E_NOMEM);
    for (auto& e : d->slot_ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return fail(CAC_E_CUDA);
    // one CTA per SM, all co-resident (cooperative launch)
    const int K = (int)(P > J ? P : J);
    d->smem = sizeof(float) * ((size_t)TS * (K + 4) + (size_t)TN * WLD + (size_t)TS * OLD);
    if (d->smem > 227 * 1024) return fail(CAC_E_UNSUPPORTED);
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaFuncSetAttribute(dec_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d->smem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dec_step_kernel, DT, d->smem) != cudaSuccess)
        return fail(CAC_E_CUDA);
    if (per_sm < 1) return fail(CAC_E_UNSUPPORTED);
    d->grid = sms;
    cudaFree(emb_d);
    cudaFree(wih_d);
    cudaFree(bih_d);
    cudaFree(bhh_d);
    for (void* a : {static_cast<void*>(emb_d), static_cast<void*>(wih_d), static_cast<void*>(bih_d),
                    static_cast<void*>(bhh_d)})
        for (auto& x : d->allocs)
            if (x == a) x = nullptr;
    *out = d;
    return CAC_OK;
}

namespace {
// Copy n host ids into the next pinned slot and queue their upload to dst.
int dec_upload_ids(cac_decoder* d, const int* ids, int n, int* dst, cudaStream_t s) {
    const int k = d->slot;
    d->slot = (d->slot + 1) % ID_SLOTS;
    if (cudaEventSynchronize(d->slot_ev[k]) != cudaSuccess) return CAC_E_CUDA;
    int* h = d->pinned + (size_t)k * d->S;
    std::memcpy(h, ids, sizeof(int) * n);
    if (cudaMemcpyAsync(dst, h, sizeof(int) * n, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaEventRecord(d->slot_ev[k], s) != cudaSuccess)
        return CAC_E_CUDA;
    return CAC_OK;
}

int check_ids(const cac_decoder* d, int n, const int* ids) {
    if (n < 0 || n > d->S || (n > 0 && !ids)) return CAC_E_INVAL;
    std::vector<char> seen(d->S, 0);
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= d->S || seen[ids[i]]) return CAC_E_INVAL;
        seen[ids[i]] = 1;
    }
    return CAC_OK;
}
}  // namespace

extern "C" int cac_decoder_reset(cac_decoder* d, int n, const int* ids, void* stream) {
    if (!d) return CAC_E_INVAL;
    int r = check_ids(d, n, ids);
    if (r != CAC_OK || n == 0) return r;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((r = dec_upload_ids(d, ids, n, d->ids, s)) != CAC_OK) return r;
    dec_reset_kernel<<<(n + 255) / 256, 256, 0, s>>>(d->ids, n, d->primed);
    return cudaGetLastError() == cudaSuccess ? CAC_OK : CAC_E_CUDA;
}

extern "C" int cac_decoder_step(cac_decoder* d, int n, const int* ids, const float* z, long long z_bstride, int T,
                                int* tokens, int* frames, int* counts, void* stream) {
    if (!d || T < 0 || T > MAX_T) return CAC_E_INVAL;
    int r = check_ids(d, n, ids);
    if (r != CAC_OK) return r;
    if (n == 0) return CAC_OK;
    if ((T > 0 && (!z || !tokens || !frames)) || !counts || z_bstride < (long long)T * d->cfg.joint_dim)
        return CAC_E_INVAL;
    if ((reinterpret_cast<uintptr_t>(z) & 15) || (z_bstride & 3) ||
        ((reinterpret_cast<uintptr_t>(tokens) | reinterpret_cast<uintptr_t>(frames) |
          reinterpret_cast<uintptr_t>(counts)) & 3))
        return CAC_E_INVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((r = dec_upload_ids(d, ids, n, d->ids, s)) != CAC_OK) return r;
    const int maxit = maxit_for(d->cfg, T);
    const int nc = 2 * (maxit + 2);
    if (cudaMemsetAsync(d->cnt, 0, sizeof(int) * (nc + 4), s) != cudaSuccess) return CAC_E_CUDA;
    DecParams p{};
    p.n = n; p.T = T; p.C = d->C; p.P = d->cfg.pred_dim; p.J = d->cfg.joint_dim; p.max_sym = d->cfg.max_symbols;
    p.blank = d->cfg.vocab; p.nct = d->nct; p.maxit = maxit;
    p.ids = d->ids; p.z = z; p.zb = z_bstride; p.tokens = tokens; p.frames = frames; p.counts = counts;
    p.tab = d->tab; p.whh = d->whh; p.wpp = d->wpp; p.bpp = d->bpp; p.wout = d->wout; p.bout = d->bout;
    p.h = d->h; p.c = d->c; p.p = d->p; p.primed = d->primed;
    p.frame = d->frame; p.sym = d->sym; p.act = d->act; p.em = d->em; p.emk = d->emk; p.cnt = d->cnt;
    p.pval = d->pval; p.pidx = d->pidx; p.hnext = d->hnext;
    p.bar = reinterpret_cast<unsigned*>(d->cnt + nc);
    p.abort_flag = d->cnt + nc + 2;
    p.status = d->status;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(d->grid);
    lc.blockDim = dim3(DT);
    lc.dynamicSmemBytes = d->smem;
    lc.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, dec_step_kernel, p) == cudaSuccess ? CAC_OK : CAC_E_CUDA;
}

extern "C" int cac_decoder_check(cac_decoder* d) {
    if (!d) return CAC_E_INVAL;
    if (cudaDeviceSynchronize() != cudaSuccess) return CAC_E_CUDA;
    int st = 0;
    if (cudaMemcpy(&st, d->status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return CAC_E_CUDA;
    if (st != 0 && cudaMemset(d->status, 0, 4) != cudaSuccess) return CAC_E_CUDA;
    return st;
}

extern "C" int cac_decoder_get_state(cac_decoder* d, int id, float* h, float* c, float* p, int* primed) {
    if (!d || id < 0 || id >= d->S) return CAC_E_INVAL;
    const size_t P = d->cfg.pred_dim, J = d->cfg.joint_dim;
    if (cudaDeviceSynchronize() != cudaSuccess) return CAC_E_CUDA;
    if ((h && cudaMemcpy(h, d->h + id * P, P * 4, cudaMemcpyDeviceToHost) != cudaSuccess) ||
        (c && cudaMemcpy(c, d->c + id * P, P * 4, cudaMemcpyDeviceToHost) != cudaSuccess) ||
        (p && cudaMemcpy(p, d->p + id * J, J * 4, cudaMemcpyDeviceToHost) != cudaSuccess) ||
        (primed && cudaMemcpy(primed, d->primed + id, 4, cudaMemcpyDeviceToHost) != cudaSuccess))
        return CAC_E_CUDA;
    return CAC_OK;
}
