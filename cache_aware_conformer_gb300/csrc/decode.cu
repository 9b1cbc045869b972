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
//      tiled (32 slots x 16 classes) over the CTAs, K = joint_dim, written as
//      per-tile partial maxima;
//   B  decisions: per active slot the first maximum over the partials; blank
//      (or max_symbols reached) moves the slot to its next frame, anything else
//      is emitted and queued for the predictor;
//   C  LSTM step of the queued slots, tiled (32 slots x 4 hidden units = 16
//      gate rows): gates = tab[token] + W_hh h, with tab = emb W_ih^T + b_ih +
//      b_hh computed once at load (the input half of the gates depends on the
//      token only), then the cell update in the tile;
//   D  predictor projection p = W_pred h' + b_pred of the queued slots, tiled
//      (32 slots x 16 outputs).
// Every tile stages its rows (weights, and slot rows when its slot tile
// changes) with one TMA bulk copy per row; the 8 warps split K and reduce
// their partial tiles through shared memory.
// h is kept twice per stream ([2][S][P]): a queued emission carries the index
// of the stream's current copy, phase C reads it and writes the new h into
// the other one, which becomes current (the index flips when the emission is
// queued, so phase D reads the new copy and nothing is copied back).
// Grid-wide barriers separate the phases: an arrival counter and a generation
// word in global memory, every spin bounded (about a second) after which the
// kernel latches CAC_E_TIMEOUT, raises an abort word that releases every
// other waiter, and returns.  Everything is fp32 on the CUDA cores (the pages
// fix fp32 for the decoder, so every argmax is decided in fp32).
#include <cfloat>
#include <climits>
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
constexpr int TN = 16;         // output columns per tile
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
    int *frame, *sym, *act, *emk, *emid, *cnt;  // emid: stream id * 2 + current h copy
    float* pval;
    int* pidx;
    int* hsel;  // [S] index of the stream's current h copy
    int S;
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

// Os[slot][col] = sum_k As[slot][k] * Ws[col][k] for the tile's 32 slots x
// TN columns.  Warp w takes the K segment [w K/8, (w + 1) K/8) for all 512
// outputs (lane = slot, 16 independent accumulators, weights broadcast to the
// warp), so the tile's latency is one segment whatever the number of live
// slots; the 8 partial tiles are summed through `red` (8 x 512 floats).  K a
// multiple of 32, rows K + 4 floats apart.
__device__ __forceinline__ void mac16(int K, const float* As, const float* Ws, float* Os, float* red) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, ld = K + 4;
    const int seg = K / 8, k0 = w * seg;
    float acc[TN];
#pragma unroll
    for (int c = 0; c < TN; ++c) acc[c] = 0.f;
    const float* ap = As + lane * ld + k0;
    const float* wp = Ws + k0;
#pragma unroll 2
    for (int k = 0; k < seg; k += 4) {
        const float4 a = *reinterpret_cast<const float4*>(ap + k);
#pragma unroll
        for (int c = 0; c < TN; ++c) {
            const float4 v = *reinterpret_cast<const float4*>(wp + c * ld + k);
            acc[c] = fmaf(a.x, v.x, acc[c]);
            acc[c] = fmaf(a.y, v.y, acc[c]);
            acc[c] = fmaf(a.z, v.z, acc[c]);
            acc[c] = fmaf(a.w, v.w, acc[c]);
        }
    }
    float4* rp = reinterpret_cast<float4*>(red + w * TS * TN + lane * TN);
#pragma unroll
    for (int q = 0; q < TN / 4; ++q) rp[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
    __syncthreads();
    for (int o = tid; o < TS * TN; o += DT) {
        float sum = 0.f;
#pragma unroll
        for (int ww = 0; ww < 8; ++ww) sum += red[ww * TS * TN + o];
        Os[(o / TN) * OLD + (o % TN)] = sum;
    }
}

// Stage one tile's rows with the TMA engine: every row is contiguous (K
// floats), so one bulk copy per row lands it in shared memory (rows K + 4
// floats apart) and completes on `bar`.  Sources: A rows from a0[r] into A0
// and, if a1, from a1[r] into A1 (only when load_a), weight rows wrow(r) into
// Ws; nullptr rows are left as they are (their outputs are never used:
// padding slots are not stored, classes past the last are masked).  Every
// thread calls; false when the wait gave up (CAC_E_TIMEOUT latched, abort
// raised).
template <class WRow>
__device__ bool stage_tile(const DecParams& d, int K, bool load_a, float* A0, const float* const* a0, float* A1,
                           const float* const* a1, float* Ws, WRow wrow, uint64_t* bar, uint32_t& phase) {
    const int ld = K + 4, tid = threadIdx.x;
    __syncthreads();  // every earlier read of these buffers is done
    if (tid < 32) {  // warp 0: lane 0 posts the byte count, the lanes issue one row each
        const uint32_t rb = (uint32_t)K * 4;
        if (tid == 0) {
            fence_proxy_async_smem();
            asm volatile("fence.proxy.async.global;" ::: "memory");
            uint32_t bytes = 0;
            for (int r = 0; r < TN; ++r) bytes += wrow(r) ? rb : 0;
            if (load_a)
                for (int r = 0; r < TS; ++r) bytes += (a0[r] ? rb : 0) + (a1 && a1[r] ? rb : 0);
            mbar_expect_tx(bar, bytes);
        }
        __syncwarp();
        if (tid < TN)
            if (const float* w = wrow(tid)) bulk_g2s(Ws + tid * ld, w, rb, bar);
        if (load_a) {
            if (a0[tid]) bulk_g2s(A0 + tid * ld, a0[tid], rb, bar);
            if (a1 && a1[tid]) bulk_g2s(A1 + tid * ld, a1[tid], rb, bar);
        }
    }
    const bool ok = __syncthreads_and(mbar_wait(bar, phase));
    phase ^= 1u;
    if (!ok && tid == 0) {
        latch_error(d.status, CAC_E_TIMEOUT);
        atomicExch(d.abort_flag, 1);
    }
    return ok;
}

// Per-tile row table in shared memory: the slot b, stream id and (phase A)
// token-independent row pointers of the tile's 32 rows, resolved once by 32
// threads so that the bulk row loads that follow are independent.
struct RowTab {
    int b[TS], id[TS], k[TS];
    const float* src[TS];  // A row source (nullptr: padding row)
    const float* aux[TS];  // phase A: the stream's predictor projection p
};

// Phase C: LSTM step of the queued emissions 0 .. ne (token emk[.], stream and h copy emid[.]):
// tile = (32 slots, 4 hidden units = the 4 x 4 gate rows of those units).
__device__ void phase_lstm(const DecParams& d, const int* emk, const int* emid, int ne, float* As, float* Ws,
                           float* Os, float* red, RowTab& rt, uint64_t* bar, uint32_t& phase) {
    const int P = d.P, tid = threadIdx.x;
    const int ut = P / 4, tiles = ((ne + TS - 1) / TS) * ut;
    int loaded = -1;  // slot tile whose h rows sit in As
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int st = t / ut, j0 = (t % ut) * 4;
        const bool load_a = st != loaded;
        if (load_a) {
            __syncthreads();
            if (tid < TS) {
                const int i = st * TS + tid;
                rt.src[tid] = nullptr;
                if (i < ne) {
                    const int e2 = __ldcg(emid + i), id = e2 >> 1, cur = e2 & 1;
                    rt.id[tid] = id;
                    rt.k[tid] = __ldcg(emk + i);
                    rt.src[tid] = d.h + ((long long)cur * d.S + id) * P;
                    rt.aux[tid] = d.h + ((long long)(cur ^ 1) * d.S + id) * P;  // the new h goes to the other copy
                }
            }
            __syncthreads();
            loaded = st;
        }
        if (!stage_tile(d, P, load_a, As, rt.src, nullptr, nullptr, Ws,
                        [&](int r) -> const float* { return d.whh + (long long)((r >> 2) * P + j0 + (r & 3)) * P; },
                        bar, phase))
            return;
        mac16(P, As, Ws, Os, red);
        __syncthreads();
        if (tid < TS * 4) {  // cell update of (slot r, unit jj)
            const int r = tid >> 2, jj = tid & 3;
            if (rt.src[r]) {
                const int id = rt.id[r], j = j0 + jj;
                const float* tb = d.tab + (long long)rt.k[r] * 4 * P;
                const float gi = Os[r * OLD + jj] + __ldg(tb + j);
                const float gf = Os[r * OLD + 4 + jj] + __ldg(tb + P + j);
                const float gg = Os[r * OLD + 8 + jj] + __ldg(tb + 2 * P + j);
                const float go = Os[r * OLD + 12 + jj] + __ldg(tb + 3 * P + j);
                float* cp = d.c + (long long)id * P + j;
                const float c2 = sigm(gf) * __ldcg(cp) + sigm(gi) * tanhf(gg);
                *cp = c2;
                const_cast<float*>(rt.aux[r])[j] = sigm(go) * tanhf(c2);
            }
        }
        __syncthreads();  // Ws, Os and the row table are reused by the next tile
    }
}

// Phase D: p = W_pred h' + b_pred for the queued slots.
__device__ void phase_proj(const DecParams& d, const int* emid, int ne, float* As, float* Ws, float* Os,
                           float* red, RowTab& rt, uint64_t* bar, uint32_t& phase) {
    const int P = d.P, J = d.J, tid = threadIdx.x;
    const int jt = J / TN, tiles = ((ne + TS - 1) / TS) * jt;
    int loaded = -1;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int st = t / jt, c0 = (t % jt) * TN;
        const bool load_a = st != loaded;
        if (load_a) {
            __syncthreads();
            if (tid < TS) {
                const int i = st * TS + tid;
                rt.src[tid] = nullptr;
                if (i < ne) {
                    const int e2 = __ldcg(emid + i), id = e2 >> 1;
                    rt.id[tid] = id;
                    rt.src[tid] = d.h + ((long long)((e2 & 1) ^ 1) * d.S + id) * P;  // the new h
                }
            }
            __syncthreads();
            loaded = st;
        }
        if (!stage_tile(d, P, load_a, As, rt.src, nullptr, nullptr, Ws,
                        [&](int r) -> const float* { return d.wpp + (long long)(c0 + r) * P; }, bar, phase))
            return;
        mac16(P, As, Ws, Os, red);
        __syncthreads();
        for (int e = tid; e < TS * TN; e += DT) {
            const int r = e / TN, cc = e % TN;
            if (rt.src[r]) d.p[(long long)rt.id[r] * J + c0 + cc] = Os[r * OLD + cc] + __ldg(d.bpp + c0 + cc);
        }
        __syncthreads();
    }
}

// Phase A: logits of the active slots act[0 .. na) at their current frame,
// partial first-maximum per TN-class tile into pval / pidx [slot][nct].
__device__ void phase_joint(const DecParams& d, const int* act, int na, float* As, float* Ws, float* Os,
                            float* Ps, float* red, RowTab& rt, uint64_t* bar, uint32_t& phase) {
    const int J = d.J, C = d.C, tid = threadIdx.x;
    const int tiles = ((na + TS - 1) / TS) * d.nct;
    int loaded = -1;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int st = t / d.nct, ct = t % d.nct, c0 = ct * TN;
        const bool load_a = st != loaded;
        if (load_a) {
            __syncthreads();
            if (tid < TS) {
                const int i = st * TS + tid;
                rt.src[tid] = nullptr;
                rt.aux[tid] = nullptr;
                if (i < na) {
                    const int b = __ldcg(act + i), id = d.ids[b], f = __ldcg(d.frame + b);
                    rt.b[tid] = b;
                    rt.src[tid] = d.z + b * d.zb + (long long)f * J;
                    rt.aux[tid] = d.p + (long long)id * J;
                }
            }
            __syncthreads();
        }
        if (!stage_tile(d, J, load_a, As, rt.src, Ps, rt.aux, Ws,
                        [&](int r) -> const float* { return c0 + r < C ? d.wout + (long long)(c0 + r) * J : nullptr; },
                        bar, phase))
            return;
        if (load_a) {
            for (int e = tid; e < TS * J / 4; e += DT) {  // As <- ReLU(z + p)
                const int r = e / (J / 4), q = e % (J / 4);
                float4* a = reinterpret_cast<float4*>(As + r * (J + 4) + 4 * q);
                const float4 pp = *reinterpret_cast<const float4*>(Ps + r * (J + 4) + 4 * q);
                const float4 zz = *a;
                *a = make_float4(fmaxf(zz.x + pp.x, 0.f), fmaxf(zz.y + pp.y, 0.f), fmaxf(zz.z + pp.z, 0.f),
                                 fmaxf(zz.w + pp.w, 0.f));
            }
            __syncthreads();
            loaded = st;
        }
        mac16(J, As, Ws, Os, red);
        __syncthreads();
        if (tid < TS && rt.src[tid]) {
            float best = -FLT_MAX;
            int bi = c0;
            for (int q = 0; q < TN && c0 + q < C; ++q) {
                const float v = Os[tid * OLD + q] + __ldg(d.bout + c0 + q);
                if (v > best) { best = v; bi = c0 + q; }
            }
            const int b = rt.b[tid];
            d.pval[(long long)b * d.nct + ct] = best;
            d.pidx[(long long)b * d.nct + ct] = bi;
        }
        __syncthreads();
    }
}

// The whole step (see the top of the file).  Iteration it reads the active
// list act[it & 1] (length cnt[2 it]) and writes the next one act[(it + 1) & 1]
// (length cnt[2 it + 2]) and its emissions emk/emid[it & 1] (length cnt[2 it +
// 1]); iteration 0 only builds the first active list and primes reset streams.
__global__ void __launch_bounds__(DT, 1) dec_step_kernel(DecParams d) {
    extern __shared__ float smem[];
    const int K = d.P > d.J ? d.P : d.J;
    float* As = smem;
    float* Ws = As + TS * (K + 4);
    float* Os = Ws + TN * (K + 4);
    float* Ps = Os + TS * OLD;  // phase A: the p rows (TS x (J + 4))
    float* red = Ps + TS * (d.J + 4);  // partial tiles of mac16 (8 x TS x TN)
    __shared__ RowTab rt;
    __shared__ __align__(8) uint64_t tbar;
    uint32_t tphase = 0;
    if (threadIdx.x == 0) {
        mbar_init(&tbar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const int gtid = blockIdx.x * DT + threadIdx.x, gstride = gridDim.x * DT;
    const long long tsym = (long long)d.T * d.max_sym;

    for (int b = gtid; b < d.n; b += gstride) {
        const int id = d.ids[b];
        d.frame[b] = 0;
        d.sym[b] = 0;
        d.counts[b] = 0;
        if (d.T > 0) d.act[d.n + atomicAdd(&d.cnt[2], 1)] = b;
        if (__ldcg(d.primed + id) == 0) {  // stream start: zero state, one predictor step on blank
            const int cur = __ldcg(d.hsel + id);
            for (int j = 0; j < d.P; ++j) {
                d.h[((long long)cur * d.S + id) * d.P + j] = 0.f;
                d.c[(long long)id * d.P + j] = 0.f;
            }
            d.primed[id] = 1;
            d.hsel[id] = cur ^ 1;
            const int q = atomicAdd(&d.cnt[1], 1);
            d.emk[q] = d.blank;
            d.emid[q] = id * 2 + cur;
        }
    }
    if (!grid_sync(d)) return;
    int ne = __ldcg(d.cnt + 1);
    if (ne > 0) {
        phase_lstm(d, d.emk, d.emid, ne, As, Ws, Os, red, rt, &tbar, tphase);
        if (!grid_sync(d)) return;
        phase_proj(d, d.emid, ne, As, Ws, Os, red, rt, &tbar, tphase);
        if (!grid_sync(d)) return;
    }
    for (int it = 1; it <= d.maxit; ++it) {
        const int na = __ldcg(d.cnt + 2 * it);
        if (na == 0) break;
        const int* act = d.act + (it & 1) * d.n;
        phase_joint(d, act, na, As, Ws, Os, Ps, red, rt, &tbar, tphase);
        if (!grid_sync(d)) return;
        int* nact = d.act + ((it + 1) & 1) * d.n;
        int* emk = d.emk + (it & 1) * d.n;
        int* emid = d.emid + (it & 1) * d.n;
        // one warp per active slot: first maximum over the slot's partials
        const int lane = threadIdx.x & 31;
        for (int i = gtid >> 5; i < na; i += gstride >> 5) {
            const int b = __ldcg(act + i);
            const long long pb = (long long)b * d.nct;
            float best = -FLT_MAX;
            int k = INT_MAX;
            for (int q = lane; q < d.nct; q += 32) {  // tiles in class order: strict > keeps the lowest index
                const float v = __ldcg(d.pval + pb + q);
                if (v > best) {
                    best = v;
                    k = __ldcg(d.pidx + pb + q);
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {  // larger value wins, equal values: the lower class
                const float ov = __shfl_xor_sync(0xffffffffu, best, o);
                const int ok = __shfl_xor_sync(0xffffffffu, k, o);
                if (ov > best || (ov == best && ok < k)) {
                    best = ov;
                    k = ok;
                }
            }
            if (lane != 0) continue;
            int f = __ldcg(d.frame + b), sy = __ldcg(d.sym + b);
            bool next = k == d.blank;
            if (!next) {
                const int cn = __ldcg(d.counts + b);
                d.tokens[b * tsym + cn] = k;
                d.frames[b * tsym + cn] = f;
                d.counts[b] = cn + 1;
                const int q = atomicAdd(&d.cnt[2 * it + 1], 1);
                const int id = d.ids[b], cur = __ldcg(d.hsel + id);
                d.hsel[id] = cur ^ 1;
                emk[q] = k;
                emid[q] = id * 2 + cur;
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
            phase_lstm(d, emk, emid, ne, As, Ws, Os, red, rt, &tbar, tphase);
            if (!grid_sync(d)) return;
            phase_proj(d, emid, ne, As, Ws, Os, red, rt, &tbar, tphase);
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

// Failure-path self-test kernels (cac_op_wait_selftest): the production waits
// with nothing that satisfies them.
__global__ void wait_selftest_mbar_kernel(int* status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        if (!mbar_wait(&bar, 0)) latch_error(status, CAC_E_TIMEOUT);  // no thread ever arrives
    }
}

__global__ void wait_selftest_grid_kernel(DecParams d) {
    if (blockIdx.x == 0) return;  // the first block never reaches the barrier
    grid_sync(d);
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
    int *ids = nullptr, *frame = nullptr, *sym = nullptr, *act = nullptr, *emk = nullptr, *emid = nullptr;
    int* cnt = nullptr;  // [2 (maxit + 2)] iteration counters, then arrivals / generation / abort
    int cnt_ints = 0;
    float* pval = nullptr;
    int* pidx = nullptr;
    int* hsel = nullptr;  // [S]
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

// free one allocation of d early (it leaves d's list, so destroy does not free it again)
void dfree(cac_decoder* d, void* p) {
    for (auto it = d->allocs.begin(); it != d->allocs.end(); ++it)
        if (*it == p) {
            cudaFree(p);
            d->allocs.erase(it);
            return;
        }
}

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
        // the embedding and the input weights live on only inside tab
        for (void* t : {static_cast<void*>(emb_d), static_cast<void*>(wih_d), static_cast<void*>(bih_d),
                        static_cast<void*>(bhh_d)})
            dfree(d, t);
    }
    const size_t S = max_streams;
    if ((r = dalloc_t(d, 2 * S * P, &d->h)) || (r = dalloc_t(d, S, &d->hsel)) || (r = dalloc_t(d, S * P, &d->c)) ||
        (r = dalloc_t(d, S * J, &d->p)) ||
        (r = dalloc_t(d, S, &d->primed)) || (r = dalloc_t(d, S, &d->ids)) || (r = dalloc_t(d, S, &d->frame)) ||
        (r = dalloc_t(d, S, &d->sym)) || (r = dalloc_t(d, 2 * S, &d->act)) || (r = dalloc_t(d, 2 * S, &d->emid)) ||
        (r = dalloc_t(d, 2 * S, &d->emk)) || (r = dalloc_t(d, S * d->nct, &d->pval)) ||
        (r = dalloc_t(d, S * d->nct, &d->pidx)) ||
        (r = dalloc_t(d, 1, &d->status)))
        return fail(r);
    d->cnt_ints = 2 * (maxit_for(*cfg, MAX_T) + 2) + 4;
    if ((r = dalloc_t(d, d->cnt_ints, &d->cnt))) return fail(r);
    if (cudaMemset(d->primed, 0, S * 4) != cudaSuccess || cudaMemset(d->status, 0, 4) != cudaSuccess ||
        cudaMemset(d->h, 0, 2 * S * P * 4) != cudaSuccess || cudaMemset(d->hsel, 0, S * 4) != cudaSuccess || cudaMemset(d->c, 0, S * P * 4) != cudaSuccess ||
        cudaMemset(d->p, 0, S * J * 4) != cudaSuccess)
        return fail(CAC_E_CUDA);
    if (cudaMallocHost(reinterpret_cast<void**>(&d->pinned), sizeof(int) * S * ID_SLOTS) != cudaSuccess)
        return fail(CAC_E_NOMEM);
    for (auto& e : d->slot_ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return fail(CAC_E_CUDA);
    // one CTA per SM, all co-resident (cooperative launch)
    const int K = (int)(P > J ? P : J);
    d->smem = sizeof(float) * ((size_t)(TS + TN) * (K + 4) + (size_t)TS * OLD + (size_t)TS * (J + 4) + 8 * TS * TN);
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
    p.h = d->h; p.c = d->c; p.p = d->p; p.primed = d->primed; p.hsel = d->hsel; p.S = d->S;
    p.frame = d->frame; p.sym = d->sym; p.act = d->act; p.emk = d->emk; p.emid = d->emid; p.cnt = d->cnt;
    p.pval = d->pval; p.pidx = d->pidx;
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
    int sel = 0;
    if (cudaMemcpy(&sel, d->hsel + id, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return CAC_E_CUDA;
    if ((h && cudaMemcpy(h, d->h + ((size_t)sel * d->S + id) * P, P * 4, cudaMemcpyDeviceToHost) != cudaSuccess) ||
        (c && cudaMemcpy(c, d->c + id * P, P * 4, cudaMemcpyDeviceToHost) != cudaSuccess) ||
        (p && cudaMemcpy(p, d->p + id * J, J * 4, cudaMemcpyDeviceToHost) != cudaSuccess) ||
        (primed && cudaMemcpy(primed, d->primed + id, 4, cudaMemcpyDeviceToHost) != cudaSuccess))
        return CAC_E_CUDA;
    return CAC_OK;
}

extern "C" int cac_op_wait_selftest(int which, void* stream) {
    if (which != 0 && which != 1) return CAC_E_INVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* buf = nullptr;  // [0] status, [1] abort, [2..3] barrier words
    if (cudaMalloc(&buf, 4 * sizeof(int)) != cudaSuccess) return CAC_E_NOMEM;
    int rc = CAC_E_CUDA;
    if (cudaMemsetAsync(buf, 0, 4 * sizeof(int), s) == cudaSuccess) {
        cudaError_t e;
        if (which == 0) {
            wait_selftest_mbar_kernel<<<1, 32, 0, s>>>(buf);
            e = cudaGetLastError();
        } else {
            int dev = 0, sms = 0;
            if (cudaGetDevice(&dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                sms = 2;
            DecParams p{};
            p.status = buf;
            p.abort_flag = buf + 1;
            p.bar = reinterpret_cast<unsigned*>(buf + 2);
            cudaLaunchConfig_t lc = {};
            lc.gridDim = dim3(sms > 1 ? sms : 2);
            lc.blockDim = dim3(DT);
            lc.stream = s;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeCooperative;
            at[0].val.cooperative = 1;
            lc.attrs = at;
            lc.numAttrs = 1;
            e = cudaLaunchKernelEx(&lc, wait_selftest_grid_kernel, p);
        }
        int st = 0;
        if (e == cudaSuccess && cudaStreamSynchronize(s) == cudaSuccess &&
            cudaMemcpy(&st, buf, sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess)
            rc = st;
    }
    cudaFree(buf);
    return rc;
}
