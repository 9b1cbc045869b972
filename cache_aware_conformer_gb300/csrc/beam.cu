// Batched modified-ALSD RNN-T beam search ("Fast Accuracy-Preserving RNNT
// Beam Search on Apple Silicon", §2.2–§2.4, §4.1; what it computes is stated
// in include/cac_beam.h), over the predictor and joint of the greedy decoder.
//
// One step (or piece of <= 64 frames of a step) is ONE cooperative launch of a
// persistent kernel (one 256-thread CTA per SM).  All streams advance in
// lockstep alignment iterations; each iteration is
//   A  joint: logits of every hypothesis that needs them (row list), tiled
//      (32 rows x 16 classes) over the CTAs, written whole to L[row][class];
//   BC one warp per running stream: fp32 log-softmax of its rows, top K per
//      hypothesis, the global top K of the K*K candidates (forced blank at the
//      symbol limit, final hypotheses as keep candidates), labels applied,
//      recombination of identical survivors (token sequences compared), new
//      predictor states allocated from the stream's pool of 2K, the new beam
//      written to the other half of its double buffer, and the rows of the
//      next iteration appended (or the stream stalls: a running hypothesis
//      needs a frame that has not arrived);
//   D  LSTM step of the new labels: gates = tab[label] + W_hh h_parent, with
//      tab = emb W_ih^T + b_ih + b_hh built once at load; the cell update
//      writes the new state into a pool entry no survivor references;
//   E  predictor projection of the new states.
// Survivors on blank or keep share their parent's pool entry (no copy).  The
// pool of 2K entries per stream suffices: at most K entries are referenced
// by the new beam, at most K parents are read and at most K entries are
// written, and parents and written entries of labels together number <= 2K
// minus the blank and keep survivors.  Projected encoder frames are kept in a
// per-stream ring of 128 frames (hypotheses of one alignment length may lag
// each other by a few frames, so a hypothesis can need a frame of an earlier
// step).  Grid-wide barriers are bounded (about a second) and latch
// CAC_E_TIMEOUT, raise an abort word and return.  Everything is fp32 on the
// CUDA cores (the pages fix fp32 for the decoder).
#include <cfloat>
#include <climits>
#include <cmath>
#include <cstring>
#include <vector>

#include "cac.h"
#include "cac_beam.h"
#include "common.cuh"
#include "status.cuh"

namespace cac {
namespace {

constexpr int BT = 256;        // threads per CTA
constexpr int TS = 32;         // rows per tile
constexpr int TN = 16;         // output columns per tile
constexpr int OLD = TN + 1;    // row stride of the output tile
constexpr int KMAX = 8;        // beam width limit
constexpr int RING = 128;      // projected frames kept per stream
constexpr int PIECE = 64;      // frames per launch (a longer step is split)
constexpr int KEEP = -2;       // candidate label of a final hypothesis kept as it is
constexpr unsigned FULL = 0xffffffffu;

struct BeamParams {
    int n, T, fin, C, P, J, K, max_sym, blank, maxit, lmax, S;
    const int* ids;          // [n] stream id of each batch slot
    const int* tb;           // [n] frames of the stream before this launch
    const int* fresh;        // [n] 1: the stream starts here
    const float* z;          // slot b's new frame t at z + b * zb + t * J
    long long zb;
    const float *tab, *whh, *wpp, *bpp, *wout, *bout;
    const float* zero;       // [P] zeros: the parent state of a stream start
    float* ring;             // [S][RING][J]
    int* cur;                // [S] current half of the beam double buffer
    float* sc;               // [2][S][K] scores (-inf: empty slot)
    int *tm, *lst, *len, *sym, *st;  // [2][S][K] time, last label, length, symbols at time, pool entry
    int* tok;                // [2][S][K][lmax]
    float *h, *c, *pp;       // [S][2K][P], [S][2K][P], [S][2K][J]
    int *rb, *rk, *rt, *rs;  // [2][n K] rows: batch slot, beam slot, frame, pool entry
    int* rmap;               // [2][n K] row of (b, k), -1 when none
    int* run;                // [2][n] stream takes the iteration
    float* L;                // [n K][C] logits of the iteration's rows
    int *jb, *jsrc, *jdst, *jlab;  // [n K (+ n)] jobs: batch slot, parent (-1: zero state), new entry, label
    int* cnt;                // [2 (maxit + 2)]: rows and jobs per iteration
    int* pending;            // [1] rows left when the iteration cap ended the launch
    unsigned* bar;           // [0] arrivals, [1] generation
    int* abort_flag;
    int* status;
    int cpad;                // C rounded up to 4
    int bcw;                 // floats of one warp's phase-BC scratch
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier of a cooperative launch.  bar[0] counts the arrivals of
// the whole launch (zeroed before it): a CTA's k-th barrier is passed once the
// count reaches k * gridDim.x (`target` carries k * gridDim.x from call to
// call).  Thread 0 arrives with a release add after the CTA's own barrier and
// polls with acquire loads; false when it gave up (timeout, latched, or
// another CTA's abort), in which case the caller returns.
__device__ bool grid_sync(const BeamParams& d, unsigned& target) {
    __shared__ int ok_s;
    __syncthreads();
    target += gridDim.x;
    if (threadIdx.x == 0) {
        int ok = 1;
        __threadfence();
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(d.bar) : "memory");
        if (ld_acquire(d.bar) < target) {
            const long long t0 = clock64();
            for (unsigned it = 1;; ++it) {
                if (ld_acquire(d.bar) >= target) break;
                if ((it & 255u) == 0u) {
                    if (*(volatile int*)d.abort_flag) { ok = 0; break; }
                    if (clock64() - t0 > (1ll << 31)) {
                        latch_error(d.status, CAC_E_TIMEOUT);
                        atomicExch(d.abort_flag, 1);
                        ok = 0;
                        break;
                    }
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

// Os[row][col] = sum_k As[row][k] * Ws[col][k] for 32 rows x TN columns: warp w
// takes K segment w of 8 for all outputs (lane = row), the 8 partial tiles are
// summed through `red`.  K a multiple of 32, rows K + 4 floats apart.
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
    for (int o = tid; o < TS * TN; o += BT) {
        float sum = 0.f;
#pragma unroll
        for (int ww = 0; ww < 8; ++ww) sum += red[ww * TS * TN + o];
        Os[(o / TN) * OLD + (o % TN)] = sum;
    }
}

// Stage one tile's rows with one TMA bulk copy per row (K floats each, rows
// K + 4 floats apart in shared memory), completing on `bar`: A rows a0[r] into
// A0 and, if a1, a1[r] into A1 (only when load_a); weight rows wrow(r) into Ws.
// nullptr rows are skipped (their outputs are never used).  Every thread
// calls; false when the wait gave up (CAC_E_TIMEOUT latched, abort raised).
template <class WRow>
__device__ bool stage_tile(const BeamParams& d, int K, bool load_a, float* A0, const float* const* a0, float* A1,
                           const float* const* a1, float* Ws, WRow wrow, uint64_t* bar, uint32_t& phase) {
    const int ld = K + 4, tid = threadIdx.x;
    __syncthreads();  // every earlier read of these buffers is done
    if (tid < 32) {
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

struct RowTab {
    int id[TS], k[TS], dst[TS];
    const float* src[TS];
    const float* aux[TS];
    const float* csrc[TS];
};

__device__ __forceinline__ long long slot_ix(const BeamParams& d, int buf, int s, int k) {
    return ((long long)buf * d.S + s) * d.K + k;
}
__device__ __forceinline__ long long pool_ix(const BeamParams& d, int s, int q) { return (long long)s * 2 * d.K + q; }

// Rows of iteration itn for batch slot b (one thread, reading the stream's
// current beam): the stream takes the iteration when a hypothesis is before
// the limit (the utterance's end on a final step) and, unless the step is
// final, none needs a frame that has not arrived; its rows are the
// hypotheses before the limit.  A row whose frame has left the ring latches
// CAC_E_LIMIT (its result is then not the search's).
__device__ void build_rows(const BeamParams& d, int b, int itn) {
    const int s = d.ids[b], K = d.K, par = itn & 1, buf = __ldcg(d.cur + s);
    const int avail = __ldg(d.tb + b) + d.T;
    const int lim = d.fin ? avail : INT_MAX;
    const long long nK = (long long)d.n * K;
    int nrow = 0;
    bool anyrun = false, wait = false;
    for (int k = 0; k < K; ++k) {
        const long long ix = slot_ix(d, buf, s, k);
        if (!(__ldcg(d.sc + ix) > -INFINITY)) continue;
        const int t = __ldcg(d.tm + ix);
        if (t < lim) {
            anyrun = true;
            ++nrow;
        }
        if (!d.fin && t >= avail) wait = true;
    }
    const bool go = anyrun && !wait;
    d.run[par * d.n + b] = go ? 1 : 0;
    int r = go ? atomicAdd(d.cnt + 2 * itn, nrow) : 0;
    for (int k = 0; k < K; ++k) {
        const long long ix = slot_ix(d, buf, s, k);
        int m = -1;
        if (go && __ldcg(d.sc + ix) > -INFINITY) {
            const int t = __ldcg(d.tm + ix);
            if (t < lim) {
                if (t < avail - RING || t < 0) latch_error(d.status, CAC_E_LIMIT);
                m = r++;
                d.rb[par * nK + m] = b;
                d.rk[par * nK + m] = k;
                d.rt[par * nK + m] = t;
                d.rs[par * nK + m] = __ldcg(d.st + ix);
            }
        }
        d.rmap[par * nK + (long long)b * K + k] = m;
    }
}

// Stream starts, the new frames into the rings, the rows of iteration 1.
__device__ void phase_init(const BeamParams& d) {
    const int gtid = blockIdx.x * BT + threadIdx.x, gstride = gridDim.x * BT;
    for (int b = gtid; b < d.n; b += gstride) {
        if (__ldg(d.fresh + b)) {  // one hypothesis: score 0, nothing emitted, last label blank, pool entry 0
            const int s = d.ids[b];
            d.cur[s] = 0;
            for (int k = 0; k < d.K; ++k) {
                const long long ix = slot_ix(d, 0, s, k);
                d.sc[ix] = k ? -INFINITY : 0.f;
                d.tm[ix] = 0;
                d.lst[ix] = d.blank;
                d.len[ix] = 0;
                d.sym[ix] = 0;
                d.st[ix] = 0;
            }
            const int j = atomicAdd(d.cnt + 1, 1);  // its predictor state: one step on blank from zero
            d.jb[j] = b;
            d.jsrc[j] = -1;
            d.jdst[j] = 0;
            d.jlab[j] = d.blank;
        }
        build_rows(d, b, 1);
    }
    const long long per = (long long)d.T * d.J, tot = (long long)d.n * per;
    for (long long e = gtid; e < tot; e += gstride) {
        const int b = (int)(e / per), t = (int)((e % per) / d.J), c = (int)(e % d.J);
        const int s = d.ids[b];
        d.ring[((long long)s * RING + (__ldg(d.tb + b) + t) % RING) * d.J + c] = __ldg(d.z + b * d.zb + (long long)t * d.J + c);
    }
}

// Phase A: logits of the iteration's rows into L (all classes).
__device__ void phase_joint(const BeamParams& d, int it, float* As, float* Ws, float* Os, float* Ps, float* red,
                            RowTab& rt, uint64_t* bar, uint32_t& phase) {
    const int J = d.J, C = d.C, tid = threadIdx.x, par = it & 1;
    const long long nK = (long long)d.n * d.K;
    const int nr = __ldcg(d.cnt + 2 * it), nct = (C + TN - 1) / TN;
    const int tiles = ((nr + TS - 1) / TS) * nct;
    int loaded = -1;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int st = t / nct, c0 = (t % nct) * TN;
        const bool load_a = st != loaded;
        if (load_a) {
            __syncthreads();
            if (tid < TS) {
                const int i = st * TS + tid;
                rt.src[tid] = nullptr;
                rt.aux[tid] = nullptr;
                if (i < nr) {
                    const int b = __ldcg(d.rb + par * nK + i), s = d.ids[b];
                    const int f = __ldcg(d.rt + par * nK + i), q = __ldcg(d.rs + par * nK + i);
                    rt.k[tid] = i;
                    rt.src[tid] = d.ring + ((long long)s * RING + (f % RING + RING) % RING) * J;
                    rt.aux[tid] = d.pp + pool_ix(d, s, q) * J;
                }
            }
            __syncthreads();
        }
        if (!stage_tile(d, J, load_a, As, rt.src, Ps, rt.aux, Ws,
                        [&](int r) -> const float* { return c0 + r < C ? d.wout + (long long)(c0 + r) * J : nullptr; },
                        bar, phase))
            return;
        if (load_a) {
            for (int e = tid; e < TS * J / 4; e += BT) {  // As <- ReLU(z + p)
                const int r = e / (J / 4), q = e % (J / 4);
                float4* a = reinterpret_cast<float4*>(As + r * (J + 4) + 4 * q);
                const float4 pq = *reinterpret_cast<const float4*>(Ps + r * (J + 4) + 4 * q);
                const float4 zz = *a;
                *a = make_float4(fmaxf(zz.x + pq.x, 0.f), fmaxf(zz.y + pq.y, 0.f), fmaxf(zz.z + pq.z, 0.f),
                                 fmaxf(zz.w + pq.w, 0.f));
            }
            __syncthreads();
            loaded = st;
        }
        mac16(J, As, Ws, Os, red);
        __syncthreads();
        for (int e = tid; e < TS * TN; e += BT) {
            const int r = e / TN, q = e % TN;
            if (rt.src[r] && c0 + q < C)
                d.L[(long long)rt.k[r] * C + c0 + q] = Os[r * OLD + q] + __ldg(d.bout + c0 + q);
        }
        __syncthreads();
    }
}

// Phase D: LSTM step of the iteration's jobs, tile = 32 jobs x 4 hidden units.
__device__ void phase_lstm(const BeamParams& d, int it, float* As, float* Ws, float* Os, float* red, RowTab& rt,
                           uint64_t* bar, uint32_t& phase) {
    const int P = d.P, tid = threadIdx.x;
    const int nj = __ldcg(d.cnt + 2 * it + 1), ut = P / 4, tiles = ((nj + TS - 1) / TS) * ut;
    int loaded = -1;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int st = t / ut, j0 = (t % ut) * 4;
        const bool load_a = st != loaded;
        if (load_a) {
            __syncthreads();
            if (tid < TS) {
                const int i = st * TS + tid;
                rt.src[tid] = nullptr;
                if (i < nj) {
                    const int b = __ldcg(d.jb + i), s = d.ids[b], src = __ldcg(d.jsrc + i);
                    rt.id[tid] = s;
                    rt.k[tid] = __ldcg(d.jlab + i);
                    rt.dst[tid] = __ldcg(d.jdst + i);
                    rt.src[tid] = src < 0 ? d.zero : d.h + pool_ix(d, s, src) * P;
                    rt.csrc[tid] = src < 0 ? d.zero : d.c + pool_ix(d, s, src) * P;
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
        if (tid < TS * 4) {  // cell update of (job r, unit jj)
            const int r = tid >> 2, jj = tid & 3;
            if (rt.src[r]) {
                const int s = rt.id[r], j = j0 + jj;
                const float* tb = d.tab + (long long)rt.k[r] * 4 * P;
                const float gi = Os[r * OLD + jj] + __ldg(tb + j);
                const float gf = Os[r * OLD + 4 + jj] + __ldg(tb + P + j);
                const float gg = Os[r * OLD + 8 + jj] + __ldg(tb + 2 * P + j);
                const float go = Os[r * OLD + 12 + jj] + __ldg(tb + 3 * P + j);
                const float c2 = sigm(gf) * __ldcg(rt.csrc[r] + j) + sigm(gi) * tanhf(gg);
                const long long o = pool_ix(d, s, rt.dst[r]) * P + j;
                d.c[o] = c2;
                d.h[o] = sigm(go) * tanhf(c2);
            }
        }
        __syncthreads();
    }
}

// Phase E: predictor projection of the new states, pp = W_pred h + b_pred.
__device__ void phase_proj(const BeamParams& d, int it, float* As, float* Ws, float* Os, float* red, RowTab& rt,
                           uint64_t* bar, uint32_t& phase) {
    const int P = d.P, J = d.J, tid = threadIdx.x;
    const int nj = __ldcg(d.cnt + 2 * it + 1), jt = J / TN, tiles = ((nj + TS - 1) / TS) * jt;
    int loaded = -1;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int st = t / jt, c0 = (t % jt) * TN;
        const bool load_a = st != loaded;
        if (load_a) {
            __syncthreads();
            if (tid < TS) {
                const int i = st * TS + tid;
                rt.src[tid] = nullptr;
                if (i < nj) {
                    const int s = d.ids[__ldcg(d.jb + i)];
                    rt.id[tid] = s;
                    rt.dst[tid] = __ldcg(d.jdst + i);
                    rt.src[tid] = d.h + pool_ix(d, s, rt.dst[tid]) * P;
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
        for (int e = tid; e < TS * TN; e += BT) {
            const int r = e / TN, q = e % TN;
            if (rt.src[r]) d.pp[pool_ix(d, rt.id[r], rt.dst[r]) * J + c0 + q] = Os[r * OLD + q] + __ldg(d.bpp + c0 + q);
        }
        __syncthreads();
    }
}

__device__ __forceinline__ int shfl(int v, int src) { return __shfl_sync(FULL, v, src); }
__device__ __forceinline__ float shflf(float v, int src) { return __shfl_sync(FULL, v, src); }

// Warp argmax by (value descending, index ascending) over the lanes' (v, i).
__device__ __forceinline__ void warp_best(float& v, int& i) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(FULL, v, o);
        const int oi = __shfl_xor_sync(FULL, i, o);
        if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
        }
    }
}

// Phase BC: one warp per stream that takes iteration `it` (see the top of the file).
__device__ void phase_bc(const BeamParams& d, int it, float* wsm) {
    const int lane = threadIdx.x & 31, K = d.K, C = d.C, par = it & 1;
    const int gw = (blockIdx.x * BT + threadIdx.x) >> 5, nw = (gridDim.x * BT) >> 5;
    float* lp = wsm + (threadIdx.x >> 5) * d.bcw;       // [cpad] log-probabilities of one row
    float* cv = lp + d.cpad;                             // [K * K] candidate scores
    int* cl = reinterpret_cast<int*>(cv + KMAX * KMAX);  // [K * K] candidate labels
    const long long nK = (long long)d.n * K;
    for (int b = gw; b < d.n; b += nw) {
        if (!__ldcg(d.run + par * d.n + b)) {
            // a stream that sits out stays out for the rest of the launch (its beam and
            // the frames it has do not change); clear its flag for the next iteration,
            // which still holds the value of two iterations ago
            if (lane == 0) d.run[(par ^ 1) * d.n + b] = 0;
            continue;
        }
        const int s = d.ids[b];
        const int lim = d.fin ? __ldg(d.tb + b) + d.T : INT_MAX;
        const int buf = __ldcg(d.cur + s), nb = buf ^ 1;
        float osc = -INFINITY;
        int otm = 0, olst = 0, oln = 0, osym = 0, ost = 0;
        if (lane < K) {  // lane k holds the old beam's slot k
            const long long ix = slot_ix(d, buf, s, lane);
            osc = __ldcg(d.sc + ix);
            otm = __ldcg(d.tm + ix);
            olst = __ldcg(d.lst + ix);
            oln = __ldcg(d.len + ix);
            osym = __ldcg(d.sym + ix);
            ost = __ldcg(d.st + ix);
        }
        for (int p = lane; p < K * K; p += 32) {
            cv[p] = -INFINITY;
            cl[p] = -1;
        }
        __syncwarp();
        // candidates of every slot, in position order parent * K + j
        for (int k = 0; k < K; ++k) {
            const float sk = shflf(osc, k);
            const int tk = shfl(otm, k), symk = shfl(osym, k);
            if (!(sk > -INFINITY)) continue;
            if (tk >= lim) {  // final: one keep candidate
                if (lane == 0) {
                    cv[k * K] = sk;
                    cl[k * K] = KEEP;
                }
                continue;
            }
            const int r = __ldcg(d.rmap + par * nK + (long long)b * K + k);
            const float* Lr = d.L + (long long)(r < 0 ? 0 : r) * C;
            float m = -INFINITY;
            for (int c = lane; c < C; c += 32) {
                const float v = __ldcg(Lr + c);
                lp[c] = v;
                m = fmaxf(m, v);
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
            float sum = 0.f;
            for (int c = lane; c < C; c += 32) sum += expf(lp[c] - m);
#pragma unroll
            for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(FULL, sum, o);
            const float lse = logf(sum);
            for (int c = lane; c < C; c += 32) lp[c] = (lp[c] - m) - lse;
            __syncwarp();
            if (symk >= d.max_sym) {  // forced blank
                if (lane == 0) {
                    cv[k * K] = sk + lp[d.blank];
                    cl[k * K] = d.blank;
                }
                __syncwarp();
                continue;
            }
            float pv = INFINITY;  // the previous pick: the next one comes strictly after it
            int pi = -1;
            for (int j = 0; j < K; ++j) {
                float bv = -INFINITY;
                int bi = INT_MAX;
                for (int c = lane; c < C; c += 32) {
                    const float v = lp[c];
                    if ((v < pv || (v == pv && c > pi)) && (v > bv || (v == bv && c < bi))) {
                        bv = v;
                        bi = c;
                    }
                }
                warp_best(bv, bi);
                if (bi == INT_MAX) break;  // fewer classes than K
                if (lane == 0) {
                    cv[k * K + j] = sk + bv;
                    cl[k * K + j] = bi;
                }
                pv = bv;
                pi = bi;
            }
            __syncwarp();
        }
        __syncwarp();  // every candidate is written (a keep candidate's path has no sync of its own)
        // the global top K (pruning); lane i takes survivor i
        float sv = -INFINITY;
        int sp = 0;
        {
            float pv = INFINITY;
            int pi = -1;
            for (int i = 0; i < K; ++i) {
                float bv = -INFINITY;
                int bp = INT_MAX;
                for (int p = lane; p < K * K; p += 32) {
                    const float v = cv[p];
                    if ((v < pv || (v == pv && p > pi)) && (v > bv || (v == bv && p < bp))) {
                        bv = v;
                        bp = p;
                    }
                }
                warp_best(bv, bp);
                if (lane == i) {
                    sv = bv;
                    sp = bp < K * K ? bp : 0;
                }
                pv = bv;
                pi = bp;
            }
        }
        const bool cand = lane < K && sv > -INFINITY;
        const int kp = cand ? sp / K : 0;
        const int lab = cand ? cl[sp] : -1;
        const int ptm = shfl(otm, kp), plst = shfl(olst, kp), pln = shfl(oln, kp), psym = shfl(osym, kp),
                  pst = shfl(ost, kp);
        bool live = cand;
        const bool islab = cand && lab != KEEP && lab != d.blank;
        int ntm = ptm, nlst = plst, nln = pln, nsym = psym, nst = pst;
        if (cand && lab == d.blank) {
            ntm = ptm + 1;
            nsym = 0;
        }
        if (islab) {
            if (pln + 1 > d.lmax) {  // transcript capacity: the label leaves the search
                live = false;
                latch_error(d.status, CAC_E_LIMIT);
            } else {
                nlst = lab;
                nln = pln + 1;
                nsym = psym + 1;
            }
        }
        float nsc = live ? sv : -INFINITY;
        // recombination: survivors with equal length, last label and tokens
        const int* T0 = d.tok + slot_ix(d, buf, s, 0) * d.lmax;
        unsigned eq = 0;  // lane i: the survivors i2 > i equal to survivor i
        for (int i = 0; i < K; ++i)
            for (int i2 = i + 1; i2 < K; ++i2) {
                if (!shfl(live, i) || !shfl(live, i2)) continue;
                const int L = shfl(nln, i);
                if (L != shfl(nln, i2) || shfl(nlst, i) != shfl(nlst, i2)) continue;
                const int ka = shfl(kp, i), kb = shfl(kp, i2), pa = shfl(pln, i), pb = shfl(pln, i2);
                const int la = shfl(lab, i), lb = shfl(lab, i2);
                const int* Ta = T0 + (long long)ka * d.lmax;
                const int* Tb = T0 + (long long)kb * d.lmax;
                bool diff = false;
                for (int x = lane; x < L; x += 32) {
                    const int va = x < pa ? __ldcg(Ta + x) : la;
                    const int vb = x < pb ? __ldcg(Tb + x) : lb;
                    diff |= va != vb;
                }
                if (!__any_sync(FULL, diff) && lane == i) eq |= 1u << i2;
            }
        unsigned done = 0;
        for (int i = 0; i < K; ++i) {
            if (!shfl(live, i) || ((done >> i) & 1u)) continue;
            const unsigned mem = ((unsigned)shfl((int)eq, i) | (1u << i)) & ~done;
            done |= mem;
            if (__popc(mem) < 2) continue;
            float m = -INFINITY;  // the best member: highest score, lowest slot on ties
            int best = i;
            for (int q = 0; q < K; ++q) {
                const float v = shflf(nsc, q);
                if (((mem >> q) & 1u) && v > m) {
                    m = v;
                    best = q;
                }
            }
            float sum = 0.f;
            for (int q = 0; q < K; ++q) {
                const float v = shflf(nsc, q);
                if ((mem >> q) & 1u) sum += expf(v - m);
            }
            const float merged = m + logf(sum);
            if ((mem >> lane) & 1u) {
                if (lane == best) {
                    nsc = merged;
                } else {
                    live = false;
                    nsc = -INFINITY;
                }
            }
        }
        // pool entries: keep and blank survivors share the parent's; labels take free ones
        unsigned busy = 0;
        for (int q = 0; q < K; ++q)
            if (shfl(live, q)) busy |= 1u << shfl(pst, q);
        for (int q = 0; q < K; ++q) {
            if (!shfl(live && islab, q)) continue;
            const int fr = __ffs(~busy) - 1;
            const int src = shfl(pst, q), lq = shfl(lab, q);
            if (fr < 0 || fr >= 2 * K) {  // cannot happen (see the top of the file); never write out of the pool
                if (lane == q) live = false;
                if (lane == 0) latch_error(d.status, CAC_E_LIMIT);
                continue;
            }
            busy |= 1u << fr;
            if (lane == q) nst = fr;
            if (lane == 0) {
                const int j = atomicAdd(d.cnt + 2 * it + 1, 1);
                d.jb[j] = b;
                d.jsrc[j] = src;
                d.jdst[j] = fr;
                d.jlab[j] = lq;
            }
        }
        // the new beam into the other half
        if (lane < K) {
            const long long ix = slot_ix(d, nb, s, lane);
            d.sc[ix] = live ? nsc : -INFINITY;
            d.tm[ix] = ntm;
            d.lst[ix] = nlst;
            d.len[ix] = nln;
            d.sym[ix] = nsym;
            d.st[ix] = nst;
        }
        int* N0 = d.tok + slot_ix(d, nb, s, 0) * d.lmax;
        for (int i = 0; i < K; ++i) {
            if (!shfl(live, i)) continue;
            const int L = shfl(nln, i), ka = shfl(kp, i), pa = shfl(pln, i), la = shfl(lab, i);
            const int* Ta = T0 + (long long)ka * d.lmax;
            int* Ni = N0 + (long long)i * d.lmax;
            for (int x = lane; x < L; x += 32) Ni[x] = x < pa ? __ldcg(Ta + x) : la;
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            d.cur[s] = nb;
            build_rows(d, b, it + 1);
        }
        __syncwarp();
    }
}

// The whole launch (see the top of the file).
__global__ void __launch_bounds__(BT, 1) beam_step_kernel(BeamParams d) {
    unsigned gt = 0;  // grid-barrier target
    extern __shared__ float smem[];
    const int Kd = d.P > d.J ? d.P : d.J;
    float* As = smem;
    float* Ws = As + TS * (Kd + 4);
    float* Os = Ws + TN * (Kd + 4);
    float* Ps = Os + TS * OLD;
    float* red = Ps + TS * (d.J + 4);
    __shared__ RowTab rt;
    __shared__ __align__(8) uint64_t tbar;
    uint32_t tphase = 0;
    if (threadIdx.x == 0) {
        mbar_init(&tbar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    phase_init(d);
    if (!grid_sync(d, gt)) return;
    if (__ldcg(d.cnt + 1) > 0) {  // predictor states of the stream starts
        phase_lstm(d, 0, As, Ws, Os, red, rt, &tbar, tphase);
        if (!grid_sync(d, gt)) return;
        phase_proj(d, 0, As, Ws, Os, red, rt, &tbar, tphase);
        if (!grid_sync(d, gt)) return;
    }
    int it = 1;
    for (; it <= d.maxit; ++it) {
        if (__ldcg(d.cnt + 2 * it) == 0) break;
        phase_joint(d, it, As, Ws, Os, Ps, red, rt, &tbar, tphase);
        if (!grid_sync(d, gt)) return;
        phase_bc(d, it, smem);
        if (!grid_sync(d, gt)) return;
        if (__ldcg(d.cnt + 2 * it + 1) > 0) {
            phase_lstm(d, it, As, Ws, Os, red, rt, &tbar, tphase);
            if (!grid_sync(d, gt)) return;
            phase_proj(d, it, As, Ws, Os, red, rt, &tbar, tphase);
            if (!grid_sync(d, gt)) return;
        }
    }
    if (it > d.maxit && blockIdx.x == 0 && threadIdx.x == 0 && __ldcg(d.cnt + 2 * it) > 0) *d.pending = 1;
}

// tab[k][r] = sum_m W_ih[r][m] emb[k][m] + b_ih[r] + b_hh[r], fp64 sums rounded to fp32
__global__ void beam_tab_kernel(const float* emb, const float* wih, const float* bih, const float* bhh, float* tab,
                                int C, int P) {
    const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= (long long)C * 4 * P) return;
    const int k = (int)(e / (4 * P)), r = (int)(e % (4 * P));
    double s = (double)bih[r] + (double)bhh[r];
    for (int m = 0; m < P; ++m) s += (double)wih[(long long)r * P + m] * (double)emb[(long long)k * P + m];
    tab[e] = (float)s;
}

}  // namespace
}  // namespace cac

using namespace cac;

namespace {
constexpr int BEAM_ID_SLOTS = 4;  // staging slots for per-launch slot tables
constexpr int BEAM_MAX_T = 1024;
}  // namespace

struct cac_beam {
    cac_dec_config cfg{};
    int C = 0, S = 0, K = 0, lmax = 0, grid = 0, cnt_ints = 0;
    size_t smem = 0;
    BeamParams proto{};               // the launch-independent fields
    std::vector<void*> allocs;
    int* slot_dev = nullptr;          // [BEAM_ID_SLOTS][3][S]: ids, tb, fresh
    int* pinned = nullptr;            // host [BEAM_ID_SLOTS][3][S]
    int* h_pending = nullptr;         // pinned host copy of the pending word
    cudaEvent_t ev[BEAM_ID_SLOTS] = {};
    int slot = 0;
    std::vector<int> tb;              // frames so far per stream
    std::vector<unsigned char> fresh, finished;
};

namespace {

int balloc(cac_beam* d, size_t bytes, void** out) {
    if (cudaMalloc(out, bytes < 16 ? 16 : bytes) != cudaSuccess) return cac::nomem();
    d->allocs.push_back(*out);
    return CAC_OK;
}

template <class T>
int balloc_t(cac_beam* d, size_t count, T** out) {
    void* v = nullptr;
    const int r = balloc(d, count * sizeof(T), &v);
    *out = static_cast<T*>(v);
    return r;
}

int maxit_for(const cac_dec_config& c, int T, int K) { return (T + 1) * (c.max_symbols + 1) + 2 * K + 2; }

// One cooperative launch over frames [off, off + T) of the call's z.
int launch_piece(cac_beam* bd, int n, const int* ids, const float* z, long long zb, int off, int T, bool fin,
                 bool first, cudaStream_t st) {
    const int k = bd->slot;
    bd->slot = (bd->slot + 1) % BEAM_ID_SLOTS;
    if (cudaEventSynchronize(bd->ev[k]) != cudaSuccess) return CAC_E_CUDA;
    int* h = bd->pinned + (size_t)k * 3 * bd->S;
    int* dv = bd->slot_dev + (size_t)k * 3 * bd->S;
    for (int b = 0; b < n; ++b) {
        h[b] = ids[b];
        h[bd->S + b] = bd->tb[ids[b]] + off;
        h[2 * bd->S + b] = first && bd->fresh[ids[b]] ? 1 : 0;
    }
    if (cudaMemcpyAsync(dv, h, sizeof(int) * 3 * bd->S, cudaMemcpyHostToDevice, st) != cudaSuccess) return CAC_E_CUDA;
    BeamParams p = bd->proto;
    p.n = n;
    p.T = T;
    p.fin = fin ? 1 : 0;
    p.maxit = maxit_for(bd->cfg, T, bd->K);
    p.ids = dv;
    p.tb = dv + bd->S;
    p.fresh = dv + 2 * bd->S;
    p.z = T > 0 ? z + (long long)off * bd->cfg.joint_dim : nullptr;
    p.zb = zb;
    if (cudaMemsetAsync(p.cnt, 0, sizeof(int) * (2 * (p.maxit + 2)), st) != cudaSuccess ||
        cudaMemsetAsync(p.bar, 0, sizeof(unsigned) * 2, st) != cudaSuccess ||
        cudaMemsetAsync(p.abort_flag, 0, sizeof(int), st) != cudaSuccess ||
        cudaMemsetAsync(p.pending, 0, sizeof(int), st) != cudaSuccess)
        return CAC_E_CUDA;
    void* args[] = {&p};
    if (cudaLaunchCooperativeKernel(reinterpret_cast<void*>(beam_step_kernel), dim3(bd->grid), dim3(BT), args,
                                    bd->smem, st) != cudaSuccess)
        return CAC_E_CUDA;
    if (cudaEventRecord(bd->ev[k], st) != cudaSuccess) return CAC_E_CUDA;
    return CAC_OK;
}

}  // namespace

extern "C" void cac_beam_destroy(cac_beam* bd) {
    if (!bd) return;
    cudaDeviceSynchronize();
    for (void* a : bd->allocs) cudaFree(a);
    if (bd->pinned) cudaFreeHost(bd->pinned);
    if (bd->h_pending) cudaFreeHost(bd->h_pending);
    for (auto& e : bd->ev)
        if (e) cudaEventDestroy(e);
    delete bd;
}

extern "C" int cac_beam_create(const cac_dec_config* cfg, const float* weights, size_t n_floats, int beam,
                               int max_streams, int max_tokens, cac_beam** out) {
    if (!cfg || !weights || !out || max_streams < 1 || cfg->vocab < 1 || cfg->max_symbols < 1 || beam < 1 ||
        beam > KMAX || max_tokens < 1 || cfg->pred_dim < 64 || cfg->joint_dim < 64)
        return CAC_E_INVAL;
    if (cfg->pred_dim % 64 || cfg->joint_dim % 64) return CAC_E_UNSUPPORTED;
    const size_t C = (size_t)cfg->vocab + 2, P = cfg->pred_dim, J = cfg->joint_dim;
    const size_t need = C * P + 2 * 4 * P * P + 2 * 4 * P + J * P + J + C * J + C;
    if (n_floats != need) return CAC_E_INVAL;
    *out = nullptr;
    cac_beam* d = new cac_beam();
    d->cfg = *cfg;
    d->C = (int)C;
    d->S = max_streams;
    d->K = beam;
    d->lmax = max_tokens;
    auto fail = [&](int code) {
        cac_beam_destroy(d);
        return code;
    };
    BeamParams& p = d->proto;
    p.C = (int)C;
    p.P = (int)P;
    p.J = (int)J;
    p.K = beam;
    p.max_sym = cfg->max_symbols;
    p.blank = cfg->vocab;
    p.lmax = max_tokens;
    p.S = max_streams;
    p.cpad = (int)((C + 3) / 4 * 4);
    p.bcw = p.cpad + 2 * KMAX * KMAX;
    const float* w = weights;
    const float *emb = w, *wih = emb + C * P, *whh = wih + 4 * P * P, *bih = whh + 4 * P * P, *bhh = bih + 4 * P,
                *wpp = bhh + 4 * P, *bpp = wpp + J * P, *wout = bpp + J, *bout = wout + C * J;
    auto upload = [&](const float* src, size_t nf, float** dst) {
        int r = balloc_t(d, nf, dst);
        if (r == CAC_OK && cudaMemcpy(*dst, src, nf * 4, cudaMemcpyHostToDevice) != cudaSuccess) r = CAC_E_CUDA;
        return r;
    };
    int r;
    float *emb_d = nullptr, *wih_d = nullptr, *bih_d = nullptr, *bhh_d = nullptr, *tab = nullptr;
    float *whh_d = nullptr, *wpp_d = nullptr, *bpp_d = nullptr, *wout_d = nullptr, *bout_d = nullptr;
    if ((r = upload(emb, C * P, &emb_d)) || (r = upload(wih, 4 * P * P, &wih_d)) || (r = upload(bih, 4 * P, &bih_d)) ||
        (r = upload(bhh, 4 * P, &bhh_d)) || (r = upload(whh, 4 * P * P, &whh_d)) || (r = upload(wpp, J * P, &wpp_d)) ||
        (r = upload(bpp, J, &bpp_d)) || (r = upload(wout, C * J, &wout_d)) || (r = upload(bout, C, &bout_d)) ||
        (r = balloc_t(d, C * 4 * P, &tab)))
        return fail(r);
    {
        const long long nt = (long long)C * 4 * P;
        beam_tab_kernel<<<(unsigned)((nt + 255) / 256), 256>>>(emb_d, wih_d, bih_d, bhh_d, tab, (int)C, (int)P);
        if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return fail(CAC_E_CUDA);
    }
    p.tab = tab;
    p.whh = whh_d;
    p.wpp = wpp_d;
    p.bpp = bpp_d;
    p.wout = wout_d;
    p.bout = bout_d;
    const size_t S = max_streams, K = beam, nK = S * K;
    float* zero = nullptr;
    if ((r = balloc_t(d, P, &zero)) || (r = balloc_t(d, S * RING * J, &p.ring)) || (r = balloc_t(d, S, &p.cur)) ||
        (r = balloc_t(d, 2 * nK, &p.sc)) || (r = balloc_t(d, 2 * nK, &p.tm)) || (r = balloc_t(d, 2 * nK, &p.lst)) ||
        (r = balloc_t(d, 2 * nK, &p.len)) || (r = balloc_t(d, 2 * nK, &p.sym)) || (r = balloc_t(d, 2 * nK, &p.st)) ||
        (r = balloc_t(d, 2 * nK * (size_t)max_tokens, &p.tok)) || (r = balloc_t(d, S * 2 * K * P, &p.h)) ||
        (r = balloc_t(d, S * 2 * K * P, &p.c)) || (r = balloc_t(d, S * 2 * K * J, &p.pp)) ||
        (r = balloc_t(d, 2 * nK, &p.rb)) || (r = balloc_t(d, 2 * nK, &p.rk)) || (r = balloc_t(d, 2 * nK, &p.rt)) ||
        (r = balloc_t(d, 2 * nK, &p.rs)) || (r = balloc_t(d, 2 * nK, &p.rmap)) || (r = balloc_t(d, 2 * S, &p.run)) ||
        (r = balloc_t(d, nK * C, &p.L)) || (r = balloc_t(d, nK, &p.jb)) || (r = balloc_t(d, nK, &p.jsrc)) ||
        (r = balloc_t(d, nK, &p.jdst)) || (r = balloc_t(d, nK, &p.jlab)) || (r = balloc_t(d, 1, &p.pending)) ||
        (r = balloc_t(d, 2, &p.bar)) || (r = balloc_t(d, 1, &p.abort_flag)) || (r = balloc_t(d, 1, &p.status)) ||
        (r = balloc_t(d, (size_t)BEAM_ID_SLOTS * 3 * S, &d->slot_dev)))
        return fail(r);
    p.zero = zero;
    // host-side frees of the load-only buffers (tab holds what they contributed)
    for (float* t : {emb_d, wih_d, bih_d, bhh_d})
        for (auto it = d->allocs.begin(); it != d->allocs.end(); ++it)
            if (*it == t) {
                cudaFree(t);
                d->allocs.erase(it);
                break;
            }
    d->cnt_ints = 2 * (maxit_for(*cfg, PIECE, beam) + 2);
    if ((r = balloc_t(d, (size_t)d->cnt_ints, &p.cnt))) return fail(r);
    if (cudaMemset(zero, 0, P * 4) != cudaSuccess || cudaMemset(p.status, 0, 4) != cudaSuccess ||
        cudaMemset(p.cur, 0, S * 4) != cudaSuccess || cudaMemset(p.ring, 0, S * RING * J * 4) != cudaSuccess)
        return fail(CAC_E_CUDA);
    if (cudaMallocHost(reinterpret_cast<void**>(&d->pinned), sizeof(int) * 3 * S * BEAM_ID_SLOTS) != cudaSuccess ||
        cudaMallocHost(reinterpret_cast<void**>(&d->h_pending), sizeof(int)) != cudaSuccess)
        return fail(cac::nomem());
    for (auto& e : d->ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return fail(CAC_E_CUDA);
    const size_t Kd = P > J ? P : J;
    const size_t tiles = sizeof(float) * ((TS + TN) * (Kd + 4) + TS * OLD + TS * (J + 4) + 8 * TS * TN);
    const size_t bc = sizeof(float) * 8 * (size_t)p.bcw;
    d->smem = tiles > bc ? tiles : bc;
    if (d->smem > 227 * 1024) return fail(CAC_E_UNSUPPORTED);
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaFuncSetAttribute(beam_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d->smem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, beam_step_kernel, BT, d->smem) != cudaSuccess)
        return fail(CAC_E_CUDA);
    if (per_sm < 1) return fail(CAC_E_UNSUPPORTED);
    d->grid = sms;
    d->tb.assign(S, 0);
    d->fresh.assign(S, 1);
    d->finished.assign(S, 0);
    *out = d;
    return CAC_OK;
}

extern "C" int cac_beam_reset(cac_beam* bd, int n, const int* ids) {
    if (!bd || n < 0 || (n > 0 && !ids)) return CAC_E_INVAL;
    for (int i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= bd->S) return CAC_E_INVAL;
    for (int i = 0; i < n; ++i) {
        bd->tb[ids[i]] = 0;
        bd->fresh[ids[i]] = 1;
        bd->finished[ids[i]] = 0;
    }
    return CAC_OK;
}

extern "C" int cac_beam_step(cac_beam* bd, int n, const int* ids, const float* z, long long z_bstride, int T,
                             int is_final, void* stream) {
    if (!bd || n < 1 || n > bd->S || !ids || T < 0 || T > BEAM_MAX_T || (is_final != 0 && is_final != 1))
        return CAC_E_INVAL;
    const int J = bd->cfg.joint_dim;
    if (T > 0 && (!z || (n > 1 && z_bstride < (long long)T * J))) return CAC_E_INVAL;
    std::vector<unsigned char> seen(bd->S, 0);
    for (int b = 0; b < n; ++b) {
        if (ids[b] < 0 || ids[b] >= bd->S || seen[ids[b]]) return CAC_E_INVAL;
        seen[ids[b]] = 1;
        if (bd->finished[ids[b]]) return CAC_E_STATE;
        if (bd->tb[ids[b]] > INT_MAX - 2 * BEAM_MAX_T) return CAC_E_LIMIT;
    }
    if (T == 0 && !is_final) return CAC_OK;  // no frames: nothing can move
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int off = 0;
    bool first = true;
    do {
        const int Tp = T - off < PIECE ? T - off : PIECE;
        const bool fin = is_final && off + Tp == T;
        int r = launch_piece(bd, n, ids, z, z_bstride, off, Tp, fin, first, st);
        if (r != CAC_OK) return r;
        first = false;
        // The last piece of an utterance runs the search to its end.  Every
        // hypothesis of alignment length i has time >= (i - max_symbols) /
        // (max_symbols + 1), so the search ends by i = (frames + 1) (max_symbols
        // + 1); the relaunches are capped accordingly (CAC_E_LIMIT beyond).
        int tmax = 0;
        for (int b = 0; b < n; ++b) tmax = bd->tb[ids[b]] > tmax ? bd->tb[ids[b]] : tmax;
        const long long bound = ((long long)tmax + T + 2) * (bd->cfg.max_symbols + 1);
        const long long cap = bound / maxit_for(bd->cfg, Tp, bd->K) + 2;
        for (long long tries = 0; fin; ++tries) {
            if (cudaMemcpyAsync(bd->h_pending, bd->proto.pending, sizeof(int), cudaMemcpyDeviceToHost, st) !=
                    cudaSuccess ||
                cudaStreamSynchronize(st) != cudaSuccess)
                return CAC_E_CUDA;
            if (!*bd->h_pending) break;
            if (tries >= cap) return CAC_E_LIMIT;
            if ((r = launch_piece(bd, n, ids, z, z_bstride, off, Tp, fin, false, st)) != CAC_OK) return r;
        }
        off += Tp;
    } while (off < T);
    for (int b = 0; b < n; ++b) {
        bd->tb[ids[b]] += T;
        bd->fresh[ids[b]] = 0;
        if (is_final) bd->finished[ids[b]] = 1;
    }
    return CAC_OK;
}

extern "C" int cac_beam_check(cac_beam* bd) {
    if (!bd) return CAC_E_INVAL;
    int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpy(&v, bd->proto.status, 4, cudaMemcpyDeviceToHost) !=
                                                       cudaSuccess ||
        cudaMemset(bd->proto.status, 0, 4) != cudaSuccess)
        return CAC_E_CUDA;
    return v;
}

extern "C" int cac_beam_get(cac_beam* bd, int id, int score_norm, float* scores, int* lengths, int* tokens,
                            int* best) {
    if (!bd || id < 0 || id >= bd->S || !scores || !lengths || !best) return CAC_E_INVAL;
    if (bd->fresh[id]) return CAC_E_STATE;  // nothing decoded since the stream's start
    const BeamParams& p = bd->proto;
    const int K = bd->K;
    int cur = 0;
    if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpy(&cur, p.cur + id, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return CAC_E_CUDA;
    const size_t base = ((size_t)cur * bd->S + id) * K;
    if (cudaMemcpy(scores, p.sc + base, sizeof(float) * K, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(lengths, p.len + base, sizeof(int) * K, cudaMemcpyDeviceToHost) != cudaSuccess ||
        (tokens && cudaMemcpy(tokens, p.tok + base * bd->lmax, sizeof(int) * K * bd->lmax, cudaMemcpyDeviceToHost) !=
                       cudaSuccess))
        return CAC_E_CUDA;
    int bi = -1;
    double bv = 0.0;
    for (int k = 0; k < K; ++k) {
        if (!(scores[k] > -INFINITY)) continue;
        const double v = score_norm ? (double)scores[k] / (lengths[k] + 1) : (double)scores[k];
        if (bi < 0 || v > bv) {
            bi = k;
            bv = v;
        }
    }
    *best = bi;
    return CAC_OK;
}
