// Batched greedy RNN-T decoding with an end-of-utterance class ("Parakeet-EOU-
// 120M — Streaming ASR Model", §Architecture: fp32 LSTM predictor on the last
// non-blank token, joint over one projected encoder frame and the predictor
// output -> vocabulary + blank + EOU, greedy loop per frame advancing the
// predictor only on non-blank emissions; "True streaming encode —
// implementation spec", §Decoder state carry: h/c persist per stream).
//
// One step decodes n streams over T frames in ONE cooperative launch of a
// persistent kernel (one 256-thread CTA per SM).  The streams advance in
// lockstep iterations, and every iteration is a short chain of latency-bound
// phases, so the kernel is built to keep each phase and each hand-off short:
//
// * Weights stay on chip.  CTA g owns a slice of the classes (joint rows of
//   W_out), of the LSTM hidden units (their 4 gate rows of W_hh) and of the
//   predictor-projection outputs (rows of W_pred); the slices are copied into
//   shared memory once per launch and every iteration only moves activation
//   rows (u = ReLU(z + p) for the joint, h for the LSTM, the new h for the
//   projection).
// * Rows arrive through a ring of TMA bulk copies: warp w consumes rows w, w +
//   8, ... and refills the ring slot it just read with the row RB further on,
//   so up to RB rows per CTA are in flight whatever the number of active slots.
// * Decisions are replicated.  Phase A ends with one 64-bit atomicMax per
//   (active slot, CTA): the key packs the logit (as an order-preserving
//   unsigned) above the complemented class id, so the maximum over the CTAs
//   is the largest logit with the lowest class on ties, independent of the
//   order of the atomics.  Every CTA then reads the keys of all active slots
//   and applies the same decisions to its own shared-memory copy of the slot
//   state (frame, symbols on the frame, emissions, current h copy, active
//   list), so no CTA has to publish decisions to the others; the owner of a
//   slot (slot mod grid) writes its outputs.
//
// Iteration: A joint + per-CTA argmax keys | grid barrier | B decisions (all
// CTAs alike) and C the LSTM step of the emitting slots (gates = tab[token] +
// W_hh h, tab = emb W_ih^T + b_ih + b_hh computed once at load; the cell
// update of the CTA's units, new h into the stream's other h copy) | grid
// barrier (only when something was emitted) | D the predictor projection
// p = W_pred h' + b_pred of the emitting slots and the next joint inputs u of
// every slot that stays active (its frame or its p changed) | grid barrier.
// Grid barriers: an arrival counter and a generation word in global memory,
// every spin bounded (about a second) after which the kernel latches
// CAC_E_TIMEOUT, raises an abort word that releases every other waiter, and
// returns.  Everything is fp32 on the CUDA cores (the pages fix fp32 for the
// decoder, so every argmax is decided in fp32).
#include <algorithm>
#include <cfloat>
#include <climits>
#include <cstring>
#include <mutex>
#include <vector>

#include "cac.h"
#include "cac_decode.h"
#include "common.cuh"
#include "status.cuh"

namespace cac {
namespace {

constexpr int DT = 256;         // threads per CTA
constexpr int NW = DT / 32;     // warps per CTA
constexpr int MAXCH = 16;       // 64-float chunks per row (pred_dim, joint_dim <= 1024)
constexpr int RB_MAX = 64;      // ring slots (rows in flight per CTA)
constexpr int STATE_INTS = 10;  // ints of replicated slot state per stream slot

// floats of the bias slices in shared memory, rounded so that the row ring
// after them stays 256-byte aligned
__host__ __device__ constexpr int bias_floats(int nc_max, int no_max) { return (nc_max + no_max + 63) / 64 * 64; }

struct DecParams {
    int n, T, C, P, J, max_sym, blank, maxit, S;
    int nc_max, nu_max, no_max;  // largest class / hidden-unit / projection-output slice of a CTA
    int RB;                      // ring slots, a multiple of 2 NW (pairs of slots for the joint)
    const int* ids;
    const float* z;
    long long zb;
    int *tokens, *frames, *counts;
    const float *tab, *whh, *wpp, *bpp, *wout, *bout;
    float *h, *c, *p;
    float* u;                    // [S][J] joint inputs ReLU(z + p) of the slots
    unsigned long long* keys;    // [2][S] packed (logit, class) maxima, one parity per iteration
    int* primed;
    int* hsel;                   // [S] index of the stream's current h copy
    unsigned* bar;               // [0] arrivals, [1] generation
    int* abort_flag;
    int* status;
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
__device__ bool grid_sync(const DecParams& d, unsigned& target) {
    __shared__ int ok_s;
    __syncthreads();
    target += gridDim.x;
    if (threadIdx.x == 0) {
        int ok = 1;
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
        ok_s = ok;
    }
    __syncthreads();
    return ok_s != 0;
}

__device__ __forceinline__ float sigm(float x) { return 1.f / (1.f + expf(-x)); }

// First index of CTA g's share of `total` items split as evenly as possible.
__device__ __forceinline__ int slice_lo(int total, int g, int G) { return (int)(((long long)total * g) / G); }

// Dot products of a group of RG rows (shared memory, K floats) with nv <= NV
// weight rows W + v * ldw (shared memory): lane l accumulates the products of
// the elements 64 ch + 2 l, 64 ch + 2 l + 1 of every 64-float chunk ch, so
// every weight element loaded serves all RG rows.
template <int RG, int NV>
__device__ __forceinline__ void group_dots(const float* const (&rows)[RG], const float* W, int ldw, int nv, int K,
                                           float (&acc)[RG][NV]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < RG; ++r)
#pragma unroll
        for (int v = 0; v < NV; ++v) acc[r][v] = 0.f;
#pragma unroll 2
    for (int c0 = 2 * lane; c0 < K; c0 += 64) {
        float2 x[RG];
#pragma unroll
        for (int r = 0; r < RG; ++r) x[r] = *reinterpret_cast<const float2*>(rows[r] + c0);
#pragma unroll
        for (int v = 0; v < NV; ++v)
            if (v < nv) {
                const float2 w = *reinterpret_cast<const float2*>(W + (size_t)v * ldw + c0);
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    acc[r][v] = fmaf(x[r].x, w.x, acc[r][v]);
                    acc[r][v] = fmaf(x[r].y, w.y, acc[r][v]);
                }
            }
    }
}

// Transposed warp reduction of 32 per-lane values: afterwards lane l holds the
// sum over the warp of value l (31 shuffles: each round a lane keeps half of
// its values and receives its partner's partial of that half).
__device__ __forceinline__ float transpose_sum32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = up ? v[i] : v[i + o];
            const float keep = up ? v[i + o] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

// The same for 16 values: lanes l and l + 16 both end with the sum of value
// l mod 16 (a plain exchange across the half-warps, then four transposed rounds).
__device__ __forceinline__ float transpose_sum16(float (&v)[16]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i], 16);
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = up ? v[i] : v[i + o];
            const float keep = up ? v[i + o] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0];
}

// Argmax key: the logit's bits made order-preserving as an unsigned (negative
// values flipped, positive ones offset), above the complemented class id, so
// that the unsigned maximum is the largest logit and, among equal logits, the
// lowest class.  Zero is below every key.
__device__ __forceinline__ unsigned long long pack_key(float v, int cls) {
    uint32_t b = __float_as_uint(v);
    b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)b << 32) | (unsigned long long)(~(uint32_t)cls);
}
__device__ __forceinline__ int key_class(unsigned long long k) { return (int)~(uint32_t)(k & 0xffffffffull); }

// Ring of RB row buffers (K floats each) filled by TMA bulk copies.  Row i of
// a pass lands in slot i mod RB and is consumed by warp i mod NW (RB is a
// multiple of NW, so a slot always belongs to the same warp); after consuming
// row i the warp refills the slot with row i + RB.  `par` holds the warp's
// slot parities (bit j: slot warp + NW j) across passes.
struct Ring {
    float* buf;
    uint64_t* full;
    int RB, K;
};

// One pass over rows 0 .. m-1 of rowK <= K floats (src(i): global address of
// row i, 16-byte aligned).  The warp takes its rows in groups of RG (RG <=
// RB / NW, so the rows of a group sit in distinct slots): use(rows, idx) gets
// the group's shared-memory rows and row indices (idx -1 and a repeat of the
// first row past the end).  False when a wait gave up (the caller latches and
// aborts).
template <int RG, class Src, class Use>
__device__ bool ring_pass(const Ring& R, uint32_t& par, int m, int rowK, Src src, Use use) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bytes = (uint32_t)rowK * 4u;
    if (lane == 0) {
        // rows were written by other CTAs (generic stores, released by the grid
        // barrier) and this warp's earlier reads of its slots are done: order
        // both before the bulk copies
        fence_proxy_async_smem();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        for (int i = warp; i < m && i < R.RB; i += NW) {
            mbar_expect_tx(&R.full[i], bytes);
            bulk_g2s(R.buf + (size_t)i * R.K, src(i), bytes, &R.full[i]);
        }
    }
    __syncwarp();
    for (int i0 = warp; i0 < m; i0 += NW * RG) {
        const float* rows[RG];
        int idx[RG];
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            const int i = i0 + NW * r;
            if (i < m) {
                const int s = i % R.RB, j = s / NW;
                if (!mbar_wait(&R.full[s], (par >> j) & 1u)) return false;
                par ^= 1u << j;
                rows[r] = R.buf + (size_t)s * R.K;
                idx[r] = i;
            } else {
                rows[r] = rows[0];
                idx[r] = -1;
            }
        }
        use(rows, idx);
        __syncwarp();
        if (lane == 0) {
            fence_proxy_async_smem();
#pragma unroll
            for (int r = 0; r < RG; ++r) {
                const int i = i0 + NW * r;
                if (i + R.RB < m) {
                    const int s = i % R.RB;
                    mbar_expect_tx(&R.full[s], bytes);
                    bulk_g2s(R.buf + (size_t)s * R.K, src(i + R.RB), bytes, &R.full[s]);
                }
            }
        }
    }
    return true;
}

// The same ring with slots of two rows (RB / 2 pair slots, a multiple of NW):
// pair p holds rows 2p and 2p + 1 of the pass (src(i) as above) and comes in
// one bulk copy when the two rows are adjacent in global memory (consecutive
// slots), in two otherwise, so that a pass over consecutive rows issues half
// as many copies.  use(rows, idx) as for RG = 2.
template <class Src, class Use>
__device__ bool ring_pass_pairs(const Ring& R, uint32_t& par, int m, int rowK, Src src, Use use) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int RBP = R.RB / 2, np = (m + 1) / 2;
    auto issue = [&](int p, int s) {
        const int i0 = 2 * p, cnt = i0 + 1 < m ? 2 : 1;
        const float* a = src(i0);
        float* dst = R.buf + (size_t)s * 2 * R.K;
        mbar_expect_tx(&R.full[s], (uint32_t)(cnt * rowK) * 4u);
        if (cnt == 2) {
            const float* b = src(i0 + 1);
            if (b == a + rowK && rowK == R.K) {
                bulk_g2s(dst, a, (uint32_t)(2 * rowK) * 4u, &R.full[s]);
                return;
            }
            bulk_g2s(dst + R.K, b, (uint32_t)rowK * 4u, &R.full[s]);
        }
        bulk_g2s(dst, a, (uint32_t)rowK * 4u, &R.full[s]);
    };
    if (lane == 0) {
        fence_proxy_async_smem();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        for (int p = warp; p < np && p < RBP; p += NW) issue(p, p);
    }
    __syncwarp();
    for (int p = warp; p < np; p += NW) {
        const int s = p % RBP, j = s / NW;
        if (!mbar_wait(&R.full[s], (par >> j) & 1u)) return false;
        par ^= 1u << j;
        const float* rows[2] = {R.buf + (size_t)s * 2 * R.K, R.buf + (size_t)s * 2 * R.K + R.K};
        const int idx[2] = {2 * p, 2 * p + 1 < m ? 2 * p + 1 : -1};
        if (idx[1] < 0) rows[1] = rows[0];
        use(rows, idx);
        __syncwarp();
        if (lane == 0 && p + RBP < np) {
            fence_proxy_async_smem();
            issue(p + RBP, s);
        }
    }
    return true;
}

__device__ __forceinline__ void fail_abort(const DecParams& d) {
    latch_error(d.status, CAC_E_TIMEOUT);
    atomicExch(d.abort_flag, 1);
}

// The whole step (see the top of the file).
__global__ void __launch_bounds__(DT, 1) dec_step_kernel(DecParams d) {
    extern __shared__ __align__(16) float sm[];
    __shared__ __align__(8) uint64_t ring_full[RB_MAX];
    __shared__ __align__(8) uint64_t wbar;
    __shared__ int s_cnt[2];  // emitted, next active
    const int G = gridDim.x, g = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = d.P, J = d.J, n = d.n, S = d.S;
    const int c_lo = slice_lo(d.C, g, G), nc = slice_lo(d.C, g + 1, G) - c_lo;
    const int u_lo = slice_lo(P, g, G), nu = slice_lo(P, g + 1, G) - u_lo;
    const int o_lo = slice_lo(J, g, G), no = slice_lo(J, g + 1, G) - o_lo;
    const int K = P > J ? P : J;
    float* Wo = sm;                                   // [nc_max][J]
    float* Wh = Wo + (size_t)d.nc_max * J;            // [4 nu][P]: row q nu + i = gate q of unit u_lo + i
    float* Wp = Wh + (size_t)4 * d.nu_max * P;        // [no_max][P]
    float* bo_s = Wp + (size_t)d.no_max * P;          // [nc_max] joint biases of the CTA's classes
    float* bp_s = bo_s + d.nc_max;                    // [no_max] projection biases
    float* rbuf = Wp + (size_t)d.no_max * P + bias_floats(d.nc_max, d.no_max);  // [RB][K]
    int* frame = reinterpret_cast<int*>(rbuf + (size_t)d.RB * K);  // replicated slot state
    int* sym = frame + S;                             // emissions on the current frame
    int* ecount = sym + S;                            // emissions of the step
    int* cur = ecount + S;                            // current h copy of the slot's stream
    int* act = cur + S;                               // [2][S] active lists
    int* dec = act + 2 * S;                           // decided class per active index
    int* eb = dec + S;                                // emitting slots, in active order
    int* ek = eb + S;                                 // their classes
    int* eh = ek + S;                                 // their h copy before the step
    const Ring R{rbuf, ring_full, d.RB, K};
    // every CTA reads the same rows (all active slots, all emitting slots): CTA
    // g starts its pass at row g m / G, so that the CTAs do not all request the
    // same lines of L2 at the same moment
    auto rot = [&](int i, int m) {
        const int j = i + (int)(((long long)g * m) / G);
        return j >= m ? j - m : j;
    };
    uint32_t par = 0;
    unsigned gt = 0;  // grid-barrier target
    const long long tsym = (long long)d.T * d.max_sym;

    // ---- weights of this CTA's slices into shared memory (TMA bulk copies)
    if (tid == 0) {
        mbar_init(&wbar, 1);
        for (int s = 0; s < d.RB; ++s) mbar_init(&ring_full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_expect_tx(&wbar, (uint32_t)(nc * J + 4 * nu * P + no * P) * 4u);
        for (int i = 0; i < nc; ++i) bulk_g2s(Wo + (size_t)i * J, d.wout + (size_t)(c_lo + i) * J, J * 4, &wbar);
        for (int q = 0; q < 4; ++q)
            for (int i = 0; i < nu; ++i)
                bulk_g2s(Wh + (size_t)(q * nu + i) * P, d.whh + ((size_t)q * P + u_lo + i) * P, P * 4, &wbar);
        for (int i = 0; i < no; ++i) bulk_g2s(Wp + (size_t)i * P, d.wpp + (size_t)(o_lo + i) * P, P * 4, &wbar);
    }
    for (int i = tid; i < nc; i += DT) bo_s[i] = __ldg(d.bout + c_lo + i);
    for (int i = tid; i < no; i += DT) bp_s[i] = __ldg(d.bpp + o_lo + i);
    // ---- replicated slot state; keys of both parities start at zero
    for (int b = tid; b < n; b += DT) {
        frame[b] = 0;
        sym[b] = 0;
        ecount[b] = 0;
        cur[b] = __ldcg(d.hsel + d.ids[b]);
        act[b] = b;
    }
    for (int b = g * DT + tid; b < 2 * n; b += G * DT) d.keys[(b >= n) * S + b % n] = 0ull;
    __syncthreads();
    // streams after a reset start from h = c = 0 with one predictor step on the
    // blank token: listed like emissions (slot order, every CTA alike)
    if (warp == 0) {
        int m = 0;
        for (int base = 0; base < n; base += 32) {
            const int b = base + lane;
            const bool pr = b < n && __ldcg(d.primed + d.ids[b]) == 0;
            const unsigned mk = __ballot_sync(0xffffffffu, pr);
            if (pr) {
                const int q = m + __popc(mk & ((1u << lane) - 1u));
                eb[q] = b;
                ek[q] = d.blank;
                eh[q] = cur[b];
                cur[b] ^= 1;
            }
            m += __popc(mk);
        }
        if (lane == 0) s_cnt[0] = m;
    }
    const bool wok = __syncthreads_and(mbar_wait(&wbar, 0));
    if (!wok) {
        if (tid == 0) fail_abort(d);
        return;
    }
    int ne = s_cnt[0];
    // priming LSTM step of this CTA's units: W_hh h = 0 and c = 0, so the gates are the blank's table row
    for (int x = tid; x < ne * nu; x += DT) {
        const int e = x / nu, j = u_lo + x % nu, id = d.ids[eb[e]];
        const float* tb = d.tab + (size_t)d.blank * 4 * P;
        const float gi = __ldg(tb + j), gg = __ldg(tb + 2 * P + j), go = __ldg(tb + 3 * P + j);
        const float c2 = sigm(gi) * tanhf(gg);  // the forget gate multiplies c = 0
        __stcg(d.c + (size_t)id * P + j, c2);
        __stcg(d.h + ((size_t)(eh[e] ^ 1) * S + id) * P + j, sigm(go) * tanhf(c2));
    }

    // ---- D: projection of the emitting slots (their new h), then the joint
    // inputs of the listed slots; shared by the priming and every iteration
    auto phase_d = [&](int ne_, const int* L, int m) -> bool {
        if (ne_ > 0 && no > 0) {
            const bool ok = ring_pass<2>(
                R, par, ne_, P,
                [&](int e) {
                    const int q = rot(e, ne_);
                    return d.h + ((size_t)(eh[q] ^ 1) * S + d.ids[eb[q]]) * P;
                },
                [&](const float* const (&rows)[2], const int (&idx)[2]) {
                    float acc[2][8];
                    group_dots<2, 8>(rows, Wp, P, no, P, acc);
                    // lane 8 r + o (< 16): output o_lo + o of row r
                    const float v = transpose_sum16(reinterpret_cast<float (&)[16]>(acc));
                    const int r = (lane >> 3) & 1, o = lane & 7;
                    if (lane < 16 && o < no && idx[r] >= 0)
                        __stcg(d.p + (size_t)d.ids[eb[rot(idx[r], ne_)]] * J + o_lo + o, v + bp_s[o]);
                });
            if (!__syncthreads_and(ok)) return false;  // also orders the p stores before the reads below
        }
        for (int x = tid; x < m * no; x += DT) {
            const int b = L[x / no], j = o_lo + x % no;
            const float zz = __ldg(d.z + b * d.zb + (long long)frame[b] * J + j);
            const float pp = __ldcg(d.p + (size_t)d.ids[b] * J + j);
            __stcg(d.u + (size_t)b * J + j, fmaxf(zz + pp, 0.f));
        }
        return true;
    };

    int na = d.T > 0 ? n : 0;
    if (ne > 0 && !grid_sync(d, gt)) return;
    if (!phase_d(ne, act, na)) {
        if (tid == 0) fail_abort(d);
        return;
    }
    if (!grid_sync(d, gt)) return;

    int cb = 0;
    for (int it = 0; it < d.maxit && na > 0; ++it) {
        const int* A = act + cb * S;
        int* N = act + (cb ^ 1) * S;
        unsigned long long* keys = d.keys + (size_t)(it & 1) * S;
        // ---- A: logits of this CTA's classes for every active slot, argmax key
        bool ok = true;
        if (nc > 0)
            ok = ring_pass_pairs(
                R, par, na, J, [&](int i) { return d.u + (size_t)A[rot(i, na)] * J; },
                [&](const float* const (&rows)[2], const int (&idx)[2]) {
                    // lane 8 r + v (and 8 r + v + 16): class c0 + v of row r; the
                    // running best of row r (largest logit, lowest class on ties)
                    // ends in lane 8 r.  Groups of two rows keep two groups of rows
                    // in flight in each warp's ring slots while one is computed.
                    const int r = (lane >> 3) & 1, v = lane & 7;
                    float best = -FLT_MAX;
                    int bi = INT_MAX;
                    for (int c0 = 0; c0 < nc; c0 += 8) {
                        const int nv = min(8, nc - c0);
                        float acc[2][8];
                        group_dots<2, 8>(rows, Wo + (size_t)c0 * J, J, nv, J, acc);
                        float x = transpose_sum16(reinterpret_cast<float (&)[16]>(acc));
                        int k = c0 + v;
                        if (v < nv) x += bo_s[c0 + v];
                        else x = -FLT_MAX, k = INT_MAX;
#pragma unroll
                        for (int o = 4; o >= 1; o >>= 1) {
                            const float ox = __shfl_xor_sync(0xffffffffu, x, o);
                            const int ok_ = __shfl_xor_sync(0xffffffffu, k, o);
                            if (ox > x || (ox == x && ok_ < k)) {
                                x = ox;
                                k = ok_;
                            }
                        }
                        if (x > best || (x == best && k < bi)) {
                            best = x;
                            bi = k;
                        }
                    }
                    if (lane < 16 && v == 0 && idx[r] >= 0)
                        atomicMax(keys + A[rot(idx[r], na)], pack_key(best, c_lo + bi));
                });
        if (!__syncthreads_and(ok)) {
            if (tid == 0) fail_abort(d);
            return;
        }
        if (!grid_sync(d, gt)) return;
        // ---- B: the decisions of every active slot, in every CTA alike.  When
        // the active list fits the ring, the LSTM's h rows of all active slots
        // are requested first (any of them may emit), so that they arrive while
        // the keys are read and the decisions taken.
        const bool pre_h = nu > 0 && na <= d.RB;
        if (pre_h && lane == 0) {
            fence_proxy_async_smem();
            asm volatile("fence.proxy.async.global;" ::: "memory");
            for (int i = warp; i < na; i += NW) {
                const int b = A[i];
                mbar_expect_tx(&R.full[i], (uint32_t)P * 4u);
                bulk_g2s(R.buf + (size_t)i * K, d.h + ((size_t)cur[b] * S + d.ids[b]) * P, (uint32_t)P * 4u,
                         &R.full[i]);
            }
        }
        for (int i = tid; i < na; i += DT) dec[i] = key_class(__ldcg(keys + A[i]));
        // the other parity's keys serve the next iteration (all its readers passed a barrier)
        for (int b = g * DT + tid; b < n; b += G * DT) d.keys[(size_t)((it + 1) & 1) * S + b] = 0ull;
        __syncthreads();
        if (warp == 0) {
            int ne_ = 0, nn = 0;
            for (int base = 0; base < na; base += 32) {
                const int i = base + lane;
                bool em = false, keep = false;
                int b = 0, k = 0;
                if (i < na) {
                    b = A[i];
                    k = dec[i];
                    int f = frame[b], sy = sym[b];
                    bool next = k == d.blank;
                    if (!next) {
                        em = true;
                        if (b % G == g) {
                            d.tokens[b * tsym + ecount[b]] = k;
                            d.frames[b * tsym + ecount[b]] = f;
                        }
                        ++ecount[b];
                        next = ++sy == d.max_sym;
                    }
                    if (next) {
                        ++f;
                        sy = 0;
                    }
                    frame[b] = f;
                    sym[b] = sy;
                    keep = f < d.T;
                }
                const unsigned lt = (1u << lane) - 1u;
                const unsigned me = __ballot_sync(0xffffffffu, em), mk = __ballot_sync(0xffffffffu, keep);
                if (em) {
                    const int q = ne_ + __popc(me & lt);
                    eb[q] = b;
                    ek[q] = k;
                    eh[q] = cur[b];
                    cur[b] ^= 1;
                }
                if (keep) N[nn + __popc(mk & lt)] = b;
                ne_ += __popc(me);
                nn += __popc(mk);
            }
            if (lane == 0) {
                s_cnt[0] = ne_;
                s_cnt[1] = nn;
            }
        }
        __syncthreads();
        ne = s_cnt[0];
        const int nn = s_cnt[1];
        // ---- C: LSTM step of this CTA's units for the emitting slots.  A group
        // of up to two rows: row r is stream id[r], class k[r], h copy hc[r] (its
        // new h goes to the other copy), live when id[r] >= 0.
        auto lstm_group = [&](const float* const (&rows)[2], const int (&idv)[2], const int (&kv)[2],
                              const int (&hcv)[2]) {
            // lane uu < nu: its unit's table entries and cell state, loaded ahead of the dot products
            float t4[2][4], cold[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                t4[r][0] = t4[r][1] = t4[r][2] = t4[r][3] = cold[r] = 0.f;
                if (lane < nu && idv[r] >= 0) {
                    const float* tb = d.tab + (size_t)kv[r] * 4 * P + u_lo + lane;
                    t4[r][0] = __ldg(tb);
                    t4[r][1] = __ldg(tb + P);
                    t4[r][2] = __ldg(tb + 2 * P);
                    t4[r][3] = __ldg(tb + 3 * P);
                    cold[r] = __ldcg(d.c + (size_t)idv[r] * P + u_lo + lane);
                }
            }
            float acc[2][32];
            group_dots<2, 32>(rows, Wh, P, 4 * nu, P, acc);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                // lane q nu + uu: gate q of unit uu; gather a unit's 4 gates in lane uu
                const float gsum = transpose_sum32(acc[r]);
                float gm[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) gm[q] = __shfl_sync(0xffffffffu, gsum, min(q * nu + lane, 31));
                if (lane < nu && idv[r] >= 0) {
                    const int id = idv[r], j = u_lo + lane;
                    const float gi = gm[0] + t4[r][0], gf = gm[1] + t4[r][1];
                    const float gg = gm[2] + t4[r][2], go = gm[3] + t4[r][3];
                    const float c2 = sigm(gf) * cold[r] + sigm(gi) * tanhf(gg);
                    __stcg(d.c + (size_t)id * P + j, c2);
                    __stcg(d.h + ((size_t)(hcv[r] ^ 1) * S + id) * P + j, sigm(go) * tanhf(c2));
                }
            }
        };
        ok = true;
        if (pre_h) {
            // the active slots' h rows were requested before the decisions (row i
            // of the active list in ring slot i): wait for every one, so that no
            // copy is left in flight, and step the emitting slots
            for (int i = warp; i < na; i += NW) {
                const int j = i / NW;
                if (!mbar_wait(&R.full[i], (par >> j) & 1u)) {
                    ok = false;
                    break;
                }
                par ^= 1u << j;
                if (dec[i] != d.blank) {
                    const int b = A[i];
                    const float* rows[2] = {R.buf + (size_t)i * K, R.buf + (size_t)i * K};
                    const int idv[2] = {d.ids[b], -1}, kv[2] = {dec[i], 0}, hcv[2] = {cur[b] ^ 1, 0};
                    lstm_group(rows, idv, kv, hcv);
                }
                __syncwarp();
            }
        } else if (ne > 0 && nu > 0) {
            ok = ring_pass<2>(
                R, par, ne, P,
                [&](int e) {
                    const int q = rot(e, ne);
                    return d.h + ((size_t)eh[q] * S + d.ids[eb[q]]) * P;
                },
                [&](const float* const (&rows)[2], const int (&idx)[2]) {
                    int idv[2], kv[2], hcv[2];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int q = idx[r] >= 0 ? rot(idx[r], ne) : 0;
                        idv[r] = idx[r] >= 0 ? d.ids[eb[q]] : -1;
                        kv[r] = idx[r] >= 0 ? ek[q] : 0;
                        hcv[r] = idx[r] >= 0 ? eh[q] : 0;
                    }
                    lstm_group(rows, idv, kv, hcv);
                });
        }
        if (!__syncthreads_and(ok)) {
            if (tid == 0) fail_abort(d);
            return;
        }
        if (ne > 0 && !grid_sync(d, gt)) return;
        // ---- D
        if (!phase_d(ne, N, nn)) {
            if (tid == 0) fail_abort(d);
            return;
        }
        if (!grid_sync(d, gt)) return;
        cb ^= 1;
        na = nn;
    }
    // ---- the owners write the per-slot results back (every CTA read hsel and
    // primed before the first barrier)
    for (int b = g + G * tid; b < n; b += G * DT) {
        d.counts[b] = ecount[b];
        d.hsel[d.ids[b]] = cur[b];
        d.primed[d.ids[b]] = 1;
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
    unsigned gt = 0;
    grid_sync(d, gt);
}

constexpr int ID_SLOTS = 4;
constexpr int MAX_T = 1024;

}  // namespace
}  // namespace cac

using namespace cac;

struct cac_decoder {
    cac_dec_config cfg{};
    int C = 0, S = 0, grid = 0;
    int nc_max = 0, nu_max = 0, no_max = 0, RB = 0;
    size_t smem = 0;
    std::vector<void*> allocs;
    float *tab = nullptr, *whh = nullptr, *wpp = nullptr, *bpp = nullptr, *wout = nullptr, *bout = nullptr;
    float *h = nullptr, *c = nullptr, *p = nullptr;
    int* primed = nullptr;
    // step scratch for up to S slots
    int* ids = nullptr;
    float* u = nullptr;                 // [S][J] joint inputs of the slots
    unsigned long long* keys = nullptr; // [2][S] argmax keys
    int* bar = nullptr;                 // arrivals, generation, abort word
    int* hsel = nullptr;  // [S]
    int* status = nullptr;
    int* pinned = nullptr;  // ID_SLOTS x S host ids
    cudaEvent_t slot_ev[ID_SLOTS] = {};
    int slot = 0;
};

namespace {

int dalloc(cac_decoder* d, size_t bytes, void** out) {
    if (cudaMalloc(out, bytes) != cudaSuccess) return cac::nomem();
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
    if (cfg->pred_dim % 64 || cfg->joint_dim % 64 || cfg->pred_dim > 64 * MAXCH || cfg->joint_dim > 64 * MAXCH)
        return CAC_E_UNSUPPORTED;
    const size_t C = (size_t)cfg->vocab + 2, P = cfg->pred_dim, J = cfg->joint_dim;
    const size_t need = C * P + 2 * 4 * P * P + 2 * 4 * P + J * P + J + C * J + C;
    if (n_floats != need) return CAC_E_INVAL;
    *out = nullptr;
    cac_decoder* d = new cac_decoder();
    d->cfg = *cfg;
    d->C = (int)C;
    d->S = max_streams;
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
        (r = dalloc_t(d, S, &d->primed)) || (r = dalloc_t(d, S, &d->ids)) || (r = dalloc_t(d, S * J, &d->u)) ||
        (r = dalloc_t(d, 2 * S, &d->keys)) || (r = dalloc_t(d, 4, &d->bar)) || (r = dalloc_t(d, 1, &d->status)))
        return fail(r);
    if (cudaMemset(d->primed, 0, S * 4) != cudaSuccess || cudaMemset(d->status, 0, 4) != cudaSuccess ||
        cudaMemset(d->h, 0, 2 * S * P * 4) != cudaSuccess || cudaMemset(d->hsel, 0, S * 4) != cudaSuccess || cudaMemset(d->c, 0, S * P * 4) != cudaSuccess ||
        cudaMemset(d->p, 0, S * J * 4) != cudaSuccess)
        return fail(CAC_E_CUDA);
    if (cudaMallocHost(reinterpret_cast<void**>(&d->pinned), sizeof(int) * S * ID_SLOTS) != cudaSuccess)
        return fail(cac::nomem());
    for (auto& e : d->slot_ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return fail(CAC_E_CUDA);
    // one CTA per SM, all co-resident (cooperative launch).  Shared memory:
    // the CTA's weight slices, the row ring (as many slots as fit, up to
    // RB_MAX, a multiple of the warp count) and the replicated slot state.
    const size_t K = P > J ? P : J;
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return fail(CAC_E_CUDA);
    d->nc_max = (int)((C + sms - 1) / sms);
    d->nu_max = (int)((P + sms - 1) / sms);
    d->no_max = (int)((J + sms - 1) / sms);
    // a CTA's gate rows (4 per unit) fill at most one warp, its projection outputs at most 8 lanes per row
    if (d->nu_max > 8 || d->no_max > 8) return fail(CAC_E_UNSUPPORTED);
    const size_t fixed = sizeof(float) * ((size_t)d->nc_max * J + (size_t)4 * d->nu_max * P + (size_t)d->no_max * P +
                                          bias_floats(d->nc_max, d->no_max)) +
                         sizeof(int) * STATE_INTS * S;
    const size_t budget = 227 * 1024 - 1024;  // less the kernel's static shared memory
    if (fixed + sizeof(float) * K * 4 * NW > budget) return fail(CAC_E_UNSUPPORTED);  // groups of 4 rows per warp
    d->RB = (int)std::min<size_t>(RB_MAX, (budget - fixed) / (sizeof(float) * K) / (2 * NW) * (2 * NW));
    d->smem = fixed + sizeof(float) * K * d->RB;
    if (cudaFuncSetAttribute(dec_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d->smem) !=
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
    if (cudaMemsetAsync(d->bar, 0, sizeof(int) * 4, s) != cudaSuccess) return CAC_E_CUDA;
    DecParams p{};
    p.n = n; p.T = T; p.C = d->C; p.P = d->cfg.pred_dim; p.J = d->cfg.joint_dim; p.max_sym = d->cfg.max_symbols;
    p.blank = d->cfg.vocab; p.maxit = maxit; p.S = d->S;
    p.nc_max = d->nc_max; p.nu_max = d->nu_max; p.no_max = d->no_max; p.RB = d->RB;
    p.ids = d->ids; p.z = z; p.zb = z_bstride; p.tokens = tokens; p.frames = frames; p.counts = counts;
    p.tab = d->tab; p.whh = d->whh; p.wpp = d->wpp; p.bpp = d->bpp; p.wout = d->wout; p.bout = d->bout;
    p.h = d->h; p.c = d->c; p.p = d->p; p.u = d->u; p.keys = d->keys; p.primed = d->primed; p.hsel = d->hsel;
    p.bar = reinterpret_cast<unsigned*>(d->bar);
    p.abort_flag = d->bar + 2;
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
    if (cudaMalloc(&buf, 4 * sizeof(int)) != cudaSuccess) return cac::nomem();
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
