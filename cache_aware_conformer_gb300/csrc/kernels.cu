// Non-GEMM kernels of the cache-aware Conformer step: LayerNorm, mel staging,
// rectangular rel-pos attention, the fused depthwise conv with its cache, and
// per-stream position bookkeeping.
#include <algorithm>
#include <cfloat>

#include "kernels.cuh"

namespace cac {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---------------------------------------------------------------------------
// LayerNorm: one warp per row, VPL = D / 32 values per lane kept in registers
// ---------------------------------------------------------------------------
template <int VPL>
__device__ __forceinline__ void ln_row(float (&v)[VPL], int lane, int D, const float* g, const float* b) {
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < VPL; ++k) s += v[k];
    const float mean = warp_sum(s) / D;
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < VPL; ++k) { const float d = v[k] - mean; q += d * d; }
    const float rstd = rsqrtf(warp_sum(q) / D + 1e-5f);
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
        const int c = lane + 32 * k;
        v[k] = (v[k] - mean) * rstd * __ldg(g + c) + __ldg(b + c);
    }
}

template <int VPL, class TA>
__global__ void __launch_bounds__(256) ln_kernel(const float* x, int M, int D, const float* g1, const float* b1,
                                                 float* y_f32, TA* y_act, const float* g2, const float* b2,
                                                 TA* z_act, int grp, int grp_stride, int row_off) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= M) return;
    float v[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k) v[k] = x[(long long)row * D + lane + 32 * k];
    ln_row<VPL>(v, lane, D, g1, b1);
    if (y_f32) {
        const long long orow = (long long)(row / grp) * grp_stride + (row % grp) + row_off;
#pragma unroll
        for (int k = 0; k < VPL; ++k) y_f32[orow * D + lane + 32 * k] = v[k];
    }
    if (y_act) {
#pragma unroll
        for (int k = 0; k < VPL; ++k) y_act[(long long)row * D + lane + 32 * k] = from_f<TA>(v[k]);
    }
    if (g2) {
        ln_row<VPL>(v, lane, D, g2, b2);
#pragma unroll
        for (int k = 0; k < VPL; ++k) z_act[(long long)row * D + lane + 32 * k] = from_f<TA>(v[k]);
    }
}

template <class TA>
static cudaError_t ln_dispatch(const float* x, int M, int D, const float* g1, const float* b1, float* y_f32,
                               void* y_act, const float* g2, const float* b2, void* z_act, int grp, int grp_stride,
                               int row_off, cudaStream_t s) {
    dim3 grid((M + 7) / 8);
    TA* ya = static_cast<TA*>(y_act);
    TA* za = static_cast<TA*>(z_act);
#define LN_CASE(V)                                                                                       \
    case V:                                                                                              \
        ln_kernel<V, TA><<<grid, 256, 0, s>>>(x, M, D, g1, b1, y_f32, ya, g2, b2, za, grp, grp_stride, row_off); \
        break;
    switch (D / 32) {
        LN_CASE(2) LN_CASE(4) LN_CASE(8) LN_CASE(16) LN_CASE(24) LN_CASE(32)
        default: return cudaErrorInvalidValue;
    }
#undef LN_CASE
    return cudaGetLastError();
}

cudaError_t launch_layernorm(const float* x, int M, int D, const float* g1, const float* b1, float* y_f32,
                             void* y_act, const float* g2, const float* b2, void* z_act, int act_bf16, int grp,
                             int grp_stride, int row_off, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    if (D % 32) return cudaErrorInvalidValue;
    return act_bf16 ? ln_dispatch<bf16>(x, M, D, g1, b1, y_f32, y_act, g2, b2, z_act, grp, grp_stride, row_off, s)
                    : ln_dispatch<float>(x, M, D, g1, b1, y_f32, y_act, g2, b2, z_act, grp, grp_stride, row_off, s);
}

// ---------------------------------------------------------------------------
// mel staging
// ---------------------------------------------------------------------------
constexpr int MEL = 128;
constexpr int TAIL = 14;

template <class T>
__global__ void __launch_bounds__(256) stage_mel_kernel(const float* mel, long long mel_bstride, const int* n_valid,
                                                        T* win, T* tail, const int* ids, const int* pos, int n,
                                                        int* status) {
    const int b = blockIdx.x;
    const int id = ids[b];
    const bool first = pos[id] == 0;
    const int W = TAIL + 8 * n;
    const int nv = n_valid ? n_valid[b] : 8 * n;
    T* w = win + (long long)b * W * MEL;
    T* tl = tail + (long long)id * TAIL * MEL;
    bool bad = false;
    for (int e = threadIdx.x; e < W * MEL; e += blockDim.x) {
        const int r = e / MEL, c = e - (e / MEL) * MEL;
        T v;
        if (r < TAIL) {
            v = first ? from_f<T>(0.f) : tl[r * MEL + c];
        } else {
            const float m = (r - TAIL < nv) ? mel[(long long)b * mel_bstride + (long long)(r - TAIL) * MEL + c] : 0.f;
            bad |= !isfinite(m);
            v = from_f<T>(m);
        }
        w[e] = v;
    }
    if (bad) latch_error(status, CAC_E_NONFINITE);
    __syncthreads();
    for (int e = threadIdx.x; e < TAIL * MEL; e += blockDim.x) tl[e] = w[8 * n * MEL + e];
}

cudaError_t launch_stage_mel(const float* mel, long long mel_bstride, const int* n_valid, void* win, void* tail,
                             const int* ids, const int* pos, int n, int nb, int act_bf16, int* status,
                             cudaStream_t s) {
    if (nb <= 0) return cudaSuccess;
    if (act_bf16)
        stage_mel_kernel<bf16><<<nb, 256, 0, s>>>(mel, mel_bstride, n_valid, static_cast<bf16*>(win),
                                                  static_cast<bf16*>(tail), ids, pos, n, status);
    else
        stage_mel_kernel<float><<<nb, 256, 0, s>>>(mel, mel_bstride, n_valid, static_cast<float*>(win),
                                                   static_cast<float*>(tail), ids, pos, n, status);
    return cudaGetLastError();
}

template <class T>
__global__ void stage_mel_offline_kernel(const float* mel, int t_mel, const int* len, T* dst, int W, int B,
                                         int* status) {
    const long long total = (long long)B * W * MEL;
    bool bad = false;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(e % MEL);
        const long long rr = e / MEL;
        const int b = (int)(rr / W), r = (int)(rr % W) - 2;
        float m = 0.f;
        if (r >= 0 && r < t_mel && r < len[b]) {
            m = mel[((long long)b * t_mel + r) * MEL + c];
            bad |= !isfinite(m);
        }
        dst[e] = from_f<T>(m);
    }
    if (bad) latch_error(status, CAC_E_NONFINITE);
}

cudaError_t launch_stage_mel_offline(const float* mel, int t_mel, const int* len, void* dst, int W, int B,
                                     int act_bf16, int* status, cudaStream_t s) {
    const int blocks = 152 * 8;
    if (act_bf16)
        stage_mel_offline_kernel<bf16><<<blocks, 256, 0, s>>>(mel, t_mel, len, static_cast<bf16*>(dst), W, B, status);
    else
        stage_mel_offline_kernel<float><<<blocks, 256, 0, s>>>(mel, t_mel, len, static_cast<float*>(dst), W, B,
                                                               status);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// rectangular rel-pos attention
//
// One warp owns (query group, head): nq queries at positions pq0 .. pq0+nq-1
// against Nk keys at positions kpos0 .. kpos0+Nk-1.
//   score[i][j] = ((q_i + u) . k_j + (q_i + v) . P[pq_i - pk_j]) * scale,
// masked (chunked-causal on absolute positions, or a window), softmax over j,
// out_i = sum_j prob[i][j] v_j.
// The warp's K and V rows are staged in shared memory by TMA bulk copies
// (cp.async.bulk on one mbarrier) issued before anything else, so the whole
// HBM read of the warp is in flight at once; the block's per-head position
// table is loaded while they land.  Scores: lane per key, 16-byte chunks of
// the key row read in a lane-rotated order (conflict-free shared loads).
// probs @ V: lane per HD/32 output dims, V rows from shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool allowed(const AttnParams& a, int pq, int pk) {
    if (pk < 0) return false;
    if (a.rc > 0) return pk >= pq - a.left && pk <= pq + a.rc;
    const int c = (pq / a.chunk) * a.chunk;
    return pk >= c - a.left && pk <= c + a.chunk - 1;
}

template <int HD, int NQ, int NK, class T>
struct AttnLayout {
    static constexpr int KV = NK * HD;                                   // elements of K (or V)
    static constexpr int WARP_BYTES = 16 + 2 * KV * (int)sizeof(T) + 4 * (2 * NQ * HD + NQ * NK);
    static constexpr int PS = HD + 4;                                    // padded position-table row
};

template <int HD, int NQ, int NK, class T>
__device__ __forceinline__ void attn_carve(uint8_t* wsm, uint64_t*& bar, T*& Ks, T*& Vs, float*& qu, float*& qv,
                                           float*& S) {
    using Lay = AttnLayout<HD, NQ, NK, T>;
    bar = reinterpret_cast<uint64_t*>(wsm);
    Ks = reinterpret_cast<T*>(wsm + 16);
    Vs = Ks + Lay::KV;
    qu = reinterpret_cast<float*>(Vs + Lay::KV);
    qv = qu + NQ * HD;
    S = qv + NQ * HD;
}

// Block prologue shared by the attention kernels: thread 0 arms the block
// barrier and bulk-copies this head's padded position table [NR][HD + 4].
template <int HD>
__device__ __forceinline__ void stage_ptable(const AttnParams& a, int h, float* Ps, uint64_t* pbar) {
    if (threadIdx.x == 0) {
        const uint32_t bytes = (uint32_t)a.NR * (HD + 4) * 4;
        mbar_init(pbar, 1);
        fence_mbar_init();
        mbar_expect_tx(pbar, bytes);
        bulk_g2s(Ps, a.P + (long long)h * a.NR * (HD + 4), bytes, pbar);
    }
}

template <class T, int EPC>
__device__ __forceinline__ void chunk_to_f(const T* src, float (&f)[EPC]);
template <>
__device__ __forceinline__ void chunk_to_f<bf16, 8>(const bf16* src, float (&f)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(src);
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 t = __bfloat1622float2(p[k]);
        f[2 * k] = t.x;
        f[2 * k + 1] = t.y;
    }
}
template <>
__device__ __forceinline__ void chunk_to_f<float, 4>(const float* src, float (&f)[4]) {
    const float4 u = *reinterpret_cast<const float4*>(src);
    f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w;
}

// Everything after the K/V copies were issued on `bar`.
template <int HD, int NQ, int NK, class T>
__device__ void attend_warp(const AttnParams& a, int h, const float* Ps, uint64_t* pbar, uint8_t* wsm, int lane,
                            const float* qsrc, int pq0, int nq, int kpos0, int Nk, T* dst, int* status) {
    using Lay = AttnLayout<HD, NQ, NK, T>;
    constexpr int PS = Lay::PS;
    constexpr int DPL = HD >= 32 ? HD / 32 : 1;
    constexpr int EPC = 16 / (int)sizeof(T);  // elements per 16-byte chunk
    constexpr int CPR = HD / EPC;             // chunks per row
    uint64_t* bar;
    T *Ks, *Vs;
    float *qu, *qv, *S;
    attn_carve<HD, NQ, NK, T>(wsm, bar, Ks, Vs, qu, qv, S);
    for (int e = lane; e < nq * HD; e += 32) {
        const int i = e / HD, d = e - (e / HD) * HD;
        const float qq = qsrc[(long long)i * a.ldq + d];
        qu[i * HD + d] = qq + __ldg(a.pbu + h * HD + d);
        qv[i * HD + d] = qq + __ldg(a.pbv + h * HD + d);
    }
    const bool landed = mbar_wait(bar, 0) && mbar_wait(pbar, 0);
    __syncwarp();
    if (!landed) {
        if (lane == 0) latch_error(status, CAC_E_TIMEOUT);
        return;
    }
    // scores
    for (int j0 = 0; j0 < Nk; j0 += 32) {
        const int j = j0 + lane;
        const bool valid = j < Nk;
        const int pk = kpos0 + j;
        float acc[NQ];
        bool ok[NQ];
        int prow[NQ];
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            acc[i] = 0.f;
            ok[i] = i < nq && valid && allowed(a, pq0 + i, pk);
            prow[i] = ok[i] ? (pq0 + i - pk - a.rmin) * PS : 0;
        }
        if (valid) {
            const T* krow = Ks + j * HD;
#pragma unroll 1
            for (int c = 0; c < CPR; ++c) {
                const int cc = (c + lane) & (CPR - 1);
                float kf[EPC];
                chunk_to_f<T, EPC>(krow + cc * EPC, kf);
#pragma unroll
                for (int i = 0; i < NQ; ++i) {
                    if (!ok[i]) continue;
                    const float* qa = qu + i * HD + cc * EPC;
                    const float* qb = qv + i * HD + cc * EPC;
                    const float* pr = Ps + prow[i] + cc * EPC;
#pragma unroll
                    for (int e = 0; e < EPC; e += 4) {
                        const float4 ua = *reinterpret_cast<const float4*>(qa + e);
                        const float4 va = *reinterpret_cast<const float4*>(qb + e);
                        const float4 p4 = *reinterpret_cast<const float4*>(pr + e);
                        acc[i] += ua.x * kf[e] + ua.y * kf[e + 1] + ua.z * kf[e + 2] + ua.w * kf[e + 3];
                        acc[i] += va.x * p4.x + va.y * p4.y + va.z * p4.z + va.w * p4.w;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < NQ; ++i)
                if (i < nq) S[i * NK + j] = ok[i] ? acc[i] * a.scale : -FLT_MAX;
        }
    }
    __syncwarp();
    // softmax over the keys of each query
#pragma unroll 1
    for (int i = 0; i < nq; ++i) {
        float m = -FLT_MAX;
        for (int j = lane; j < Nk; j += 32) m = fmaxf(m, S[i * NK + j]);
        m = warp_max(m);
        float sum = 0.f;
        for (int j = lane; j < Nk; j += 32) {
            const float s = S[i * NK + j];
            const float e = (s == -FLT_MAX) ? 0.f : __expf(s - m);
            S[i * NK + j] = e;
            sum += e;
        }
        sum = warp_sum(sum);
        const float inv = 1.f / sum;
        for (int j = lane; j < Nk; j += 32) S[i * NK + j] *= inv;
    }
    __syncwarp();
    // probs @ V
    float acc[NQ][DPL];
#pragma unroll
    for (int i = 0; i < NQ; ++i)
#pragma unroll
        for (int t = 0; t < DPL; ++t) acc[i][t] = 0.f;
    const int d0 = lane * DPL;
    const bool dl = d0 < HD;
#pragma unroll 4
    for (int j = 0; j < Nk; ++j) {
        float vv[DPL];
#pragma unroll
        for (int t = 0; t < DPL; ++t) vv[t] = dl ? to_f(Vs[j * HD + d0 + t]) : 0.f;
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            if (i >= nq) break;
            const float pij = S[i * NK + j];
#pragma unroll
            for (int t = 0; t < DPL; ++t) acc[i][t] = fmaf(pij, vv[t], acc[i][t]);
        }
    }
    if (dl) {
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            if (i >= nq) break;
#pragma unroll
            for (int t = 0; t < DPL; ++t) dst[(long long)i * a.ldo + d0 + t] = from_f<T>(acc[i][t]);
        }
    }
}

constexpr int ATT_WARPS = 4;

// streaming: block = (ATT_WARPS batch slots, head); keys = [cache | new] from the ring,
// whose rows for one stream and head are contiguous modulo R: at most two copies each.
template <int HD, int NQ, int NK, class T>
__global__ void __launch_bounds__(ATT_WARPS * 32) attn_stream_kernel(AttnParams a, int* status) {
    using Lay = AttnLayout<HD, NQ, NK, T>;
    extern __shared__ float4 sm4[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(sm4);
    const int h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * ATT_WARPS + warp;
    const bool live = b < a.nb;
    uint64_t* pbar = reinterpret_cast<uint64_t*>(sm);
    float* Ps = reinterpret_cast<float*>(sm + 16);
    uint8_t* wsm = sm + 16 + ((a.NR * Lay::PS * 4 + 15) & ~15) + warp * Lay::WARP_BYTES;
    stage_ptable<HD>(a, h, Ps, pbar);
    int id = 0, p0 = 0, Lc = 0, Nk = 0;
    if (live) {
        id = a.ids[b];
        p0 = a.pos[id];
        Lc = min(p0, a.left);
        Nk = min(Lc + a.nq, NK);
        if (lane == 0) {
            uint64_t* bar;
            T *Ks, *Vs;
            float *qu, *qv, *S;
            attn_carve<HD, NQ, NK, T>(wsm, bar, Ks, Vs, qu, qv, S);
            mbar_init(bar, 1);
            fence_mbar_init();
            constexpr uint32_t ROW = HD * sizeof(T);
            mbar_expect_tx(bar, 2u * ROW * Nk);
            const long long base = (long long)id * a.sstride + (long long)h * a.R * HD;
            const T* kb = static_cast<const T*>(a.k) + base;
            const T* vb = static_cast<const T*>(a.v) + base;
            const int s0 = (p0 - Lc) % a.R;
            const int n1 = min(Nk, a.R - s0);
            bulk_g2s(Ks, kb + (long long)s0 * HD, ROW * n1, bar);
            bulk_g2s(Vs, vb + (long long)s0 * HD, ROW * n1, bar);
            if (Nk > n1) {
                bulk_g2s(Ks + n1 * HD, kb, ROW * (Nk - n1), bar);
                bulk_g2s(Vs + n1 * HD, vb, ROW * (Nk - n1), bar);
            }
        }
    }
    __syncthreads();
    if (!live) return;
    attend_warp<HD, NQ, NK, T>(a, h, Ps, pbar, wsm, lane, a.q + (long long)b * a.nq * a.ldq + h * HD, p0, a.nq, p0 - Lc,
                               Nk, static_cast<T*>(a.out) + (long long)b * a.nq * a.ldo + h * HD, status);
}

// offline: block = (ATT_WARPS query groups of one sequence, head); keys from dense K/V
// rows (one bulk copy per row, issued by the lanes of the warp).
template <int HD, int NQ, int NK, class T>
__global__ void __launch_bounds__(ATT_WARPS * 32) attn_offline_kernel(AttnParams a, int qgroup, int* status) {
    using Lay = AttnLayout<HD, NQ, NK, T>;
    extern __shared__ float4 sm4[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(sm4);
    const int h = blockIdx.y, seq = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int len = a.seq_len[seq];
    const int pq0 = (blockIdx.x * ATT_WARPS + warp) * qgroup;
    const bool live = pq0 < len;
    uint64_t* pbar = reinterpret_cast<uint64_t*>(sm);
    float* Ps = reinterpret_cast<float*>(sm + 16);
    uint8_t* wsm = sm + 16 + ((a.NR * Lay::PS * 4 + 15) & ~15) + warp * Lay::WARP_BYTES;
    stage_ptable<HD>(a, h, Ps, pbar);
    int nq = 0, klo = 0, Nk = 0;
    const long long rb = (long long)seq * a.T;
    if (live) {
        nq = min(qgroup, len - pq0);
        const int pql = pq0 + nq - 1;
        int khi;
        if (a.rc > 0) {
            klo = max(pq0 - a.left, 0);
            khi = min(pql + a.rc, len - 1);
        } else {
            klo = max((pq0 / a.chunk) * a.chunk - a.left, 0);
            khi = min((pql / a.chunk) * a.chunk + a.chunk - 1, len - 1);
        }
        Nk = min(khi - klo + 1, NK);
        uint64_t* bar;
        T *Ks, *Vs;
        float *qu, *qv, *S;
        attn_carve<HD, NQ, NK, T>(wsm, bar, Ks, Vs, qu, qv, S);
        constexpr uint32_t ROW = HD * sizeof(T);
        if (lane == 0) {
            mbar_init(bar, 1);
            fence_mbar_init();
            mbar_expect_tx(bar, 2u * ROW * Nk);
        }
        __syncwarp();
        const T* kb = static_cast<const T*>(a.k) + rb * a.ldk + h * HD;
        const T* vb = static_cast<const T*>(a.v) + rb * a.ldk + h * HD;
        for (int j = lane; j < Nk; j += 32) {
            bulk_g2s(Ks + j * HD, kb + (long long)(klo + j) * a.ldk, ROW, bar);
            bulk_g2s(Vs + j * HD, vb + (long long)(klo + j) * a.ldk, ROW, bar);
        }
    }
    __syncthreads();
    if (!live) return;
    attend_warp<HD, NQ, NK, T>(a, h, Ps, pbar, wsm, lane, a.q + (rb + pq0) * a.ldq + h * HD, pq0, nq, klo, Nk,
                               static_cast<T*>(a.out) + (rb + pq0) * a.ldo + h * HD, status);
}

template <int HD, int NQ, int NK, class T>
static size_t attn_smem(const AttnParams& a) {
    using Lay = AttnLayout<HD, NQ, NK, T>;
    return 16 + ((size_t)a.NR * Lay::PS * 4 + 15) / 16 * 16 + (size_t)ATT_WARPS * Lay::WARP_BYTES;
}

template <class K>
static cudaError_t raise_smem(K kern, size_t smem, size_t& attr) {
    if (smem <= attr) return cudaSuccess;
    constexpr size_t kMax = 227 * 1024;  // per-block dynamic shared memory limit of sm_10x
    if (smem > kMax) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMax);
    if (e == cudaSuccess) attr = kMax;
    return e;
}

template <int HD, int NQ, int NK, class T>
static cudaError_t attn_stream_launch(const AttnParams& a, int* status, cudaStream_t s) {
    const size_t smem = attn_smem<HD, NQ, NK, T>(a);
    auto kern = attn_stream_kernel<HD, NQ, NK, T>;
    static size_t attr = 48 * 1024;  // dynamic shared memory limit set so far for this instantiation
    cudaError_t e = raise_smem(kern, smem, attr);
    if (e != cudaSuccess) return e;
    dim3 grid((a.nb + ATT_WARPS - 1) / ATT_WARPS, a.H);
    kern<<<grid, ATT_WARPS * 32, smem, s>>>(a, status);
    return cudaGetLastError();
}

template <int HD, int NQ, int NK, class T>
static cudaError_t attn_offline_launch(const AttnParams& a, int qgroup, int* status, cudaStream_t s) {
    const size_t smem = attn_smem<HD, NQ, NK, T>(a);
    auto kern = attn_offline_kernel<HD, NQ, NK, T>;
    static size_t attr = 48 * 1024;
    cudaError_t e = raise_smem(kern, smem, attr);
    if (e != cudaSuccess) return e;
    const int groups = (a.T + qgroup - 1) / qgroup;
    dim3 grid((groups + ATT_WARPS - 1) / ATT_WARPS, a.H, a.nb);
    kern<<<grid, ATT_WARPS * 32, smem, s>>>(a, qgroup, status);
    return cudaGetLastError();
}

#define ATT_DISPATCH(LAUNCH, NQ, NK, ...)                                                                  \
    do {                                                                                                   \
        if (a.HD == 64)                                                                                    \
            return act_bf16 ? LAUNCH<64, NQ, NK, bf16>(__VA_ARGS__) : LAUNCH<64, NQ, NK, float>(__VA_ARGS__); \
        if (a.HD == 16)                                                                                    \
            return act_bf16 ? LAUNCH<16, NQ, NK, bf16>(__VA_ARGS__) : LAUNCH<16, NQ, NK, float>(__VA_ARGS__); \
    } while (0)

// NQ x NK instantiations: 160 ms pushes (2 queries, keys <= left + 2), chunked
// pushes of up to 8 frames (keys <= left + 8), provisional passes (up to 24
// queries, keys <= left + 24); offline groups of up to 8 queries.
cudaError_t launch_attention_stream(const AttnParams& a, int act_bf16, int* status, cudaStream_t s) {
    if (a.nb <= 0) return cudaSuccess;
    const int nk_need = a.left + a.nq;
    if (a.nq <= 2 && nk_need <= 80) ATT_DISPATCH(attn_stream_launch, 2, 80, a, status, s);
    if (a.nq <= 8 && nk_need <= 80) ATT_DISPATCH(attn_stream_launch, 8, 80, a, status, s);
    if (a.nq <= 24 && nk_need <= 96) ATT_DISPATCH(attn_stream_launch, 24, 96, a, status, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attention_offline(const AttnParams& a, int act_bf16, int* status, cudaStream_t s) {
    if (a.nb <= 0) return cudaSuccess;
    // queries per warp: one chunk of the chunked mask, or 8 consecutive frames of a window mask
    const int qgroup = a.rc > 0 ? 8 : a.chunk;
    const int nk_need = a.rc > 0 ? a.left + qgroup + a.rc : a.left + a.chunk;
    if (qgroup > 8 || nk_need > 96) return cudaErrorInvalidValue;
    if (qgroup <= 2 && nk_need <= 80) ATT_DISPATCH(attn_offline_launch, 2, 80, a, qgroup, status, s);
    ATT_DISPATCH(attn_offline_launch, 8, 96, a, qgroup, status, s);
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// causal depthwise conv (k = 9) over [conv cache | glu_new] + affine + SiLU
// one thread per (batch slot, channel); the 8-slot cache ring is indexed by
// absolute position mod 8 and reads as zero before the stream start.
// ---------------------------------------------------------------------------
template <class T>
__global__ void __launch_bounds__(256) dwconv_kernel(const T* glu, T* cache, long long cs_stride, const int* ids,
                                                     const int* pos, int nq, int n_commit, const float* wT,
                                                     const float* bdw, const float* bng, const float* bnb, T* out,
                                                     int D, int nb) {
    const long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (idx >= (long long)nb * D) return;
    const int b = (int)(idx / D), c = (int)(idx % D);
    float w[9];
#pragma unroll
    for (int k = 0; k < 9; ++k) w[k] = __ldg(wT + k * D + c);
    const float bias = __ldg(bdw + c), gam = __ldg(bng + c), bet = __ldg(bnb + c);
    float win[9];
    int p0 = 0;
    T* cs = nullptr;
    if (cache) {
        const int id = ids[b];
        p0 = pos[id];
        cs = cache + (long long)id * cs_stride;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int p = p0 - 8 + k;
            win[k] = p >= 0 ? to_f(cs[(long long)(p & 7) * D + c]) : 0.f;
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) win[k] = 0.f;
    }
    const T* g = glu + (long long)b * nq * D + c;
    T* o = out + (long long)b * nq * D + c;
    for (int t = 0; t < nq; ++t) {
        win[8] = to_f(g[(long long)t * D]);
        float acc = bias;
#pragma unroll
        for (int k = 0; k < 9; ++k) acc = fmaf(w[k], win[k], acc);
        o[(long long)t * D] = from_f<T>(siluf_(gam * acc + bet));
#pragma unroll
        for (int k = 0; k < 8; ++k) win[k] = win[k + 1];
    }
    if (cs) {
        for (int t = max(0, n_commit - 8); t < n_commit; ++t) cs[(long long)((p0 + t) & 7) * D + c] = g[(long long)t * D];
    }
}

cudaError_t launch_dwconv(const void* glu, void* cache, long long cs_stride, const int* ids, const int* pos, int nq,
                          int n_commit, const float* wT, const float* bdw, const float* bng, const float* bnb,
                          void* out, int D, int nb, int act_bf16, cudaStream_t s) {
    if (nb <= 0) return cudaSuccess;
    const long long threads = (long long)nb * D;
    const int blocks = (int)((threads + 255) / 256);
    if (act_bf16)
        dwconv_kernel<bf16><<<blocks, 256, 0, s>>>(static_cast<const bf16*>(glu), static_cast<bf16*>(cache), cs_stride,
                                                   ids, pos, nq, n_commit, wT, bdw, bng, bnb, static_cast<bf16*>(out),
                                                   D, nb);
    else
        dwconv_kernel<float><<<blocks, 256, 0, s>>>(static_cast<const float*>(glu), static_cast<float*>(cache),
                                                    cs_stride, ids, pos, nq, n_commit, wT, bdw, bng, bnb,
                                                    static_cast<float*>(out), D, nb);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// bookkeeping and small utilities
// ---------------------------------------------------------------------------
__global__ void advance_kernel(int* pos, const int* ids, int nb, int n) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < nb) pos[ids[b]] += n;
}
__global__ void set_pos_kernel(int* pos, const int* ids, int nb, int value) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < nb) pos[ids[b]] = value;
}

cudaError_t launch_advance(int* pos, const int* ids, int nb, int n, cudaStream_t s) {
    if (nb <= 0) return cudaSuccess;
    advance_kernel<<<(nb + 255) / 256, 256, 0, s>>>(pos, ids, nb, n);
    return cudaGetLastError();
}
cudaError_t launch_set_pos(int* pos, const int* ids, int nb, int value, cudaStream_t s) {
    if (nb <= 0) return cudaSuccess;
    set_pos_kernel<<<(nb + 255) / 256, 256, 0, s>>>(pos, ids, nb, value);
    return cudaGetLastError();
}

__global__ void sinusoid_kernel(float* pe, int NR, int rmin, int D) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= NR * (D / 2)) return;
    const int row = idx / (D / 2), m = idx % (D / 2);
    const double w = pow(10000.0, -2.0 * m / D);
    const double ang = (double)(rmin + row) * w;
    pe[(long long)row * D + 2 * m] = (float)sin(ang);
    pe[(long long)row * D + 2 * m + 1] = (float)cos(ang);
}

cudaError_t launch_sinusoid(float* pe, int NR, int rmin, int D, cudaStream_t s) {
    const int n = NR * (D / 2);
    sinusoid_kernel<<<(n + 255) / 256, 256, 0, s>>>(pe, NR, rmin, D);
    return cudaGetLastError();
}

template <class T>
__global__ void to_f32_kernel(const T* src, float* dst, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        dst[i] = to_f(src[i]);
}

cudaError_t launch_to_f32(const void* src, float* dst, long long n, int src_bf16, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int blocks = (int)std::min<long long>((n + 255) / 256, 152 * 16);
    if (src_bf16)
        to_f32_kernel<bf16><<<blocks, 256, 0, s>>>(static_cast<const bf16*>(src), dst, n);
    else
        to_f32_kernel<float><<<blocks, 256, 0, s>>>(static_cast<const float*>(src), dst, n);
    return cudaGetLastError();
}

}  // namespace cac
