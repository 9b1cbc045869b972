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
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= M) return;
    float v[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k) v[k] = x[(long long)row * D + lane + 32 * k];
    pdl_trigger();
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
        return launch_k(ln_kernel<V, TA>, grid, dim3(256), 0, s, 1, x, M, D, g1, b1, y_f32, ya, g2, b2, za, grp,   \
                        grp_stride, row_off);
    switch (D / 32) {
        LN_CASE(2) LN_CASE(4) LN_CASE(8) LN_CASE(16) LN_CASE(24) LN_CASE(32)
        default: return cudaErrorInvalidValue;
    }
#undef LN_CASE
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
    pdl_trigger();
    pdl_wait();
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
        return launch_k(stage_mel_kernel<bf16>, dim3(nb), dim3(256), 0, s, 1, mel, mel_bstride, n_valid,
                        static_cast<bf16*>(win), static_cast<bf16*>(tail), ids, pos, n, status);
    return launch_k(stage_mel_kernel<float>, dim3(nb), dim3(256), 0, s, 1, mel, mel_bstride, n_valid,
                    static_cast<float*>(win), static_cast<float*>(tail), ids, pos, n, status);
}

template <class T>
__global__ void stage_mel_offline_kernel(const float* mel, int t_mel, const int* len, T* dst, int W, int B,
                                         int* status) {
    pdl_trigger();
    pdl_wait();
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
        return launch_k(stage_mel_offline_kernel<bf16>, dim3(blocks), dim3(256), 0, s, 1, mel, t_mel, len,
                        static_cast<bf16*>(dst), W, B, status);
    return launch_k(stage_mel_offline_kernel<float>, dim3(blocks), dim3(256), 0, s, 1, mel, t_mel, len,
                    static_cast<float*>(dst), W, B, status);
}

// ---------------------------------------------------------------------------
// rectangular rel-pos attention
//
// Work unit: (query group, head) — the n new frames of one stream (or one
// chunk of an offline sequence) against their Nk keys at positions
// kpos0 .. kpos0+Nk-1:
//   score[i][j] = ((q_i + u) . k_j + (q_i + v) . P[pq_i - pk_j]) * scale,
// masked (chunked-causal on absolute positions, or a window), softmax over j,
// out_i = sum_j prob[i][j] v_j.
//
// A block serves SPB units of one head with WPS warps each (the queries of a
// unit are dealt round-robin to its warps).  Per unit, one lane issues TMA
// bulk copies of all K and V rows into shared memory on one mbarrier (the ring
// span of a stream is at most two contiguous pieces); thread 0 bulk-copies the
// head's padded position table on a block barrier.  Inside a warp, LPK =
// HD / 8 lanes share a key: each lane holds 8 dims of (q + u) and (q + v) in
// registers, reads the matching 8 dims of k_j and of P[rel] from shared
// memory, and the partial dots are combined with log2(LPK) shuffles.  probs @ V
// uses the same lane layout over the keys, then reduces across key groups.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool allowed(const AttnParams& a, int pq, int pk) {
    if (pk < 0) return false;
    if (a.rc > 0) return pk >= pq - a.left && pk <= pq + a.rc;
    const int c = (pq / a.chunk) * a.chunk;
    return pk >= c - a.left && pk <= c + a.chunk - 1;
}

template <int HD, int NQW, int WPS, int SPB, int NK, class T>
struct Attn {
    static constexpr int NQ = NQW * WPS;              // queries per unit
    static constexpr int THREADS = SPB * WPS * 32;
    static constexpr int PS = HD + 4;                 // padded position-table row (floats)
    static constexpr int LPK = HD / 8;                // lanes per key
    static constexpr int KPS = 32 / LPK;              // keys per warp step
    static constexpr int KV = NK * HD;                // elements of K (or V) per unit
    static constexpr int UNIT_BYTES = 16 + 2 * KV * (int)sizeof(T) + 4 * NQ * NK;
    static size_t smem(int NR) { return 16 + ((size_t)NR * PS * 4 + 15) / 16 * 16 + (size_t)SPB * UNIT_BYTES; }
};

// 4 consecutive elements -> float
__device__ __forceinline__ void ld4f(const bf16* p, float* f) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}
__device__ __forceinline__ void ld4f(const float* p, float* f) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w;
}
__device__ __forceinline__ void st4(bf16* p, const float* f) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(f[2], f[3]);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t*>(&a);
    u.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ void st4(float* p, const float* f) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
}

// The 8 dims of a row that lane c (of LPK) owns: [c*4, c*4+4) and [HD/2 + c*4, ..+4).
// Rows of odd keys read the two halves in the other order so that the two keys
// sharing a half-warp request hit different banks.
template <int HD, class T>
__device__ __forceinline__ void ld8(const T* row, int c, int odd, float* lo, float* hi) {
    float a[4], b[4];
    ld4f(row + (odd ? HD / 2 : 0) + c * 4, a);
    ld4f(row + (odd ? 0 : HD / 2) + c * 4, b);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        lo[e] = odd ? b[e] : a[e];
        hi[e] = odd ? a[e] : b[e];
    }
}

// One warp: its queries (i = wsub, wsub + WPS, ...) of one unit, after the
// unit's K/V copies and the position table were issued.
template <int HD, int NQW, int WPS, int SPB, int NK, class T>
__device__ void attend(const AttnParams& a, int h, const float* Ps, uint64_t* pbar, uint8_t* usm, int wsub, int lane,
                       const float* qsrc, int pq0, int nq, int kpos0, int Nk, T* dst, int* status) {
    using A = Attn<HD, NQW, WPS, SPB, NK, T>;
    constexpr int LPK = A::LPK, KPS = A::KPS, PS = A::PS;
    uint64_t* bar = reinterpret_cast<uint64_t*>(usm);
    const T* Ks = reinterpret_cast<const T*>(usm + 16);
    const T* Vs = Ks + A::KV;
    float* S = reinterpret_cast<float*>(const_cast<T*>(Vs + A::KV));
    const int c = lane % LPK, g = lane / LPK;
    // this warp's queries, with both biases folded in, 8 dims per lane in registers
    float qu[NQW][8], qv[NQW][8];
#pragma unroll
    for (int t = 0; t < NQW; ++t) {
        const int i = wsub + WPS * t;
        if (i >= nq) break;
        const float* qr = qsrc + (long long)i * a.ldq;
        const float* ub = a.pbu + h * HD;
        const float* vb = a.pbv + h * HD;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int d = half * (HD / 2) + c * 4;
            const float4 q4 = *reinterpret_cast<const float4*>(qr + d);
            const float4 u4 = __ldg(reinterpret_cast<const float4*>(ub + d));
            const float4 v4 = __ldg(reinterpret_cast<const float4*>(vb + d));
            const float qq[4] = {q4.x, q4.y, q4.z, q4.w}, uu[4] = {u4.x, u4.y, u4.z, u4.w},
                        vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                qu[t][half * 4 + e] = qq[e] + uu[e];
                qv[t][half * 4 + e] = qq[e] + vv[e];
            }
        }
    }
    const bool landed = mbar_wait(bar, 0) && mbar_wait(pbar, 0);
    __syncwarp();
    if (!landed) {
        if (lane == 0) latch_error(status, CAC_E_TIMEOUT);
        return;
    }
    // scores
    for (int j0 = 0; j0 < Nk; j0 += KPS) {
        const int j = j0 + g;
        const bool valid = j < Nk;
        const int pk = kpos0 + j;
        float k8[8];
        {
            float lo[4], hi[4];
            ld8<HD>(Ks + (valid ? j : 0) * HD, c, j & 1, lo, hi);
#pragma unroll
            for (int e = 0; e < 4; ++e) { k8[e] = lo[e]; k8[4 + e] = hi[e]; }
        }
#pragma unroll
        for (int t = 0; t < NQW; ++t) {
            const int i = wsub + WPS * t;
            if (i >= nq) break;
            const int pq = pq0 + i;
            const bool ok = valid && allowed(a, pq, pk);
            float part = 0.f;
            if (ok) {
                float p8[8];
                const float* pr = Ps + (pq - pk - a.rmin) * PS;
                ld4f(pr + c * 4, p8);
                ld4f(pr + HD / 2 + c * 4, p8 + 4);
#pragma unroll
                for (int e = 0; e < 8; ++e) part = fmaf(qu[t][e], k8[e], fmaf(qv[t][e], p8[e], part));
            }
#pragma unroll
            for (int o = 1; o < LPK; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
            if (valid && c == 0) S[i * NK + j] = ok ? part * a.scale : -FLT_MAX;
        }
    }
    __syncwarp();
    // softmax over the keys of each of this warp's queries
#pragma unroll 1
    for (int t = 0; t < NQW; ++t) {
        const int i = wsub + WPS * t;
        if (i >= nq) break;
        float* Si = S + i * NK;
        float m = -FLT_MAX;
        for (int j = lane; j < Nk; j += 32) m = fmaxf(m, Si[j]);
        m = warp_max(m);
        float sum = 0.f;
        for (int j = lane; j < Nk; j += 32) {
            const float e = (Si[j] == -FLT_MAX) ? 0.f : __expf(Si[j] - m);
            Si[j] = e;
            sum += e;
        }
        sum = warp_sum(sum);
        const float inv = 1.f / sum;
        for (int j = lane; j < Nk; j += 32) Si[j] *= inv;
    }
    __syncwarp();
    pdl_trigger();
    // probs @ V: key group g takes keys j = g, g + KPS, ...; each lane 8 dims
    float acc[NQW][8];
#pragma unroll
    for (int t = 0; t < NQW; ++t)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[t][e] = 0.f;
#pragma unroll 2
    for (int j = g; j < Nk; j += KPS) {
        float lo[4], hi[4];
        ld8<HD>(Vs + j * HD, c, j & 1, lo, hi);
#pragma unroll
        for (int t = 0; t < NQW; ++t) {
            const int i = wsub + WPS * t;
            if (i >= nq) break;
            const float pij = S[i * NK + j];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[t][e] = fmaf(pij, lo[e], acc[t][e]);
                acc[t][4 + e] = fmaf(pij, hi[e], acc[t][4 + e]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NQW; ++t) {
        const int i = wsub + WPS * t;
        if (i >= nq) break;
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
            for (int o = LPK; o < 32; o <<= 1) acc[t][e] += __shfl_xor_sync(0xffffffffu, acc[t][e], o);
        if (g == 0) {
            T* o = dst + (long long)i * a.ldo;
            st4(o + c * 4, acc[t]);
            st4(o + HD / 2 + c * 4, acc[t] + 4);
        }
    }
}

// Block prologue: thread 0 arms the block barrier and bulk-copies this head's
// padded position table [NR][HD + 4].
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

// streaming: units = batch slots; keys = [cache | new] from the stream's ring
template <int HD, int NQW, int WPS, int SPB, int NK, class T>
__global__ void __launch_bounds__(SPB * WPS * 32) attn_stream_kernel(AttnParams a, int* status) {
    using A = Attn<HD, NQW, WPS, SPB, NK, T>;
    extern __shared__ float4 sm4[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(sm4);
    const int h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = warp / WPS, wsub = warp % WPS;
    const int b = blockIdx.x * SPB + slot;
    const bool live = b < a.nb;
    uint64_t* pbar = reinterpret_cast<uint64_t*>(sm);
    float* Ps = reinterpret_cast<float*>(sm + 16);
    uint8_t* usm = sm + 16 + ((a.NR * A::PS * 4 + 15) & ~15) + slot * A::UNIT_BYTES;
    stage_ptable<HD>(a, h, Ps, pbar);  // weights: before waiting for the QKV projection
    pdl_wait();
    int id = 0, p0 = 0, Lc = 0, Nk = 0;
    if (live) {
        id = a.ids[b];
        p0 = a.pos[id];
        Lc = min(p0, a.left);
        Nk = min(Lc + a.nq, NK);
        if (wsub == 0 && lane == 0) {
            uint64_t* bar = reinterpret_cast<uint64_t*>(usm);
            T* Ks = reinterpret_cast<T*>(usm + 16);
            T* Vs = Ks + A::KV;
            constexpr uint32_t ROW = HD * sizeof(T);
            mbar_init(bar, 1);
            fence_mbar_init();
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
    attend<HD, NQW, WPS, SPB, NK, T>(a, h, Ps, pbar, usm, wsub, lane, a.q + (long long)b * a.nq * a.ldq + h * HD, p0,
                                     a.nq, p0 - Lc, Nk, static_cast<T*>(a.out) + (long long)b * a.nq * a.ldo + h * HD,
                                     status);
}

// offline: units = query groups (one mask chunk, or `qgroup` frames of a window
// mask) of one sequence; keys from the dense K/V rows, one bulk copy per row.
template <int HD, int NQW, int WPS, int SPB, int NK, class T>
__global__ void __launch_bounds__(SPB * WPS * 32) attn_offline_kernel(AttnParams a, int qgroup, int* status) {
    using A = Attn<HD, NQW, WPS, SPB, NK, T>;
    extern __shared__ float4 sm4[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(sm4);
    const int h = blockIdx.y, seq = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = warp / WPS, wsub = warp % WPS;
    const int len = a.seq_len[seq];
    const int pq0 = (blockIdx.x * SPB + slot) * qgroup;
    const bool live = pq0 < len;
    uint64_t* pbar = reinterpret_cast<uint64_t*>(sm);
    float* Ps = reinterpret_cast<float*>(sm + 16);
    uint8_t* usm = sm + 16 + ((a.NR * A::PS * 4 + 15) & ~15) + slot * A::UNIT_BYTES;
    stage_ptable<HD>(a, h, Ps, pbar);
    pdl_wait();
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
        if (wsub == 0) {
            uint64_t* bar = reinterpret_cast<uint64_t*>(usm);
            T* Ks = reinterpret_cast<T*>(usm + 16);
            T* Vs = Ks + A::KV;
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
    }
    __syncthreads();
    if (!live) return;
    attend<HD, NQW, WPS, SPB, NK, T>(a, h, Ps, pbar, usm, wsub, lane, a.q + (rb + pq0) * a.ldq + h * HD, pq0, nq, klo,
                                     Nk, static_cast<T*>(a.out) + (rb + pq0) * a.ldo + h * HD, status);
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

template <int HD, int NQW, int WPS, int SPB, int NK, class T>
static cudaError_t attn_stream_launch(const AttnParams& a, int* status, cudaStream_t s) {
    using A = Attn<HD, NQW, WPS, SPB, NK, T>;
    const size_t smem = A::smem(a.NR);
    auto kern = attn_stream_kernel<HD, NQW, WPS, SPB, NK, T>;
    static size_t attr = 48 * 1024;  // dynamic shared memory limit set so far for this instantiation
    cudaError_t e = raise_smem(kern, smem, attr);
    if (e != cudaSuccess) return e;
    dim3 grid((a.nb + SPB - 1) / SPB, a.H);
    return launch_k(kern, grid, dim3(A::THREADS), smem, s, 1, a, status);
}

template <int HD, int NQW, int WPS, int SPB, int NK, class T>
static cudaError_t attn_offline_launch(const AttnParams& a, int qgroup, int* status, cudaStream_t s) {
    using A = Attn<HD, NQW, WPS, SPB, NK, T>;
    const size_t smem = A::smem(a.NR);
    auto kern = attn_offline_kernel<HD, NQW, WPS, SPB, NK, T>;
    static size_t attr = 48 * 1024;
    cudaError_t e = raise_smem(kern, smem, attr);
    if (e != cudaSuccess) return e;
    const int groups = (a.T + qgroup - 1) / qgroup;
    dim3 grid((groups + SPB - 1) / SPB, a.H, a.nb);
    return launch_k(kern, grid, dim3(A::THREADS), smem, s, 1, a, qgroup, status);
}

#define ATT_DISPATCH(LAUNCH, NQW, WPS, SPB, NK, ...)                                                     \
    do {                                                                                                 \
        if (a.HD == 64)                                                                                  \
            return act_bf16 ? LAUNCH<64, NQW, WPS, SPB, NK, bf16>(__VA_ARGS__)                           \
                            : LAUNCH<64, NQW, WPS, SPB, NK, float>(__VA_ARGS__);                         \
        if (a.HD == 16)                                                                                  \
            return act_bf16 ? LAUNCH<16, NQW, WPS, SPB, NK, bf16>(__VA_ARGS__)                           \
                            : LAUNCH<16, NQW, WPS, SPB, NK, float>(__VA_ARGS__);                         \
    } while (0)

// Instantiations (queries per unit = NQW * WPS): 160 ms pushes (2 queries,
// keys <= left + 2: 4 units x 2 warps per block), chunked pushes of up to 8
// frames (keys <= left + 8: 2 units x 4 warps), provisional passes (up to 24
// queries, keys <= left + 24: 1 unit x 8 warps); offline groups of <= 8.
cudaError_t launch_attention_stream(const AttnParams& a, int act_bf16, int* status, cudaStream_t s) {
    if (a.nb <= 0) return cudaSuccess;
    const int nk_need = a.left + a.nq;
    if (a.nq <= 2 && nk_need <= 80) ATT_DISPATCH(attn_stream_launch, 1, 2, 4, 80, a, status, s);
    if (a.nq <= 8 && nk_need <= 80) ATT_DISPATCH(attn_stream_launch, 2, 4, 2, 80, a, status, s);
    if (a.nq <= 24 && nk_need <= 96) ATT_DISPATCH(attn_stream_launch, 3, 8, 1, 96, a, status, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attention_offline(const AttnParams& a, int act_bf16, int* status, cudaStream_t s) {
    if (a.nb <= 0) return cudaSuccess;
    // queries per unit: one chunk of the chunked mask, or 8 consecutive frames of a window mask
    const int qgroup = a.rc > 0 ? 8 : a.chunk;
    const int nk_need = a.rc > 0 ? a.left + qgroup + a.rc : a.left + a.chunk;
    if (qgroup > 8 || nk_need > 96) return cudaErrorInvalidValue;
    if (qgroup <= 2 && nk_need <= 80) ATT_DISPATCH(attn_offline_launch, 1, 2, 4, 80, a, qgroup, status, s);
    ATT_DISPATCH(attn_offline_launch, 2, 4, 2, 96, a, qgroup, status, s);
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
    const int b = (int)(idx / D), c = (int)(idx % D);
    float w[9];
    const int cw = idx < (long long)nb * D ? c : 0;
#pragma unroll
    for (int k = 0; k < 9; ++k) w[k] = __ldg(wT + k * D + cw);
    const float bias = __ldg(bdw + cw), gam = __ldg(bng + cw), bet = __ldg(bnb + cw);
    pdl_wait();
    if (idx >= (long long)nb * D) return;
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
    pdl_trigger();
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
        return launch_k(dwconv_kernel<bf16>, dim3(blocks), dim3(256), 0, s, 1, static_cast<const bf16*>(glu),
                        static_cast<bf16*>(cache), cs_stride, ids, pos, nq, n_commit, wT, bdw, bng, bnb,
                        static_cast<bf16*>(out), D, nb);
    return launch_k(dwconv_kernel<float>, dim3(blocks), dim3(256), 0, s, 1, static_cast<const float*>(glu),
                    static_cast<float*>(cache), cs_stride, ids, pos, nq, n_commit, wT, bdw, bng, bnb,
                    static_cast<float*>(out), D, nb);
}

// ---------------------------------------------------------------------------
// bookkeeping and small utilities
// ---------------------------------------------------------------------------
__global__ void advance_kernel(int* pos, const int* ids, int nb, int n) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < nb) pos[ids[b]] += n;
}
__global__ void set_pos_kernel(int* pos, const int* ids, int nb, int value) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < nb) pos[ids[b]] = value;
}

cudaError_t launch_advance(int* pos, const int* ids, int nb, int n, cudaStream_t s) {
    if (nb <= 0) return cudaSuccess;
    return launch_k(advance_kernel, dim3((nb + 255) / 256), dim3(256), 0, s, 1, pos, ids, nb, n);
}
cudaError_t launch_set_pos(int* pos, const int* ids, int nb, int value, cudaStream_t s) {
    if (nb <= 0) return cudaSuccess;
    return launch_k(set_pos_kernel, dim3((nb + 255) / 256), dim3(256), 0, s, 1, pos, ids, nb, value);
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
    pdl_wait();
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
