// GEMM interface: C[M,N] = A[M,K] * B[N,K]^T with a fused epilogue.
//
// A holds activations (row-major, K contiguous).  For a stride-2, kernel-3
// convolution over time A is a window buffer read in im2col form: GEMM row t,
// K index k*C + c is window row 2t + k, channel c (the SIMT kernel reads it as
// overlapping rows with row stride 2C; the tcgen05 kernel through a 3-D tensor
// map).  B holds weights stored [out][in] (K-major).  Each epilogue call
// receives one output row's 32 consecutive fp32 accumulators (col0 is a
// multiple of 32).
#pragma once

#include "common.cuh"

namespace cac {

enum EpiKind : int {
    EPI_STORE = 0,  // out = act(acc + bias) to fp32 and/or activation-dtype buffers, optional row remap
    EPI_RESID = 1,  // x += scale * (acc + bias)                      (fp32 residual stream)
    EPI_GLU = 2,    // 32-column segments [16 value | 16 gate] -> 16 outputs value * sigmoid(gate)
    EPI_QKV = 3,    // Q (fp32) and K/V written into per-stream rings (or dense buffers)
    EPI_SUB = 4,    // subsampling stage: ReLU(acc + bias), zero before stream start, row remap
    EPI_GLUDW = 5,  // EPI_GLU, then the causal depthwise conv + affine + SiLU and the conv-ring commit
};
enum ActKind : int { ACT_NONE = 0, ACT_RELU = 1, ACT_SILU = 2 };

struct EpiParams {
    int kind = EPI_STORE;
    int act = ACT_NONE;
    int act_bf16 = 1;            // activation-dtype outputs are bf16 (1) or fp32 (0)
    const float* bias = nullptr;
    // EPI_STORE / EPI_GLU / EPI_SUB destination
    float* out_f32 = nullptr;
    void* out_act = nullptr;
    int ldo = 0;
    // EPI_STORE row remap: out row = g' * grp_stride + (r % grp) + row_off with
    // g = r / grp and g' = grp_map ? grp_map[g] : g
    int grp = 1 << 30, grp_stride = 0, row_off = 0;
    const int* grp_map = nullptr;
    // EPI_RESID
    float* x = nullptr;
    int ldx = 0;
    float scale = 1.f;
    // EPI_QKV (also uses ids / pos / nq)
    int D = 0, HD = 0, R = 0;
    long long ring_sstride = 0;  // elements between consecutive stream ids in a ring
    void* kring = nullptr;       // ring base already offset to this layer
    void* vring = nullptr;
    int dense = 0;               // 1: K/V rows go to kring/vring as dense [M][D]
    float* q = nullptr;
    int ldq = 0;
    const int* ids = nullptr;    // batch slot -> stream id
    const int* pos = nullptr;    // stream id -> absolute position of its first new frame
    int nq = 1;                  // rows per batch slot
    // EPI_SUB
    int P = 1;                   // A rows (pairs) per group
    int T_out = 1;               // valid outputs per group (the rest are seams between groups)
    int dst_rows = 1, dst_off = 0;
    int tmult = 0, toff = 0;     // absolute time = tmult * pos[id] - toff + t (zeroed when < 0)
    int split_out = 0;           // bf16 only, > 0: also store lo = bf16(v - hi) at column split_out + c
    // EPI_GLUDW (tcgen05 path, streaming steps): rows b * nq + i (frame i of
    // batch slot b, 32 % nq == 0, so a stream's rows lie in one warp).  The GLU
    // value g (rounded to the activation dtype, as stored) goes to out_act
    // (when set); then, per channel c,
    //   y = SiLU(dw_gamma[c] * (dw_bias[c] + sum_k dw_wT[k][c] * win_k) + dw_beta[c]) -> dw_out,
    // win_k = g of frame i - 8 + k: from the conv ring (dw_ring + id * dw_sstride,
    // slot = absolute frame mod 8, zero before the stream start) or from this
    // step's rows; afterwards the step's g rows are committed to the ring.
    void* dw_ring = nullptr;
    long long dw_sstride = 0;
    const float* dw_wT = nullptr;   // [9][D]
    const float* dw_bias = nullptr;
    const float* dw_gamma = nullptr;
    const float* dw_beta = nullptr;
    void* dw_out = nullptr;
    int dw_rows = 0;                // rows of the GEMM (M): rows past it have no stream
    // LayerNorm folded into this GEMM (EPI_STORE / EPI_GLU / EPI_QKV / EPI_GLUDW):
    // A is the split operand of gamma * x (x the residual rows), bias = b + W beta
    // and ln_colsum[n] = sum_k gamma_k W[n][k], so that LN(x) W^T + b =
    // rstd_r (acc - mean_r ln_colsum) + bias.  Before the bias: v = rstd_r * (acc -
    // mean_r * ln_colsum[c]), with mean_r and rstd_r of x from the row's ln_parts
    // partials (sum, centred sum of squares of 32 columns each) at ln_stats + r *
    // ln_parts; rows >= ln_rows are not read.
    const float2* ln_stats = nullptr;
    const float* ln_colsum = nullptr;
    int ln_parts = 0, ln_rows = 0;
    // EPI_RESID (bf16): also emit the split operand of xs_gamma * (updated x) (hi
    // at xs + r * ldxs + c, lo xs_lo columns further) and the per-32-column
    // partials of x at stats_out + r * stats_parts + c / 32, for a GEMM that
    // folds the next LayerNorm (xs_gamma: that LayerNorm's gain)
    bf16* xs = nullptr;
    const float* xs_gamma = nullptr;
    long long ldxs = 0;
    int xs_lo = 0;
    float2* stats_out = nullptr;
    int stats_parts = 0;
    // checked build: ids index n_streams streams and positions are >= 0; a
    // violation latches CAC_E_BOUNDS in status and the row is not written
    int n_streams = 1 << 30;
    int* status = nullptr;
};

// host helpers ---------------------------------------------------------------
// Encode a 2-D bf16 tensor map [rows][inner] with `row_stride_bytes` between
// rows, box [box_rows][64], 128-byte swizzle.  Returns false on failure.
bool make_tmap_bf16(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows,
                    uint64_t row_stride_bytes, uint32_t box_rows);

// Blocks of 64-wide bf16 rows: 3-D map {64, rows, blocks} (row stride 128 B,
// block stride block_stride_bytes), box {64, box_rows, 1}, 128-byte swizzle —
// e.g. one head's K or V ring of one stream and layer, or one head's position
// table, per copy.
bool make_tmap_bf16_blocks(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t blocks,
                           uint64_t block_stride_bytes, uint32_t box_rows);

// Convolution view of a window buffer [rows][C] for a stride-2, kernel-3
// convolution: 3-D map {C, 2, rows/2} (channel, row parity, row pair), box
// {64, 1, box_rows}.  GEMM row t, K index k*C + c reads window row 2t + k.
bool make_tmap_bf16_conv(CUtensorMap* tm, const void* base, uint64_t C, uint64_t pairs, uint32_t box_rows);

// tcgen05/TMEM GEMM, bf16 operands.  K % 64 == 0, N % BN == 0, BN in {64, 128, 256}.
// conv_C > 0 selects the convolution view of A (tmA from make_tmap_bf16_conv, K = 3 * conv_C;
// with a_split the window rows are 2 * conv_C wide, hi | lo).
// splits in 1..4: split-K over a cluster of `splits` CTAs per output tile,
// reduced deterministically through distributed shared memory.
// a_split: A is a split operand [M][2K] (hi in columns [0, K), lo = residual of
// the bf16 rounding in [K, 2K)); the product is (hi + lo) * B^T.
// pal_tab (palette weights, BN = 64): tmB is a make_tmap_packed map over the
// 6-bit indices [N][3K/4] bytes and pal_tab holds N/64 tables of 64 bf16 values,
// one per 64-row block of the output columns.
cudaError_t launch_gemm_tc(const CUtensorMap* tmA, const CUtensorMap* tmB, int M, int N, int K, int BN, int conv_C,
                           int splits, int a_split, const EpiParams& ep, int* status, cudaStream_t s,
                           const uint16_t* pal_tab = nullptr);

// Packed 6-bit indices [rows][row_bytes] (a row's indices as a little-endian bit
// stream, row_bytes = 3K/4 a multiple of 16), box 48 bytes x 64 rows.
bool make_tmap_packed(CUtensorMap* tm, const void* base, uint64_t row_bytes, uint64_t rows);

// Persistent tcgen05 GEMM for many output tiles (128 x 128 tiles, one CTA per
// SM, two TMEM accumulators so epilogue and main loop overlap).  tmB128: the
// weight map with 128-row boxes.  N % 128 == 0; other rules as launch_gemm_tc
// (no split-K, no EPI_GLUDW).
cudaError_t launch_gemm_tc_persistent(const CUtensorMap* tmA, const CUtensorMap* tmB128, int M, int N, int K,
                                      int conv_C, int a_split, const EpiParams& ep, int* status, cudaStream_t s);

// SIMT GEMM (fp32 or bf16 operands, fp32 accumulate).  N % 32 == 0.  a_split
// (bf16 only): A row r holds hi at A + r * lda and lo at A + r * lda + K.
// conv_C > 0: A is a stride-2 convolution window (lda = row-pair stride), K
// index k * conv_C + c reads channel c of window row 2r + k; window rows are
// conv_C wide, or 2 * conv_C (hi | lo) with a_split.
cudaError_t launch_gemm_simt(int bf16_operands, const void* A, long long lda, const void* B, long long ldb, int M,
                             int N, int K, int conv_C, int a_split, const EpiParams& ep, cudaStream_t s);

// ---------------------------------------------------------------------------
// epilogue, applied to one row segment of 32 accumulators
// ---------------------------------------------------------------------------
template <class T>
__device__ __forceinline__ void store32(T* dst, const float (&v)[32]);

template <>
__device__ __forceinline__ void store32<float>(float* dst, const float (&v)[32]) {
    float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int i = 0; i < 8; ++i) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

template <>
__device__ __forceinline__ void store32<bf16>(bf16* dst, const float (&v)[32]) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 u;
        __nv_bfloat162 p0 = __floats2bfloat162_rn(v[8 * i + 0], v[8 * i + 1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(v[8 * i + 2], v[8 * i + 3]);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(v[8 * i + 4], v[8 * i + 5]);
        __nv_bfloat162 p3 = __floats2bfloat162_rn(v[8 * i + 6], v[8 * i + 7]);
        u.x = *reinterpret_cast<uint32_t*>(&p0);
        u.y = *reinterpret_cast<uint32_t*>(&p1);
        u.z = *reinterpret_cast<uint32_t*>(&p2);
        u.w = *reinterpret_cast<uint32_t*>(&p3);
        d[i] = u;
    }
}

// Warp-cooperative row stores: lane l holds 32 consecutive elements of its
// own row, to be written at dst (lane's row pointer).  The rows go through the
// warp's shared-memory slice `stage` (EPI_STAGE_FLOATS floats) so that every
// global store instruction writes whole lines: 4 rows x 128 B (fp32) or 8 rows x
// 64 B (bf16) per instruction instead of 32 scattered 16-byte pieces.  Rows
// whose lane has live == false are not written.  Every lane of the warp calls.
constexpr int EPI_STAGE_FLOATS = 32 * 36;

__device__ __forceinline__ void rows_store(float* stage, float* dst, const float (&v)[32], bool live) {
    const int lane = threadIdx.x & 31;
    float4* s = reinterpret_cast<float4*>(stage + lane * 36);  // 144-byte rows: conflict-free v4 writes
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    __syncwarp();
    const unsigned live_mask = __ballot_sync(0xffffffffu, live);
    const unsigned long long p = reinterpret_cast<unsigned long long>(dst);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = 4 * i + (lane >> 3), c = lane & 7;
        const unsigned long long pr = __shfl_sync(0xffffffffu, p, r);
        const float4 q = reinterpret_cast<const float4*>(stage + r * 36)[c];
        if ((live_mask >> r) & 1u) reinterpret_cast<float4*>(pr)[c] = q;
    }
    __syncwarp();  // the slice is free for the next call
}

__device__ __forceinline__ void rows_store(float* stage, bf16* dst, const float (&v)[32], bool live) {
    const int lane = threadIdx.x & 31;
    uint32_t* su = reinterpret_cast<uint32_t*>(stage);
    uint4* s = reinterpret_cast<uint4*>(su + lane * 20);  // 80-byte rows
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 u;
        __nv_bfloat162 p0 = __floats2bfloat162_rn(v[8 * j + 0], v[8 * j + 1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(v[8 * j + 2], v[8 * j + 3]);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(v[8 * j + 4], v[8 * j + 5]);
        __nv_bfloat162 p3 = __floats2bfloat162_rn(v[8 * j + 6], v[8 * j + 7]);
        u.x = *reinterpret_cast<uint32_t*>(&p0);
        u.y = *reinterpret_cast<uint32_t*>(&p1);
        u.z = *reinterpret_cast<uint32_t*>(&p2);
        u.w = *reinterpret_cast<uint32_t*>(&p3);
        s[j] = u;
    }
    __syncwarp();
    const unsigned live_mask = __ballot_sync(0xffffffffu, live);
    const unsigned long long p = reinterpret_cast<unsigned long long>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = 8 * i + (lane >> 2), c = lane & 3;
        const unsigned long long pr = __shfl_sync(0xffffffffu, p, r);
        const uint4 q = reinterpret_cast<const uint4*>(su + r * 20)[c];
        if ((live_mask >> r) & 1u) reinterpret_cast<uint4*>(pr)[c] = q;
    }
    __syncwarp();
}

// store32 through the warp's staging slice when there is one (every lane
// calls), else directly (live lanes only)
template <class T>
__device__ __forceinline__ void put32(float* stage, T* dst, const float (&v)[32], bool live) {
    if (stage)
        rows_store(stage, dst, v, live);
    else if (live)
        store32<T>(dst, v);
}

// Operands of the epilogue that do not depend on the accumulators (bias, and
// the residual rows for EPI_RESID): loaded ahead, while the main loop runs.
struct EpiPre {
    float4 b[8];
    float4 x[8];
    float4 g[8];  // EPI_RESID with xs: the next LayerNorm's gain
    float ln_mean, ln_rstd;
    int dw_id, dw_p0;  // EPI_GLUDW: the row's stream id and position of its first new frame
};

// mean and 1/sqrt(var + 1e-5) of a row from its partials (sum_j, M2_j) over 32
// columns each (parts even, <= 32): var = (sum_j M2_j + 32 sum_j (mean_j -
// mean)^2) / (32 parts).  The loads are issued together (one float4 = two parts).
__device__ __forceinline__ void ln_row_stats(const float2* st, int parts, float& mean, float& rstd) {
    const float4* s4 = reinterpret_cast<const float4*>(st);
    float4 q[16];
    // through L2: the partials may come from another CTA of the same launch
#pragma unroll
    for (int j = 0; j < 16; ++j) q[j] = 2 * j < parts ? __ldcg(s4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) s += q[j].x + q[j].z;
    const float n = 32.f * (float)parts;
    mean = s / n;
    float m2 = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if (2 * j < parts) {
            const float d0 = q[j].x * (1.f / 32.f) - mean, d1 = q[j].z * (1.f / 32.f) - mean;
            m2 += q[j].y + q[j].w + 32.f * (d0 * d0 + d1 * d1);
        }
    }
    rstd = rsqrtf(m2 / n + 1e-5f);
}

__device__ __forceinline__ void ln_fold32(const EpiParams& e, int col0, const EpiPre& pre, float (&v)[32]) {
    const float4* c4 = reinterpret_cast<const float4*>(e.ln_colsum + col0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 c = __ldg(c4 + i);
        v[4 * i] = pre.ln_rstd * fmaf(-pre.ln_mean, c.x, v[4 * i]);
        v[4 * i + 1] = pre.ln_rstd * fmaf(-pre.ln_mean, c.y, v[4 * i + 1]);
        v[4 * i + 2] = pre.ln_rstd * fmaf(-pre.ln_mean, c.z, v[4 * i + 2]);
        v[4 * i + 3] = pre.ln_rstd * fmaf(-pre.ln_mean, c.w, v[4 * i + 3]);
    }
}

// mean and rstd of a row's LayerNorm (folded into the GEMM) from the partials
// at ln_stats; (0, 1) when there is none.
__device__ __forceinline__ float2 epi_row_stats(const EpiParams& e, int row) {
    float2 r = make_float2(0.f, 1.f);
    if (e.ln_stats && row < e.ln_rows) ln_row_stats(e.ln_stats + (long long)row * e.ln_parts, e.ln_parts, r.x, r.y);
    return r;
}

__device__ __forceinline__ void epi_apply_stats(float2 st, EpiPre& pre) {
    pre.ln_mean = st.x;
    pre.ln_rstd = st.y;
}

// stats = false: the caller supplies the row's LayerNorm statistics later
// through epi_apply_stats (computed once per row elsewhere).
template <int KIND>
__device__ __forceinline__ void epi_prefetch(const EpiParams& e, int row, int col0, EpiPre& pre, bool stats = true) {
    if (e.bias) {
        const float4* b4 = reinterpret_cast<const float4*>(e.bias + col0);
#pragma unroll
        for (int i = 0; i < 8; ++i) pre.b[i] = __ldg(b4 + i);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) pre.b[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if constexpr (KIND == EPI_RESID) {
        const float4* x4 = reinterpret_cast<const float4*>(e.x + (long long)row * e.ldx + col0);
#pragma unroll
        for (int i = 0; i < 8; ++i) pre.x[i] = __ldcg(x4 + i);  // L2: may be another CTA's write
        if (e.xs) {
            const float4* g4 = reinterpret_cast<const float4*>(e.xs_gamma + col0);
#pragma unroll
            for (int i = 0; i < 8; ++i) pre.g[i] = __ldg(g4 + i);
        }
    } else {
        pre.ln_mean = 0.f;
        pre.ln_rstd = 1.f;
        if (stats && e.ln_stats && row < e.ln_rows) epi_apply_stats(epi_row_stats(e, row), pre);
        if constexpr (KIND == EPI_GLUDW) {
            pre.dw_id = 0;
            pre.dw_p0 = 0;
            if (row < e.dw_rows) {
                pre.dw_id = e.ids[row / e.nq];
                if (!in_range(pre.dw_id, e.n_streams, e.status)) {
                    pre.dw_id = -1;  // checked build: the row is skipped
                } else {
                    pre.dw_p0 = e.pos[pre.dw_id];
                    if (!in_range(pre.dw_p0, 1 << 30, e.status)) {
                        pre.dw_id = -1;
                    } else {
                        // warm L2 with the conv-ring rows the epilogue reads (written a
                        // step ago, usually evicted since); this runs during the main loop
                        const int fi = row % e.nq;
                        const bf16* ring = static_cast<const bf16*>(e.dw_ring) + (long long)pre.dw_id * e.dw_sstride +
                                           (col0 >> 1);
                        for (int d = fi + 1; d <= 8; ++d) {
                            const int pabs = pre.dw_p0 + fi - d;
                            if (pabs >= 0)
                                asm volatile("prefetch.global.L2 [%0];" ::"l"(ring + (long long)(pabs & 7) * e.D));
                        }
                    }
                }
            }
        }
    }
}

// stage == nullptr: called by live lanes only, per-thread stores.  stage !=
// nullptr: called by every lane of the warp (live marks rows < M), row stores
// through the warp's staging slice.
template <int KIND, class TAct>
__device__ __forceinline__ void epilogue32(const EpiParams& e, int row, int col0, float (&v)[32], const EpiPre& pre,
                                           float* stage = nullptr, bool live = true) {
    if constexpr (KIND != EPI_RESID) {
        if (e.ln_stats) ln_fold32(e, col0, pre, v);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 b = pre.b[i];
        v[4 * i] += b.x; v[4 * i + 1] += b.y; v[4 * i + 2] += b.z; v[4 * i + 3] += b.w;
    }
    if constexpr (KIND == EPI_STORE) {
        if (e.act == ACT_SILU) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = siluf_(v[i]);
        } else if (e.act == ACT_RELU) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = fmaxf(v[i], 0.f);
        }
        long long orow = 0;
        if (live) {
            const int g = row / e.grp;
            orow = (long long)(e.grp_map ? e.grp_map[g] : g) * e.grp_stride + (row % e.grp) + e.row_off;
        }
        if (e.out_f32) put32<float>(stage, e.out_f32 + orow * e.ldo + col0, v, live);
        if (e.out_act) {
            TAct* dst = reinterpret_cast<TAct*>(e.out_act) + orow * e.ldo + col0;
            put32<TAct>(stage, dst, v, live);
            if (e.split_out > 0) {  // split operand for the next GEMM: lo = bf16(v - hi)
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] -= to_f(from_f<TAct>(v[i]));
                put32<TAct>(stage, dst + e.split_out, v, live);
            }
        }
    } else if constexpr (KIND == EPI_RESID) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 a = pre.x[i];
            v[4 * i] = fmaf(e.scale, v[4 * i], a.x);
            v[4 * i + 1] = fmaf(e.scale, v[4 * i + 1], a.y);
            v[4 * i + 2] = fmaf(e.scale, v[4 * i + 2], a.z);
            v[4 * i + 3] = fmaf(e.scale, v[4 * i + 3], a.w);
        }
        put32<float>(stage, e.x + (long long)row * e.ldx + col0, v, live);
        if (e.xs) {
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) sum += v[i];
            const float mu = sum * (1.f / 32.f);
            float m2 = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) m2 = fmaf(v[i] - mu, v[i] - mu, m2);
            if (live) e.stats_out[(long long)row * e.stats_parts + (col0 >> 5)] = make_float2(sum, m2);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 g = pre.g[i];
                v[4 * i] *= g.x; v[4 * i + 1] *= g.y; v[4 * i + 2] *= g.z; v[4 * i + 3] *= g.w;
            }
            bf16* dst = e.xs + (long long)row * e.ldxs + col0;
            put32<bf16>(stage, dst, v, live);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] -= __bfloat162float(__float2bfloat16_rn(v[i]));
            put32<bf16>(stage, dst + e.xs_lo, v, live);
        }
    } else if constexpr (KIND == EPI_GLU) {
        if (live) {
            TAct* o = reinterpret_cast<TAct*>(e.out_act) + (long long)row * e.ldo + (col0 >> 1);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = from_f<TAct>(v[i] * sigmoidf_(v[16 + i]));
        }
    } else if constexpr (KIND == EPI_QKV) {
        const int region = col0 / e.D;
        const int cc = col0 - region * e.D;
        if (region == 0) {
            put32<float>(stage, e.q + (long long)row * e.ldq + cc, v, live);
            return;
        }
        TAct* base = reinterpret_cast<TAct*>(region == 1 ? e.kring : e.vring);
        if (e.dense) {
            put32<TAct>(stage, base + (long long)row * e.D + cc, v, live);
            return;
        }
        int id = 0, slot = 0;
        if (live) {
            const int b = row / e.nq, i = row - (row / e.nq) * e.nq;
            id = e.ids[b];
            if (!in_range(id, e.n_streams, e.status)) {
                live = false;  // checked build: the row is skipped
                id = 0;
            } else {
                const int p = e.pos[id];
                if (!in_range(p, 1 << 30, e.status)) live = false;
                slot = live ? (p + i) % e.R : 0;
            }
        }
        TAct* sbase = base + (long long)id * e.ring_sstride;
        if (e.HD >= 32) {
            const int h = cc / e.HD, d0 = cc - h * e.HD;
            put32<TAct>(stage, sbase + ((long long)h * e.R + slot) * e.HD + d0, v, live);
        } else if (live) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const int d = cc + k, h = d / e.HD, dd = d - h * e.HD;
                sbase[((long long)h * e.R + slot) * e.HD + dd] = from_f<TAct>(v[k]);
            }
        }
    } else if constexpr (KIND == EPI_SUB) {
        const int g = row / e.P, t = row - (row / e.P) * e.P;
        bool on = live && t < e.T_out;  // seam rows spanning two groups are not written
        bool zero = false;
        if (on && e.ids) {
            if (in_range(e.ids[g], e.n_streams, e.status))
                zero = (e.tmult * e.pos[e.ids[g]] - e.toff + t) < 0;
            else
                on = false;  // checked build: the row is skipped
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = zero ? 0.f : fmaxf(v[i], 0.f);
        TAct* dst = reinterpret_cast<TAct*>(e.out_act) + ((long long)g * e.dst_rows + e.dst_off + t) * e.ldo + col0;
        put32<TAct>(stage, dst, v, on);
        if (e.split_out > 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] -= to_f(from_f<TAct>(v[i]));
            put32<TAct>(stage, dst + e.split_out, v, on);
        }
    }
}

// EPI_GLUDW for one 32-column accumulator segment (16 output channels); every
// lane of the warp calls it (shuffles), `live` marks rows < M.
// win: the lane's stream in the GEMM's shared-memory copy of the conv ring
// ([slot][32 channels], offset to this chunk's 16 channels), or nullptr to
// read the ring in global memory.  prm: the GEMM's shared-memory copy of the
// per-channel constants offset to this chunk's channels (rows of 32 floats:
// 0-8 the taps, 9 the conv bias, 10 gamma, 11 beta), csum: its copy of
// ln_colsum offset to this chunk's columns; both nullptr to read them in
// global memory.
__device__ __forceinline__ void epilogue_gludw(const EpiParams& e, int row, bool live, int col0, float (&v)[32],
                                               const EpiPre& pre, const bf16* win, const float* prm,
                                               const float* csum) {
    const int lane = threadIdx.x & 31;
    const int D = e.D, C = col0 >> 1, nq = e.nq;
    if (kChecked && pre.dw_id < 0) live = false;  // an id or position out of range (latched)
    if (e.ln_stats) {
        if (csum) {
            const float4* c4 = reinterpret_cast<const float4*>(csum);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 c = c4[i];
                v[4 * i] = pre.ln_rstd * fmaf(-pre.ln_mean, c.x, v[4 * i]);
                v[4 * i + 1] = pre.ln_rstd * fmaf(-pre.ln_mean, c.y, v[4 * i + 1]);
                v[4 * i + 2] = pre.ln_rstd * fmaf(-pre.ln_mean, c.z, v[4 * i + 2]);
                v[4 * i + 3] = pre.ln_rstd * fmaf(-pre.ln_mean, c.w, v[4 * i + 3]);
            }
        } else {
            ln_fold32(e, col0, pre, v);
        }
    }
    // per-channel constant rows: shared memory (row stride 32) or global (row stride D)
    auto cvec = [&](int r, int q) -> float4 {
        if (prm) return reinterpret_cast<const float4*>(prm + r * 32)[q];
        const float* g = r < 9 ? e.dw_wT + (long long)r * D : (r == 9 ? e.dw_bias : (r == 10 ? e.dw_gamma : e.dw_beta));
        return __ldg(reinterpret_cast<const float4*>(g + C) + q);
    };
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 b = pre.b[i];
        v[4 * i] += b.x; v[4 * i + 1] += b.y; v[4 * i + 2] += b.z; v[4 * i + 3] += b.w;
    }
    float g[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) g[i] = __bfloat162float(__float2bfloat16_rn(v[i] * sigmoidf_(v[16 + i])));
    const int fi = row % nq;
    const int id = live ? pre.dw_id : 0, p0 = live ? pre.dw_p0 : 0;  // loaded ahead (epi_prefetch)
    bf16* ring = static_cast<bf16*>(e.dw_ring) + (long long)id * e.dw_sstride;
    float acc[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 t = cvec(9, q);
        acc[4 * q] = t.x; acc[4 * q + 1] = t.y; acc[4 * q + 2] = t.z; acc[4 * q + 3] = t.w;
    }
    // taps k = 0 .. 7 (d = 8 - k frames back): this step's earlier rows by
    // shuffle, older frames from the conv ring (slot = frame mod 8, zero before
    // the stream start); the ring rows of four taps are loaded before any is used
    constexpr int TB = 4;  // taps whose ring rows are in flight together
#pragma unroll
    for (int k0 = 0; k0 < 8; k0 += TB) {
        uint4 r[TB][2];
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            const int d = 8 - (k0 + j), pabs = p0 + fi - d;
            if (d > fi && live && pabs >= 0) {
                const uint4* src = win ? reinterpret_cast<const uint4*>(win + (pabs & 7) * 32)
                                       : reinterpret_cast<const uint4*>(ring + (long long)(pabs & 7) * D + C);
                r[j][0] = src[0];
                r[j][1] = src[1];
            } else {
                r[j][0] = make_uint4(0u, 0u, 0u, 0u);  // bf16 zeros
                r[j][1] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int j = 0; j < TB; ++j) {
            const int k = k0 + j, d = 8 - k;
            float sh[16], win[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) sh[i] = d < nq ? __shfl_sync(0xffffffffu, g[i], (lane - d) & 31) : 0.f;
            if (d <= fi) {
#pragma unroll
                for (int i = 0; i < 16; ++i) win[i] = sh[i];
            } else {
                const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&r[j][0]);
                const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&r[j][1]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 a0 = __bfloat1622float2(h0[i]), a1 = __bfloat1622float2(h1[i]);
                    win[2 * i] = a0.x; win[2 * i + 1] = a0.y; win[8 + 2 * i] = a1.x; win[8 + 2 * i + 1] = a1.y;
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 w = cvec(k, q);
                acc[4 * q] = fmaf(w.x, win[4 * q], acc[4 * q]);
                acc[4 * q + 1] = fmaf(w.y, win[4 * q + 1], acc[4 * q + 1]);
                acc[4 * q + 2] = fmaf(w.z, win[4 * q + 2], acc[4 * q + 2]);
                acc[4 * q + 3] = fmaf(w.w, win[4 * q + 3], acc[4 * q + 3]);
            }
        }
    }
    {   // tap 8 (d = 0): this row's own GLU value
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 w = cvec(8, q);
            acc[4 * q] = fmaf(w.x, g[4 * q], acc[4 * q]);
            acc[4 * q + 1] = fmaf(w.y, g[4 * q + 1], acc[4 * q + 1]);
            acc[4 * q + 2] = fmaf(w.z, g[4 * q + 2], acc[4 * q + 2]);
            acc[4 * q + 3] = fmaf(w.w, g[4 * q + 3], acc[4 * q + 3]);
        }
    }
    __syncwarp();  // every lane has read the ring before this step's rows are committed
    if (!live) return;
    float y[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 gg = cvec(10, q), bb = cvec(11, q);
        y[4 * q] = siluf_(fmaf(gg.x, acc[4 * q], bb.x));
        y[4 * q + 1] = siluf_(fmaf(gg.y, acc[4 * q + 1], bb.y));
        y[4 * q + 2] = siluf_(fmaf(gg.z, acc[4 * q + 2], bb.z));
        y[4 * q + 3] = siluf_(fmaf(gg.w, acc[4 * q + 3], bb.w));
    }
    auto pack16 = [](const float (&f)[16], uint4& u0, uint4& u1) {
        uint32_t* w0 = reinterpret_cast<uint32_t*>(&u0);
        uint32_t* w1 = reinterpret_cast<uint32_t*>(&u1);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 a = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            const __nv_bfloat162 c = __floats2bfloat162_rn(f[8 + 2 * i], f[8 + 2 * i + 1]);
            w0[i] = *reinterpret_cast<const uint32_t*>(&a);
            w1[i] = *reinterpret_cast<const uint32_t*>(&c);
        }
    };
    uint4 u0, u1;
    pack16(y, u0, u1);
    uint4* yo = reinterpret_cast<uint4*>(static_cast<bf16*>(e.dw_out) + (long long)row * D + C);
    yo[0] = u0;
    yo[1] = u1;
    pack16(g, u0, u1);
    uint4* rs = reinterpret_cast<uint4*>(ring + (long long)((p0 + fi) & 7) * D + C);
    rs[0] = u0;
    rs[1] = u1;
    if (e.out_act) {
        uint4* go = reinterpret_cast<uint4*>(static_cast<bf16*>(e.out_act) + (long long)row * D + C);
        go[0] = u0;
        go[1] = u1;
    }
}

}  // namespace cac
