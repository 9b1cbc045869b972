// Rectangular rel-pos attention of a streaming step on the tensor cores
// (mma.sync m16n8k16, bf16 operands, fp32 accumulation).
//
// Work unit: one (stream, head) with nq <= 4 new queries at absolute
// positions p0 .. p0 + nq - 1 and the Nk = Lc + nq <= 80 keys p0 - Lc .. p0 +
// nq - 1 (cache + new rows of the stream's K/V rings).  One warp per unit:
//
//   ac[j][i] = K[j] . (q_i + u)      A = K rows (16 keys per tile),   B = q + u
//   bd[r][i] = P[r] . (q_i + v)      A = position-table rows r,       B = q + v
//   score[i][j] = (ac[j][i] + bd[p_i - p_j - rmin][i]) * scale, masked to the
//                 query's key window, softmax over j
//   out[i][d]   = sum_j prob[i][j] V[j][d]      A = V^T (ldmatrix.trans),  B = prob
//
// The queries and the probabilities are fp32; each enters the MMA as a split
// pair (hi = bf16(x), lo = bf16(x - hi)) occupying two of the eight B columns
// (columns 0..3: hi of queries 0..3, columns 4..7: lo), so one MMA per tile
// carries them at ~16 significant bits and hi + lo is recombined from the
// fp32 accumulators with one shuffle.  K, V and the position table are bf16
// already (exact operands).
//
// Staging: cp.async 16-byte copies into 128-byte-swizzled shared rows (chunk
// c of row r at chunk position c ^ (r & 7)), so the ldmatrix row reads are
// conflict-free.  Keys are stored in logical order (ring slot (s0 + j) mod R
// -> row j); rows j >= Nk and table rows r >= NR are zero-filled.  The
// position table is weights: it is copied before the wait on the previous
// kernel, the K/V rows after it.
#include <cfloat>

#include "kernels.cuh"

namespace cac {

namespace {
constexpr int AM_WARPS = 4;                      // units per block
constexpr int AM_ROWS = 80;                      // key / rel rows per unit (5 tiles of 16)
constexpr int AM_ROWB = 128;                     // bytes per row (64 bf16)
constexpr int AM_MAT = AM_ROWS * AM_ROWB;        // one [80][64] bf16 matrix
constexpr int AM_SLD = 84;                       // fp32 row stride of the score arrays
constexpr int AM_UNIT = 2 * AM_MAT + 2 * 4 * AM_SLD * 4;
constexpr int AM_SMEM = AM_MAT + AM_WARPS * AM_UNIT;

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)(row * AM_ROWB + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D += A * B, m16n8k16, bf16 in, fp32 accumulate
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// half 0: bf16(x); half 1: bf16(x - bf16(x))
__device__ __forceinline__ bf16 split_part(float x, int half) {
    const bf16 hi = __float2bfloat16_rn(x);
    return half ? __float2bfloat16_rn(x - __bfloat162float(hi)) : hi;
}
__device__ __forceinline__ uint32_t pack2(bf16 lo16, bf16 hi16) {
    return (uint32_t)__bfloat16_as_ushort(lo16) | ((uint32_t)__bfloat16_as_ushort(hi16) << 16);
}

// ac or bd for the five 16-row tiles of one [80][64] matrix against the
// split-query B fragments; result rows (keys / rels) x queries into S[i][row].
__device__ __forceinline__ void score_tiles(uint32_t mat, const uint32_t (&b)[4][2], float* S, int lane) {
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int mt = 0; mt < AM_ROWS / 16; ++mt) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int row = mt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t a[4];
            ldsm_x4(mat + swz(row, ks * 2 + (lane >> 4)), a);
            mma16816(acc, a, b[ks][0], b[ks][1]);
        }
        // columns 2c, 2c+1 (c < 2: hi of queries 2c, 2c+1; c >= 2: their lo)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], 2);
        if (c < 2) {
            const int r0 = mt * 16 + g;
            S[(2 * c) * AM_SLD + r0] = acc[0];
            S[(2 * c + 1) * AM_SLD + r0] = acc[1];
            S[(2 * c) * AM_SLD + r0 + 8] = acc[2];
            S[(2 * c + 1) * AM_SLD + r0 + 8] = acc[3];
        }
    }
}

__global__ void __launch_bounds__(AM_WARPS * 32) attn_stream_mma_kernel(AttnParams a, int* status) {
    extern __shared__ __align__(1024) uint8_t sm[];
    const int h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int b = blockIdx.x * AM_WARPS + warp;
    const bool live = b < a.nb;
    const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(sm);
    const uint32_t Pm = sbase;
    uint8_t* usm = sm + AM_MAT + warp * AM_UNIT;
    const uint32_t Km = sbase + AM_MAT + warp * AM_UNIT, Vm = Km + AM_MAT;
    float* Sac = reinterpret_cast<float*>(usm + 2 * AM_MAT);  // [4][AM_SLD]: ac, then probabilities
    float* Sbd = Sac + 4 * AM_SLD;                           // [4][AM_SLD]: bd, then the output staging
    constexpr int HD = 64;

    // position table of this head (weights): rows >= NR zero
    {
        const bf16* P = static_cast<const bf16*>(a.P) + (long long)h * a.NR * HD;
        for (int e = threadIdx.x; e < AM_ROWS * 8; e += blockDim.x) {
            const int r = e >> 3, ch = e & 7;
            const bool ok = r < a.NR;
            cp_async16(Pm + swz(r, ch), P + (ok ? r : 0) * HD + ch * 8, ok);
        }
    }
    pdl_wait();
    int p0 = 0, Lc = 0, Nk = 0, nq = a.nq;
    const float* q = nullptr;
    if (live) {
        const int id = a.ids[b];
        p0 = a.pos[id];
        Lc = min(p0, a.left);
        Nk = Lc + nq;
        const int s0 = (p0 - Lc) % a.R;
        const long long base = (long long)id * a.sstride + (long long)h * a.R * HD;
        const bf16* kb = static_cast<const bf16*>(a.k) + base;
        const bf16* vb = static_cast<const bf16*>(a.v) + base;
        for (int e = lane; e < AM_ROWS * 8; e += 32) {
            const int j = e >> 3, ch = e & 7;
            const bool ok = j < Nk;
            int sl = s0 + j;
            if (sl >= a.R) sl -= a.R;
            const long long off = (long long)(ok ? sl : 0) * HD + ch * 8;
            cp_async16(Km + swz(j, ch), kb + off, ok);
            cp_async16(Vm + swz(j, ch), vb + off, ok);
        }
        q = a.q + (long long)b * nq * a.ldq + h * HD;
    }
    cp_async_wait_all();
    __syncthreads();
    if (!live) return;

    // B fragments of the split queries: column g -> query g & 3, half g >> 2;
    // rows (dims) 16 ks + 2c, +1 and 16 ks + 2c + 8, +9
    uint32_t bu[4][2], bv[4][2];
    {
        const int qi = g & 3, half = g >> 2;
        const bool has = qi < nq;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int d = ks * 16 + 2 * c + 8 * hh;
                float2 qq = make_float2(0.f, 0.f);
                if (has) qq = *reinterpret_cast<const float2*>(q + (long long)qi * a.ldq + d);
                const float2 uu = *reinterpret_cast<const float2*>(a.pbu + h * HD + d);
                const float2 vv = *reinterpret_cast<const float2*>(a.pbv + h * HD + d);
                bu[ks][hh] = has ? pack2(split_part(qq.x + uu.x, half), split_part(qq.y + uu.y, half)) : 0u;
                bv[ks][hh] = has ? pack2(split_part(qq.x + vv.x, half), split_part(qq.y + vv.y, half)) : 0u;
            }
        }
    }
    score_tiles(Km, bu, Sac, lane);
    score_tiles(Pm, bv, Sbd, lane);
    __syncwarp();

    // masked softmax per query over its key window (absolute positions)
    const int kpos0 = p0 - Lc;
    for (int i = 0; i < nq; ++i) {
        const int pq = p0 + i;
        int lo, hi;
        if (a.rc > 0) {
            lo = max(pq - a.left, 0);
            hi = pq + a.rc;
        } else {
            const int cc = (pq / a.chunk) * a.chunk;
            lo = max(cc - a.left, 0);
            hi = cc + a.chunk - 1;
        }
        float sv[3];
        float m = -FLT_MAX;
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            const int j = lane + 32 * t, pk = kpos0 + j;
            const bool ok = j < Nk && pk >= lo && pk <= hi;
            sv[t] = ok ? (Sac[i * AM_SLD + j] + Sbd[i * AM_SLD + (pq - pk - a.rmin)]) * a.scale : -FLT_MAX;
            m = fmaxf(m, sv[t]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float sum = 0.f;
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            sv[t] = sv[t] == -FLT_MAX ? 0.f : __expf(sv[t] - m);
            sum += sv[t];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float inv = 1.f / sum;
        __syncwarp();  // every lane has read Sac row i before it is overwritten
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            const int j = lane + 32 * t;
            if (j < AM_ROWS) Sac[i * AM_SLD + j] = sv[t] * inv;
        }
    }
    __syncwarp();
    pdl_trigger();

    // out^T[d][col] = V^T[d][:] . prob^T[:][col]; B column g -> query g & 3, half g >> 2
    float acc[4][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[mt][k] = 0.f;
    {
        const int qi = g & 3, half = g >> 2;
        const bool has = qi < nq;
#pragma unroll
        for (int ks = 0; ks < AM_ROWS / 16; ++ks) {
            uint32_t bp[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int j = ks * 16 + 2 * c + 8 * hh;
                const float p0v = has ? Sac[qi * AM_SLD + j] : 0.f;
                const float p1v = has ? Sac[qi * AM_SLD + j + 1] : 0.f;
                bp[hh] = pack2(split_part(p0v, half), split_part(p1v, half));
            }
            const int key = ks * 16 + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                uint32_t av[4];
                ldsm_x4_t(Vm + swz(key, mt * 2 + ((lane >> 3) & 1)), av);
                mma16816(acc[mt], av, bp[0], bp[1]);
            }
        }
    }
    // recombine hi + lo, stage out[i][d] (fp32) in Sbd, then write the rows
    float* O = Sbd;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[mt][k] += __shfl_xor_sync(0xffffffffu, acc[mt][k], 2);
    }
    __syncwarp();  // Sbd (bd scores) fully consumed by the softmax
    if (c < 2) {
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            const int d = mt * 16 + g;
            O[(2 * c) * 64 + d] = acc[mt][0];
            O[(2 * c + 1) * 64 + d] = acc[mt][1];
            O[(2 * c) * 64 + d + 8] = acc[mt][2];
            O[(2 * c + 1) * 64 + d + 8] = acc[mt][3];
        }
    }
    __syncwarp();
    bf16* dst = static_cast<bf16*>(a.out) + (long long)b * nq * a.ldo + h * HD;
    for (int i = 0; i < nq; ++i) {
        const float2 o = *reinterpret_cast<const float2*>(O + i * 64 + 2 * lane);
        const __nv_bfloat162 hi2 = __floats2bfloat162_rn(o.x, o.y);
        bf16* row = dst + (long long)i * a.ldo + 2 * lane;
        *reinterpret_cast<__nv_bfloat162*>(row) = hi2;
        if (a.out_split > 0) {
            const float2 hf = __bfloat1622float2(hi2);
            *reinterpret_cast<__nv_bfloat162*>(row + a.out_split) = __floats2bfloat162_rn(o.x - hf.x, o.y - hf.y);
        }
    }
}
}  // namespace

bool attention_stream_mma_ok(const AttnParams& a, int act_bf16) {
    return act_bf16 && a.HD == 64 && a.nq >= 1 && a.nq <= 4 && a.left + a.nq <= AM_ROWS && a.NR <= AM_ROWS &&
           a.rmin <= 0 && a.ldq % 2 == 0 && a.ldo % 2 == 0 && a.out_split % 2 == 0;
}

cudaError_t launch_attention_stream_mma(const AttnParams& a, int* status, cudaStream_t s) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attn_stream_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             AM_SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 grid((a.nb + AM_WARPS - 1) / AM_WARPS, a.H);
    return launch_k(attn_stream_mma_kernel, grid, dim3(AM_WARPS * 32), AM_SMEM, s, 1, a, status);
}

}  // namespace cac
